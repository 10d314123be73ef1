/*
 * Plain CPU oracle for the virtual-rank sum all-reduce.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library: every conversion below is written from the IEEE 754
 * definitions of binary32, binary16 and bfloat16, and the packet layout from
 * its prose description.
 *
 * What it computes, and where that comes from:
 *
 *  - The collective is a SUM all-reduce over the R tensor-parallel ranks
 *    ("SGLang 中的 MSCCL++ All-Reduce 基准测试与推理集成指南", §1: every
 *    layer's attention and MLP output is summed across all TP ranks; §4.3,
 *    guard items 2 and 4: dtypes float32/float16/bfloat16, ReduceOp.SUM only).
 *    The drop-in NCCL-style statement of the call is in "【论文分享】MSCCL++：
 *    让 GPU 通信像 CUDA 一样可编程", section "第一层：Collective API".
 *  - The pages fix neither the accumulation order nor its precision.  The
 *    reading used here: widen every element to binary32 exactly, fold the R
 *    ranks left to right (rank 0 first, acc starts at rank 0's value, never at
 *    +0.0), one IEEE binary32 round-to-nearest-even add per rank, then round
 *    once to the buffer dtype with round-to-nearest-even.  No flush-to-zero.
 *  - One-shot and two-shot schedules ("SGLang ..." §4.4: the packet algorithm
 *    and the reduce-scatter + all-gather "rsag" algorithm) compute this same
 *    function; only the reduce-scatter intermediate has its own definition
 *    (oracle_reduce_scatter).
 *  - LL packets ("【论文分享】MSCCL++..." section "MemoryChannel", protocol
 *    table: LL = frequent synchronisation at small granularity).  The page
 *    gives no layout; the reading used here is an 8-byte little-endian word
 *    whose low 4 bytes carry 4 bytes of the message and whose high 4 bytes
 *    carry the flag.  Packet p carries message bytes [4p, 4p+4); bytes past
 *    the end of the message are zero.
 *
 * Every function is pinned by tests under tests/ (exhaustive comparison of
 * the conversions with torch's CPU casts, exact integer sums, hand-derived
 * IEEE cases, brute-force binary64 sums within the rounding-error bound, and
 * packet round trips).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math (see oracle/__init__.py).
 */
#include <float.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float expressions evaluated in IEEE binary32"
#endif

enum { OR_BF16 = 0, OR_FP16 = 1, OR_FP32 = 2 };

static float f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t bits_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

size_t oracle_elem_size(int dtype)
{
    switch (dtype) {
    case OR_BF16: return 2;
    case OR_FP16: return 2;
    case OR_FP32: return 4;
    default: return 0;
    }
}

/* ---------------------------------------------------------------------------
 * Widening conversions (exact).
 * ------------------------------------------------------------------------- */

/* bfloat16 is, by definition, the upper 16 bits of a binary32 pattern:
 * same sign, same 8-bit exponent, the top 7 of the 23 fraction bits. */
float oracle_bf16_to_f32(uint16_t h)
{
    return f32_from_bits((uint32_t)h << 16);
}

/* binary16: sign s, 5-bit exponent e (bias 15), 10-bit fraction m.
 *   e == 0      : (-1)^s * m * 2^-24                 (zero / subnormal)
 *   1 <= e <= 30: (-1)^s * (1024 + m) * 2^(e - 25)    (normal)
 *   e == 31     : infinity (m == 0) or NaN (m != 0)
 * Every binary16 value is exactly representable in binary32, and ldexpf of
 * an integer below 2^11 by these exponents is exact. */
float oracle_fp16_to_f32(uint16_t h)
{
    uint32_t s = (uint32_t)(h >> 15);
    uint32_t e = (uint32_t)((h >> 10) & 0x1Fu);
    uint32_t m = (uint32_t)(h & 0x3FFu);
    float mag;
    if (e == 31u) {
        /* keep the payload in the top fraction bits, as a widening cast does */
        return f32_from_bits((s << 31) | 0x7F800000u | (m << 13));
    }
    if (e == 0u)
        mag = ldexpf((float)m, -24);
    else
        mag = ldexpf((float)(1024u + m), (int)e - 25);
    return s ? -mag : mag;
}

/* ---------------------------------------------------------------------------
 * Narrowing conversions, IEEE roundTiesToEven.
 * ------------------------------------------------------------------------- */

/* binary32 -> bfloat16.
 * Non-negative binary32 patterns are ordered like the values they encode, and
 * the bfloat16 values are exactly the binary32 patterns whose low 16 bits are
 * zero.  So for a finite magnitude pattern |x| = K * 2^16 + D (0 <= D < 2^16):
 *   lo = pattern K * 2^16       is the largest bfloat16 magnitude <= |x|,
 *   hi = pattern (K + 1) * 2^16 is the next one up (possibly the next binade,
 *        or infinity after the largest finite value),
 * and within one binade the distance from lo to |x| is D/2^16 of the distance
 * from lo to hi.  Round-to-nearest picks hi when D > 2^15, lo when D < 2^15,
 * and on a tie the one whose last kept bit (bit 0 of K) is 0.  Rounding the
 * largest finite value upward gives the infinity pattern, which is IEEE's
 * overflow rule under roundTiesToEven. */
uint16_t oracle_f32_to_bf16(float x)
{
    uint32_t u = bits_from_f32(x);
    uint32_t sign = u & 0x80000000u;
    uint32_t mag = u & 0x7FFFFFFFu;
    uint32_t K, D;
    if (mag > 0x7F800000u) {
        /* NaN stays NaN: keep sign and top payload bits, force the quiet bit */
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    K = mag >> 16;
    D = mag & 0xFFFFu;
    if (D > 0x8000u || (D == 0x8000u && (K & 1u) != 0u))
        K += 1u;
    return (uint16_t)((sign >> 16) | K);
}

/* binary32 -> binary16.
 * Write |x| = M * 2^E with M the integer significand (24 bits for normal
 * binary32 values, including the hidden bit).  The binary16 values in the
 * binade [2^k, 2^(k+1)) are the multiples of the quantum 2^(k-10); below 2^-14
 * (the subnormal range) the quantum is 2^-24.  So the quantum exponent is
 * Q = max(k - 10, -24), and rounding |x| is rounding the rational M * 2^(E-Q)
 * to the nearest integer q, ties to even q.  The result q * 2^Q is then
 * encoded: q < 1024 only happens with Q = -24 (subnormal, exponent field 0);
 * otherwise q is in [1024, 2048] and a carry to 2048 moves to the next binade.
 * An exponent field of 31 or more is an overflow to infinity, which under
 * roundTiesToEven is exactly the case |x| >= 65520. */
uint16_t oracle_f32_to_fp16(float x)
{
    uint32_t u = bits_from_f32(x);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t ebits = (u >> 23) & 0xFFu;
    uint32_t frac = u & 0x7FFFFFu;
    uint32_t M;
    int E, k, Q, shift;
    uint32_t q, rest, half;
    int field;

    if (ebits == 0xFFu) {
        if (frac == 0u)
            return (uint16_t)(sign | 0x7C00u);                 /* infinity */
        return (uint16_t)(sign | 0x7E00u | (frac >> 13));      /* quiet NaN */
    }
    if (ebits == 0u) {
        if (frac == 0u)
            return (uint16_t)sign;                             /* signed zero */
        /* binary32 subnormals are below 2^-126, far under half of 2^-24 */
        return (uint16_t)sign;
    }
    M = 0x800000u | frac;              /* |x| = M * 2^(ebits - 150) */
    E = (int)ebits - 150;
    k = (int)ebits - 127;              /* |x| lies in [2^k, 2^(k+1)) */
    Q = k - 10;
    if (Q < -24)
        Q = -24;
    shift = Q - E;                     /* >= 13 because k - 10 >= k - 23 */
    if (shift > 30) {
        /* M < 2^24 so M / 2^shift < 2^-6: rounds to zero */
        return (uint16_t)sign;
    }
    q = M >> shift;
    rest = M & ((1u << shift) - 1u);
    half = 1u << (shift - 1);
    if (rest > half || (rest == half && (q & 1u) != 0u))
        q += 1u;
    if (q == 0u)
        return (uint16_t)sign;
    if (q < 1024u)                     /* only reachable with Q == -24 */
        return (uint16_t)(sign | q);
    if (q == 2048u) {                  /* carry into the next binade */
        q = 1024u;
        Q += 1;
    }
    field = Q + 25;                    /* value = q * 2^Q, q in [1024, 2048) */
    if (field >= 31)
        return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | ((uint32_t)field << 10) | (q - 1024u));
}

/* ---------------------------------------------------------------------------
 * Element access by dtype.
 * ------------------------------------------------------------------------- */

static float load_widened(int dtype, const void *buf, size_t i)
{
    if (dtype == OR_FP32) {
        float f;
        memcpy(&f, (const unsigned char *)buf + 4 * i, 4);
        return f;
    } else {
        uint16_t h;
        memcpy(&h, (const unsigned char *)buf + 2 * i, 2);
        return dtype == OR_BF16 ? oracle_bf16_to_f32(h) : oracle_fp16_to_f32(h);
    }
}

static void store_narrowed(int dtype, void *buf, size_t i, float y)
{
    if (dtype == OR_FP32) {
        memcpy((unsigned char *)buf + 4 * i, &y, 4);
    } else {
        uint16_t h = dtype == OR_BF16 ? oracle_f32_to_bf16(y) : oracle_f32_to_fp16(y);
        memcpy((unsigned char *)buf + 2 * i, &h, 2);
    }
}

/* ---------------------------------------------------------------------------
 * The all-reduce.
 * ------------------------------------------------------------------------- */

/* One element of the sum: widen, fold buffers 0..R-1 left to right in
 * binary32 starting from buffer 0's value (the caller rounds once to the
 * dtype).  Used by the all-reduce (the R ranks' inputs) and by plan reduce
 * steps (the step's sources in their listed order). */
static float fold_element(int R, int dtype, const void *const *in, size_t i)
{
    float acc = load_widened(dtype, in[0], i);
    int k;
    for (k = 1; k < R; ++k) {
        float x = load_widened(dtype, in[k], i);
        acc = acc + x;
    }
    return acc;
}

/* out[r][i] = round_dtype( in[0][i] + in[1][i] + ... + in[R-1][i] ) for every
 * rank r and element i, the sum folded left to right in binary32.
 * Returns 0, or -1 on a bad argument.  Inputs and outputs may alias only
 * element for element (in[r] == out[r]); the whole input element is read
 * before any output element with the same index is written. */
int oracle_allreduce(int R, size_t N, int dtype, const void *const *in, void *const *out)
{
    size_t i;
    int r;
    if (R < 1 || oracle_elem_size(dtype) == 0 || in == NULL || out == NULL)
        return -1;
    for (i = 0; i < N; ++i) {
        float acc = fold_element(R, dtype, in, i);
        for (r = 0; r < R; ++r)
            store_narrowed(dtype, out[r], i, acc);
    }
    return 0;
}

/* The shard boundaries of the two-shot schedule.  The pages name the
 * reduce-scatter + all-gather algorithm but not its split; the reading used
 * here: every shard holds S = ceil(N / R) elements rounded up to a whole
 * 16-byte vector (8 two-byte or 4 four-byte elements), shard j covers
 * [j*S, min((j+1)*S, N)), and the last shards may be short or empty. */
void oracle_shard_bounds(int R, size_t N, int dtype, int j, size_t *lo, size_t *hi)
{
    size_t per_vec = 16 / oracle_elem_size(dtype);
    size_t S = (N + (size_t)R - 1) / (size_t)R;
    size_t a, b;
    S = (S + per_vec - 1) / per_vec * per_vec;
    a = (size_t)j * S;
    b = a + S;
    if (a > N)
        a = N;
    if (b > N)
        b = N;
    *lo = a;
    *hi = b;
}

/* Reduce-scatter step of the two-shot schedule: for every shard j, out[j]
 * receives the reduced elements of shard j; nothing else is written. */
int oracle_reduce_scatter(int R, size_t N, int dtype, const void *const *in, void *const *out)
{
    int j;
    if (R < 1 || oracle_elem_size(dtype) == 0 || in == NULL || out == NULL)
        return -1;
    for (j = 0; j < R; ++j) {
        size_t lo, hi, i;
        oracle_shard_bounds(R, N, dtype, j, &lo, &hi);
        for (i = lo; i < hi; ++i)
            store_narrowed(dtype, out[j], i, fold_element(R, dtype, in, i));
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Plans: sequences of reduce / copy steps over chunks of the rank buffers.
 *
 * "【论文分享】MSCCL++：让 GPU 通信像 CUDA 一样可编程", section
 * "第二层：DSL API": an algorithm is written as channel put / wait / reduce
 * steps; the compiler finds the data dependencies and inserts the
 * synchronisation, and the runtime interprets the plan.  The meaning of a
 * plan is therefore its steps executed one after another in the order
 * written; that sequential execution is what this function does (a
 * correctly synchronised parallel execution must give the same bits).
 *
 * A plan cuts every buffer into `nchunks` chunks: chunk c holds elements
 * [c*C, min((c+1)*C, N)), C = ceil(N / nchunks) rounded up to a whole
 * 16-byte vector.  Step k is described by the integers
 *   kind[k]   0 = copy, 1 = reduce
 *   dst[k]    buffer id of the destination
 *   nsrc[k]   number of sources (1 for a copy)
 *   src[k*32 + i], i < nsrc[k]: buffer ids of the sources, folded in order
 *   cbeg[k], cend[k]: the chunk range [cbeg, cend)
 * where buffer id b < R names in[b] and R <= b < 2R names out[b - R].
 * A reduce widens every source element to binary32, folds them left to
 * right, and rounds once to the dtype (the all-reduce fold above); a copy
 * moves the bits.  Returns 0, or -1 on a bad step.
 * ------------------------------------------------------------------------- */
int oracle_plan_run(int R, size_t N, int dtype, int nchunks, int nsteps, const int *kind,
                    const int *dst, const int *nsrc, const int *src, const int *cbeg,
                    const int *cend, void *const *in, void *const *out)
{
    size_t per_vec, C;
    int k;
    if (R < 1 || nchunks < 1 || oracle_elem_size(dtype) == 0)
        return -1;
    per_vec = 16 / oracle_elem_size(dtype);
    C = (N + (size_t)nchunks - 1) / (size_t)nchunks;
    C = (C + per_vec - 1) / per_vec * per_vec;
    for (k = 0; k < nsteps; ++k) {
        void *d;
        const void *srcs[32];
        int i, c;
        if (dst[k] < 0 || dst[k] >= 2 * R || nsrc[k] < 1 || nsrc[k] > 32 ||
            (kind[k] == 0 && nsrc[k] != 1) || cbeg[k] < 0 || cend[k] > nchunks)
            return -1;
        d = dst[k] < R ? (void *)in[dst[k]] : out[dst[k] - R];
        for (i = 0; i < nsrc[k]; ++i) {
            int b = src[k * 32 + i];
            if (b < 0 || b >= 2 * R)
                return -1;
            srcs[i] = b < R ? in[b] : out[b - R];
        }
        for (c = cbeg[k]; c < cend[k]; ++c) {
            size_t lo = (size_t)c * C, hi = lo + C, e;
            if (lo > N)
                lo = N;
            if (hi > N)
                hi = N;
            for (e = lo; e < hi; ++e) {
                if (kind[k] == 0) {
                    size_t s = oracle_elem_size(dtype);
                    memmove((unsigned char *)d + e * s, (const unsigned char *)srcs[0] + e * s, s);
                } else {
                    store_narrowed(dtype, d, e, fold_element(nsrc[k], dtype, srcs, e));
                }
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Weighted per-token combine.
 *
 * "NCCL EP统一MoE通信生态", section 3.1 and Table III: in the low-latency
 * mode the combine reduces every token at the receiver, weighting each
 * expert's output.  Reading used here: K sources y[k] hold T tokens of H
 * elements (row-major), w holds T x K binary32 weights (row-major), and
 *   out[t][h] = round_dtype( fold over k = 0..K-1 of  w[t][k] * y[k][t][h] )
 * with every product rounded to binary32 on its own (no fused multiply-add),
 * the products folded left to right from k = 0, and one final rounding to
 * the dtype -- the all-reduce fold with a weight per (token, source).
 * ------------------------------------------------------------------------- */
int oracle_combine(int K, size_t T, size_t H, int dtype, const void *const *y, const float *w,
                   void *out)
{
    size_t t, h;
    int k;
    if (K < 1 || oracle_elem_size(dtype) == 0)
        return -1;
    for (t = 0; t < T; ++t) {
        for (h = 0; h < H; ++h) {
            size_t i = t * H + h;
            float acc = w[t * (size_t)K] * load_widened(dtype, y[0], i);
            for (k = 1; k < K; ++k) {
                float p = w[t * (size_t)K + (size_t)k] * load_widened(dtype, y[k], i);
                acc = acc + p;
            }
            store_narrowed(dtype, out, i, acc);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * LL packets.
 * ------------------------------------------------------------------------- */

size_t oracle_ll_packets(int dtype, size_t n)
{
    size_t bytes = n * oracle_elem_size(dtype);
    return (bytes + 3) / 4;
}

/* Packet p = (flag << 32) | payload, payload = message bytes [4p, 4p+4) read
 * little-endian, zero past the end of the n-element message.  For two-byte
 * dtypes element 2p is the low half and element 2p+1 the high half; for
 * binary32 the payload is element p's bit pattern. */
int oracle_ll_pack(int dtype, const void *src, size_t n, uint32_t flag, uint64_t *pkts)
{
    size_t bytes = n * oracle_elem_size(dtype);
    size_t P = oracle_ll_packets(dtype, n);
    const unsigned char *b = (const unsigned char *)src;
    size_t p;
    int j;
    if (oracle_elem_size(dtype) == 0)
        return -1;
    for (p = 0; p < P; ++p) {
        uint32_t payload = 0;
        for (j = 0; j < 4; ++j) {
            size_t at = 4 * p + (size_t)j;
            uint32_t byte = at < bytes ? (uint32_t)b[at] : 0u;
            payload |= byte << (8 * j);
        }
        pkts[p] = ((uint64_t)flag << 32) | (uint64_t)payload;
    }
    return 0;
}

/* Inverse of oracle_ll_pack.  A packet whose flag differs from `flag` is
 * counted and its bytes are not written.  Returns the mismatch count. */
size_t oracle_ll_unpack(int dtype, const uint64_t *pkts, size_t n, uint32_t flag, void *dst)
{
    size_t bytes = n * oracle_elem_size(dtype);
    size_t P = oracle_ll_packets(dtype, n);
    unsigned char *b = (unsigned char *)dst;
    size_t p, bad = 0;
    int j;
    for (p = 0; p < P; ++p) {
        uint32_t f = (uint32_t)(pkts[p] >> 32);
        uint32_t payload = (uint32_t)(pkts[p] & 0xFFFFFFFFu);
        if (f != flag) {
            ++bad;
            continue;
        }
        for (j = 0; j < 4; ++j) {
            size_t at = 4 * p + (size_t)j;
            if (at < bytes)
                b[at] = (unsigned char)((payload >> (8 * j)) & 0xFFu);
        }
    }
    return bad;
}

/* ---------------------------------------------------------------------------
 * Bulk conversions (used by the tests' exhaustive checks).
 * ------------------------------------------------------------------------- */

void oracle_round_f32(int dtype, const float *src, size_t n, void *dst)
{
    size_t i;
    for (i = 0; i < n; ++i)
        store_narrowed(dtype, dst, i, src[i]);
}

void oracle_widen(int dtype, const void *src, size_t n, float *dst)
{
    size_t i;
    for (i = 0; i < n; ++i)
        dst[i] = load_widened(dtype, src, i);
}
