// The C ABI (include/ar.h): handle life cycle, argument checks and the choice
// of kernel for each (algo, proto, alignment).  Nothing here allocates,
// copies or synchronises on the hot path, so every call can be captured in a
// CUDA graph.  The NCCL-style drop-in statement of the call follows
// "【论文分享】MSCCL++：让 GPU 通信像 CUDA 一样可编程", section
// "第一层：Collective API"; its guards (dtypes, SUM only) "SGLang 中的 MSCCL++
// All-Reduce 基准测试与推理集成指南", section 4.3.
#include <new>

#include "ar_internal.h"

using namespace ar;

// AUTO lookup: messages are bucketed by bytes per rank, rounded up to a power
// of two and clamped to [512 B, 256 MiB] (SGLang guide, section 4.4).
constexpr int kMinBucketLog2 = 9;
constexpr int kMaxBucketLog2 = 28;
constexpr int kBuckets = kMaxBucketLog2 - kMinBucketLog2 + 1;
// ar_tune times 15 sizes, 2^9 .. 2^23 bytes per rank (the page's [2^9, 2^24)).
constexpr int kTuneMaxLog2 = 23;
// CTA-cap divisors ar_tune times for every path (the launch-shape dimension).
constexpr int kTuneDiv[] = {1, 2, 4};
constexpr int kTuneDivs = 3;
constexpr float kTuneDivMargin = 0.02f;
// Two-shot HB calls moving at least this many bytes (with R >= 4) run the
// TMA staging in its one-stage form.
constexpr uint64_t kTmaLargeBytes = (uint64_t)1 << 30;
// Two-shot HB with AR_HB_STAGING_AUTO before ar_tune (and above the tuned
// sizes): TMA staging where it measured faster on GB300, direct staging
// elsewhere.  T = bytes moved per call, 2 R n elem_size.
static bool tma_band(int R, uint64_t T) {
    const uint64_t KiB = 1024, MiB = KiB * KiB;
    if (R >= 4 && R <= 16 && T >= kTmaLargeBytes)
        return true;                         // the one-stage form (at R = 32 the
                                             // direct staging measured as fast or faster)
    if (R >= 32)
        return T >= 64 * KiB && T <= 128 * MiB;
    if (R >= 16)
        return (T >= 128 * KiB && T <= MiB) || (T >= 16 * MiB && T <= 64 * MiB);
    if (R >= 8)
        return T >= 16 * MiB && T <= 64 * MiB;
    return false;
}

struct ar_handle {
    int R;
    size_t N;
    int dtype;
    size_t esz;
    int device;
    int num_sms;
    void *dev_mem;
    size_t dev_bytes;
    Ctl ctl;
    uint64_t *slots;        // LL scratch, NULL if the handle is not LL capable
    uint64_t ppad;          // packets per slot
    uint64_t shard;         // two-shot shard S, elements
    int ll_cap[2];          // co-resident CTAs of the per-rank LL kernel [two_shot]
    int ll_staged_cap[2];   // co-resident CTAs of the staged LL kernels [two_shot]
    int one_shot_warps;     // warps per CTA of the one-shot HB kernel
    int one_shot_cap;       // CTAs of the one-shot HB kernel per launch
    int reg_cap;            // CTAs of the 256-thread kernels per launch
    int tma_tile;
    int tma_stages;
    int tma_tile_large;     // per-rank tile of the one-stage form for calls
                            // moving >= kTmaLargeBytes, 0 = not used
    // AUTO choice per message-size bucket (bucket b: messages of at most
    // 2^(9+b) bytes per rank), timed by ar_tune; us[algo][proto], 0 = untimed
    float tuned_us[kBuckets][2][2];
    int tuned_max;          // largest tuned bucket, -1 before ar_tune
    // two-shot HB staging per bucket, timed by ar_tune: enum ar_hb_staging,
    // AR_HB_STAGING_AUTO = not timed
    int tuned_hb2[kBuckets];
    // divisor of each path's CTA cap per bucket, timed by ar_tune (1: the
    // full cap); [bucket][algo][proto]
    int tuned_div[kBuckets][2][2];
    int grid_div;           // forced divisor (ar_set_grid_divisor), 0 = tuned
    int pdl;                // launch with programmatic dependent launch
    int ll_transport;       // enum ar_ll_transport
    int hb_staging;         // enum ar_hb_staging
    bool cluster_ok;        // the cluster LL kernel can run for this R
    uint64_t cluster_uc;    // its 16-byte units per rank per chunk (largest)
    int cluster_max;        // co-resident clusters at that chunk size
};

namespace {

const uint64_t kDefaultTimeoutNs = 1000000000ull;

bool valid_dtype(int d) { return d == AR_BF16 || d == AR_FP16 || d == AR_FP32; }

uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

int clamp_grid(uint64_t want, int cap) {
    if (want < 1)
        want = 1;
    if (want > (uint64_t)cap)
        want = (uint64_t)cap;
    return (int)want;
}

bool on_device(const ar_handle *h) {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev == h->device;
}

bool ranges_overlap(uintptr_t a, uintptr_t b, size_t len) { return a < b + len && b < a + len; }

// Checks shared by the calls that take R output pointers and, optionally, R
// input pointers.  Sets *vec16 / *vec8 (all pointers 16- / 8-byte aligned)
// and *inplace (some in[r] == out[r]).
int check_buffers(const ar_handle *h, const void *const in[], void *const out[], uint64_t n,
                  bool *vec16, bool *vec8, bool *inplace) {
    if (!h || !out)
        return AR_ERR_INVALID;
    if (!on_device(h))
        return AR_ERR_INVALID;
    const int R = h->R;
    const size_t len = n * h->esz;
    uintptr_t all = 0;
    for (int r = 0; r < R; ++r) {
        if (!out[r] || (in && !in[r]))
            return AR_ERR_INVALID;
        const uintptr_t o = (uintptr_t)out[r];
        const uintptr_t i = in ? (uintptr_t)in[r] : 0;
        if ((o % h->esz) != 0 || (i % h->esz) != 0)
            return AR_ERR_INVALID;
        all |= o | i;
    }
    *vec16 = (all & 15u) == 0;
    *vec8 = (all & 7u) == 0;
    *inplace = false;
    for (int a = 0; a < R; ++a) {
        const uintptr_t oa = (uintptr_t)out[a];
        for (int b = a + 1; b < R; ++b)
            if (ranges_overlap(oa, (uintptr_t)out[b], len))
                return AR_ERR_INVALID;            // outputs must be disjoint
        if (!in)
            continue;
        for (int b = 0; b < R; ++b) {
            const uintptr_t ib = (uintptr_t)in[b];
            if (!ranges_overlap(oa, ib, len))
                continue;
            if (a == b && ib == oa)
                *inplace = true;                  // same rank, exactly in place
            else
                return AR_ERR_INVALID;
        }
    }
    return AR_OK;
}

void fill_ptrs(const ar_handle *h, const void *const in[], void *const out[], RankPtrs *p) {
    for (int r = 0; r < AR_MAX_RANKS; ++r) {
        p->in[r] = (in && r < h->R) ? in[r] : nullptr;
        p->out[r] = r < h->R ? out[r] : nullptr;
    }
}

// One call: its buffers, its message length n (<= the handle's N) and what
// the checks found.
struct Call {
    const void *const *in;
    void *const *out;
    uint64_t n;
    uint64_t shard;         // two-shot shard of n elements
    bool vec16, vec8, inplace;
    bool host = false;      // some buffer is page-locked host memory
    cudaStream_t s;
};

// ceil(n / R) rounded up to a whole 16-byte vector
uint64_t shard_of(uint64_t n, int R, size_t esz) {
    const uint64_t per_vec = 16 / esz;
    return ceil_div(ceil_div(n, (uint64_t)R), per_vec) * per_vec;
}

HbArgs hb_args(const ar_handle *h, const Call &c) {
    HbArgs a;
    fill_ptrs(h, c.in, c.out, &a.p);
    a.n = c.n;
    a.shard = c.shard;
    a.R = h->R;
    a.inplace = c.inplace ? 1 : 0;
    return a;
}

int from_cuda(cudaError_t e) {
    if (e == cudaSuccess)
        return AR_OK;
    (void)cudaGetLastError();   // clear a non-sticky launch error
    return AR_ERR_CUDA;
}

// ---- the four all-reduce paths ---------------------------------------------

int bucket_of(uint64_t bytes);

// Divisor of a path's CTA cap for a message of n elements per rank (the
// launch-shape dimension of the tuner): the handle's forced one, else the one
// ar_tune timed fastest at the message's size bucket, else 1.  Threads per
// CTA are fixed per kernel by its launch bounds.
// 0 when the handle neither forces a divisor nor has one tuned for the size.
int grid_div_set(const ar_handle *h, uint64_t n, int algo, int proto) {
    if (h->grid_div > 0)
        return h->grid_div;
    if (h->tuned_max >= 0) {
        const int b = bucket_of(n * h->esz);
        if (b <= h->tuned_max)
            return h->tuned_div[b][algo][proto];
    }
    return 0;
}

int grid_div(const ar_handle *h, uint64_t n, int algo, int proto) {
    const int d = grid_div_set(h, n, algo, proto);
    return d > 0 ? d : 1;
}

int div_cap(int cap, int div) {
    const int c = cap / div;
    return c > 0 ? c : 1;
}

// One-shot HB: runs of the message (a run: 32 units of every rank for one
// CTA's warps) and the divisor of the CTA cap.  Without a forced or tuned
// divisor, a message of R <= 16 ranks with more runs than a quarter of the
// cap and at most twice the cap runs on a quarter of the cap: at up to one
// run per CTA the full grid folds without the shared-memory ring, and at up
// to two it keeps too few runs in each ring; a quarter of the cap measured
// 3-30% faster (R = 4 at 512 KiB-2 MiB per rank, R = 8 at 256 KiB-1 MiB,
// R = 16 at 128-512 KiB) and slower beyond twice the cap.  Above 16 ranks
// the one-run form stages its inputs once and keeps the full grid.
uint64_t one_shot_runs(const ar_handle *h, uint64_t n, bool vec16) {
    const uint64_t units = vec16 ? n / (16 / h->esz) : n;
    const uint64_t per_blk = (uint64_t)(h->one_shot_warps / h->R) * 32;
    return ceil_div(units, per_blk);
}

int one_shot_div(const ar_handle *h, uint64_t n, bool vec16) {
    const int d = grid_div_set(h, n, AR_ONE_SHOT, AR_HB);
    if (d > 0)
        return d;
    const uint64_t runs = one_shot_runs(h, n, vec16);
    if (vec16 && h->R <= 16 && runs <= 2 * (uint64_t)h->one_shot_cap &&
        runs > (uint64_t)(h->one_shot_cap / 4))
        return 4;                            // measured with 16-byte vectors only
    return 1;
}

int one_shot_hb(ar_handle *h, const Call &c) {
    const HbArgs a = hb_args(h, c);
    // host memory: the element-wise form, whose loads and stores are plain
    // ones (the vector forms stage their inputs with cp.async)
    const bool vec = c.vec16 && !c.host;
    const uint64_t runs = one_shot_runs(h, c.n, vec);
    const int grid = clamp_grid(runs, div_cap(h->one_shot_cap, one_shot_div(h, c.n, vec)));
    return from_cuda(launch_one_shot_hb(a, h->dtype, vec, runs <= (uint64_t)grid, grid,
                                        32 * h->one_shot_warps, c.s, h->pdl));
}

// Staging of a two-shot HB call of n elements per rank whose buffers are all
// 16-byte aligned: the handle's setting; with AR_HB_STAGING_AUTO the faster
// one timed by ar_tune at the message's size bucket, else the fixed rule of
// tma_band.
int hb2_staging(const ar_handle *h, uint64_t n) {
    if (h->hb_staging != AR_HB_STAGING_AUTO)
        return h->hb_staging;
    const uint64_t bytes = n * h->esz;
    if (h->tuned_max >= 0) {
        const int b = bucket_of(bytes);
        if (b <= h->tuned_max && h->tuned_hb2[b] != AR_HB_STAGING_AUTO)
            return h->tuned_hb2[b];
    }
    return tma_band(h->R, 2 * (uint64_t)h->R * bytes) ? AR_HB_STAGING_TMA : AR_HB_STAGING_DIRECT;
}

int two_shot_hb(ar_handle *h, const Call &c) {
    const int div = grid_div(h, c.n, AR_TWO_SHOT, AR_HB);
    const uint64_t body = (c.n * h->esz) / 16 * 16;
    if (c.vec16 && !c.host && body > 0 && hb2_staging(h, c.n) == AR_HB_STAGING_TMA) {
        // far beyond L2 (>= 1 GiB moved) one stage of 128 KiB per CTA and two
        // CTAs per SM in turn streamed faster than several stages filling the
        // SM's shared memory (R = 16 x 128 MiB: 635 against 676 us); below
        // that, the handle's stages
        const bool large =
            h->tma_tile_large > 0 && 2 * (uint64_t)h->R * c.n * h->esz >= kTmaLargeBytes;
        const int tile = large ? h->tma_tile_large : h->tma_tile;
        TmaArgs a;
        fill_ptrs(h, c.in, c.out, &a.p);
        a.n = c.n;
        a.body_bytes = body;
        a.shard_bytes = c.shard * h->esz;
        a.tiles_per_shard = ceil_div(a.shard_bytes, (uint64_t)tile);
        a.R = h->R;
        a.tile_bytes = tile;
        a.stages = large ? 1 : h->tma_stages;
        a.c = h->ctl;
        const uint64_t items = ceil_div(body, (uint64_t)tile) + (uint64_t)h->R;
        const int grid = clamp_grid(items, div_cap((large ? 2 : 1) * h->num_sms, div));
        return from_cuda(launch_two_shot_tma(a, h->dtype, grid, c.s, h->pdl));
    }
    // direct staging, or unaligned buffers: one thread per 16-byte vector (or
    // per element) folds the R inputs once and stores R copies; up to 64 MiB
    // moved per call the vector form runs held to four CTAs per SM; above
    // that, binary32 vectors run in kWideThreads-thread CTAs (768 threads per
    // SM, as the 16-bit forms) when that grid fills its cap, the same thread
    // count as the 256-thread grid's (a partly filled last wave of the wider
    // CTAs measured slower)
    const HbArgs a = hb_args(h, c);
    const uint64_t units = c.vec16 ? c.n / (16 / h->esz) : c.n;
    const bool occupancy4 = 2 * (uint64_t)h->R * c.n * h->esz <= ((uint64_t)64 << 20);
    if (c.vec16 && !occupancy4 && h->dtype == AR_FP32) {
        const int wide_cap = h->reg_cap * kRegThreads / kWideThreads;
        if (wide_cap > 0 && ceil_div(units, kWideThreads) >= (uint64_t)wide_cap)
            return from_cuda(launch_reduce(a, h->dtype, true, false, div_cap(wide_cap, div), c.s,
                                           h->pdl, kReduceWide));
    }
    const int grid = clamp_grid(ceil_div(units, kRegThreads), div_cap(h->reg_cap, div));
    return from_cuda(launch_reduce(a, h->dtype, c.vec16, false, grid, c.s, h->pdl,
                                   occupancy4 ? kReduceOcc4 : kReducePlain));
}

// One-shot LL through thread-block clusters (R peers per cluster exchange
// packets in distributed shared memory).
int ll_cluster(ar_handle *h, const Call &c) {
    LlClusterArgs a;
    fill_ptrs(h, c.in, c.out, &a.p);
    a.n = c.n;
    a.R = h->R;
    a.c = h->ctl;
    const uint64_t U = c.n * h->esz / 16;
    a.units_per_chunk = U < h->cluster_uc ? (U > 0 ? U : 1) : h->cluster_uc;
    const uint64_t nchunks = U > 0 ? ceil_div(U, a.units_per_chunk) : 1;
    int cap = h->cluster_max;
    if (cap > kEpochWords / h->R)
        cap = kEpochWords / h->R;
    cap = div_cap(cap, grid_div(h, c.n, AR_ONE_SHOT, AR_LL));
    return from_cuda(launch_ll_cluster(a, h->dtype, clamp_grid(nchunks, cap), c.s, h->pdl));
}

// LL: the staged kernels need every buffer 8-byte aligned, the cluster
// kernel 16-byte aligned; other buffers take the per-rank kernel.
int ll(ar_handle *h, const Call &c, bool two) {
    if (!h->slots)
        return AR_ERR_UNSUPPORTED;
    if (!two && c.vec16 && !c.host && h->cluster_ok && h->ll_transport == AR_LL_CLUSTER)
        return ll_cluster(h, c);
    LlArgs a;
    fill_ptrs(h, c.in, c.out, &a.p);
    a.n = c.n;
    a.shard = c.shard;
    a.slots = h->slots;
    a.ppad = h->ppad;
    a.R = h->R;
    a.c = h->ctl;
    const uint64_t nbytes = c.n * h->esz;
    if (c.vec8) {
        // aligned: CTAs serving all R ranks a block of units each, the
        // receivers of a unit sharing its packets' polls
        const uint64_t ub = kLlStagedThreads / h->R;
        int cap = h->ll_staged_cap[two ? 1 : 0];
        if (cap > kEpochWords)
            cap = kEpochWords;
        if (cap < 1)
            return AR_ERR_UNSUPPORTED;
        cap = div_cap(cap, grid_div(h, c.n, two ? AR_TWO_SHOT : AR_ONE_SHOT, AR_LL));
        a.G = 0;
        const int ctas = clamp_grid(ceil_div(nbytes / 8, ub), cap);
        return from_cuda(launch_ll_staged(a, h->dtype, two, ctas, c.s, h->pdl));
    }
    // not 8-byte aligned: per-rank CTAs, one packet per unit
    const uint64_t work = (nbytes + 3) / 4;
    int gmax = h->ll_cap[two ? 1 : 0] / h->R;
    if (gmax > kEpochWords / h->R)
        gmax = kEpochWords / h->R;
    if (gmax < 1)
        return AR_ERR_UNSUPPORTED;                 // cannot keep R CTAs resident
    gmax = div_cap(gmax, grid_div(h, c.n, two ? AR_TWO_SHOT : AR_ONE_SHOT, AR_LL));
    a.G = clamp_grid(ceil_div(work, kLlThreads), gmax);
    return from_cuda(launch_ll(a, h->dtype, two, c.s, h->pdl));
}

int run_path(ar_handle *h, const Call &c, int algo, int proto) {
    if (proto == AR_HB)
        return algo == AR_ONE_SHOT ? one_shot_hb(h, c) : two_shot_hb(h, c);
    return ll(h, c, algo == AR_TWO_SHOT);
}

// ---- AUTO -------------------------------------------------------------------

int bucket_of(uint64_t bytes) {
    int b = kMinBucketLog2;
    while (b < kMaxBucketLog2 && ((uint64_t)1 << b) < bytes)
        ++b;
    return b - kMinBucketLog2;
}

// Resolve AR_ALGO_AUTO / AR_PROTO_AUTO for a message of `bytes` per rank:
// the fastest tuned (algo, proto) allowed by the fixed half of the request,
// or, before ar_tune, a fixed rule from GB300 measurements (10-call graphs,
// L2 flushed; R = 2 to 32):
//   - LL only for the one-shot at R >= 24 up to 4 KiB per rank, HB
//     otherwise;
//   - with HB, the one-shot for R <= 2 at every size, for R = 4 up to
//     256 KiB per rank, for R = 16 up to 128 KiB and for the other
//     8 <= R <= 24 up to 64 KiB, the two-shot otherwise.  Against the
//     two-shot with its AUTO staging the one-shot, whose fold work grows
//     with R^2, wins only there; R = 3, 5 and 6, without an unrolled ring,
//     were faster or tied two-shot;
//   - with LL forced, the one-shot up to 2 MiB.
void resolve(const ar_handle *h, uint64_t bytes, int *algo, int *proto) {
    const bool ll_ok = h->slots != nullptr;
    if (h->tuned_max >= 0) {
        int b = bucket_of(bytes);
        if (b > h->tuned_max)
            b = h->tuned_max;
        float best = 0.f;
        int ba = -1, bp = -1;
        for (int a = 0; a < 2; ++a)
            for (int p = 0; p < 2; ++p) {
                if ((*algo != AR_ALGO_AUTO && *algo != a) || (*proto != AR_PROTO_AUTO && *proto != p))
                    continue;
                if (p == AR_LL && !ll_ok)
                    continue;
                const float us = h->tuned_us[b][a][p];
                if (us > 0.f && (ba < 0 || us < best)) {
                    best = us;
                    ba = a;
                    bp = p;
                }
            }
        if (ba >= 0) {
            *algo = ba;
            *proto = bp;
            return;
        }
    }
    if (*proto == AR_PROTO_AUTO)
        *proto = ll_ok && h->R >= 24 && bytes <= (4u << 10) && *algo != AR_TWO_SHOT ? AR_LL
                                                                                  : AR_HB;
    if (*algo == AR_ALGO_AUTO) {
        bool one;
        if (*proto == AR_LL)
            one = bytes <= (2u << 20);
        else if (h->R <= 2)
            one = true;
        else if (h->R == 4)
            one = bytes <= (256u << 10);
        else if (h->R == 16)
            one = bytes <= (128u << 10);
        else
            one = h->R >= 8 && h->R <= 24 && bytes <= (64u << 10);
        *algo = one ? AR_ONE_SHOT : AR_TWO_SHOT;
    }
}

}  // namespace

namespace ar {
Ctl handle_ctl(ar_handle_t h) { return h->ctl; }
}  // namespace ar

// ---------------------------------------------------------------------------

extern "C" {

const char *ar_strerror(int code) {
    switch (code) {
    case AR_OK: return "AR_OK";
    case AR_ERR_INVALID: return "AR_ERR_INVALID: invalid argument";
    case AR_ERR_UNSUPPORTED: return "AR_ERR_UNSUPPORTED: request not supported";
    case AR_ERR_CUDA: return "AR_ERR_CUDA: CUDA runtime error";
    case AR_ERR_NOMEM: return "AR_ERR_NOMEM: device allocation failed";
    case AR_ERR_TIMEOUT: return "AR_ERR_TIMEOUT: a device-side wait timed out";
    case AR_ERR_FLAG_MISMATCH: return "AR_ERR_FLAG_MISMATCH: LL packet with an unexpected flag";
    default: return "unknown ar status code";
    }
}

int ar_create(int R, size_t N, int dtype, ar_handle_t *out) {
    if (!out)
        return AR_ERR_INVALID;
    *out = nullptr;
    if (R < 1 || R > AR_MAX_RANKS || N < 1 || !valid_dtype(dtype))
        return AR_ERR_INVALID;
    const size_t esz = elem_size(dtype);
    if (N > ((size_t)1 << 40) / esz)
        return AR_ERR_INVALID;

    ar_handle *h = new (std::nothrow) ar_handle();
    if (!h)
        return AR_ERR_NOMEM;
    h->R = R;
    h->N = N;
    h->dtype = dtype;
    h->esz = esz;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) !=
            cudaSuccess) {
        delete h;
        return AR_ERR_CUDA;
    }

    // two-shot shard: ceil(N / R) rounded up to a whole 16-byte vector
    const uint64_t per_vec = 16 / esz;
    h->shard = ceil_div(ceil_div(N, (uint64_t)R), per_vec) * per_vec;

    // device memory: [status, abort | epoch words | LL slots]
    const size_t ctl_bytes = 256;
    const size_t epoch_bytes = sizeof(uint32_t) * kEpochWords;
    const bool ll_capable = N * esz <= AR_LL_MAX_BYTES;
    h->ppad = ll_capable ? ceil_div(ceil_div(N * esz, 4), 4) * 4 : 0;
    const size_t slot_bytes = ll_capable ? (size_t)(R + 1) * h->ppad * sizeof(uint64_t) : 0;
    h->dev_bytes = ctl_bytes + epoch_bytes + slot_bytes;
    if (cudaMalloc(&h->dev_mem, h->dev_bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        delete h;
        return AR_ERR_NOMEM;
    }
    if (cudaMemset(h->dev_mem, 0, h->dev_bytes) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(h->dev_mem);
        delete h;
        return AR_ERR_CUDA;
    }
    uint8_t *base = static_cast<uint8_t *>(h->dev_mem);
    h->ctl.status = reinterpret_cast<int *>(base);
    h->ctl.abort = reinterpret_cast<uint32_t *>(base + 4);
    h->ctl.epoch = reinterpret_cast<uint32_t *>(base + ctl_bytes);
    h->ctl.timeout_ns = kDefaultTimeoutNs;
    h->ctl.drop_rank = -1;
    h->slots = ll_capable ? reinterpret_cast<uint64_t *>(base + ctl_bytes + epoch_bytes) : nullptr;

    // launch shapes
    int err = 0;
    for (int t = 0; t < 2; ++t) {
        int per_sm = 0;
        err |= ll_occupancy(dtype, t != 0, &per_sm) != cudaSuccess;
        h->ll_cap[t] = per_sm * h->num_sms;
        err |= ll_staged_occupancy(dtype, t != 0, &per_sm) != cudaSuccess;
        h->ll_staged_cap[t] = per_sm * h->num_sms;
    }
    h->one_shot_warps = R <= 8 ? R * ((8 + R - 1) / R) : R;
    h->one_shot_cap = h->num_sms * (2048 / (32 * h->one_shot_warps));
    err |= one_shot_prepare() != cudaSuccess;
    h->reg_cap = h->num_sms * (2048 / kRegThreads);
    int smem_limit = 0;
    err |= tma_prepare(dtype, &smem_limit) != cudaSuccess;
    // per-rank tile: a 64 KiB stage over R ranks, 1..8 KiB; then as many
    // stages (2..4) as the shared memory holds
    int tile = (int)((64 * 1024 / R) / 16 * 16);
    if (tile > 8192)
        tile = 8192;
    if (tile < 1024)
        tile = 1024;
    int stages = kTmaMaxStages;
    while (stages > 2 && tma_smem_bytes(R, tile, stages) > (size_t)smem_limit)
        --stages;
    while (tile > 1024 && tma_smem_bytes(R, tile, stages) > (size_t)smem_limit)
        tile -= 1024;
    h->tma_tile = tile;
    h->tma_stages = stages;
    // calls moving kTmaLargeBytes or more: one stage of 128 KiB over R ranks
    // (R >= 4: where it measured), two CTAs per SM in turn
    const int large = (int)((128 * 1024 / R) / 16 * 16);
    h->tma_tile_large =
        R >= 4 && tma_smem_bytes(R, large, 1) <= (size_t)smem_limit ? large : 0;

    h->tuned_max = -1;                       // AUTO uses the fixed rule until ar_tune
    for (int b = 0; b < kBuckets; ++b) {
        for (int a = 0; a < 2; ++a)
            for (int p = 0; p < 2; ++p) {
                h->tuned_us[b][a][p] = 0.f;
                h->tuned_div[b][a][p] = 1;
            }
        h->tuned_hb2[b] = AR_HB_STAGING_AUTO;
    }
    h->grid_div = 0;
    h->pdl = 1;
    h->ll_transport = AR_LL_AUTO;
    h->hb_staging = AR_HB_STAGING_AUTO;

    // cluster LL: one CTA per virtual rank in a cluster (portable up to 8,
    // 16 with the non-portable size); receive buffers of ~64 KiB per CTA
    h->cluster_ok = false;
    if (ll_capable && R <= 16) {
        uint64_t uc = ((uint64_t)kLlClusterTargetSmem / (8u * R) - 4) / 4;
        if (uc > 1024)
            uc = 1024;
        LlClusterArgs probe = {};
        probe.R = R;
        probe.units_per_chunk = uc;
        int clusters = 0;
        if (ll_cluster_prepare(dtype, R) == cudaSuccess &&
            ll_cluster_max_clusters(probe, dtype, &clusters) == cudaSuccess && clusters > 0) {
            h->cluster_ok = true;
            h->cluster_uc = uc;
            h->cluster_max = clusters;
        }
        (void)cudaGetLastError();   // a refused cluster shape only disables the path
    }
    if (err) {
        (void)cudaGetLastError();
        cudaFree(h->dev_mem);
        delete h;
        return AR_ERR_CUDA;
    }
    *out = h;
    return AR_OK;
}

int ar_destroy(ar_handle_t h) {
    if (!h)
        return AR_OK;
    int rc = AR_OK;
    DeviceScope on(h->device);
    if (!on.ok() || cudaDeviceSynchronize() != cudaSuccess)
        rc = AR_ERR_CUDA;
    if (cudaFree(h->dev_mem) != cudaSuccess)
        rc = AR_ERR_CUDA;
    delete h;
    return rc;
}

// The checks and the Call shared by ar_allreduce_n and ar_allreduce_host.
static int prepare_call(ar_handle_t h, const void *const in[], void *const out[], size_t n,
                        int algo, int proto, cudaStream_t stream, Call *c) {
    if (!in || !h || n < 1 || n > h->N)
        return AR_ERR_INVALID;
    if (algo != AR_ONE_SHOT && algo != AR_TWO_SHOT && algo != AR_ALGO_AUTO)
        return AR_ERR_INVALID;
    if (proto != AR_LL && proto != AR_HB && proto != AR_PROTO_AUTO)
        return AR_ERR_INVALID;
    const int rc = check_buffers(h, in, out, n, &c->vec16, &c->vec8, &c->inplace);
    if (rc != AR_OK)
        return rc;
    c->in = in;
    c->out = out;
    c->n = n;
    c->shard = shard_of(n, h->R, h->esz);
    c->s = stream;
    return AR_OK;
}

int ar_allreduce_n(ar_handle_t h, const void *const in[], void *const out[], size_t n, int algo,
                   int proto, cudaStream_t stream) {
    Call c;
    const int rc = prepare_call(h, in, out, n, algo, proto, stream, &c);
    if (rc != AR_OK)
        return rc;
    if (algo == AR_ALGO_AUTO || proto == AR_PROTO_AUTO)
        resolve(h, n * h->esz, &algo, &proto);
    return run_path(h, c, algo, proto);
}

// Every buffer must be memory the device reaches at the buffer's own
// address: device memory of the handle's device, managed memory, or
// page-locked host memory mapped at its host address.  *host tells whether
// any buffer is host memory.  Pageable host memory is refused.
static int check_reachable(const ar_handle *h, const void *const in[], void *const out[],
                           bool *host) {
    *host = false;
    for (int r = 0; r < h->R; ++r) {
        const void *ptrs[2] = {in[r], out[r]};
        for (const void *p : ptrs) {
            cudaPointerAttributes at;
            if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
                (void)cudaGetLastError();
                return AR_ERR_INVALID;
            }
            if (at.type == cudaMemoryTypeHost) {
                if (at.devicePointer != p)
                    return AR_ERR_INVALID;
                *host = true;
            } else if (at.type == cudaMemoryTypeDevice) {
                if (at.device != h->device)
                    return AR_ERR_INVALID;
            } else if (at.type != cudaMemoryTypeManaged) {
                return AR_ERR_INVALID;
            }
        }
    }
    return AR_OK;
}

int ar_allreduce_host(ar_handle_t h, const void *const in[], void *const out[], size_t n,
                      int algo, int proto, cudaStream_t stream) {
    Call c;
    int rc = prepare_call(h, in, out, n, algo, proto, stream, &c);
    if (rc != AR_OK)
        return rc;
    rc = check_reachable(h, in, out, &c.host);
    if (rc != AR_OK)
        return rc;
    if (!c.host) {
        if (algo == AR_ALGO_AUTO || proto == AR_PROTO_AUTO)
            resolve(h, n * h->esz, &algo, &proto);
        return run_path(h, c, algo, proto);
    }
    // AUTO with host buffers, a fixed rule from GB300 measurements (one-call
    // graphs, bf16, R = 2 to 32, 1 KiB to 4 MiB per rank, the kernels
    // reading and writing host memory): the one-shot LL for R >= 24 up to
    // 16 KiB per rank (R = 32, 1 KiB: 7.7 against 9.9 us), the one-shot HB
    // for R <= 4 from 1 MiB (7-9% faster), the two-shot HB otherwise (R = 8:
    // 0.91-1.00 of the one-shot LL's time from 1 to 512 KiB; R = 2 and 4 up
    // to 128 KiB: 5.8 against 7.2-7.9 us).  A half fixed by the caller is
    // kept: with AR_LL the one-shot, with AR_ONE_SHOT LL on an LL-capable
    // handle (HB for R <= 4 from 1 MiB), with AR_TWO_SHOT HB.
    const uint64_t bytes = n * h->esz;
    const bool ll_ok = h->slots != nullptr;
    const bool one_hb = h->R <= 4 && bytes >= ((uint64_t)1 << 20);
    if (algo == AR_ALGO_AUTO && proto == AR_PROTO_AUTO) {
        if (ll_ok && h->R >= 24 && bytes <= 16384) {
            algo = AR_ONE_SHOT;
            proto = AR_LL;
        } else {
            algo = one_hb ? AR_ONE_SHOT : AR_TWO_SHOT;
            proto = AR_HB;
        }
    } else if (algo == AR_ALGO_AUTO) {
        algo = proto == AR_LL || one_hb ? AR_ONE_SHOT : AR_TWO_SHOT;
    } else if (proto == AR_PROTO_AUTO) {
        proto = algo == AR_ONE_SHOT && ll_ok && !one_hb ? AR_LL : AR_HB;
    }
    return run_path(h, c, algo, proto);
}

int ar_allreduce(ar_handle_t h, const void *const in[], void *const out[], int algo, int proto,
                 cudaStream_t stream) {
    if (!h)
        return AR_ERR_INVALID;
    return ar_allreduce_n(h, in, out, h->N, algo, proto, stream);
}

int ar_reduce_scatter(ar_handle_t h, const void *const in[], void *const out[],
                      cudaStream_t stream) {
    if (!in || !h)
        return AR_ERR_INVALID;
    Call c;
    const int rc = check_buffers(h, in, out, h->N, &c.vec16, &c.vec8, &c.inplace);
    if (rc != AR_OK)
        return rc;
    c.in = in;
    c.out = out;
    c.n = h->N;
    c.shard = h->shard;
    c.s = stream;
    const HbArgs a = hb_args(h, c);
    const uint64_t units = c.vec16 ? h->N / (16 / h->esz) : h->N;
    const int grid = clamp_grid(ceil_div(units, kRegThreads), h->reg_cap);
    return from_cuda(launch_reduce(a, h->dtype, c.vec16, true, grid, stream, h->pdl));
}

int ar_all_gather(ar_handle_t h, void *const out[], cudaStream_t stream) {
    if (!h)
        return AR_ERR_INVALID;
    Call c;
    const int rc = check_buffers(h, nullptr, out, h->N, &c.vec16, &c.vec8, &c.inplace);
    if (rc != AR_OK)
        return rc;
    c.in = nullptr;
    c.out = out;
    c.n = h->N;
    c.shard = h->shard;
    c.s = stream;
    const HbArgs a = hb_args(h, c);
    const uint64_t units = c.vec16 ? h->N / (16 / h->esz) : h->N;
    const int grid = clamp_grid(ceil_div(units, kRegThreads), h->reg_cap);
    return from_cuda(launch_all_gather(a, h->dtype, c.vec16, grid, stream, h->pdl));
}

int ar_combine(ar_handle_t h, const void *const y[], const float *w, void *out, size_t T,
               size_t H, cudaStream_t stream) {
    if (!h || !y || !w || !out || T < 1 || H < 1 || !on_device(h))
        return AR_ERR_INVALID;
    if (T > h->N / H)
        return AR_ERR_INVALID;                       // T * H elements must fit the handle
    const int K = h->R;
    const size_t len = T * H * h->esz;
    const uintptr_t o = (uintptr_t)out, wb = (uintptr_t)w;
    const size_t wlen = T * (size_t)K * sizeof(float);
    if ((o % h->esz) != 0 || (wb % 4) != 0 || (o < wb + wlen && wb < o + len))
        return AR_ERR_INVALID;                       // misaligned, or out overlaps w
    uintptr_t all = o;
    for (int k = 0; k < K; ++k) {
        const uintptr_t a = (uintptr_t)y[k];
        if (!y[k] || (a % h->esz) != 0)
            return AR_ERR_INVALID;
        if (ranges_overlap(a, o, len) && a != o)
            return AR_ERR_INVALID;                   // out may only be a source exactly
        all |= a;
    }
    const bool vec = (all & 15u) == 0 && (H * h->esz) % 16 == 0;
    CombineArgs a;
    for (int r = 0; r < AR_MAX_RANKS; ++r) {
        a.p.in[r] = r < K ? y[r] : nullptr;
        a.p.out[r] = r == 0 ? out : nullptr;
    }
    a.w = w;
    a.T = T;
    a.H = H;
    a.K = K;
    const uint64_t units = vec ? T * (H / (16 / h->esz)) : T * H;
    const int grid = clamp_grid(ceil_div(units, kRegThreads), h->reg_cap);
    return from_cuda(launch_combine(a, h->dtype, vec, grid, stream, h->pdl));
}

int ar_tune(ar_handle_t h, cudaStream_t stream) {
    if (!h || !on_device(h))
        return AR_ERR_INVALID;
    const size_t esz = h->esz;
    uint64_t max_bytes = (uint64_t)1 << kTuneMaxLog2;
    if (max_bytes > h->N * esz)
        max_bytes = h->N * esz;
    const uint64_t nmax = max_bytes / esz > 0 ? max_bytes / esz : 1;
    const size_t buf_bytes = (nmax * esz + 255) / 256 * 256;
    void *mem = nullptr;
    if (cudaStreamSynchronize(stream) != cudaSuccess)
        return from_cuda(cudaErrorUnknown);
    if (cudaMalloc(&mem, buf_bytes * 2 * h->R) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ERR_NOMEM;
    }
    const void *ins[AR_MAX_RANKS];
    void *outs[AR_MAX_RANKS];
    for (int r = 0; r < h->R; ++r) {
        ins[r] = static_cast<uint8_t *>(mem) + buf_bytes * r;
        outs[r] = static_cast<uint8_t *>(mem) + buf_bytes * (h->R + r);
    }
    cudaStream_t ts = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int rc = AR_OK;
    if (cudaMemset(mem, 0, buf_bytes * 2 * h->R) != cudaSuccess ||
        cudaStreamCreateWithFlags(&ts, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)
        rc = AR_ERR_CUDA;
    int last = -1;
    // every power of two from 512 B to max_bytes per rank (at least one size)
    for (int lg = kMinBucketLog2; rc == AR_OK && lg <= kTuneMaxLog2; ++lg) {
        const uint64_t bytes = (uint64_t)1 << lg;
        if (bytes > max_bytes && lg > kMinBucketLog2)
            break;
        const uint64_t n = bytes <= max_bytes ? bytes / esz : nmax;
        const int b = lg - kMinBucketLog2;
        Call c;
        c.in = ins;
        c.out = outs;
        c.n = n > 0 ? n : 1;
        c.shard = shard_of(c.n, h->R, esz);
        c.vec16 = c.vec8 = true;
        c.inplace = false;
        c.s = ts;
        // µs per call of (a, p): a graph of 10 calls, 5 warm-up replays, 20
        // timed replays; < 0 on a CUDA failure
        auto time_path = [&](int a, int p) -> float {
            cudaGraph_t g = nullptr;
            cudaGraphExec_t ge = nullptr;
            if (run_path(h, c, a, p) != AR_OK ||
                cudaStreamBeginCapture(ts, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
                return -1.f;
            int crc = AR_OK;
            for (int k = 0; k < 10 && crc == AR_OK; ++k)
                crc = run_path(h, c, a, p);
            if (cudaStreamEndCapture(ts, &g) != cudaSuccess || crc != AR_OK ||
                cudaGraphInstantiate(&ge, g, 0) != cudaSuccess) {
                if (g)
                    cudaGraphDestroy(g);
                return -1.f;
            }
            float ms = 0.f;
            bool okc = true;
            for (int k = 0; k < 5 && okc; ++k)
                okc = cudaGraphLaunch(ge, ts) == cudaSuccess;
            okc = okc && cudaEventRecord(e0, ts) == cudaSuccess;
            for (int k = 0; k < 20 && okc; ++k)
                okc = cudaGraphLaunch(ge, ts) == cudaSuccess;
            okc = okc && cudaEventRecord(e1, ts) == cudaSuccess &&
                  cudaEventSynchronize(e1) == cudaSuccess &&
                  cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess;
            cudaGraphExecDestroy(ge);
            cudaGraphDestroy(g);
            return okc ? ms * 1000.f / 200.f : -1.f;
        };
        // every (algo, proto) with each CTA-cap divisor, and two-shot HB with
        // both stagings (the buffers here are 16-byte aligned); the fastest
        // launch is kept for this size
        const int user_div = h->grid_div, user_staging = h->hb_staging;
        for (int a = 0; a < 2 && rc == AR_OK; ++a)
            for (int p = 0; p < 2 && rc == AR_OK; ++p) {
                h->tuned_us[b][a][p] = 0.f;
                h->tuned_div[b][a][p] = 1;
                if (p == AR_LL && !h->slots)
                    continue;
                const bool stagings = a == AR_TWO_SHOT && p == AR_HB;
                float best = -1.f;
                int best_div = 1, best_staging = AR_HB_STAGING_AUTO;
                for (int k = 0; k < kTuneDivs && rc == AR_OK; ++k) {
                    // the fastest staging at this divisor; a larger divisor
                    // is kept only when it beats the smaller ones by more
                    // than kTuneDivMargin (where the message never reaches
                    // the cap the launches are the same, and only noise
                    // would tell them apart)
                    float us_k = -1.f;
                    int staging_k = AR_HB_STAGING_AUTO;
                    for (int st = 0; st < (stagings ? 2 : 1); ++st) {
                        h->grid_div = kTuneDiv[k];
                        if (stagings)
                            h->hb_staging = st == 0 ? AR_HB_STAGING_TMA : AR_HB_STAGING_DIRECT;
                        const float us = time_path(a, p);
                        if (us < 0.f) {
                            rc = AR_ERR_CUDA;
                            break;
                        }
                        if (us_k < 0.f || us < us_k) {
                            us_k = us;
                            staging_k = h->hb_staging;
                        }
                    }
                    if (rc == AR_OK && (best < 0.f || us_k < best * (1.f - kTuneDivMargin))) {
                        best = us_k;
                        best_div = kTuneDiv[k];
                        best_staging = staging_k;
                    }
                }
                h->grid_div = user_div;
                h->hb_staging = user_staging;
                if (rc != AR_OK)
                    break;
                h->tuned_us[b][a][p] = best;
                h->tuned_div[b][a][p] = best_div;
                if (stagings)
                    h->tuned_hb2[b] = best_staging;
            }
        if (rc == AR_OK)
            last = b;
    }
    if (ts) {
        cudaStreamSynchronize(ts);
        cudaStreamDestroy(ts);
    }
    if (e0)
        cudaEventDestroy(e0);
    if (e1)
        cudaEventDestroy(e1);
    cudaFree(mem);
    if (rc != AR_OK) {
        (void)cudaGetLastError();
        h->tuned_max = -1;
        return rc;
    }
    h->tuned_max = last;
    // a timed-out wait during tuning would show in the status word
    const int st = ar_status(h, stream);
    return st;
}

int ar_get_tuning(ar_handle_t h, size_t bytes, int *algo, int *proto, float us[4]) {
    if (!h || !algo || !proto)
        return AR_ERR_INVALID;
    int a = AR_ALGO_AUTO, p = AR_PROTO_AUTO;
    resolve(h, bytes, &a, &p);
    *algo = a;
    *proto = p;
    if (us) {
        int b = bucket_of(bytes);
        if (h->tuned_max >= 0 && b > h->tuned_max)
            b = h->tuned_max;
        for (int k = 0; k < 4; ++k)
            us[k] = h->tuned_max >= 0 ? h->tuned_us[b][k / 2][k % 2] : 0.f;
    }
    return AR_OK;
}

int ar_ll_pack(ar_handle_t h, const void *src, uint64_t *pkts, size_t n, uint32_t flag,
               cudaStream_t stream) {
    if (!h || !src || !pkts || !on_device(h))
        return AR_ERR_INVALID;
    if (((uintptr_t)src % h->esz) != 0 || ((uintptr_t)pkts % 8) != 0)
        return AR_ERR_INVALID;
    if (n == 0)
        return AR_OK;
    PackArgs a = {};
    a.src = src;
    a.pkts = pkts;
    a.n = n;
    a.flag = flag;
    a.status = h->ctl.status;
    const bool vec = ((uintptr_t)src % 8) == 0 && ((uintptr_t)pkts % 16) == 0;
    const int grid = clamp_grid(ceil_div(ceil_div(n * h->esz, 8), kRegThreads), h->reg_cap);
    return from_cuda(launch_pack(a, h->dtype, vec, grid, stream, h->pdl));
}

int ar_ll_unpack(ar_handle_t h, const uint64_t *pkts, void *dst, size_t n, uint32_t flag,
                 cudaStream_t stream) {
    if (!h || !dst || !pkts || !on_device(h))
        return AR_ERR_INVALID;
    if (((uintptr_t)dst % h->esz) != 0 || ((uintptr_t)pkts % 8) != 0)
        return AR_ERR_INVALID;
    if (n == 0)
        return AR_OK;
    PackArgs a = {};
    a.dst = dst;
    a.cpkts = pkts;
    a.n = n;
    a.flag = flag;
    a.status = h->ctl.status;
    const bool vec = ((uintptr_t)dst % 8) == 0 && ((uintptr_t)pkts % 16) == 0;
    const int grid = clamp_grid(ceil_div(ceil_div(n * h->esz, 8), kRegThreads), h->reg_cap);
    return from_cuda(launch_unpack(a, h->dtype, vec, grid, stream, h->pdl));
}

int ar_status(ar_handle_t h, cudaStream_t stream) {
    if (!h)
        return AR_ERR_INVALID;
    if (cudaStreamSynchronize(stream) != cudaSuccess)
        return from_cuda(cudaErrorUnknown);
    int code = 0;
    if (cudaMemcpyAsync(&code, h->ctl.status, sizeof(int), cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaMemsetAsync(h->ctl.status, 0, sizeof(int), stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return from_cuda(cudaErrorUnknown);
    return code;
}

int ar_set_timeout(ar_handle_t h, uint64_t ns) {
    if (!h)
        return AR_ERR_INVALID;
    h->ctl.timeout_ns = ns ? ns : kDefaultTimeoutNs;
    return AR_OK;
}

int ar_set_pdl(ar_handle_t h, int enable) {
    if (!h || (enable != 0 && enable != 1))
        return AR_ERR_INVALID;
    h->pdl = enable;
    return AR_OK;
}

int ar_set_ll_transport(ar_handle_t h, int transport) {
    if (!h || (transport != AR_LL_AUTO && transport != AR_LL_GLOBAL && transport != AR_LL_CLUSTER))
        return AR_ERR_INVALID;
    h->ll_transport = transport;
    return AR_OK;
}

int ar_set_hb_staging(ar_handle_t h, int staging) {
    if (!h || (staging != AR_HB_STAGING_AUTO && staging != AR_HB_STAGING_TMA &&
               staging != AR_HB_STAGING_DIRECT))
        return AR_ERR_INVALID;
    h->hb_staging = staging;
    return AR_OK;
}

int ar_get_hb_staging(ar_handle_t h, size_t bytes, int *staging) {
    if (!h || !staging || bytes == 0 || bytes > h->N * h->esz)
        return AR_ERR_INVALID;
    *staging = hb2_staging(h, bytes / h->esz > 0 ? bytes / h->esz : 1);
    return AR_OK;
}

int ar_set_grid_divisor(ar_handle_t h, int divisor) {
    if (!h || (divisor != 0 && divisor != 1 && divisor != 2 && divisor != 4 && divisor != 8))
        return AR_ERR_INVALID;
    h->grid_div = divisor;
    return AR_OK;
}

int ar_get_grid_divisor(ar_handle_t h, size_t bytes, int algo, int proto, int *divisor) {
    if (!h || !divisor || bytes == 0 || bytes > h->N * h->esz ||
        (algo != AR_ONE_SHOT && algo != AR_TWO_SHOT) || (proto != AR_LL && proto != AR_HB))
        return AR_ERR_INVALID;
    const uint64_t n = bytes / h->esz > 0 ? bytes / h->esz : 1;
    *divisor = algo == AR_ONE_SHOT && proto == AR_HB ? one_shot_div(h, n, true)
                                                     : grid_div(h, n, algo, proto);
    return AR_OK;
}

int ar_debug_drop_rank(ar_handle_t h, int rank) {
    if (!h || rank < -1 || rank >= h->R)
        return AR_ERR_INVALID;
    h->ctl.drop_rank = rank;
    return AR_OK;
}

int ar_round(int dtype, const float *src, void *dst, size_t n, cudaStream_t stream) {
    if (!valid_dtype(dtype) || !src || !dst)
        return AR_ERR_INVALID;
    if (((uintptr_t)src % 4) != 0 || ((uintptr_t)dst % elem_size(dtype)) != 0)
        return AR_ERR_INVALID;
    if (n == 0)
        return AR_OK;
    const int grid = clamp_grid(ceil_div(n, kRegThreads), 4096);
    return from_cuda(launch_round(dtype, src, dst, n, grid, stream));
}

int ar_get_info(ar_handle_t h, ar_info *info) {
    if (!h || !info)
        return AR_ERR_INVALID;
    info->R = h->R;
    info->dtype = h->dtype;
    info->N = h->N;
    info->elem_size = h->esz;
    info->ll_capable = h->slots != nullptr;
    info->ll_packets_per_rank = (h->N * h->esz + 3) / 4;
    info->scratch_bytes = h->dev_bytes;
    info->num_sms = h->num_sms;
    info->ll_ctas_per_rank_max = h->ll_cap[0] / h->R;
    info->tma_tile_bytes = h->tma_tile;
    info->tma_stages = h->tma_stages;
    info->timeout_ns = h->ctl.timeout_ns;
    info->ll_transport = h->ll_transport;
    info->hb_staging = h->hb_staging;
    info->pdl = h->pdl;
    info->ll_cluster_ok = h->cluster_ok ? 1 : 0;
    info->ll_cluster_units = h->cluster_ok ? (int)h->cluster_uc : 0;
    info->ll_cluster_max = h->cluster_ok ? h->cluster_max : 0;
    info->ll_staged_ctas_max = h->ll_staged_cap[0] < kEpochWords ? h->ll_staged_cap[0] : kEpochWords;
    return AR_OK;
}

}  // extern "C"
