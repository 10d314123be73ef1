/*
 * ar.h -- C ABI of a GB300 (sm_103a) sum all-reduce over R virtual ranks.
 *
 * The R ranks' buffers all live in one GPU's HBM ("virtual peers").  The
 * library sums them element by element and writes the sum into every rank's
 * output, with the schedules and protocols the MSCCL++ pages describe:
 *
 *   - the collective: a SUM all-reduce over the tensor-parallel ranks, called
 *     after every attention and MLP output ("SGLang 中的 MSCCL++ All-Reduce
 *     基准测试与推理集成指南", section 1), as a drop-in NCCL-style call
 *     ("【论文分享】MSCCL++：让 GPU 通信像 CUDA 一样可编程", section
 *     "第一层：Collective API");
 *   - dtypes float32 / float16 / bfloat16 and the SUM operation only (SGLang
 *     guide, section 4.3, run-time guard items 2 and 4);
 *   - the one-shot packet algorithm and the reduce-scatter + all-gather
 *     ("rsag") algorithm (SGLang guide, section 4.4);
 *   - the LL (low latency: small granularity, frequent synchronisation) and
 *     HB (high bandwidth: bulk transfer, little synchronisation) protocols of
 *     the MemoryChannel (MSCCL++ summary, section "MemoryChannel", protocol
 *     table);
 *   - capture in a CUDA graph (SGLang guide, section 1, first selling point).
 *
 * Arithmetic: every element is widened to binary32, the ranks are folded
 * left to right (rank 0 first, starting from rank 0's value) with one IEEE
 * binary32 round-to-nearest-even add per rank, and the result is rounded once
 * to the buffer dtype with round-to-nearest-even; no flush to zero.  Every
 * schedule and protocol gives bit-identical results.
 *
 * Conventions for every function:
 *   - The return value is an ar_status_code; AR_OK is 0.
 *   - "Device pointer": memory the current CUDA device can read/write with
 *     ordinary loads and stores (cudaMalloc, torch CUDA tensors, ...).  The
 *     library does not check that a pointer is a device pointer.  Buffers
 *     in page-locked host memory go through ar_allreduce_host, which checks
 *     them and keeps them off the kernels that copy with TMA or cp.async.
 *   - "Host array": a plain C array in host memory, read during the call only.
 *   - Work is enqueued on `stream` and nothing waits for it, except in
 *     ar_create, ar_destroy and ar_status.  No entry point used on the hot
 *     path (ar_allreduce, ar_reduce_scatter, ar_all_gather, ar_ll_pack,
 *     ar_ll_unpack, ar_round) allocates memory, copies between host and
 *     device, or synchronises, so all of them can be captured in a CUDA graph.
 *   - Calls on one handle must be ordered on the device (one stream, or
 *     streams joined by events): the handle's scratch and its epoch words are
 *     shared by all its calls.
 *   - Call with the device that was current at ar_create current; otherwise
 *     AR_ERR_INVALID.  ar_destroy and ar_plan_destroy make that device
 *     current themselves for the call, and restore the caller's.
 *   - A handle holds host state (its tuning table and settings) without
 *     locks: calls on one handle come from one host thread at a time.
 *     Distinct handles are independent.
 *   - Errors detected on the host are returned immediately and nothing is
 *     enqueued.  Errors detected on the device (a timed-out wait, a packet
 *     with the wrong flag) are recorded in the handle's status word and
 *     returned, then cleared, by ar_status.
 */
#ifndef AR_H
#define AR_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Largest number of virtual ranks one handle serves. */
#define AR_MAX_RANKS 32

/* Largest message, in bytes per rank, the LL protocol accepts.  LL is the
 * small-message protocol (MSCCL++ summary, "MemoryChannel" table: decode,
 * sampling, small messages); its packets double the bytes moved, and larger
 * messages belong to HB.  A handle whose N * sizeof(dtype) exceeds this
 * gets AR_ERR_UNSUPPORTED for LL calls and allocates no LL scratch. */
#define AR_LL_MAX_BYTES (64ull << 20)

typedef struct ar_handle *ar_handle_t;

/* Buffer element types (SGLang guide, section 4.3, guard item 2). */
enum ar_dtype {
    AR_BF16 = 0,
    AR_FP16 = 1,
    AR_FP32 = 2
};

/* Schedules (SGLang guide, section 4.4).
 *   AR_ONE_SHOT: every virtual rank r reads all R inputs and writes its own
 *                output out[r].
 *   AR_TWO_SHOT: reduce-scatter then all-gather.  The elements are cut into
 *                R shards (shard j: [j*S, min((j+1)*S, N)), S = ceil(N/R)
 *                rounded up to a whole 16-byte vector); rank j reduces shard
 *                j, then the reduced shard is copied to every output. */
enum ar_algo {
    AR_ONE_SHOT = 0,
    AR_TWO_SHOT = 1,
    AR_ALGO_AUTO = 2           /* chosen per message size, see ar_tune */
};

/* Protocols (MSCCL++ summary, section "MemoryChannel", protocol table).
 *   AR_LL: inputs travel as 8-byte packets, 4 message bytes in the low half
 *          and a 4-byte flag in the high half, written with one store; a
 *          receiver polls each packet until its flag equals the call's flag,
 *          so producers and consumers synchronise per packet inside one
 *          kernel.  The flag comes from epoch words kept on the device, so
 *          replays of a captured graph use a fresh flag every time.
 *   AR_HB: bulk path.  Two-shot HB stages tiles through shared memory with
 *          the Tensor Memory Accelerator (cp.async.bulk + mbarrier, no
 *          multicast) when every buffer is 16-byte aligned. */
enum ar_proto {
    AR_LL = 0,
    AR_HB = 1,
    AR_PROTO_AUTO = 2          /* chosen per message size, see ar_tune */
};

/* How one-shot LL packets travel between virtual peers.
 *   AR_LL_GLOBAL:  through per-sender slots in the handle's scratch (HBM/L2),
 *                  the layout real peers over NVLink would use; one
 *                  cooperative kernel for all ranks.
 *   AR_LL_CLUSTER: the R peers of a chunk form one thread-block cluster and
 *                  store their packets straight into each other's shared
 *                  memory (distributed shared memory), each receiver polling
 *                  its own; used where it applies (one-shot, R <= 16, every
 *                  buffer 16-byte aligned), AR_LL_GLOBAL elsewhere.
 *   AR_LL_AUTO:    AR_LL_GLOBAL (default; on GB300 the global-memory
 *                  exchange measured faster at every message size).
 * All three give identical results. */
enum ar_ll_transport {
    AR_LL_AUTO = 0,
    AR_LL_GLOBAL = 1,
    AR_LL_CLUSTER = 2
};

/* How two-shot HB calls move their data when every buffer is 16-byte aligned
 * (other buffers always take the direct form, element by element).
 *   AR_HB_STAGING_TMA:    bulk copies (the Tensor Memory Accelerator) bring
 *                         tiles of the R inputs into shared memory; each
 *                         thread folds its vectors of the tile once and
 *                         stores them to the R outputs; one CTA per SM with
 *                         several stages, or, for R >= 4 and calls moving
 *                         1 GiB or more, one stage of 128 KiB and two CTAs
 *                         per SM in turn.  Best for mid-sized messages at
 *                         larger R and for messages far beyond L2.
 *   AR_HB_STAGING_DIRECT: one thread per 16-byte vector loads the R inputs
 *                         into registers, folds them once and stores R copies;
 *                         as many CTAs as the message needs.  Lower latency
 *                         for small and mid-sized messages.
 *   AR_HB_STAGING_AUTO:   per message size: after ar_tune, the one timed
 *                         faster at that size; before it, and above the
 *                         largest tuned size, a fixed rule from GB300
 *                         measurements: with T = 2 * R * n * elem_size bytes
 *                         moved per call, TMA for 4 <= R <= 16 and
 *                         T >= 1 GiB; for R >= 32 and 64 KiB <= T <= 128 MiB;
 *                         for 16 <= R < 32 and T in [128 KiB, 1 MiB] or
 *                         [16 MiB, 64 MiB]; for 8 <= R < 16 and T in
 *                         [16 MiB, 64 MiB]; DIRECT otherwise.
 * Both are the reduce-scatter + all-gather schedule fused per unit (each
 * unit reduced once, by its shard's owner, and replicated) and give
 * identical results.  Source: the SGLang guide, section 4.4 (each algorithm
 * is timed over candidate launch configurations and the fastest kept per
 * message size). */
enum ar_hb_staging {
    AR_HB_STAGING_AUTO = 0,
    AR_HB_STAGING_TMA = 1,
    AR_HB_STAGING_DIRECT = 2
};

enum ar_status_code {
    AR_OK = 0,
    AR_ERR_INVALID = 1,        /* bad argument (null, range, aliasing, device) */
    AR_ERR_UNSUPPORTED = 2,    /* valid request this library does not serve   */
    AR_ERR_CUDA = 3,           /* a CUDA runtime call failed                   */
    AR_ERR_NOMEM = 4,          /* device allocation failed in ar_create        */
    AR_ERR_TIMEOUT = 5,        /* device: a wait ran past the handle's timeout */
    AR_ERR_FLAG_MISMATCH = 6   /* device: ar_ll_unpack met a packet whose flag
                                  differs from the expected one               */
};

/* Description of a handle, filled by ar_get_info. */
typedef struct ar_info {
    int R;                     /* virtual ranks                                */
    int dtype;                 /* enum ar_dtype                                */
    size_t N;                  /* elements per rank                            */
    size_t elem_size;          /* bytes per element                            */
    int ll_capable;            /* 1 if N * elem_size <= AR_LL_MAX_BYTES        */
    size_t ll_packets_per_rank;/* ceil(N * elem_size / 4)                      */
    size_t scratch_bytes;      /* device bytes the handle owns                 */
    int num_sms;               /* SMs of the handle's device                   */
    int ll_ctas_per_rank_max;  /* co-resident CTAs per rank of the per-rank LL
                                  kernel (buffers not all 8-byte aligned)     */
    int tma_tile_bytes;        /* per-rank tile of the two-shot TMA kernel     */
    int tma_stages;            /* pipeline stages of the two-shot TMA kernel   */
    uint64_t timeout_ns;       /* current device-side wait limit               */
    int ll_transport;          /* enum ar_ll_transport in force                */
    int ll_cluster_ok;         /* 1 if the cluster LL kernel can run           */
    int ll_cluster_units;      /* its 16-byte units per rank per chunk         */
    int ll_cluster_max;        /* its co-resident clusters                     */
    int pdl;                   /* 1 if launches use programmatic dependent launch */
    int ll_staged_ctas_max;    /* CTAs of the staged one-shot LL kernel (every
                                  buffer 8-byte aligned), each serving all R
                                  ranks                                       */
    int hb_staging;            /* enum ar_hb_staging in force                  */
} ar_info;

/* Create a handle for R virtual ranks of N elements of `dtype` each, on the
 * current device.  Source: the communication objects are set up once, on the
 * host, before device code uses them ("microsoft/mscclpp" project page, "How
 * it works": channels are defined on the host and called from kernels; SGLang
 * guide, section 4.4: the communicator is built once at start-up).  What it
 * allocates (packet scratch, epoch and status words) is this library's own
 * design; the pages size no such buffers.
 *   R:     1 .. AR_MAX_RANKS.
 *   N:     >= 1 elements per rank.
 *   dtype: enum ar_dtype.
 *   out:   receives the handle (host pointer, must not be NULL).
 * Allocates the handle's device memory (status word, epoch words and, when
 * N * elem_size <= AR_LL_MAX_BYTES, the LL packet scratch of (R + 1) slots of
 * ceil(N * elem_size / 4) packets, rounded up to 4 packets), zeroes it and
 * waits for that to finish.  Errors: AR_ERR_INVALID (R or N out of range,
 * bad dtype, out == NULL), AR_ERR_NOMEM, AR_ERR_CUDA. */
int ar_create(int R, size_t N, int dtype, ar_handle_t *out);

/* Free the handle and its device memory.  Waits for the handle's device
 * first (whichever device is current; the caller's is restored).  NULL is
 * accepted and ignored.  The pages define no teardown call: library
 * plumbing. */
int ar_destroy(ar_handle_t h);

/* Sum all-reduce: for every rank r and element i < N,
 *   out[r][i] = round_dtype( in[0][i] + in[1][i] + ... + in[R-1][i] )
 * with the binary32 left fold described at the top of this file.
 *   in:    host array of R device pointers, N elements each.
 *   out:   host array of R device pointers, N elements each.
 *   algo:  enum ar_algo.   proto: enum ar_proto.
 *   stream: the CUDA stream to enqueue on (0 = legacy default stream).
 * Every pointer must be non-NULL and aligned to the element size; 16-byte
 * alignment of all 2R pointers enables the vector paths, other alignments
 * run an element-wise GPU path (same results).  Outputs must not overlap
 * each other.  An input may overlap an output only as the same rank's
 * buffer exactly (in[r] == out[r], in place); inputs may overlap each other.
 * Errors: AR_ERR_INVALID (NULL handle or pointer, misaligned pointer,
 * forbidden overlap, wrong device, bad algo/proto), AR_ERR_UNSUPPORTED (LL on
 * a handle without LL scratch), AR_ERR_CUDA (launch failure).  Device-side
 * errors (AR_ERR_TIMEOUT) are reported by ar_status. */
int ar_allreduce(ar_handle_t h, const void *const in[], void *const out[],
                 int algo, int proto, cudaStream_t stream);

/* ar_allreduce on the first n elements of every buffer, 1 <= n <= N (the
 * handle's N is the largest message it serves, as one SGLang communicator
 * serves every message size it was tuned for: SGLang guide, section 4.4;
 * n has its own shards, S =
 * ceil(n/R) rounded up to a 16-byte vector).  Buffers need n elements.
 * With AR_ALGO_AUTO and/or AR_PROTO_AUTO the library picks the half left
 * open, per message size: the tuned fastest choice after ar_tune, else a
 * fixed rule from GB300 measurements (LL only for the one-shot at R >= 24
 * up to 4 KiB per rank on an LL-capable handle, HB otherwise; with HB,
 * one-shot for R <= 2 at every size, for R = 4 up to 256 KiB per rank, for
 * R = 16 up to 128 KiB and for other 8 <= R <= 24 up to 64 KiB, two-shot
 * otherwise; with AR_LL forced, one-shot up to 2 MiB).
 * Errors: as ar_allreduce; AR_ERR_INVALID also for n == 0 or n > N. */
int ar_allreduce_n(ar_handle_t h, const void *const in[], void *const out[], size_t n,
                   int algo, int proto, cudaStream_t stream);

/* ar_allreduce_n whose buffers may be in host memory: each of the 2R
 * pointers is device memory of the handle's device, managed memory, or
 * page-locked host memory that the device reaches at the same address
 * (cudaHostAlloc, cudaMallocHost or cudaHostRegister on a system with
 * unified addressing; on GB300 the kernels then read and write it through
 * the CPU-GPU link, so no copy is enqueued).  The pages' collective runs on
 * GPU buffers (MSCCL++ summary, section "第一层：Collective API"); host
 * buffers are a library addition for callers whose data sits in host memory.
 * With some buffer in host memory the call takes only kernels whose loads
 * and stores are plain ones: the two-shot HB in its direct staging, the
 * one-shot HB in its element-wise form, and the LL protocol over HBM packet
 * slots.  AUTO then follows a fixed rule from GB300 measurements: the
 * one-shot LL for R >= 24 up to 16 KiB per rank, the one-shot HB for R <= 4
 * from 1 MiB, the two-shot HB otherwise (a half fixed by the caller is kept:
 * with AR_LL the one-shot; with AR_ONE_SHOT LL on an LL-capable handle, HB
 * for R <= 4 from 1 MiB; with AR_TWO_SHOT HB).  With every
 * buffer in device memory the call is ar_allreduce_n.  Results are the same
 * bits either way.  Each call queries every pointer
 * (cudaPointerGetAttributes).
 * Errors: as ar_allreduce_n; AR_ERR_INVALID also for pageable host memory,
 * host memory mapped at another address, or another device's memory. */
int ar_allreduce_host(ar_handle_t h, const void *const in[], void *const out[], size_t n,
                      int algo, int proto, cudaStream_t stream);

/* Autotune AUTO for this handle (SGLang guide, section 4.4: every
 * (algorithm, configuration) is timed inside a CUDA graph at 15
 * power-of-two message sizes in [2^9, 2^24) bytes, and later calls map their
 * size, rounded up to a power of two and clamped to [512 B, 256 MiB], to the
 * fastest).  Here: each (algo, proto) pair is timed at every power of two
 * from 512 B to min(8 MiB, N * elem_size) bytes per rank as a graph of 10
 * calls, 5 warm-up replays then 20 timed replays, with each CTA-cap divisor
 * 1, 2 and 4 (see ar_set_grid_divisor; a larger one is kept only when more
 * than 2% faster) and two-shot HB also once per staging (enum ar_hb_staging).
 * The fastest launch of each pair is kept for that size: its divisor for
 * later calls of that pair, its staging for later two-shot HB calls with
 * AR_HB_STAGING_AUTO; sizes above the largest tuned one use its (algo, proto)
 * choice.  Not a hot-path call: it waits for `stream`, allocates and frees
 * 2 * R temporary buffers, creates a private stream and synchronises.
 * Returns AR_OK or the first error (including a device-side one, as
 * ar_status would). */
int ar_tune(ar_handle_t h, cudaStream_t stream);

/* The AUTO choice for a message of `bytes` per rank (*algo, *proto) and,
 * if `us` is not NULL, the tuned µs per call of the four pairs in the order
 * one-shot LL, one-shot HB, two-shot LL, two-shot HB (0 = not timed).  The
 * lookup follows the tuned-configuration cache of the SGLang guide, section
 * 4.4 (size rounded up to a power of two, clamped to [512 B, 256 MiB]). */
int ar_get_tuning(ar_handle_t h, size_t bytes, int *algo, int *proto, float us[4]);

/* Weighted per-token combine ("NCCL EP统一MoE通信生态", section 3.1 and
 * Table III: the low-latency mode reduces each token at the receiver with a
 * weight per expert).  With K = the handle's R sources:
 *   out[t*H + h] = round_dtype( fold over k = 0..K-1 of w[t*K + k] * y[k][t*H + h] )
 * every product rounded to binary32 on its own (no fused multiply-add), the
 * products folded left to right from k = 0, one final rounding.
 *   y:   host array of K device pointers, T*H elements each (row-major).
 *   w:   device pointer, T*K binary32 weights (row-major), 4-byte aligned.
 *   out: device pointer, T*H elements; may be one of the y[k] exactly,
 *        otherwise must not overlap them or w.
 *   T*H <= the handle's N.  16-byte aligned buffers with H*elem_size a
 *   multiple of 16 take the vector path.  Errors: AR_ERR_INVALID. */
int ar_combine(ar_handle_t h, const void *const y[], const float *w, void *out, size_t T,
               size_t H, cudaStream_t stream);

/* Reduce-scatter step of the two-shot schedule (the "rsag" algorithm of the
 * SGLang guide, section 4.4), HB: for every shard j,
 *   out[j][i] = round_dtype(fold of in[0..R-1][i])  for i in shard j,
 * and nothing else is written.  Shards as in enum ar_algo.  Arguments,
 * alignment and aliasing rules as in ar_allreduce. */
int ar_reduce_scatter(ar_handle_t h, const void *const in[], void *const out[],
                      cudaStream_t stream);

/* All-gather step of the two-shot schedule (SGLang guide, section 4.4,
 * "rsag"): for every shard j and rank
 * r != j, copies out[j]'s shard j into out[r]'s shard j (bits unchanged).
 *   out: host array of R device pointers, N elements each, not overlapping.
 * ar_reduce_scatter followed by ar_all_gather on the same outputs equals
 * ar_allreduce. */
int ar_all_gather(ar_handle_t h, void *const out[], cudaStream_t stream);

/* LL encode of one message of n elements of the handle's dtype (the LL
 * protocol of the MSCCL++ summary, section "MemoryChannel", protocol table).
 *   src:  device pointer, n elements.
 *   pkts: device pointer, ceil(n * elem_size / 4) 8-byte packets, 8-byte
 *         aligned.  Packet p = ((uint64_t)flag << 32) | payload, payload =
 *         message bytes [4p, 4p + 4) little-endian, zero past the end; so
 *         two-byte elements 2p and 2p + 1 are its low and high halves and a
 *         binary32 element p is its whole payload.
 *   n:    0 is accepted and does nothing.
 * Each packet is written with a single 8-byte store.  (Layout: the pages
 * name the LL protocol but print no layout; this is the library's reading.)
 * Errors: AR_ERR_INVALID (NULL, misaligned pointer). */
int ar_ll_pack(ar_handle_t h, const void *src, uint64_t *pkts, size_t n,
               uint32_t flag, cudaStream_t stream);

/* LL decode (MSCCL++ summary, section "MemoryChannel", LL protocol): the
 * inverse of ar_ll_pack.  A packet whose flag differs from
 * `flag` leaves its bytes of dst unwritten and records AR_ERR_FLAG_MISMATCH
 * in the handle's status word (read it with ar_status).  No waiting. */
int ar_ll_unpack(ar_handle_t h, const uint64_t *pkts, void *dst, size_t n,
                 uint32_t flag, cudaStream_t stream);

/* Wait for `stream`, then return and clear the handle's device status word:
 * AR_OK, AR_ERR_TIMEOUT or AR_ERR_FLAG_MISMATCH (the first error recorded
 * since the last ar_status), or AR_ERR_CUDA if the stream reports a CUDA
 * error.  The pages define no device-side error reporting (their waits are
 * unbounded): library plumbing for this library's bounded waits. */
int ar_status(ar_handle_t h, cudaStream_t stream);

/* Limit, in nanoseconds, of every device-side wait (LL packet polls, TMA
 * barrier waits) of later calls.  Default 1e9 (one second); 0 restores the
 * default.  A wait past the limit records AR_ERR_TIMEOUT, makes the other
 * waiters of the same call give up, and the kernel returns normally.  The
 * pages define no such limit: library plumbing. */
int ar_set_timeout(ar_handle_t h, uint64_t ns);

/* Programmatic dependent launch for the handle's later calls (1 = on, the
 * default; 0 = off).  On, a call's kernel may begin launching while the
 * previous kernel of the stream is still draining; it waits for that
 * kernel's completion before its first global-memory access, so results
 * are unchanged and only launch latency is hidden -- the per-call overhead
 * that dominates the small messages the LL protocol serves (SGLang guide,
 * section 1: latency enters every generated token).  Errors: AR_ERR_INVALID. */
int ar_set_pdl(ar_handle_t h, int enable);

/* Choose how later one-shot LL calls move packets (enum ar_ll_transport).
 * The MemoryChannel lets GPU threads write a peer's memory directly
 * (MSCCL++ summary, section "MemoryChannel"); for virtual peers on one GPU
 * that memory can be HBM or a cluster peer's shared memory.
 * Errors: AR_ERR_INVALID. */
int ar_set_ll_transport(ar_handle_t h, int transport);

/* Choose how later two-shot HB calls move their data (enum ar_hb_staging;
 * AR_HB_STAGING_AUTO is the default).  The HB protocol is the bulk row of the
 * MemoryChannel's protocol table (MSCCL++ summary, section "MemoryChannel");
 * the pages name no staging for it: a library choice, identical bits either
 * way.  Errors: AR_ERR_INVALID. */
int ar_set_hb_staging(ar_handle_t h, int staging);

/* The staging (AR_HB_STAGING_TMA or AR_HB_STAGING_DIRECT) a two-shot HB call
 * of `bytes` per rank (1 .. N * elem_size) on this handle would use now, with
 * every buffer 16-byte aligned.  The pages define no such query: library
 * plumbing.  Errors: AR_ERR_INVALID (NULL, bytes out of range). */
int ar_get_hb_staging(ar_handle_t h, size_t bytes, int *staging);

/* Launch shape: the number of CTAs.  The SGLang guide's tuner (section 4.4)
 * times launch configurations (blocks, threads per block) for each
 * algorithm; here the threads per CTA are fixed per kernel by its launch
 * bounds, and the CTA count is the path's cap (what the message needs, at
 * most the co-resident or per-SM limit the path uses) divided by a divisor.
 * ar_tune times divisors 1, 2 and 4 for every (algo, proto) at each tuned
 * size and keeps the fastest; calls of any algo/proto then use it.
 *
 * Force the divisor for later calls: 1, 2, 4 or 8; 0 (the default) uses the
 * tuned divisor, or 1 before ar_tune and above the tuned sizes.  Results are
 * the same bits whatever the divisor.  Errors: AR_ERR_INVALID. */
int ar_set_grid_divisor(ar_handle_t h, int divisor);

/* The divisor a call of `bytes` per rank (1 .. N * elem_size) with this algo
 * (AR_ONE_SHOT or AR_TWO_SHOT) and proto (AR_LL or AR_HB) would use now.
 * Errors: AR_ERR_INVALID (NULL, bytes out of range, AUTO or unknown
 * algo/proto). */
int ar_get_grid_divisor(ar_handle_t h, size_t bytes, int algo, int proto, int *divisor);

/* Fault injection for tests: virtual rank `rank` (0..R-1) writes no LL
 * packets in later LL calls, so its peers' polls time out (AR_ERR_TIMEOUT
 * from ar_status) and the kernel returns.  -1 turns it off.  The pages
 * define no such call: test plumbing. */
int ar_debug_drop_rank(ar_handle_t h, int rank);

/* The final rounding step on its own: dst[i] = round_dtype(src[i]) for n
 * binary32 values, with the same conversion the all-reduce kernels use
 * (round to nearest even, no flush to zero).  src, dst: device pointers.
 * Errors: AR_ERR_INVALID.  The pages print no rounding rule; this exposes
 * the library's reading (one round-to-nearest-even narrowing) so that it can
 * be checked exhaustively. */
int ar_round(int dtype, const float *src, void *dst, size_t n, cudaStream_t stream);

/* Fill *info (host pointer) with the handle's description.  The pages define
 * no such call: library plumbing. */
int ar_get_info(ar_handle_t h, ar_info *info);

/* Static string naming an ar_status_code.  The pages define no such call:
 * library plumbing. */
const char *ar_strerror(int code);

/* ---------------------------------------------------------------------------
 * Plans: an algorithm written as steps, compiled, then executed.
 *
 * "【论文分享】MSCCL++：让 GPU 通信像 CUDA 一样可编程", section
 * "第二层：DSL API": an algorithm author writes channel put / wait / reduce
 * steps; a compiler analyses the data dependencies, inserts the
 * synchronisation and emits an execution plan that a runtime interprets.
 * Here a step is a copy (a put into a peer's buffer; every virtual peer's
 * buffer is in this GPU's memory) or a reduce over chunks of the rank
 * buffers; ar_plan_compile adds the waits and signals; ar_plan_execute runs
 * the plan as one cooperative kernel in which every CTA interprets its own
 * instruction stream.  A plan means exactly its steps executed one after
 * another in the order written.
 * ------------------------------------------------------------------------- */
enum ar_op_kind {
    AR_OP_COPY = 0,            /* dst[c] = src[0][c] (bits unchanged)          */
    AR_OP_REDUCE = 1           /* dst[c] = round(fold of src[0..nsrc-1][c])    */
};
enum ar_buf_kind {
    AR_BUF_IN = 0,             /* the in[] buffer of a rank                   */
    AR_BUF_OUT = 1             /* the out[] buffer of a rank                  */
};

/* One step.  Buffers are cut into `nchunks` chunks (ar_plan_compile): chunk
 * c holds elements [c*C, min((c+1)*C, N)), C = ceil(N / nchunks) rounded up
 * to a whole 16-byte vector.  The step runs on chunks [chunk_begin,
 * chunk_end) in the program of virtual rank `rank`.  A reduce folds its
 * sources in the order listed (binary32, left to right) and rounds once. */
typedef struct ar_op {
    int kind;                  /* enum ar_op_kind                              */
    int rank;                  /* whose program runs the step, 0..R-1         */
    int dst_buf, dst_rank;     /* destination: enum ar_buf_kind, rank         */
    int src_buf;               /* sources' buffer kind                        */
    int nsrc;                  /* 1 for a copy, 1..R for a reduce             */
    int src_rank[AR_MAX_RANKS];/* sources' ranks, in fold order               */
    int chunk_begin, chunk_end;
} ar_op;

typedef struct ar_plan *ar_plan_t;

/* Compile `nops` steps for the handle's R, N and dtype ("【论文分享】MSCCL++：
 * 让 GPU 通信像 CUDA 一样可编程", section "第二层：DSL API": dependency analysis,
 * synchronisation, operator fusion, an execution plan).  Each step over k
 * chunks becomes k tasks; task (step, c) runs on CTA rank * ctas_per_rank +
 * c % ctas_per_rank.  A copy task whose source chunk was last written by an
 * earlier task t, and whose destination chunk no task has touched since t,
 * is fused into t (t also stores its result there) and disappears; the
 * results are those of running the steps one after another.  A task waits
 * for every earlier task in another CTA whose chunk it reads after a write,
 * writes after a read, or writes after a write; those producers signal a
 * semaphore.  Allocates the plan's device memory and waits for the upload
 * (not a hot-path call).
 * Errors: AR_ERR_INVALID (bad step, range), AR_ERR_UNSUPPORTED (R *
 * ctas_per_rank CTAs cannot all be resident, or the steps make more than
 * 2^20 tasks), AR_ERR_NOMEM (device or host memory), AR_ERR_CUDA. */
int ar_plan_compile(ar_handle_t h, const ar_op *ops, int nops, int nchunks,
                    int ctas_per_rank, ar_plan_t *out);
/* (ctas_per_rank == 0: as many as can be resident together, R * that <= the
 * device's capacity for the interpreter kernel.) */

/* The two all-reduce algorithms of the SGLang guide, section 4.4 (one-shot
 * packet and "rsag"), as plans with chunks_per_rank * R chunks:
 *   AR_ONE_SHOT: rank r reduces every input into out[r];
 *   AR_TWO_SHOT: rank j reduces shard j (chunks [j*K, (j+1)*K)) into out[j],
 *                then every rank copies every other shard into its output.
 * Same results as ar_allreduce.  chunks_per_rank == 0 picks ctas_per_rank
 * chunks, except for AR_TWO_SHOT with R >= 8: there a multiple of
 * ctas_per_rank (1 to 16 per CTA) that makes a chunk about 8 KiB of a rank
 * buffer.  ctas_per_rank == 0 fills the resident capacity, except for
 * AR_TWO_SHOT with R >= 16: there two CTAs per SM.  Errors as
 * ar_plan_compile. */
int ar_plan_builtin(ar_handle_t h, int algo, int chunks_per_rank, int ctas_per_rank,
                    ar_plan_t *out);

/* Run the plan once (the runtime that interprets an execution plan, section
 * "第二层：DSL API" above) on these buffers (host arrays of R device pointers, N
 * elements each; the 2R buffers must not overlap).  Capturable in a CUDA
 * graph: the run index comes from device-side epoch words.  Waits are
 * bounded by the handle's timeout; a timed-out run reports AR_ERR_TIMEOUT
 * through ar_status on the handle, and the plan must then be rebuilt. */
int ar_plan_execute(ar_plan_t p, const void *const in[], void *const out[], cudaStream_t stream);

/* Tasks (after fusion), inserted waits and signalling tasks of a compiled
 * plan (any pointer may be NULL).  The pages define no such call: library
 * plumbing that exposes what the compiler of section "第二层：DSL API" did. */
int ar_plan_stats(ar_plan_t p, int *tasks, int *waits, int *signals);

/* Free a plan (waits for the device first).  NULL is accepted.  The pages
 * define no teardown call: library plumbing. */
int ar_plan_destroy(ar_plan_t p);

/* Bytes of packet scratch compiled into the library for
 * ar_allreduce_ll_static (every GPU that loads the library holds this much
 * static device memory, plus 8.25 KiB of control words, until the process
 * exits). */
#define AR_NOALLOC_SCRATCH_BYTES (8u << 20)

/* One-shot LL all-reduce that allocates nothing.  The pages have no
 * counterpart of this call; it exists for callers that cannot allocate
 * device memory where they run the collective: an inference engine that
 * reserves nearly all of the GPU's memory up front for its own pool (KV
 * cache, activations) and accounts for every byte, so a side allocation
 * would fail or break its memory plan; or a hook on a latency-critical path
 * that must not pay for cudaMalloc/cudaFree, which can synchronise the whole
 * device.  ar_create's scratch is unavailable to them; this call uses a
 * fixed array of static device memory inside the library instead.
 *   R, N, dtype: as in ar_create.   in, out, stream: as in ar_allreduce
 *   (same alignment and aliasing rules).
 * Computes exactly what ar_allreduce(h, in, out, AR_ONE_SHOT, AR_LL, stream)
 * computes.  Limit: R * ceil(ceil(N * elem_size / 4) / 4) * 32 bytes of
 * packets must fit in AR_NOALLOC_SCRATCH_BYTES (8 MiB: for example R = 8
 * ranks of up to 512 KiB each); larger messages return AR_ERR_UNSUPPORTED
 * and nothing is enqueued.  It calls no cudaMalloc/cudaFree and no
 * allocating library routine.
 * The first call on each device sets the array up (resolves its device
 * address, zeroes its control words and waits for that to finish, so that
 * call synchronises the device); make it with that device current.
 * All calls share the one array and it keeps the last call's contents, so
 * calls whose kernels overlap on the GPU race: order them on one stream (or
 * with events).  Device-side wait limits are fixed at one second and a
 * timed-out wait is not reported (there is no handle to query).
 * Errors: AR_ERR_INVALID (arguments), AR_ERR_UNSUPPORTED (too large),
 * AR_ERR_CUDA. */
int ar_allreduce_ll_static(int R, size_t N, int dtype, const void *const in[],
                           void *const out[], cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* AR_H */
