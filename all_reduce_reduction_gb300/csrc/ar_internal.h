// Internal declarations shared by the library's translation units: kernel
// argument blocks (passed by value as __grid_constant__ parameters, so a
// launch copies nothing to the device and stays legal inside graph capture)
// and the host-side launchers each kernel file exports.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ar.h"

namespace ar {

// Words in a handle's epoch array.  Every LL kernel launch uses at most this
// many CTAs (see the epoch scheme in ar_device.cuh).  Every call rewrites all
// of them, so the array is kept just above the largest grid the LL kernels
// use on GB300 (1216 co-resident CTAs of the staged kernel: 152 SMs x 8).
constexpr int kEpochWords = 2048;

// Threads per CTA of the register (non-TMA) kernels and the LL kernels.
constexpr int kRegThreads = 256;
// Threads per CTA of the fused two-shot's wide form (binary32, large calls).
constexpr int kWideThreads = 384;
constexpr int kLlThreads = 128;
constexpr int kLlStagedThreads = 256;   // one-shot LL with shared receive staging

// One-shot HB: slots of the shared-memory ring that stages the inputs.
constexpr int kOneShotStages = 4;

// TMA two-shot kernel: one producer warp and kTmaConsumerWarps consumer warps.
constexpr int kTmaConsumerWarps = 8;
constexpr int kTmaThreads = 32 * (1 + kTmaConsumerWarps);
constexpr int kTmaMaxStages = 4;

inline size_t elem_size(int dtype) { return dtype == AR_FP32 ? 4 : 2; }

// Makes `device` current for the scope and restores the caller's device.
class DeviceScope {
  public:
    explicit DeviceScope(int device) {
        ok_ = cudaGetDevice(&prev_) == cudaSuccess &&
              (prev_ == device || cudaSetDevice(device) == cudaSuccess);
        if (!ok_)
            prev_ = -1;
    }
    ~DeviceScope() {
        int cur = -1;
        if (prev_ >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev_)
            (void)cudaSetDevice(prev_);
    }
    bool ok() const { return ok_; }
    DeviceScope(const DeviceScope &) = delete;
    DeviceScope &operator=(const DeviceScope &) = delete;

  private:
    int prev_ = -1;
    bool ok_ = false;
};

// Launch kernel(args...) on stream s.  With `pdl` the launch allows
// programmatic dependent launch: it may start while the previous kernel in
// the stream drains, and every kernel of this library waits (griddepcontrol
// .wait) before its first global-memory access, so only the launch latency
// overlaps, never the data.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = 0;
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 1;
    }
    cfg.attrs = attr;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// The R ranks' buffers.  512 bytes for R = 32.
struct RankPtrs {
    const void *in[AR_MAX_RANKS];
    void *out[AR_MAX_RANKS];
};

// Device-side control words of a handle, shared by all its calls.
struct Ctl {
    uint32_t *epoch;      // kEpochWords words, all equal between calls
    int *status;          // first device-side error since the last ar_status
    uint32_t *abort;      // flag of the call whose waiters must give up
    uint64_t timeout_ns;  // limit of one wait
    int drop_rank;        // test fault injection: this rank writes no packets
};

// Register-path kernels (one-shot HB, reduce-scatter, fused two-shot,
// all-gather).
struct HbArgs {
    RankPtrs p;
    uint64_t n;           // elements per rank
    uint64_t shard;       // elements per shard S (two-shot split)
    int R;
    int inplace;          // some in[r] == out[r]
};

// Two-shot TMA kernel.
struct TmaArgs {
    RankPtrs p;
    uint64_t n;             // elements per rank
    uint64_t body_bytes;    // bytes per rank moved by TMA (multiple of 16)
    uint64_t shard_bytes;   // bytes per shard (multiple of 16)
    uint64_t tiles_per_shard;
    int R;
    int tile_bytes;         // per-rank tile (multiple of 16)
    int stages;
    Ctl c;
};

// LL kernels.
struct LlArgs {
    RankPtrs p;
    uint64_t n;           // elements per rank
    uint64_t shard;       // elements per shard S (two-shot split)
    uint64_t *slots;      // (R + 1) slots of `ppad` packets; slot R = results
    uint64_t ppad;        // packets per slot (multiple of 4)
    int R;
    int G;                // CTAs per virtual rank; gridDim.x == R * G
    Ctl c;
};

// LL one-shot through thread-block clusters (distributed shared memory).
struct LlClusterArgs {
    RankPtrs p;
    uint64_t n;               // elements per rank
    uint64_t units_per_chunk; // 16-byte units per rank per chunk (Uc)
    int R;                    // cluster size = virtual ranks
    Ctl c;
};
// Receive-buffer budget per CTA of the cluster LL kernel.
constexpr int kLlClusterMaxSmem = 96 * 1024;
constexpr int kLlClusterTargetSmem = 64 * 1024;

// Weighted per-token combine: K sources in p.in[0..K-1], the output in p.out[0].
struct CombineArgs {
    RankPtrs p;
    const float *w;          // T x K weights, row-major
    uint64_t T, H;           // tokens, elements per token
    int K;
};

// Standalone packet encode/decode and rounding.
struct PackArgs {
    const void *src;
    void *dst;
    uint64_t *pkts;
    const uint64_t *cpkts;
    uint64_t n;
    uint32_t flag;
    int *status;
};

// ---- launchers (return the launch's cudaError_t) ----------------------------

// ar_api.cu: a handle's device control words (status, abort, epoch, limit)
Ctl handle_ctl(ar_handle_t h);

// ar_hb.cu
cudaError_t one_shot_prepare();                 // opt in to the one-shot ring's shared memory
// `single`: the grid covers the message, every CTA has at most one run
cudaError_t launch_one_shot_hb(const HbArgs &a, int dtype, bool vec, bool single, int grid,
                               int block, cudaStream_t s, bool pdl = false);
// Launch forms of the fused two-shot (vectors, not scatter_only): 256-thread
// CTAs as the registers allow, 256-thread CTAs held to four per SM, or
// kWideThreads-thread CTAs (binary32 only; `grid` then counts those).
enum ReduceForm { kReducePlain = 0, kReduceOcc4 = 1, kReduceWide = 2 };
cudaError_t launch_reduce(const HbArgs &a, int dtype, bool vec, bool scatter_only, int grid,
                          cudaStream_t s, bool pdl = false, int form = kReducePlain);
cudaError_t launch_all_gather(const HbArgs &a, int dtype, bool vec, int grid, cudaStream_t s,
                              bool pdl = false);
cudaError_t launch_round(int dtype, const float *src, void *dst, uint64_t n, int grid,
                         cudaStream_t s);

// ar_tma.cu
cudaError_t tma_prepare(int dtype, int *max_dynamic_smem);   // opt in to large shared memory
size_t tma_smem_bytes(int R, int tile_bytes, int stages);
cudaError_t launch_two_shot_tma(const TmaArgs &a, int dtype, int grid, cudaStream_t s,
                                bool pdl = false);

// ar_ll.cu
// the per-rank kernel (buffers not all 8-byte aligned)
cudaError_t ll_occupancy(int dtype, bool two_shot, int *blocks_per_sm);
cudaError_t launch_ll(const LlArgs &a, int dtype, bool two_shot, cudaStream_t s, bool pdl = false);
// the staged kernels (every buffer 8-byte aligned)
cudaError_t ll_staged_occupancy(int dtype, bool two_shot, int *blocks_per_sm);
cudaError_t launch_ll_staged(const LlArgs &a, int dtype, bool two_shot, int ctas, cudaStream_t s,
                             bool pdl = false);
cudaError_t launch_pack(const PackArgs &a, int dtype, bool vec, int grid, cudaStream_t s,
                        bool pdl = false);
cudaError_t launch_unpack(const PackArgs &a, int dtype, bool vec, int grid, cudaStream_t s,
                          bool pdl = false);

// ar_combine.cu
cudaError_t launch_combine(const CombineArgs &a, int dtype, bool vec, int grid, cudaStream_t s,
                           bool pdl = false);

// ar_ll_cluster.cu
size_t ll_cluster_smem_bytes(int R, uint64_t units_per_chunk);
cudaError_t ll_cluster_prepare(int dtype, int R);
cudaError_t ll_cluster_max_clusters(const LlClusterArgs &a, int dtype, int *clusters);
cudaError_t launch_ll_cluster(const LlClusterArgs &a, int dtype, int nclusters, cudaStream_t s,
                              bool pdl = false);

}  // namespace ar
