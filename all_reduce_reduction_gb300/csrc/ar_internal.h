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
// many CTAs (see the epoch scheme in ar_device.cuh).
constexpr int kEpochWords = 8192;

// Threads per CTA of the register (non-TMA) kernels and the LL kernels.
constexpr int kRegThreads = 256;
constexpr int kLlThreads = 128;

// TMA two-shot kernel: one producer warp and kTmaConsumerWarps consumer warps.
constexpr int kTmaConsumerWarps = 8;
constexpr int kTmaThreads = 32 * (1 + kTmaConsumerWarps);
constexpr int kTmaMaxStages = 4;

inline size_t elem_size(int dtype) { return dtype == AR_FP32 ? 4 : 2; }

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

// ar_hb.cu
cudaError_t launch_one_shot_hb(const HbArgs &a, int dtype, bool vec, int grid, int block,
                               cudaStream_t s);
cudaError_t launch_reduce(const HbArgs &a, int dtype, bool vec, bool scatter_only, int grid,
                          cudaStream_t s);
cudaError_t launch_all_gather(const HbArgs &a, int dtype, bool vec, int grid, cudaStream_t s);
cudaError_t launch_round(int dtype, const float *src, void *dst, uint64_t n, int grid,
                         cudaStream_t s);

// ar_tma.cu
cudaError_t tma_prepare(int dtype, int *max_dynamic_smem);   // opt in to large shared memory
size_t tma_smem_bytes(int R, int tile_bytes, int stages);
cudaError_t launch_two_shot_tma(const TmaArgs &a, int dtype, int grid, cudaStream_t s);

// ar_ll.cu
cudaError_t ll_occupancy(int dtype, bool vec, bool two_shot, int *blocks_per_sm);
cudaError_t launch_ll(const LlArgs &a, int dtype, bool vec, bool two_shot, cudaStream_t s);
cudaError_t launch_pack(const PackArgs &a, int dtype, bool vec, int grid, cudaStream_t s);
cudaError_t launch_unpack(const PackArgs &a, int dtype, bool vec, int grid, cudaStream_t s);

}  // namespace ar
