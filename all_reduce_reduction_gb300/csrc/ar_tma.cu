// Two-shot HB all-reduce with TMA staging: reduce-scatter and all-gather
// fused per tile through shared memory.
//
// Sources: the reduce-scatter + all-gather ("rsag") all-reduce of
// "SGLang 中的 MSCCL++ All-Reduce 基准测试与推理集成指南", section 4.4, and the HB
// protocol (bulk transfer, little synchronisation) of "【论文分享】MSCCL++：
// 让 GPU 通信像 CUDA 一样可编程", section "MemoryChannel", protocol table.
//
// Work item = (shard j, tile t): bytes [j*shard_bytes + t*T, ...) of every
// rank's buffer, clipped to shard j.  Shard j is the part virtual rank j
// reduces in the reduce-scatter step.  Per item:
//   producer (warp 0, one thread): R bulk copies global -> shared of the
//     item's tile of every input into one pipeline stage, completing on the
//     stage's "full" mbarrier (expect_tx = R * len);
//   consumers (8 warps): each thread folds its 16-byte vectors of the R
//     staged tiles in rank order (binary32), rounds, and stores the result
//     straight from registers to all R outputs (the all-gather step, fed
//     without re-reading the reduced shard); each warp then releases the
//     stage ("empty" mbarrier: one arrival per consumer warp).  For R = 8,
//     16 and 32 the fold is instantiated with R fixed, fully unrolled, its
//     shared-memory reads issued eight at a time.
// The consumer warps never wait for one another: no named barrier.  No
// multicast.  Minimal traffic: R reads + R writes of every byte.  The tile
// size, the number of stages and the grid come from the launcher per call:
// several stages on one CTA per SM, or, for calls moving 1 GiB or more, one
// stage of 128 KiB on two CTAs per SM that run one after the other.
//
// Every wait is bounded by the handle's timeout; a timed-out wait records
// AR_ERR_TIMEOUT and raises a shared abort flag that every other waiter of
// the CTA reads, so all of them give up.  Before the CTA exits, bulk loads
// still in flight are waited for.
#include "ar_device.cuh"

namespace ar {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// The consumer warps: every thread of the block but the producer warp.  The
// stages' "empty" barriers count one arrival per consumer warp.
constexpr int kConsumerThreads = 32 * kTmaConsumerWarps;
static_assert(kTmaThreads == 32 + kConsumerThreads,
              "the block is one producer warp plus the consumer warps");

// Bounded wait on an mbarrier phase.  Gives up when *abort is raised or the
// limit passes (then records AR_ERR_TIMEOUT and raises *abort).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Ctl &c,
                                       volatile int *abort) {
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t deadline = globaltimer_ns() + c.timeout_ns;
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort)
            return false;
        if (globaltimer_ns() > deadline) {
            record_error(c.status, AR_ERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

// Byte range of item i inside every rank's buffer; false if it is empty.
__device__ __forceinline__ bool item_range(const TmaArgs &a, uint64_t i, uint64_t &off,
                                           uint32_t &len) {
    const uint64_t j = i / a.tiles_per_shard;
    const uint64_t t = i - j * a.tiles_per_shard;
    const uint64_t lo = j * a.shard_bytes + t * (uint64_t)a.tile_bytes;
    uint64_t end = (j + 1) * a.shard_bytes;
    if (end > a.body_bytes)
        end = a.body_bytes;
    if (lo >= end)
        return false;
    off = lo;
    len = (uint32_t)((end - lo) < (uint64_t)a.tile_bytes ? (end - lo) : (uint64_t)a.tile_bytes);
    return true;
}

template <int DT, int RC>
__global__ void __launch_bounds__(kTmaThreads, 1) k_two_shot_tma(const __grid_constant__ TmaArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_flag;
    __shared__ uint64_t consumed_items;

    const int R = RC ? RC : a.R;
    const int T = a.tile_bytes, S = a.stages;
    uint8_t *in_tiles = smem;                                   // [S][R][T]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)S * R * T);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t items = a.tiles_per_shard * (uint64_t)R;
    volatile int *abortp = &abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kTmaConsumerWarps);
        }
        abort_flag = 0;
        consumed_items = 0;
        fence_mbar_init();
    }
    __syncthreads();
    kernel_prologue();

    uint64_t issued = 0;   // producer: items whose loads were issued
    if (warp == 0) {
        if (lane == 0) {
            for (uint64_t i = blockIdx.x; i < items; i += gridDim.x) {
                uint64_t off;
                uint32_t len;
                if (!item_range(a, i, off, len))
                    continue;
                const int stage = (int)(issued % S);
                const uint32_t parity = (uint32_t)((issued / S) & 1u);
                // the stage is free once the consumers released its previous use
                if (issued >= (uint64_t)S && !mbar_wait(empty0 + 8 * stage, parity ^ 1u, a.c, abortp))
                    break;
                if (*abortp)
                    break;
                mbar_arrive_expect_tx(full0 + 8 * stage, (uint32_t)R * len);
                const uint32_t dst = smem_u32(in_tiles + (size_t)stage * R * T);
                for (int k = 0; k < R; ++k)
                    bulk_g2s(dst + (uint32_t)(k * T), static_cast<const uint8_t *>(a.p.in[k]) + off,
                             len, full0 + 8 * stage);
                ++issued;
            }
        }
        __syncwarp();
    } else {
        const int ct = threadIdx.x - 32;
        const bool elected = ct == 0;
        uint64_t done = 0;
        for (uint64_t i = blockIdx.x; i < items; i += gridDim.x) {
            uint64_t off;
            uint32_t len;
            if (!item_range(a, i, off, len))
                continue;
            const int stage = (int)(done % S);
            const uint32_t parity = (uint32_t)((done / S) & 1u);
            const bool ok = mbar_wait(full0 + 8 * stage, parity, a.c, abortp);
            // leave as a whole warp (a lane that gave up and a lane that saw
            // the stage land must not part ways: both pass the same
            // __syncwarp calls)
            if (__any_sync(0xffffffffu, !ok))
                break;
            const uint8_t *tile = in_tiles + (size_t)stage * R * T;
            for (uint32_t p = (uint32_t)ct * 16u; p < len; p += 16u * kConsumerThreads) {
                VecAcc<DT> acc;
                acc.init(*reinterpret_cast<const uint4 *>(tile + p));
                if constexpr (RC > 0) {
#pragma unroll
                    for (int k0 = 1; k0 < RC; k0 += 8) {
                        uint4 x[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (k0 + j < RC)
                                x[j] = *reinterpret_cast<const uint4 *>(tile + (size_t)(k0 + j) * T + p);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (k0 + j < RC)
                                acc.add(x[j]);
                    }
                } else {
#pragma unroll 4
                    for (int k = 1; k < R; ++k)
                        acc.add(*reinterpret_cast<const uint4 *>(tile + (size_t)k * T + p));
                }
                const uint4 y = acc.result();
                for (int r = 0; r < R; ++r)
                    st_v4(static_cast<uint8_t *>(a.p.out[r]) + off + p, y);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty0 + 8 * stage);
            ++done;
        }
        if (elected)
            consumed_items = done;
        __syncwarp();

        // Ragged tail (< 16 bytes per rank): block 0, one thread per element,
        // every input read before the outputs are written.
        if (blockIdx.x == 0) {
            const uint64_t first = a.body_bytes / Elem<DT>::kSize;
            const uint64_t e = first + (uint64_t)ct;
            if (e < a.n) {
                ElemAcc<DT> acc;
                acc.init(ld_elem<DT>(a.p.in[0], e));
                for (int k = 1; k < R; ++k)
                    acc.add(ld_elem<DT>(a.p.in[k], e));
                const uint32_t y = acc.result();
                for (int r = 0; r < R; ++r)
                    st_elem<DT>(a.p.out[r], e, y);
            }
        }
        __syncwarp();
    }

    __syncthreads();
    // After an abort, loads may have been issued that no consumer waited
    // for; wait (bounded) until they have landed before shared memory is
    // released.  At most one item per stage can be outstanding.
    if (threadIdx.x == 0) {
        for (uint64_t k = consumed_items; k < issued; ++k) {
            const int stage = (int)(k % S);
            const uint32_t parity = (uint32_t)((k / S) & 1u);
            const uint64_t deadline = globaltimer_ns() + a.c.timeout_ns;
            while (!mbar_try_wait(full0 + 8 * stage, parity) && globaltimer_ns() < deadline) {
            }
        }
    }
}

size_t tma_smem_bytes(int R, int tile_bytes, int stages) {
    return (size_t)stages * R * tile_bytes + 2 * sizeof(uint64_t) * stages;
}

// R fixed at compile time for the rank counts of the workloads (fold fully
// unrolled, shared-memory reads eight at a time); other R loop.
template <int DT> static void *tma_kernel_for(int R) {
    switch (R) {
    case 8: return reinterpret_cast<void *>(&k_two_shot_tma<DT, 8>);
    case 16: return reinterpret_cast<void *>(&k_two_shot_tma<DT, 16>);
    case 32: return reinterpret_cast<void *>(&k_two_shot_tma<DT, 32>);
    default: return reinterpret_cast<void *>(&k_two_shot_tma<DT, 0>);
    }
}

// Dynamic shared memory the kernel may opt in to: the device's per-block
// opt-in maximum less what the kernel declares statically.
template <int DT> static cudaError_t prepare_dt(int *limit) {
    int dev = 0, optin = 0;
    cudaFuncAttributes fa;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess)
        e = cudaFuncGetAttributes(&fa, tma_kernel_for<DT>(0));
    if (e != cudaSuccess)
        return e;
    *limit = optin - (int)fa.sharedSizeBytes;
    for (int R : {0, 8, 16, 32}) {
        e = cudaFuncSetAttribute(tma_kernel_for<DT>(R), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 *limit);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t tma_prepare(int dtype, int *max_dynamic_smem) {
    switch (dtype) {
    case AR_BF16: return prepare_dt<AR_BF16>(max_dynamic_smem);
    case AR_FP16: return prepare_dt<AR_FP16>(max_dynamic_smem);
    default: return prepare_dt<AR_FP32>(max_dynamic_smem);
    }
}

cudaError_t launch_two_shot_tma(const TmaArgs &a, int dtype, int grid, cudaStream_t s, bool pdl) {
    const size_t smem = tma_smem_bytes(a.R, a.tile_bytes, a.stages);
    void *k = dtype == AR_BF16 ? tma_kernel_for<AR_BF16>(a.R)
            : dtype == AR_FP16 ? tma_kernel_for<AR_FP16>(a.R) : tma_kernel_for<AR_FP32>(a.R);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kTmaThreads);
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
    void *args[] = {const_cast<TmaArgs *>(&a)};
    return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace ar
