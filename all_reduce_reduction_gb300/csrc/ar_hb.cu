// Register-path kernels: one-shot HB, the reduce-scatter step, a fused
// two-shot (reduce once, store to every output) used where TMA cannot be
// (unaligned buffers), the all-gather step, and the standalone rounding.
//
// Sources: the one-shot and the reduce-scatter + all-gather ("rsag")
// all-reduce algorithms of "SGLang 中的 MSCCL++ All-Reduce 基准测试与推理集成指南",
// section 4.4; HB = bulk transfer with little synchronisation ("【论文分享】
// MSCCL++：让 GPU 通信像 CUDA 一样可编程", section "MemoryChannel", protocol
// table).
#include "ar_device.cuh"

namespace ar {

// Fold R ranks' 16-byte vectors at vector index u, ranks 0..R-1 in order.
// Loads are issued eight ranks at a time so that they overlap.
template <int DT, bool L1>
__device__ __forceinline__ uint4 fold_vec(const void *const *in, int R, uint64_t u) {
    VecAcc<DT> acc;
#pragma unroll 1
    for (int k0 = 0; k0 < R; k0 += 8) {
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (k0 + j < R) {
                const uint4 *p = reinterpret_cast<const uint4 *>(in[k0 + j]) + u;
                v[j] = L1 ? ld_v4_l1(p) : ld_v4_stream(p);
            }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (k0 + j < R) {
                if (k0 + j == 0)
                    acc.init(v[j]);
                else
                    acc.add(v[j]);
            }
    }
    return acc.result();
}

// Fold one element i.
template <int DT>
__device__ __forceinline__ uint32_t fold_elem(const void *const *in, int R, uint64_t i) {
    ElemAcc<DT> acc;
    acc.init(ld_elem<DT>(in[0], i));
    for (int k = 1; k < R; ++k)
        acc.add(ld_elem<DT>(in[k], i));
    return acc.result();
}

// ---------------------------------------------------------------------------
// One-shot HB.  Virtual rank r's output reads all R inputs: warp w of a CTA
// computes out[w % R] for a run of 32 units (16-byte vectors, or elements
// when some buffer is not 16-byte aligned).
//
// With vectors the CTA stages the inputs in shared memory through a ring of
// kOneShotStages slots filled by cp.async: in each slot, warp w holds rank
// w % R's 512 bytes of its run, loaded once, and after a barrier every warp
// folds all R staged vectors of its run in rank order.  So each input byte
// crosses L2 once per CTA instead of R times, and the loads of the next
// kOneShotStages - 1 iterations are in flight while one is folded.  When the
// grid covers the message (small messages: every CTA has one run) the host
// launches the SINGLE instantiation instead, which skips the ring.  In place
// (in[r] == out[r]) is safe: a CTA's units belong to it alone, an iteration
// stores only units whose loads have completed, and the loads in flight are
// of later iterations' units.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"((uint32_t)__cvta_generic_to_shared(smem)), "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int PENDING> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" :: "n"(PENDING) : "memory");
}

// RC > 0: the kernel is instantiated for R == RC, so the ring path's fold is
// unrolled and its shared-memory reads are issued eight at a time.
template <int DT, bool VEC, bool SINGLE, int RC = 0>
__global__ void __launch_bounds__(1024) k_one_shot_hb(const __grid_constant__ HbArgs a) {
    extern __shared__ uint4 ring[];                      // VEC: [kOneShotStages][W * 32]
    kernel_prologue();
    constexpr int PV = VEC ? Elem<DT>::kPerVec : 1;
    const int R = RC ? RC : a.R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = blockDim.x >> 5;
    const int r = warp % R;
    const int g = warp / R;
    const int m = W / R;
    const uint64_t units = a.n / PV;
    const uint64_t per_blk = (uint64_t)m * 32;
    const uint64_t nblk = (units + per_blk - 1) / per_blk;

    if constexpr (VEC && SINGLE) {
        // Every CTA has at most one run (the grid covers the message), so
        // there is nothing to overlap.  Up to 16 ranks, fold straight from
        // global memory (the R warps of a run read the same lines side by
        // side, and all but the first read hit L1); above, the R^2 loads
        // through L1 cost more than one staging pass.
        if (blockIdx.x < nblk) {
            const uint64_t u = (uint64_t)blockIdx.x * per_blk + (uint64_t)g * 32 + lane;
            const bool live = g < m && u < units;
            uint4 res = make_uint4(0, 0, 0, 0);
            if (R <= 16) {
                if (live)
                    res = fold_vec<DT, true>(a.p.in, R, u);
            } else {
                if (live)
                    ring[threadIdx.x] =
                        ld_v4_stream(reinterpret_cast<const uint4 *>(a.p.in[r]) + u);
                __syncthreads();
                if (live) {
                    const uint4 *run = ring + g * R * 32 + lane;
                    VecAcc<DT> acc;
                    acc.init(run[0]);
                    for (int k = 1; k < R; ++k)
                        acc.add(run[k * 32]);
                    res = acc.result();
                }
            }
            if (a.inplace)
                __syncthreads();
            if (live)
                st_v4(reinterpret_cast<uint4 *>(a.p.out[r]) + u, res);
        }
    } else if constexpr (VEC) {
        constexpr int S = kOneShotStages;
        const uint64_t iters =
            blockIdx.x < nblk ? (nblk - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        if (iters > 0) {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.p.in[r]);
            // iteration j: this warp's run of rank r into slot j % S (one
            // group per iteration, empty past the last so the wait count
            // stays fixed)
            auto issue = [&](uint64_t j) {
                if (j < iters && g < m) {
                    const uint64_t u =
                        (blockIdx.x + j * gridDim.x) * per_blk + (uint64_t)g * 32 + lane;
                    if (u < units)
                        cp_async16(&ring[(int)(j % S) * (W * 32) + threadIdx.x], src + u);
                }
                cp_async_commit();
            };
#pragma unroll
            for (int j = 0; j < S - 1; ++j)
                issue(j);
            for (uint64_t it = 0; it < iters; ++it) {
                cp_async_wait<S - 2>();                  // this thread's copies of iteration it
                __syncthreads();                         // ... and everyone's; slot (it-1) % S is free
                issue(it + S - 1);
                const uint64_t u =
                    (blockIdx.x + it * gridDim.x) * per_blk + (uint64_t)g * 32 + lane;
                if (g < m && u < units) {
                    const uint4 *slot = ring + (int)(it % S) * (W * 32) + g * R * 32 + lane;
                    VecAcc<DT> acc;
                    acc.init(slot[0]);
                    if constexpr (RC > 0) {
#pragma unroll
                        for (int k0 = 1; k0 < RC; k0 += 8) {
                            uint4 x[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (k0 + j < RC)
                                    x[j] = slot[(k0 + j) * 32];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (k0 + j < RC)
                                    acc.add(x[j]);
                        }
                    } else {
                        for (int k = 1; k < R; ++k)
                            acc.add(slot[k * 32]);
                    }
                    st_v4(reinterpret_cast<uint4 *>(a.p.out[r]) + u, acc.result());
                }
            }
            cp_async_wait<0>();
        }
    } else {
        for (uint64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
            const uint64_t u = blk * per_blk + (uint64_t)g * 32 + lane;
            const bool live = u < units && g < m;
            uint32_t res = 0;
            if (live)
                res = fold_elem<DT>(a.p.in, R, u);
            if (a.inplace)
                __syncthreads();
            if (live)
                st_elem<DT>(a.p.out[r], u, res);
        }
    }

    // Ragged tail (fewer than one vector of elements): the last CTA, one
    // thread per (element, rank), all reads before any store.
    if (VEC && blockIdx.x == gridDim.x - 1) {
        const uint64_t first = units * PV;
        const int tail = (int)(a.n - first);
        const int t = threadIdx.x;
        const bool live = t < tail * R;
        uint32_t res = 0;
        if (live)
            res = fold_elem<DT>(a.p.in, R, first + t / R);
        __syncthreads();
        if (live)
            st_elem<DT>(a.p.out[t % R], first + t / R, res);
    }
}

// ---------------------------------------------------------------------------
// Reduce: one thread per unit folds the R inputs once, then stores either to
// the output of the unit's shard owner only (reduce-scatter step) or to all
// R outputs (fused two-shot: the direct staging of the two-shot HB).  The
// thread reads everything before it writes and no other thread touches its
// unit, so in place is safe.  k_reduce_o4 is the fused vector form held to
// 64 registers (four CTAs per SM instead of three): more loads in flight,
// which the direct staging wants up to 64 MiB moved per call (L2-sized work)
// and not above, where the extra concurrency measured slower.
// ---------------------------------------------------------------------------
template <int DT, bool VEC, bool SCATTER>
__device__ __forceinline__ void reduce_body(const HbArgs &a) {
    kernel_prologue();
    constexpr int PV = VEC ? Elem<DT>::kPerVec : 1;
    const int R = a.R;
    const uint64_t units = a.n / PV;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += stride) {
        const int owner = (int)((u * PV) / a.shard);
        if (VEC) {
            const uint4 res = fold_vec<DT, false>(a.p.in, R, u);
            if (SCATTER) {
                st_v4(reinterpret_cast<uint4 *>(a.p.out[owner]) + u, res);
            } else {
                for (int r = 0; r < R; ++r)
                    st_v4(reinterpret_cast<uint4 *>(a.p.out[r]) + u, res);
            }
        } else {
            const uint32_t res = fold_elem<DT>(a.p.in, R, u);
            if (SCATTER) {
                st_elem<DT>(a.p.out[owner], u, res);
            } else {
                for (int r = 0; r < R; ++r)
                    st_elem<DT>(a.p.out[r], u, res);
            }
        }
    }
    if (VEC && blockIdx.x == 0) {
        const uint64_t i = units * PV + threadIdx.x;
        if (i < a.n) {
            const uint32_t res = fold_elem<DT>(a.p.in, R, i);
            const int owner = (int)(i / a.shard);
            if (SCATTER) {
                st_elem<DT>(a.p.out[owner], i, res);
            } else {
                for (int r = 0; r < R; ++r)
                    st_elem<DT>(a.p.out[r], i, res);
            }
        }
    }
}

template <int DT, bool VEC, bool SCATTER>
__global__ void __launch_bounds__(kRegThreads) k_reduce(const __grid_constant__ HbArgs a) {
    reduce_body<DT, VEC, SCATTER>(a);
}

template <int DT>
__global__ void __launch_bounds__(kRegThreads, 4) k_reduce_o4(const __grid_constant__ HbArgs a) {
    reduce_body<DT, true, false>(a);
}

// The fused form in kWideThreads-thread CTAs, for binary32.  Its fold needs
// fewer registers than the 16-bit ones (no widening), so four 256-thread CTAs
// fit on an SM (1024 threads); two of these fit (768 threads, as three
// 256-thread CTAs of the 16-bit forms), which streams large messages faster.
template <int DT>
__global__ void __launch_bounds__(kWideThreads) k_reduce_wide(const __grid_constant__ HbArgs a) {
    reduce_body<DT, true, false>(a);
}

// ---------------------------------------------------------------------------
// All-gather: every unit of shard j is read once from out[j] and stored to
// the R - 1 other outputs (a copy: bits unchanged).
// ---------------------------------------------------------------------------
template <int ESZ, bool VEC>
__global__ void __launch_bounds__(kRegThreads) k_all_gather(const __grid_constant__ HbArgs a) {
    kernel_prologue();
    constexpr int PV = VEC ? 16 / ESZ : 1;
    const int R = a.R;
    const uint64_t units = a.n / PV;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += stride) {
        const int owner = (int)((u * PV) / a.shard);
        if (VEC) {
            const uint4 v = ld_v4_stream(reinterpret_cast<const uint4 *>(a.p.out[owner]) + u);
            for (int r = 0; r < R; ++r)
                if (r != owner)
                    st_v4(reinterpret_cast<uint4 *>(a.p.out[r]) + u, v);
        } else if (ESZ == 2) {
            const uint16_t v = reinterpret_cast<const uint16_t *>(a.p.out[owner])[u];
            for (int r = 0; r < R; ++r)
                if (r != owner)
                    reinterpret_cast<uint16_t *>(a.p.out[r])[u] = v;
        } else {
            const uint32_t v = reinterpret_cast<const uint32_t *>(a.p.out[owner])[u];
            for (int r = 0; r < R; ++r)
                if (r != owner)
                    reinterpret_cast<uint32_t *>(a.p.out[r])[u] = v;
        }
    }
    if (VEC && blockIdx.x == 0) {
        const uint64_t i = units * PV + threadIdx.x;
        if (i < a.n) {
            const int owner = (int)(i / a.shard);
            for (int r = 0; r < R; ++r) {
                if (r == owner)
                    continue;
                if (ESZ == 2)
                    reinterpret_cast<uint16_t *>(a.p.out[r])[i] =
                        reinterpret_cast<const uint16_t *>(a.p.out[owner])[i];
                else
                    reinterpret_cast<uint32_t *>(a.p.out[r])[i] =
                        reinterpret_cast<const uint32_t *>(a.p.out[owner])[i];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// The final rounding on its own (exposes narrow1 for exhaustive checks).
// ---------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kRegThreads) k_round(const float *src, void *dst, uint64_t n) {
    kernel_prologue();
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        st_elem<DT>(dst, i, narrow1<DT>(src[i]));
}

// ---------------------------------------------------------------------------
// Launchers.
// ---------------------------------------------------------------------------
// Dynamic shared memory of a one-shot launch: the ring's kOneShotStages
// slots of one 16-byte vector per thread, or one slot when a single run is
// staged (more than 16 ranks), or none.
static size_t one_shot_smem(bool vec, bool single, int R, int block) {
    if (!vec || (single && R <= 16))
        return 0;
    return (size_t)(single ? 1 : kOneShotStages) * block * sizeof(uint4);
}

// Rank counts whose ring instantiation folds with R fixed (unrolled); R = 4
// and 32 only for one run per CTA (with several, the loop over R measured
// faster at R = 4; at R = 32 the one-shot is not the schedule for them).
static bool one_shot_unrolled(int R, bool single) {
    return R == 2 || R == 8 || R == 16 || ((R == 4 || R == 32) && single);
}

// `single`: the grid covers the message (one run per CTA at most).  The
// one-run form then runs only for rank counts without an unrolled ring: with
// one run per CTA the unrolled ring (each input staged once, the fold
// unrolled) measured 8-23% faster than folding through L1 over a runtime R
// (R = 2, 8, 16 at 1-64 KiB per rank); the ring's runtime-R loop did not.
template <int DT>
static cudaError_t one_shot_dt(const HbArgs &a, bool vec, bool single, int grid, int block,
                               cudaStream_t s, bool pdl) {
    const bool one_run = vec && single && !one_shot_unrolled(a.R, single);
    const size_t smem = one_shot_smem(vec, one_run, a.R, block);
    if (one_run)
        return launch_kernel(k_one_shot_hb<DT, true, true>, grid, block, smem, s, pdl, a);
    if (vec) {
        // rank counts with an unrolled fold: those where it measured faster
        // (R = 4 and 32 only with one run per CTA)
        switch (a.R) {
        case 2: return launch_kernel(k_one_shot_hb<DT, true, false, 2>, grid, block, smem, s, pdl, a);
        case 4:
            if (single)
                return launch_kernel(k_one_shot_hb<DT, true, false, 4>, grid, block, smem, s, pdl, a);
            return launch_kernel(k_one_shot_hb<DT, true, false>, grid, block, smem, s, pdl, a);
        case 32:
            if (single)
                return launch_kernel(k_one_shot_hb<DT, true, false, 32>, grid, block, smem, s, pdl, a);
            return launch_kernel(k_one_shot_hb<DT, true, false>, grid, block, smem, s, pdl, a);
        case 8: return launch_kernel(k_one_shot_hb<DT, true, false, 8>, grid, block, smem, s, pdl, a);
        case 16: return launch_kernel(k_one_shot_hb<DT, true, false, 16>, grid, block, smem, s, pdl, a);
        default: return launch_kernel(k_one_shot_hb<DT, true, false>, grid, block, smem, s, pdl, a);
        }
    }
    return launch_kernel(k_one_shot_hb<DT, false, false>, grid, block, smem, s, pdl, a);
}

template <int DT> static cudaError_t one_shot_prepare_dt(int bytes) {
    const void *fns[] = {reinterpret_cast<const void *>(&k_one_shot_hb<DT, true, false>),
                         reinterpret_cast<const void *>(&k_one_shot_hb<DT, true, false, 2>),
                         reinterpret_cast<const void *>(&k_one_shot_hb<DT, true, false, 4>),
                         reinterpret_cast<const void *>(&k_one_shot_hb<DT, true, false, 32>),
                         reinterpret_cast<const void *>(&k_one_shot_hb<DT, true, false, 8>),
                         reinterpret_cast<const void *>(&k_one_shot_hb<DT, true, false, 16>)};
    for (const void *f : fns) {
        const cudaError_t e =
            cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t one_shot_prepare() {
    const int bytes = (int)one_shot_smem(true, false, 0, 1024);
    cudaError_t e = one_shot_prepare_dt<AR_BF16>(bytes);
    if (e == cudaSuccess)
        e = one_shot_prepare_dt<AR_FP16>(bytes);
    if (e == cudaSuccess)
        e = one_shot_prepare_dt<AR_FP32>(bytes);
    return e;
}

cudaError_t launch_one_shot_hb(const HbArgs &a, int dtype, bool vec, bool single, int grid,
                               int block, cudaStream_t s, bool pdl) {
    switch (dtype) {
    case AR_BF16: return one_shot_dt<AR_BF16>(a, vec, single, grid, block, s, pdl);
    case AR_FP16: return one_shot_dt<AR_FP16>(a, vec, single, grid, block, s, pdl);
    default: return one_shot_dt<AR_FP32>(a, vec, single, grid, block, s, pdl);
    }
}

template <int DT>
static cudaError_t reduce_dt(const HbArgs &a, bool vec, bool scatter, int form, int grid,
                             cudaStream_t s, bool pdl) {
    if (vec && scatter)
        return launch_kernel(k_reduce<DT, true, true>, grid, kRegThreads, 0, s, pdl, a);
    if (vec && form == kReduceWide) {
        if constexpr (DT == AR_FP32)
            return launch_kernel(k_reduce_wide<DT>, grid, kWideThreads, 0, s, pdl, a);
        else
            return cudaErrorInvalidValue;
    }
    if (vec && form == kReduceOcc4)
        return launch_kernel(k_reduce_o4<DT>, grid, kRegThreads, 0, s, pdl, a);
    if (vec)
        return launch_kernel(k_reduce<DT, true, false>, grid, kRegThreads, 0, s, pdl, a);
    if (scatter)
        return launch_kernel(k_reduce<DT, false, true>, grid, kRegThreads, 0, s, pdl, a);
    return launch_kernel(k_reduce<DT, false, false>, grid, kRegThreads, 0, s, pdl, a);
}

cudaError_t launch_reduce(const HbArgs &a, int dtype, bool vec, bool scatter_only, int grid,
                          cudaStream_t s, bool pdl, int form) {
    switch (dtype) {
    case AR_BF16: return reduce_dt<AR_BF16>(a, vec, scatter_only, form, grid, s, pdl);
    case AR_FP16: return reduce_dt<AR_FP16>(a, vec, scatter_only, form, grid, s, pdl);
    default: return reduce_dt<AR_FP32>(a, vec, scatter_only, form, grid, s, pdl);
    }
}

cudaError_t launch_all_gather(const HbArgs &a, int dtype, bool vec, int grid, cudaStream_t s,
                              bool pdl) {
    if (elem_size(dtype) == 2)
        return vec ? launch_kernel(k_all_gather<2, true>, grid, kRegThreads, 0, s, pdl, a)
                   : launch_kernel(k_all_gather<2, false>, grid, kRegThreads, 0, s, pdl, a);
    return vec ? launch_kernel(k_all_gather<4, true>, grid, kRegThreads, 0, s, pdl, a)
               : launch_kernel(k_all_gather<4, false>, grid, kRegThreads, 0, s, pdl, a);
}

cudaError_t launch_round(int dtype, const float *src, void *dst, uint64_t n, int grid,
                         cudaStream_t s) {
    switch (dtype) {
    case AR_BF16: return launch_kernel(k_round<AR_BF16>, grid, kRegThreads, 0, s, false, src, dst, n);
    case AR_FP16: return launch_kernel(k_round<AR_FP16>, grid, kRegThreads, 0, s, false, src, dst, n);
    default: return launch_kernel(k_round<AR_FP32>, grid, kRegThreads, 0, s, false, src, dst, n);
    }
}

}  // namespace ar
