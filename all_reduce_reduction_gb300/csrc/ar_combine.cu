// Weighted per-token combine: out[t][h] = round(fold_k w[t][k] * y[k][t][h]).
//
// Source: "NCCL EP统一MoE通信生态", section 3.1 and Table III: in the
// low-latency mode the combine reduces every token at the receiver with a
// weight per expert.  The same ordered binary32 fold as the all-reduce, with
// each source first multiplied by its token's weight: every product is
// rounded on its own (__fmul_rn) and added with __fadd_rn, so nothing is
// contracted into a fused multiply-add and the bits equal the plain
// definition.  One thread per 16-byte vector of a token's row (or per
// element when the rows are not 16-byte aligned), eight sources' loads in
// flight at a time.  A thread reads every source element of its unit before
// it writes the output, so out may be one of the sources exactly.
#include "ar_device.cuh"

namespace ar {

// Weighted lanes: the word accumulators of ar_device.cuh with a factor.
template <int DT> struct WWordAcc;

template <> struct WWordAcc<AR_BF16> {
    float lo, hi;
    __device__ __forceinline__ void init(uint32_t x, float w) {
        lo = __fmul_rn(w, __uint_as_float(x << 16));
        hi = __fmul_rn(w, __uint_as_float(x & 0xFFFF0000u));
    }
    __device__ __forceinline__ void add(uint32_t x, float w) {
        lo = __fadd_rn(lo, __fmul_rn(w, __uint_as_float(x << 16)));
        hi = __fadd_rn(hi, __fmul_rn(w, __uint_as_float(x & 0xFFFF0000u)));
    }
    __device__ __forceinline__ uint32_t result() const {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&b);
    }
};

template <> struct WWordAcc<AR_FP16> {
    float lo, hi;
    __device__ __forceinline__ void init(uint32_t x, float w) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&x));
        lo = __fmul_rn(w, f.x);
        hi = __fmul_rn(w, f.y);
    }
    __device__ __forceinline__ void add(uint32_t x, float w) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&x));
        lo = __fadd_rn(lo, __fmul_rn(w, f.x));
        hi = __fadd_rn(hi, __fmul_rn(w, f.y));
    }
    __device__ __forceinline__ uint32_t result() const {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
};

template <> struct WWordAcc<AR_FP32> {
    float v;
    __device__ __forceinline__ void init(uint32_t x, float w) { v = __fmul_rn(w, __uint_as_float(x)); }
    __device__ __forceinline__ void add(uint32_t x, float w) {
        v = __fadd_rn(v, __fmul_rn(w, __uint_as_float(x)));
    }
    __device__ __forceinline__ uint32_t result() const { return __float_as_uint(v); }
};

template <int DT> struct WVecAcc {
    WWordAcc<DT> q[4];
    __device__ __forceinline__ void init(uint4 v, float w) {
        q[0].init(v.x, w); q[1].init(v.y, w); q[2].init(v.z, w); q[3].init(v.w, w);
    }
    __device__ __forceinline__ void add(uint4 v, float w) {
        q[0].add(v.x, w); q[1].add(v.y, w); q[2].add(v.z, w); q[3].add(v.w, w);
    }
    __device__ __forceinline__ uint4 result() const {
        return make_uint4(q[0].result(), q[1].result(), q[2].result(), q[3].result());
    }
};

template <int DT, bool VEC>
__global__ void __launch_bounds__(kRegThreads) k_combine(const __grid_constant__ CombineArgs a) {
    kernel_prologue();
    constexpr int PV = VEC ? Elem<DT>::kPerVec : 1;
    const int K = a.K;
    const uint64_t row = a.H / PV;                       // units per token
    const uint64_t units = a.T * row;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += stride) {
        const uint64_t t = u / row;
        const float *wt = a.w + t * (uint64_t)K;
        if (VEC) {
            WVecAcc<DT> acc;
            for (int k0 = 0; k0 < K; k0 += 8) {
                uint4 v[8];
                float w[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (k0 + j < K) {
                        v[j] = ld_v4_stream(reinterpret_cast<const uint4 *>(a.p.in[k0 + j]) + u);
                        w[j] = __ldg(wt + k0 + j);
                    }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (k0 + j < K) {
                        if (k0 + j == 0)
                            acc.init(v[j], w[j]);
                        else
                            acc.add(v[j], w[j]);
                    }
            }
            st_v4(reinterpret_cast<uint4 *>(a.p.out[0]) + u, acc.result());
        } else {
            float acc = __fmul_rn(__ldg(wt), widen1<DT>(ld_elem<DT>(a.p.in[0], u)));
            for (int k = 1; k < K; ++k)
                acc = __fadd_rn(acc, __fmul_rn(__ldg(wt + k), widen1<DT>(ld_elem<DT>(a.p.in[k], u))));
            st_elem<DT>(a.p.out[0], u, narrow1<DT>(acc));
        }
    }
}

template <int DT>
static cudaError_t combine_dt(const CombineArgs &a, bool vec, int grid, cudaStream_t s, bool pdl) {
    if (vec)
        return launch_kernel(k_combine<DT, true>, grid, kRegThreads, 0, s, pdl, a);
    return launch_kernel(k_combine<DT, false>, grid, kRegThreads, 0, s, pdl, a);
}

cudaError_t launch_combine(const CombineArgs &a, int dtype, bool vec, int grid, cudaStream_t s,
                           bool pdl) {
    switch (dtype) {
    case AR_BF16: return combine_dt<AR_BF16>(a, vec, grid, s, pdl);
    case AR_FP16: return combine_dt<AR_FP16>(a, vec, grid, s, pdl);
    default: return combine_dt<AR_FP32>(a, vec, grid, s, pdl);
    }
}

}  // namespace ar
