// Device-side building blocks shared by the kernels: dtype lanes, the ordered
// binary32 fold, LL packet memory operations, bounded waits and the epoch
// scheme that gives every call a fresh packet flag.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ar_internal.h"

namespace ar {

// ---------------------------------------------------------------------------
// Element types.  A 16-byte vector holds kPerVec elements; a 4-byte LL
// payload word holds kPerWord.
// ---------------------------------------------------------------------------
template <int DT> struct Elem;
template <> struct Elem<AR_BF16> { enum { kSize = 2, kPerVec = 8, kPerWord = 2 }; };
template <> struct Elem<AR_FP16> { enum { kSize = 2, kPerVec = 8, kPerWord = 2 }; };
template <> struct Elem<AR_FP32> { enum { kSize = 4, kPerVec = 4, kPerWord = 1 }; };

// Exact widening of one element's bit pattern to binary32.
template <int DT> __device__ __forceinline__ float widen1(uint32_t bits);
template <> __device__ __forceinline__ float widen1<AR_BF16>(uint32_t b) {
    return __uint_as_float(b << 16);
}
template <> __device__ __forceinline__ float widen1<AR_FP16>(uint32_t b) {
    return __half2float(__ushort_as_half((unsigned short)b));
}
template <> __device__ __forceinline__ float widen1<AR_FP32>(uint32_t b) {
    return __uint_as_float(b);
}

// Round-to-nearest-even narrowing of one binary32 value (cvt.rn, no .ftz).
template <int DT> __device__ __forceinline__ uint32_t narrow1(float f);
template <> __device__ __forceinline__ uint32_t narrow1<AR_BF16>(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
template <> __device__ __forceinline__ uint32_t narrow1<AR_FP16>(float f) {
    return __half_as_ushort(__float2half_rn(f));
}
template <> __device__ __forceinline__ uint32_t narrow1<AR_FP32>(float f) {
    return __float_as_uint(f);
}

// A 4-byte word of elements (element 2p in the low half for two-byte types).
// WordAcc folds words rank by rank: init with rank 0, add ranks 1..R-1 in
// order, one binary32 add (__fadd_rn: never contracted) per element.
template <int DT> struct WordAcc;

template <> struct WordAcc<AR_BF16> {
    float lo, hi;
    __device__ __forceinline__ void init(uint32_t w) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xFFFF0000u);
    }
    __device__ __forceinline__ void add(uint32_t w) {
        lo = __fadd_rn(lo, __uint_as_float(w << 16));
        hi = __fadd_rn(hi, __uint_as_float(w & 0xFFFF0000u));
    }
    __device__ __forceinline__ uint32_t result() const {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);   // .x (low) <- lo
        return *reinterpret_cast<const uint32_t *>(&b);
    }
};

template <> struct WordAcc<AR_FP16> {
    float lo, hi;
    __device__ __forceinline__ void init(uint32_t w) {
        float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
        lo = f.x;
        hi = f.y;
    }
    __device__ __forceinline__ void add(uint32_t w) {
        float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
        lo = __fadd_rn(lo, f.x);
        hi = __fadd_rn(hi, f.y);
    }
    __device__ __forceinline__ uint32_t result() const {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
};

template <> struct WordAcc<AR_FP32> {
    float v;
    __device__ __forceinline__ void init(uint32_t w) { v = __uint_as_float(w); }
    __device__ __forceinline__ void add(uint32_t w) { v = __fadd_rn(v, __uint_as_float(w)); }
    __device__ __forceinline__ uint32_t result() const { return __float_as_uint(v); }
};

// 16-byte vector = four words.
template <int DT> struct VecAcc {
    WordAcc<DT> w[4];
    __device__ __forceinline__ void init(uint4 v) {
        w[0].init(v.x); w[1].init(v.y); w[2].init(v.z); w[3].init(v.w);
    }
    __device__ __forceinline__ void add(uint4 v) {
        w[0].add(v.x); w[1].add(v.y); w[2].add(v.z); w[3].add(v.w);
    }
    __device__ __forceinline__ uint4 result() const {
        return make_uint4(w[0].result(), w[1].result(), w[2].result(), w[3].result());
    }
};

// One element.
template <int DT> struct ElemAcc {
    float v;
    __device__ __forceinline__ void init(uint32_t b) { v = widen1<DT>(b); }
    __device__ __forceinline__ void add(uint32_t b) { v = __fadd_rn(v, widen1<DT>(b)); }
    __device__ __forceinline__ uint32_t result() const { return narrow1<DT>(v); }
};

// ---------------------------------------------------------------------------
// Global memory access.
// ---------------------------------------------------------------------------

// 16-byte load that allocates in L1 (re-read by the other ranks' warps).
__device__ __forceinline__ uint4 ld_v4_l1(const void *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte streaming load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_v4_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Element-granular access (2 or 4 bytes), for misaligned buffers and tails.
template <int DT> __device__ __forceinline__ uint32_t ld_elem(const void *base, uint64_t i) {
    if (Elem<DT>::kSize == 2)
        return reinterpret_cast<const uint16_t *>(base)[i];
    return reinterpret_cast<const uint32_t *>(base)[i];
}
template <int DT> __device__ __forceinline__ void st_elem(void *base, uint64_t i, uint32_t b) {
    if (Elem<DT>::kSize == 2)
        reinterpret_cast<uint16_t *>(base)[i] = (uint16_t)b;
    else
        reinterpret_cast<uint32_t *>(base)[i] = b;
}

// LL packets: every packet is written by one naturally aligned 8-byte store
// and read by one 8-byte load, so its payload and its flag are always seen
// together.  A v2.u64 access is two such 8-byte accesses.  The .relaxed.gpu
// qualifiers make the polls see other CTAs' stores (L1 is not coherent).
__device__ __forceinline__ void st_pkt2(uint64_t *p, uint64_t a, uint64_t b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" :: "l"(p), "l"(a), "l"(b)
                 : "memory");
}
__device__ __forceinline__ void st_pkt(uint64_t *p, uint64_t a) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(a) : "memory");
}
__device__ __forceinline__ void ld_pkt2(const uint64_t *p, uint64_t &a, uint64_t &b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];"
                 : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ uint64_t ld_pkt(const uint64_t *p) {
    uint64_t a;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
    return a;
}
__device__ __forceinline__ uint32_t ld_u32_relaxed(const uint32_t *p) {
    uint32_t a;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(a) : "l"(p) : "memory");
    return a;
}
__device__ __forceinline__ void st_u32_relaxed(uint32_t *p, uint32_t a) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(a) : "memory");
}

// Payload word q (message bytes [4q, 4q + 4), zero past the end) of an
// n-element buffer, element by element (any alignment of the buffer).
template <int ESZ>
__device__ __forceinline__ uint32_t load_payload(const void *base, uint64_t n, uint64_t q) {
    if (ESZ == 4)
        return reinterpret_cast<const uint32_t *>(base)[q];
    const uint16_t *b = reinterpret_cast<const uint16_t *>(base);
    const uint32_t lo = b[2 * q];
    const uint32_t hi = (2 * q + 1 < n) ? (uint32_t)b[2 * q + 1] : 0u;
    return lo | (hi << 16);
}

template <int ESZ>
__device__ __forceinline__ void store_payload(void *base, uint64_t n, uint64_t q, uint32_t pl) {
    if (ESZ == 4) {
        reinterpret_cast<uint32_t *>(base)[q] = pl;
        return;
    }
    uint16_t *b = reinterpret_cast<uint16_t *>(base);
    b[2 * q] = (uint16_t)pl;
    if (2 * q + 1 < n)
        b[2 * q + 1] = (uint16_t)(pl >> 16);
}

__device__ __forceinline__ uint64_t make_pkt(uint32_t payload, uint32_t flag) {
    return ((uint64_t)flag << 32) | (uint64_t)payload;
}
__device__ __forceinline__ uint32_t pkt_flag(uint64_t p) { return (uint32_t)(p >> 32); }
__device__ __forceinline__ uint32_t pkt_payload(uint64_t p) { return (uint32_t)p; }

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel starts with kernel_prologue():
// it lets the next kernel of the stream begin launching, then waits until
// the kernels it depends on have completed and their writes are visible.
// Both instructions do nothing when the launch did not ask for it.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void kernel_prologue() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Errors and bounded waits.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void record_error(int *status, int code) {
    atomicCAS(status, 0, code);
}

// Poll state of one thread within one call.  A wait that finds its data at
// once costs one load.  Otherwise the thread re-polls, backing off with
// __nanosleep after the first few tries; every 16 tries it checks the call's
// abort word (another waiter gave up) and the clock.  Past the handle's limit
// it records AR_ERR_TIMEOUT, raises the abort word for this call's flag and
// returns false: nothing spins without bound.
struct Poller {
    const Ctl *c;
    uint32_t flag;
    uint64_t deadline;   // 0 until the first failed poll

    __device__ __forceinline__ bool keep_waiting(uint32_t tries) {
        if (tries > 8)
            __nanosleep(tries > 64 ? 256 : 32);
        if ((tries & 15u) != 15u)
            return true;
        if (ld_u32_relaxed(c->abort) == flag)
            return false;
        uint64_t now = globaltimer_ns();
        if (deadline == 0) {
            deadline = now + c->timeout_ns;
            return true;
        }
        if (now > deadline) {
            record_error(c->status, AR_ERR_TIMEOUT);
            st_u32_relaxed(c->abort, flag);
            return false;
        }
        return true;
    }
};

// Wait until both packets at p carry the flag; returns false on give-up.
__device__ __forceinline__ bool poll_pkt2(Poller &w, const uint64_t *p, uint64_t &a,
                                          uint64_t &b) {
    ld_pkt2(p, a, b);
    uint32_t tries = 0;
    while (pkt_flag(a) != w.flag || pkt_flag(b) != w.flag) {
        if (!w.keep_waiting(++tries))
            return false;
        ld_pkt2(p, a, b);
    }
    return true;
}

__device__ __forceinline__ bool poll_pkt(Poller &w, const uint64_t *p, uint64_t &a) {
    a = ld_pkt(p);
    uint32_t tries = 0;
    while (pkt_flag(a) != w.flag) {
        if (!w.keep_waiting(++tries))
            return false;
        a = ld_pkt(p);
    }
    return true;
}

// Wait for the four packets [p, p + 4) (one 16-byte payload vector).
__device__ __forceinline__ bool poll_vec(Poller &w, const uint64_t *p, uint4 &v) {
    uint64_t a, b, c, d;
    ld_pkt2(p, a, b);
    ld_pkt2(p + 2, c, d);
    if (pkt_flag(a) != w.flag || pkt_flag(b) != w.flag) {
        if (!poll_pkt2(w, p, a, b))
            return false;
    }
    if (pkt_flag(c) != w.flag || pkt_flag(d) != w.flag) {
        if (!poll_pkt2(w, p + 2, c, d))
            return false;
    }
    v = make_uint4(pkt_payload(a), pkt_payload(b), pkt_payload(c), pkt_payload(d));
    return true;
}

// ---------------------------------------------------------------------------
// Epochs: a fresh LL flag for every call, kept on the device so that graph
// replays (whose kernel parameters are frozen) never reuse one.
//
// The handle keeps kEpochWords words, all equal to the last call's flag E
// between calls.  CTA b of a launch with g CTAs reads word b at its start and
// uses flag E + 1 (0 is skipped: zeroed scratch means "empty").  CTA b writes
// the new flag to words b, b + g, b + 2g, ...  Those sets are disjoint and
// together cover every word, so each word is written exactly once per call
// and all words are equal again when the kernel ends; no atomics, no
// last-block detection, whatever the grid size of each call.
//
// No CTA of a call reads any word but its own, so the words b + g, b + 2g,
// ... are written as soon as the CTA has its flag (publish_epoch_others,
// early in the kernel, overlapping the rest of its work); word b itself is
// written last, once every thread of the CTA has read it
// (publish_epoch_own).  The next call reads the words only after this grid
// has completed (griddepcontrol.wait, or plain stream order).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t call_flag(const Ctl &c) {
    uint32_t f = ld_u32_relaxed(c.epoch + blockIdx.x) + 1u;
    return f == 0u ? 1u : f;
}

__device__ __forceinline__ void publish_epoch_others(const Ctl &c, uint32_t flag) {
    for (uint32_t w = blockIdx.x + (threadIdx.x + 1) * gridDim.x; w < (uint32_t)kEpochWords;
         w += blockDim.x * gridDim.x)
        st_u32_relaxed(c.epoch + w, flag);
}

__device__ __forceinline__ void publish_epoch_own(const Ctl &c, uint32_t flag) {
    __syncthreads();   // every thread of this CTA has read word blockIdx.x
    if (threadIdx.x == 0)
        st_u32_relaxed(c.epoch + blockIdx.x, flag);
}

}  // namespace ar
