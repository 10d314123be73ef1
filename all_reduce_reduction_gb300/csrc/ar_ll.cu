// LL protocol kernels: one-shot and two-shot all-reduce through flag-tagged
// 8-byte packets, and the standalone packet encode/decode.
//
// Sources: the LL protocol (small granularity, frequent synchronisation, for
// decode, sampling and small messages) of the MemoryChannel in
// "【论文分享】MSCCL++：让 GPU 通信像 CUDA 一样可编程", section "MemoryChannel",
// protocol table; its one-sided put/signal/wait primitives ("microsoft/mscclpp"
// project page, "How it works"); the one-shot packet and the reduce-scatter +
// all-gather all-reduce algorithms of "SGLang 中的 MSCCL++ All-Reduce 基准测试与
// 推理集成指南", section 4.4.
//
// Kernels.  When every buffer is 8-byte aligned, k_ll_staged (one-shot) and
// k_ll2_staged (two-shot) run: their CTAs serve all R ranks for a block of
// units, and the R receivers of a unit share one poll of each packet (see
// their comments).  Otherwise k_ll runs either schedule with per-rank CTAs
// and one packet per unit, as follows.
//
// Virtual peers.  The R ranks' kernels are emulated as one kernel over all
// ranks' data: CTA b works for virtual rank r = b % R (CTA gi = b / R of its
// G CTAs).  A rank "puts" its input into its own slot of the handle's
// scratch as packets (payload + this call's flag in one 8-byte store); the
// peers' CTAs poll those packets until the flag matches.  All peers share
// one HBM, so one slot per sender serves every receiver.  There is no grid
// barrier: producers and consumers meet only through packet flags.
//
// Forward progress.  Consumers wait for packets that other CTAs produce, so
// all CTAs must be resident together: the launch is cooperative and its grid
// never exceeds the occupancy-derived capacity.  Every CTA performs all of
// its puts before any of its waits, and in the two-shot kernel all of its
// reduce-scatter work before any all-gather wait, so every wait depends only
// on work that resident CTAs do without waiting.  Waits are bounded anyway.
//
// In place (in[r] == out[r]) is safe: the CTA that writes out[r]'s unit u is
// the CTA that read in[r]'s unit u into packets, earlier.
#include "ar_device.cuh"

namespace ar {

__device__ __forceinline__ uint2 ld_v2(const void *p) {
    uint2 v;
    asm volatile("ld.global.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ void st_v2(void *p, uint2 v) {
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// Fold the packet at `base` (packet offset inside a slot) of slots 0..R-1,
// in rank order.  Loads of eight ranks are issued before any flag is
// checked, so a ready message costs one round trip per eight ranks.
template <int DT>
__device__ __forceinline__ bool fold_one(Poller &w, const uint64_t *base, uint32_t ppad, int R,
                                         uint32_t &out) {
    WordAcc<DT> acc;
#pragma unroll 1
    for (int k0 = 0; k0 < R; k0 += 8) {
        uint64_t p[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (k0 + j < R)
                p[j] = ld_pkt(base + (uint32_t)(k0 + j) * ppad);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (k0 + j < R) {
                if (pkt_flag(p[j]) != w.flag && !poll_pkt(w, base + (uint32_t)(k0 + j) * ppad, p[j]))
                    return false;
                if (k0 + j == 0)
                    acc.init(pkt_payload(p[j]));
                else
                    acc.add(pkt_payload(p[j]));
            }
        }
    }
    out = acc.result();
    return true;
}

// Per-rank kernel for buffers that are not all 8-byte aligned: a unit is one
// packet (4 message bytes; the last one may be partial).
template <int DT, bool TWO>
__global__ void __launch_bounds__(kLlThreads) k_ll(const __grid_constant__ LlArgs a) {
    constexpr int ESZ = Elem<DT>::kSize;
    const int R = a.R, G = a.G;
    const int r = blockIdx.x % R, gi = blockIdx.x / R;
    const uint32_t tid = threadIdx.x, T = blockDim.x;
    kernel_prologue();
    const uint32_t flag = call_flag(a.c);
    Poller w{&a.c, flag, 0};

    const uint32_t nbytes = (uint32_t)a.n * ESZ;
    const uint32_t P = (nbytes + 3) / 4;                  // packets per rank
    // this thread's packets (the same set in every phase that uses them)
    const uint32_t q0 = (uint32_t)gi * T + tid, qstep = (uint32_t)G * T;

    const uint32_t ppad = (uint32_t)a.ppad;
    uint64_t *const slot_r = a.slots + (uint32_t)r * ppad;
    uint64_t *const res = a.slots + (uint32_t)R * ppad;   // two-shot results
    bool ok = true;

    // ---- put: rank r's input -> slot r (one 8-byte store per packet) -------
    if (a.c.drop_rank != r) {
        for (uint32_t q = q0; q < P; q += qstep)
            st_pkt(slot_r + q, make_pkt(load_payload<ESZ>(a.p.in[r], a.n, q), flag));
    }

    publish_epoch_others(a.c, flag);

    if (!TWO) {
        // ---- one-shot: out[r] = fold of every slot -------------------------
        for (uint32_t q = q0; ok && q < P; q += qstep) {
            uint32_t y;
            ok = fold_one<DT>(w, a.slots + q, ppad, R, y);
            if (ok)
                store_payload<ESZ>(a.p.out[r], a.n, q, y);
        }
    } else {
        // ---- reduce-scatter: rank r folds shard r into result packets ------
        const uint32_t shard_pk = (uint32_t)(a.shard * ESZ / 4);   // packets per shard
        const uint32_t lo = (uint32_t)r * shard_pk;
        uint32_t hi = lo + shard_pk;
        if (hi > P)
            hi = P;
        for (uint32_t q = lo + q0; ok && q < hi; q += qstep) {
            uint32_t y;
            ok = fold_one<DT>(w, a.slots + q, ppad, R, y);
            if (ok)
                st_pkt(res + q, make_pkt(y, flag));
        }
        // ---- all-gather: out[r] <- result packets (same units as the put) --
        for (uint32_t q = q0; ok && q < P; q += qstep) {
            uint64_t p;
            ok = poll_pkt(w, res + q, p);
            if (ok)
                store_payload<ESZ>(a.p.out[r], a.n, q, pkt_payload(p));
        }
    }

    publish_epoch_own(a.c, flag);
}

// ---------------------------------------------------------------------------
// One-shot LL with shared receive staging (every buffer 8-byte aligned).  A
// CTA serves blocks of UB = blockDim / R units for all R virtual ranks.
// Thread (k, j) = (tid / UB, tid % UB):
//   put:     stores rank k's packet pair of unit j of the block after each
//            of its blocks (block b + 1 mod nblk), so the packets a CTA
//            receives were stored by another CTA;
//   receive: polls sender k's pair of unit j of its own block once (bounded)
//            and stages the payload in shared memory; after a barrier the
//            same thread, now receiver k, folds the R staged payloads of
//            unit j in rank order into out[k].
// Every receiver still folds every sender's payload itself; the R receivers
// of a unit share the one poll of each packet, as the one-shot HB shares its
// input loads, so the packets cross L2 R times less often.  The last (< 8)
// message bytes travel as single packets, put by the last CTA and received
// by CTA 0.  Forward progress and in place: as for k_ll (all puts precede
// all waits; out[k]'s unit is written only after its packet, hence its input
// read, has been seen).
// ---------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kLlStagedThreads) k_ll_staged(const __grid_constant__ LlArgs a) {
    constexpr int ESZ = Elem<DT>::kSize;
    __shared__ uint2 stage[kLlStagedThreads];
    __shared__ uint32_t stage1[2 * AR_MAX_RANKS];        // single packets: [rank][0..1]
    kernel_prologue();
    const uint32_t flag = call_flag(a.c);
    Poller w{&a.c, flag, 0};
    const int R = a.R;
    const uint32_t tid = threadIdx.x;
    const uint32_t UB = blockDim.x / (uint32_t)R;         // units per block
    const uint32_t k = tid / UB, j = tid - k * UB;
    const bool member = k < (uint32_t)R;                  // tid < R * UB
    const uint32_t nbytes = (uint32_t)a.n * ESZ;
    const uint32_t U = nbytes / 8;                        // packet pairs per rank
    const uint32_t ntail = (nbytes + 3) / 4 - 2 * U;      // 0, 1 or 2 single packets
    const uint32_t nblk = (U + UB - 1) / UB;
    const uint32_t ppad = (uint32_t)a.ppad;
    uint64_t *const slot_k = a.slots + (member ? k : 0) * ppad;

    // ---- put -----------------------------------------------------------------
    if (member && a.c.drop_rank != (int)k) {
        const uint2 *src = reinterpret_cast<const uint2 *>(a.p.in[k]);
        for (uint32_t b = blockIdx.x; b < nblk; b += gridDim.x) {
            const uint32_t u = (b + 1 == nblk ? 0 : b + 1) * UB + j;
            if (u < U) {
                const uint2 v = ld_v2(src + u);
                st_pkt2(slot_k + 2 * u, make_pkt(v.x, flag), make_pkt(v.y, flag));
            }
        }
        if (blockIdx.x == gridDim.x - 1 && j < ntail)
            st_pkt(slot_k + 2 * U + j,
                   make_pkt(load_payload<ESZ>(a.p.in[k], a.n, 2 * U + j), flag));
    }

    publish_epoch_others(a.c, flag);

    // ---- receive -----------------------------------------------------------------
    bool ok = true, aborted = false;
    for (uint32_t b = blockIdx.x; b < nblk; b += gridDim.x) {        // uniform per CTA
        const uint32_t u = b * UB + j;
        const bool live = member && u < U;
        if (live && ok) {
            uint64_t p0, p1;
            ok = poll_pkt2(w, slot_k + 2 * u, p0, p1);
            stage[tid] = make_uint2(pkt_payload(p0), pkt_payload(p1));
        }
        if (__syncthreads_or(!ok)) {
            aborted = true;                               // someone gave up: all leave
            break;
        }
        if (live) {
            WordAcc<DT> a0, a1;
            a0.init(stage[j].x);
            a1.init(stage[j].y);
            for (int s = 1; s < R; ++s) {
                const uint2 x = stage[(uint32_t)s * UB + j];
                a0.add(x.x);
                a1.add(x.y);
            }
            st_v2(reinterpret_cast<uint2 *>(a.p.out[k]) + u, make_uint2(a0.result(), a1.result()));
        }
        __syncthreads();                                  // the stage is refilled next block
    }
    if (!aborted && blockIdx.x == 0 && ntail > 0) {
        const bool tl = member && j < ntail;
        if (tl) {
            uint64_t p = 0;
            ok = poll_pkt(w, slot_k + 2 * U + j, p);
            stage1[2 * k + j] = pkt_payload(p);
        }
        if (!__syncthreads_or(!ok) && tl) {
            WordAcc<DT> acc;
            acc.init(stage1[j]);
            for (int s = 1; s < R; ++s)
                acc.add(stage1[2 * s + j]);
            store_payload<ESZ>(a.p.out[k], a.n, 2 * U + j, acc.result());
        }
    }

    publish_epoch_own(a.c, flag);
}

// ---------------------------------------------------------------------------
// Two-shot LL with shared staging (every buffer 8-byte aligned), on the same
// blocks and thread roles as k_ll_staged:
//   put:            as k_ll_staged (block b + 1 of every rank);
//   reduce-scatter: for each of its blocks, thread (k, j) polls sender k's
//                   pair of unit j once and stages it; after a barrier the
//                   thread of the unit's shard owner folds the R payloads in
//                   rank order and writes the reduced pair as a result
//                   packet (slot R);
//   all-gather:     for the block after each of its blocks (whose results
//                   another CTA reduced), R blocks per pass: thread (k, j)
//                   polls the result pair of unit j of the pass's k-th block
//                   once and stages it; after a barrier thread (k, j) stores
//                   unit j of every block of the pass to out[k].
// Every wait depends only on work each CTA finishes before its own waits
// (puts before reductions, reductions before gathers), so the cooperative
// grid makes progress.  In place: out[k]'s units of block b + 1 are written
// by the CTA that read in[k]'s units of that block in its put.  The last
// (< 8) message bytes travel as single packets: put by the last CTA,
// reduced by CTA 0, gathered by the last CTA.
// ---------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kLlStagedThreads) k_ll2_staged(const __grid_constant__ LlArgs a) {
    constexpr int ESZ = Elem<DT>::kSize;
    __shared__ uint2 stage[kLlStagedThreads];
    __shared__ uint32_t stage1[2 * AR_MAX_RANKS];        // single packets: [rank][0..1]
    __shared__ uint32_t gather1[2];                      // their reduced values
    kernel_prologue();
    const uint32_t flag = call_flag(a.c);
    Poller w{&a.c, flag, 0};
    const int R = a.R;
    const uint32_t tid = threadIdx.x;
    const uint32_t UB = blockDim.x / (uint32_t)R;         // units per block
    const uint32_t k = tid / UB, j = tid - k * UB;
    const bool member = k < (uint32_t)R;                  // tid < R * UB
    const uint32_t nbytes = (uint32_t)a.n * ESZ;
    const uint32_t U = nbytes / 8;                        // packet pairs per rank
    const uint32_t ntail = (nbytes + 3) / 4 - 2 * U;      // 0, 1 or 2 single packets
    const uint32_t nblk = (U + UB - 1) / UB;
    const uint32_t G = gridDim.x;
    const uint32_t ppad = (uint32_t)a.ppad;
    const uint32_t shard_pk = (uint32_t)(a.shard * ESZ / 4);   // packets per shard (even)
    uint64_t *const slot_k = a.slots + (member ? k : 0) * ppad;
    uint64_t *const res = a.slots + (uint32_t)R * ppad;         // result packets
    auto owner = [&](uint32_t q) {                        // shard owner of packet q
        const uint32_t o = q / shard_pk;
        return o < (uint32_t)R ? o : (uint32_t)R - 1u;
    };

    // ---- put -----------------------------------------------------------------
    if (member && a.c.drop_rank != (int)k) {
        const uint2 *src = reinterpret_cast<const uint2 *>(a.p.in[k]);
        for (uint32_t b = blockIdx.x; b < nblk; b += G) {
            const uint32_t u = (b + 1 == nblk ? 0 : b + 1) * UB + j;
            if (u < U) {
                const uint2 v = ld_v2(src + u);
                st_pkt2(slot_k + 2 * u, make_pkt(v.x, flag), make_pkt(v.y, flag));
            }
        }
        if (blockIdx.x == G - 1 && j < ntail)
            st_pkt(slot_k + 2 * U + j,
                   make_pkt(load_payload<ESZ>(a.p.in[k], a.n, 2 * U + j), flag));
    }

    publish_epoch_others(a.c, flag);

    // ---- reduce-scatter: this CTA's blocks ----------------------------------
    bool ok = true, aborted = false;
    for (uint32_t b = blockIdx.x; b < nblk; b += G) {                // uniform per CTA
        const uint32_t u = b * UB + j;
        const bool live = member && u < U;
        if (live && ok) {
            uint64_t p0, p1;
            ok = poll_pkt2(w, slot_k + 2 * u, p0, p1);
            stage[tid] = make_uint2(pkt_payload(p0), pkt_payload(p1));
        }
        if (__syncthreads_or(!ok)) {
            aborted = true;
            break;
        }
        if (live && k == owner(2 * u)) {
            WordAcc<DT> a0, a1;
            a0.init(stage[j].x);
            a1.init(stage[j].y);
            for (int s = 1; s < R; ++s) {
                const uint2 x = stage[(uint32_t)s * UB + j];
                a0.add(x.x);
                a1.add(x.y);
            }
            st_pkt2(res + 2 * u, make_pkt(a0.result(), flag), make_pkt(a1.result(), flag));
        }
        __syncthreads();                                  // the stage is refilled next block
    }
    if (!aborted && blockIdx.x == 0 && ntail > 0) {
        const bool tl = member && j < ntail;
        if (tl) {
            uint64_t p = 0;
            ok = poll_pkt(w, slot_k + 2 * U + j, p);
            stage1[2 * k + j] = pkt_payload(p);
        }
        if (__syncthreads_or(!ok)) {
            aborted = true;
        } else if (tl && k == owner(2 * U + j)) {
            WordAcc<DT> acc;
            acc.init(stage1[j]);
            for (int s = 1; s < R; ++s)
                acc.add(stage1[2 * s + j]);
            st_pkt(res + 2 * U + j, make_pkt(acc.result(), flag));
        }
    }

    // ---- all-gather: the block after each of this CTA's blocks, R blocks per
    // pass: thread (k, j) polls the result pair of unit j of the pass's k-th
    // block once and stages it; after a barrier it stores unit j of every
    // block of the pass to out[k] --------------------------------------------
    const uint32_t mine = blockIdx.x < nblk ? (nblk - 1 - blockIdx.x) / G + 1 : 0;
    auto gather_unit = [&](uint32_t i) {                  // unit j of gather block i
        const uint32_t b = blockIdx.x + i * G;            // this CTA's i-th block
        return (b + 1 == nblk ? 0 : b + 1) * UB + j;
    };
    for (uint32_t i0 = 0; !aborted && i0 < mine; i0 += (uint32_t)R) {   // uniform per CTA
        if (member && i0 + k < mine && ok) {
            const uint32_t u = gather_unit(i0 + k);
            if (u < U) {
                uint64_t p0, p1;
                ok = poll_pkt2(w, res + 2 * u, p0, p1);
                stage[tid] = make_uint2(pkt_payload(p0), pkt_payload(p1));
            }
        }
        if (__syncthreads_or(!ok)) {
            aborted = true;
            break;
        }
        if (member) {
            uint2 *dst = reinterpret_cast<uint2 *>(a.p.out[k]);
            for (uint32_t s = 0; s < (uint32_t)R && i0 + s < mine; ++s) {
                const uint32_t u = gather_unit(i0 + s);
                if (u < U)
                    st_v2(dst + u, stage[s * UB + j]);
            }
        }
        __syncthreads();                                  // the stage is refilled next pass
    }
    if (!aborted && blockIdx.x == G - 1 && ntail > 0) {
        if (k == 0 && j < ntail) {
            uint64_t p = 0;
            ok = poll_pkt(w, res + 2 * U + j, p);
            gather1[j] = pkt_payload(p);
        }
        if (!__syncthreads_or(!ok) && member && j < ntail)
            store_payload<ESZ>(a.p.out[k], a.n, 2 * U + j, gather1[j]);
    }

    publish_epoch_own(a.c, flag);
}

template <int DT> static const void *ll2_staged_kernel() {
    return reinterpret_cast<const void *>(&k_ll2_staged<DT>);
}

template <int DT> static const void *ll_staged_kernel() {
    return reinterpret_cast<const void *>(&k_ll_staged<DT>);
}

static const void *ll_staged_for(int dtype, bool two) {
    switch (dtype) {
    case AR_BF16: return two ? ll2_staged_kernel<AR_BF16>() : ll_staged_kernel<AR_BF16>();
    case AR_FP16: return two ? ll2_staged_kernel<AR_FP16>() : ll_staged_kernel<AR_FP16>();
    default: return two ? ll2_staged_kernel<AR_FP32>() : ll_staged_kernel<AR_FP32>();
    }
}

cudaError_t ll_staged_occupancy(int dtype, bool two_shot, int *blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        blocks_per_sm, ll_staged_for(dtype, two_shot), kLlStagedThreads, 0);
}

// gridDim = ctas, each serving all R ranks (a.G is not used).
cudaError_t launch_ll_staged(const LlArgs &a, int dtype, bool two_shot, int ctas, cudaStream_t s,
                             bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kLlStagedThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.numAttrs = 1;
    if (pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    cfg.attrs = attr;
    void *args[] = {const_cast<LlArgs *>(&a)};
    return cudaLaunchKernelExC(&cfg, ll_staged_for(dtype, two_shot), args);
}

template <int DT, bool TWO> static const void *ll_kernel() {
    return reinterpret_cast<const void *>(&k_ll<DT, TWO>);
}

static const void *ll_kernel_for(int dtype, bool two) {
    switch (dtype) {
    case AR_BF16: return two ? ll_kernel<AR_BF16, true>() : ll_kernel<AR_BF16, false>();
    case AR_FP16: return two ? ll_kernel<AR_FP16, true>() : ll_kernel<AR_FP16, false>();
    default: return two ? ll_kernel<AR_FP32, true>() : ll_kernel<AR_FP32, false>();
    }
}

cudaError_t ll_occupancy(int dtype, bool two_shot, int *blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm,
                                                         ll_kernel_for(dtype, two_shot),
                                                         kLlThreads, 0);
}

cudaError_t launch_ll(const LlArgs &a, int dtype, bool two_shot, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.R * a.G));
    cfg.blockDim = dim3(kLlThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.numAttrs = 1;
    if (pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    cfg.attrs = attr;
    void *args[] = {const_cast<LlArgs *>(&a)};
    return cudaLaunchKernelExC(&cfg, ll_kernel_for(dtype, two_shot), args);
}

// ---------------------------------------------------------------------------
// Standalone encode / decode (ar_ll_pack, ar_ll_unpack).  With VEC the
// message buffer is 8-byte aligned and the packets 16-byte aligned.
// ---------------------------------------------------------------------------
template <int ESZ, bool VEC>
__global__ void __launch_bounds__(kRegThreads) k_pack(const __grid_constant__ PackArgs a) {
    kernel_prologue();
    const uint64_t nbytes = a.n * ESZ, P = (nbytes + 3) / 4;
    const uint64_t U = VEC ? nbytes / 8 : 0;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t t0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (uint64_t u = t0; VEC && u < U; u += stride) {
        const uint2 v = ld_v2(reinterpret_cast<const uint2 *>(a.src) + u);
        st_pkt2(a.pkts + 2 * u, make_pkt(v.x, a.flag), make_pkt(v.y, a.flag));
    }
    for (uint64_t q = 2 * U + t0; q < P; q += stride)
        st_pkt(a.pkts + q, make_pkt(load_payload<ESZ>(a.src, a.n, q), a.flag));
}

template <int ESZ, bool VEC>
__global__ void __launch_bounds__(kRegThreads) k_unpack(const __grid_constant__ PackArgs a) {
    kernel_prologue();
    const uint64_t nbytes = a.n * ESZ, P = (nbytes + 3) / 4;
    const uint64_t U = VEC ? nbytes / 8 : 0;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t t0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    bool bad = false;
    for (uint64_t u = t0; VEC && u < U; u += stride) {
        uint64_t p0, p1;
        ld_pkt2(a.cpkts + 2 * u, p0, p1);
        const bool g0 = pkt_flag(p0) == a.flag, g1 = pkt_flag(p1) == a.flag;
        if (g0 && g1) {
            st_v2(reinterpret_cast<uint2 *>(a.dst) + u, make_uint2(pkt_payload(p0), pkt_payload(p1)));
        } else {
            bad = true;
            if (g0)
                reinterpret_cast<uint32_t *>(a.dst)[2 * u] = pkt_payload(p0);
            if (g1)
                reinterpret_cast<uint32_t *>(a.dst)[2 * u + 1] = pkt_payload(p1);
        }
    }
    for (uint64_t q = 2 * U + t0; q < P; q += stride) {
        const uint64_t p = ld_pkt(a.cpkts + q);
        if (pkt_flag(p) == a.flag)
            store_payload<ESZ>(a.dst, a.n, q, pkt_payload(p));
        else
            bad = true;
    }
    if (bad)
        record_error(a.status, AR_ERR_FLAG_MISMATCH);
}

cudaError_t launch_pack(const PackArgs &a, int dtype, bool vec, int grid, cudaStream_t s,
                        bool pdl) {
    if (elem_size(dtype) == 2)
        return vec ? launch_kernel(k_pack<2, true>, grid, kRegThreads, 0, s, pdl, a)
                   : launch_kernel(k_pack<2, false>, grid, kRegThreads, 0, s, pdl, a);
    return vec ? launch_kernel(k_pack<4, true>, grid, kRegThreads, 0, s, pdl, a)
               : launch_kernel(k_pack<4, false>, grid, kRegThreads, 0, s, pdl, a);
}

cudaError_t launch_unpack(const PackArgs &a, int dtype, bool vec, int grid, cudaStream_t s,
                          bool pdl) {
    if (elem_size(dtype) == 2)
        return vec ? launch_kernel(k_unpack<2, true>, grid, kRegThreads, 0, s, pdl, a)
                   : launch_kernel(k_unpack<2, false>, grid, kRegThreads, 0, s, pdl, a);
    return vec ? launch_kernel(k_unpack<4, true>, grid, kRegThreads, 0, s, pdl, a)
               : launch_kernel(k_unpack<4, false>, grid, kRegThreads, 0, s, pdl, a);
}

}  // namespace ar
