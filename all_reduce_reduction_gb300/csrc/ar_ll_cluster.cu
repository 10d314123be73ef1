// LL one-shot all-reduce with the virtual peers of a chunk in one thread-block
// cluster: packets travel between the peers' SMs through distributed shared
// memory instead of L2.
//
// Sources: the LL protocol of the MemoryChannel ("【论文分享】MSCCL++：让 GPU 通信
// 像 CUDA 一样可编程", section "MemoryChannel": GPU threads write the peer's
// memory directly; LL = small granularity, frequent synchronisation); the
// one-sided put / wait primitives ("microsoft/mscclpp" project page, "How it
// works"); the one-shot packet all-reduce ("SGLang 中的 MSCCL++ All-Reduce 基准
// 测试与推理集成指南", section 4.4).
//
// Layout.  A cluster of R CTAs handles chunks of Uc 16-byte units of every
// rank's buffer; CTA rank r of the cluster is virtual rank r.  Each CTA owns
// a receive buffer in shared memory with one slot per sender: [R][Uc * 4 + 4]
// packets (the last 4 of a slot carry the < 16-byte tail, in chunk 0 only).
// Per chunk, rank r loads its 16-byte units, turns each into four 8-byte
// packets (payload + flag) and stores them into slot r of EVERY peer's
// receive buffer (st.shared::cluster, one 8-byte packet per store half); each
// peer polls its own buffer until the four flags of every sender match, folds
// the R payloads in rank order and writes its output.  There is no barrier
// between the puts and the polls; the packets' flags are the synchronisation.
//
// Flags and reuse.  The receive buffers are zeroed at kernel start, then one
// cluster barrier makes every peer's zeroing (and its start) visible before
// any remote store.  Chunk iteration i uses flag i + 1, so a packet left from
// the previous iteration never matches.  Before a buffer slot is written for
// chunk i + 1, a cluster barrier ensures every peer consumed chunk i (the one
// write-after-read hazard of the reuse).  A CTA never exits before it has
// received all the packets addressed to it, so no remote store targets an
// exited CTA.
//
// Waits are bounded like the global-memory LL kernel's: a timed-out poll
// records AR_ERR_TIMEOUT and raises the call's abort word (the call is named
// by the handle's epoch flag); a thread that gives up skips its remaining
// work but still takes part in every cluster barrier, so the kernel ends.
#include "ar_device.cuh"

namespace ar {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    return remote;
}

__device__ __forceinline__ void st_cluster_pkt2(uint32_t addr, uint64_t a, uint64_t b) {
    asm volatile("st.relaxed.cluster.shared::cluster.v2.u64 [%0], {%1, %2};"
                 :: "r"(addr), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void st_cluster_pkt(uint32_t addr, uint64_t a) {
    asm volatile("st.relaxed.cluster.shared::cluster.u64 [%0], %1;" :: "r"(addr), "l"(a) : "memory");
}
__device__ __forceinline__ void ld_local_pkt2(uint32_t addr, uint64_t &a, uint64_t &b) {
    asm volatile("ld.relaxed.cluster.shared::cta.v2.u64 {%0, %1}, [%2];"
                 : "=l"(a), "=l"(b) : "r"(addr) : "memory");
}
__device__ __forceinline__ uint64_t ld_local_pkt(uint32_t addr) {
    uint64_t a;
    asm volatile("ld.relaxed.cluster.shared::cta.u64 %0, [%1];" : "=l"(a) : "r"(addr) : "memory");
    return a;
}
// Cluster-wide barrier (all threads of all R CTAs); the warp is reconverged
// first because the .aligned form needs every lane at the same instruction.
__device__ __forceinline__ void cluster_sync() {
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Poll until the packet pair at a local shared address carries `want`.
__device__ __forceinline__ bool poll_local2(Poller &w, uint32_t addr, uint32_t want, uint64_t &a,
                                            uint64_t &b) {
    uint32_t tries = 0;
    ld_local_pkt2(addr, a, b);
    while (pkt_flag(a) != want || pkt_flag(b) != want) {
        if (!w.keep_waiting(++tries))
            return false;
        ld_local_pkt2(addr, a, b);
    }
    return true;
}

template <int DT>
__global__ void __launch_bounds__(kLlThreads) k_ll_cluster(const __grid_constant__ LlClusterArgs a) {
    constexpr int ESZ = Elem<DT>::kSize;
    extern __shared__ __align__(16) uint64_t rbuf[];
    const int R = a.R;
    const uint32_t r = blockIdx.x % R;                   // == %cluster_ctarank
    const uint64_t cluster = blockIdx.x / R, nclusters = gridDim.x / R;
    const uint32_t tid = threadIdx.x, T = blockDim.x;
    const uint64_t Uc = a.units_per_chunk;
    const uint64_t slot_pk = Uc * 4 + 4;                 // packets per sender slot

    kernel_prologue();
    const uint32_t call = call_flag(a.c);                // names this call for the abort word
    Poller w{&a.c, call, 0};
    publish_epoch_others(a.c, call);

    const uint64_t nbytes = a.n * ESZ;
    const uint64_t P = (nbytes + 3) / 4;
    const uint64_t U = nbytes / 16;
    const uint64_t tail = P - 4 * U;                     // 0..3 single packets
    const uint64_t nchunks = (U + Uc - 1) / Uc > 0 ? (U + Uc - 1) / Uc : 1;
    const bool drop = a.c.drop_rank == (int)r;

    // zero the receive buffer, then make every peer's zeroing visible
    for (uint64_t i = tid; i < (uint64_t)R * slot_pk; i += T)
        rbuf[i] = 0;
    cluster_sync();

    const uint32_t base = smem_addr(rbuf);
    const uint4 *src = reinterpret_cast<const uint4 *>(a.p.in[r]);
    uint4 *dst = reinterpret_cast<uint4 *>(a.p.out[r]);
    bool ok = true;
    uint32_t iter = 0;
    for (uint64_t ch = cluster; ch < nchunks; ch += nclusters, ++iter) {
        if (iter > 0)
            cluster_sync();                              // every peer consumed the last chunk
        const uint32_t flag = iter + 1;
        const uint64_t u0 = ch * Uc;
        // ---- put: my units into slot r of every peer ---------------------
        if (!drop) {
            for (uint64_t j = tid; j < Uc && u0 + j < U; j += T) {
                const uint4 v = ld_v4_stream(src + u0 + j);
                const uint64_t p0 = make_pkt(v.x, flag), p1 = make_pkt(v.y, flag);
                const uint64_t p2 = make_pkt(v.z, flag), p3 = make_pkt(v.w, flag);
                const uint32_t local = base + (uint32_t)((r * slot_pk + 4 * j) * 8);
                for (int q = 0; q < R; ++q) {
                    const uint32_t rem = map_to_rank(local, (uint32_t)q);
                    st_cluster_pkt2(rem, p0, p1);
                    st_cluster_pkt2(rem + 16, p2, p3);
                }
            }
            if (ch == 0 && tid < tail) {
                const uint64_t q = 4 * U + tid;
                const uint64_t pk = make_pkt(load_payload<ESZ>(a.p.in[r], a.n, q), flag);
                const uint32_t local = base + (uint32_t)((r * slot_pk + 4 * Uc + tid) * 8);
                for (int q2 = 0; q2 < R; ++q2)
                    st_cluster_pkt(map_to_rank(local, (uint32_t)q2), pk);
            }
        }
        // ---- wait + fold: every sender's packets in my own buffer ---------
        for (uint64_t j = tid; ok && j < Uc && u0 + j < U; j += T) {
            VecAcc<DT> acc;
            for (int k = 0; k < R; ++k) {
                const uint32_t at = base + (uint32_t)((k * slot_pk + 4 * j) * 8);
                uint64_t q0, q1, q2, q3;
                ld_local_pkt2(at, q0, q1);
                ld_local_pkt2(at + 16, q2, q3);
                if (pkt_flag(q0) != flag || pkt_flag(q1) != flag)
                    ok = poll_local2(w, at, flag, q0, q1);
                if (ok && (pkt_flag(q2) != flag || pkt_flag(q3) != flag))
                    ok = poll_local2(w, at + 16, flag, q2, q3);
                if (!ok)
                    break;
                const uint4 v = make_uint4(pkt_payload(q0), pkt_payload(q1), pkt_payload(q2),
                                           pkt_payload(q3));
                if (k == 0)
                    acc.init(v);
                else
                    acc.add(v);
            }
            if (ok)
                st_v4(dst + u0 + j, acc.result());
        }
        if (ch == 0 && ok && tid < tail) {
            WordAcc<DT> acc;
            for (int k = 0; ok && k < R; ++k) {
                const uint32_t at = base + (uint32_t)((k * slot_pk + 4 * Uc + tid) * 8);
                uint64_t pk = ld_local_pkt(at);
                uint32_t tries = 0;
                while (pkt_flag(pk) != flag) {
                    if (!w.keep_waiting(++tries)) {
                        ok = false;
                        break;
                    }
                    pk = ld_local_pkt(at);
                }
                if (!ok)
                    break;
                if (k == 0)
                    acc.init(pkt_payload(pk));
                else
                    acc.add(pkt_payload(pk));
            }
            if (ok)
                store_payload<ESZ>(a.p.out[r], a.n, 4 * U + tid, acc.result());
        }
        __syncwarp();
    }
    // A CTA leaves only when every packet addressed to it has arrived (or the
    // call gave up); the final barrier also keeps peers' smem alive while
    // remote stores of a given-up call may still be in flight.
    cluster_sync();
    publish_epoch_own(a.c, call);
}

template <int DT> static const void *cluster_kernel() {
    return reinterpret_cast<const void *>(&k_ll_cluster<DT>);
}

static const void *cluster_kernel_for(int dtype) {
    switch (dtype) {
    case AR_BF16: return cluster_kernel<AR_BF16>();
    case AR_FP16: return cluster_kernel<AR_FP16>();
    default: return cluster_kernel<AR_FP32>();
    }
}

size_t ll_cluster_smem_bytes(int R, uint64_t units_per_chunk) {
    return (size_t)R * (units_per_chunk * 4 + 4) * sizeof(uint64_t);
}

cudaError_t ll_cluster_prepare(int dtype, int R) {
    const void *k = cluster_kernel_for(dtype);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kLlClusterMaxSmem);
    if (e == cudaSuccess && R > 8)
        e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

cudaError_t ll_cluster_max_clusters(const LlClusterArgs &a, int dtype, int *clusters) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.R);
    cfg.blockDim = dim3(kLlThreads);
    cfg.dynamicSmemBytes = ll_cluster_smem_bytes(a.R, a.units_per_chunk);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.R;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, cluster_kernel_for(dtype), &cfg);
}

cudaError_t launch_ll_cluster(const LlClusterArgs &a, int dtype, int nclusters, cudaStream_t s,
                              bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.R * nclusters));
    cfg.blockDim = dim3(kLlThreads);
    cfg.dynamicSmemBytes = ll_cluster_smem_bytes(a.R, a.units_per_chunk);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.R;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
    if (pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    cfg.attrs = attr;
    void *args[] = {const_cast<LlClusterArgs *>(&a)};
    return cudaLaunchKernelExC(&cfg, cluster_kernel_for(dtype), args);
}

}  // namespace ar
