// Plans: an algorithm written as copy / reduce steps over chunks of the rank
// buffers, compiled on the host into one instruction stream per CTA (with the
// synchronisation the data dependencies need), and interpreted on the device
// by one cooperative kernel.
//
// Source: "【论文分享】MSCCL++：让 GPU 通信像 CUDA 一样可编程", section
// "第二层：DSL API": an algorithm author writes channel put / wait / reduce
// steps; the DSL compiler analyses the data dependencies, inserts the
// synchronisation and produces an execution plan that the runtime
// interprets.  Here a step is a copy (a put into a peer's buffer: every
// virtual peer's buffer is in this GPU's memory) or a reduce; the waits and
// signals are what the compiler inserts.
//
// Compilation.
//   * Buffers are cut into nchunks chunks (16-byte aligned boundaries).  Step
//     k over chunks [b, e) becomes tasks (k, c), c in [b, e).  Task (k, c)
//     runs on CTA rank_k * G + c % G: each virtual rank owns G CTAs.
//   * Program order is the order of the steps.  For every (buffer, chunk)
//     region the compiler tracks the last writer and the readers since; a
//     task depends on the last writer of every region it reads or writes
//     (read-after-write, write-after-write) and on the readers since that
//     write of every region it writes (write-after-read).
//   * Fusion (the DSL compiler's operator fusion): a copy task whose source
//     region was last written by task t, and whose destination region no
//     task has touched since t, becomes an extra destination of t: t stores
//     its result there too and the copy disappears.  The copy would have
//     stored exactly t's result, and nothing in between could tell the
//     difference, so the final state is the sequential one.  A two-shot
//     plan's all-gather copies fuse into the shard reductions this way: no
//     re-read of the reduced shards, and no semaphores left.
//   * A dependency inside one CTA needs nothing beyond program order (the
//     CTA syncs its threads between tasks, except between tasks of one step
//     on different chunks, which share no region).  One across CTAs gets a
//     semaphore: the producer task signals it once per run, the consumer
//     waits for it.  Every wait targets a task earlier in program order, and
//     all CTAs are resident at once (cooperative launch), so every wait ends.
//
// Runs.  Semaphores count completed producer tasks over all runs; run m
// (read from per-CTA epoch words like the LL flag) waits for the value
// m + 1, compared modulo 2^32.  A run whose wait timed out leaves the counts
// out of step: such a plan reports AR_ERR_TIMEOUT and must be rebuilt.
#include <algorithm>
#include <map>
#include <new>
#include <vector>

#include "ar_device.cuh"

namespace ar {

enum : int { kInstrWait = 0, kInstrTask = 1, kInstrSignal = 2 };

// Most destinations a task can gain by fusion: every other buffer.
constexpr int kPlanMaxExtraDst = 2 * AR_MAX_RANKS - 1;

struct PlanStep {            // device copy of one step
    int kind;                // AR_OP_COPY / AR_OP_REDUCE
    int dst;                 // buffer id: < R in[], else out[id - R]
    int nsrc;
    int src[AR_MAX_RANKS];
};

struct PlanArgs {
    RankPtrs p;
    uint64_t n;
    uint64_t chunk;          // elements per chunk (multiple of a 16-byte vector)
    const PlanStep *steps;
    const int4 *instr;       // {kind, a, b, x}: wait(sem a) / task(step a, chunk b, extra
                             // destinations at xdst[x] when x >= 0) / signal(sem a)
    const int *xdst;         // extra destination lists: count, then buffer ids
    const int *start;        // instr[start[b] .. start[b + 1]) belong to CTA b
    uint32_t *sems;
    uint32_t *epoch;         // one word per CTA: completed runs
    int R;
    int vec;                 // every buffer 16-byte aligned
    Ctl c;
};

__device__ __forceinline__ const void *buf_ptr(const PlanArgs &a, int id) {
    return id < a.R ? a.p.in[id] : a.p.out[id - a.R];
}

// The step's buffer pointers, resolved once per task into shared memory (the
// step table itself lives in global memory).
struct TaskPtrs {
    const void *src[AR_MAX_RANKS];
    void *dst;
    void *xdst[kPlanMaxExtraDst];   // fused copies' destinations
    int kind, nsrc, nx;
};

template <int DT>
__device__ void run_task(const PlanArgs &a, const TaskPtrs &t, uint64_t chunk) {
    constexpr int PV = Elem<DT>::kPerVec;
    const uint64_t lo = chunk * a.chunk;
    uint64_t hi = lo + a.chunk;
    if (hi > a.n)
        hi = a.n;
    if (lo >= hi)
        return;
    const int nsrc = t.nsrc;
    uint64_t vhi = lo;                                   // [lo, vhi): whole vectors
    if (a.vec) {
        vhi = lo + (hi - lo) / PV * PV;
        for (uint64_t u = lo / PV + threadIdx.x; u < vhi / PV; u += blockDim.x) {
            uint4 y;
            if (t.kind == AR_OP_COPY) {
                y = ld_v4_stream(reinterpret_cast<const uint4 *>(t.src[0]) + u);
            } else {
                // fold the sources in their order, eight loads in flight at a time
                VecAcc<DT> acc;
                for (int k0 = 0; k0 < nsrc; k0 += 8) {
                    uint4 v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (k0 + j < nsrc)
                            v[j] = ld_v4_stream(reinterpret_cast<const uint4 *>(t.src[k0 + j]) + u);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (k0 + j < nsrc) {
                            if (k0 + j == 0)
                                acc.init(v[j]);
                            else
                                acc.add(v[j]);
                        }
                }
                y = acc.result();
            }
            st_v4(reinterpret_cast<uint4 *>(t.dst) + u, y);
            for (int d = 0; d < t.nx; ++d)
                st_v4(reinterpret_cast<uint4 *>(t.xdst[d]) + u, y);
        }
    }
    for (uint64_t e = vhi + threadIdx.x; e < hi; e += blockDim.x) {
        uint32_t y;
        if (t.kind == AR_OP_COPY) {
            y = ld_elem<DT>(t.src[0], e);
        } else {
            ElemAcc<DT> acc;
            acc.init(ld_elem<DT>(t.src[0], e));
            for (int k = 1; k < nsrc; ++k)
                acc.add(ld_elem<DT>(t.src[k], e));
            y = acc.result();
        }
        st_elem<DT>(t.dst, e, y);
        for (int d = 0; d < t.nx; ++d)
            st_elem<DT>(t.xdst[d], e, y);
    }
}

// Occupancy as measured: binary32 held to 64 registers (four CTAs per SM;
// the compiler takes 80 otherwise), the 16-bit forms to three CTAs per SM
template <int DT>
__global__ void __launch_bounds__(kRegThreads, DT == AR_FP32 ? 4 : 3)
    k_plan(const __grid_constant__ PlanArgs a) {
    __shared__ int give_up;
    __shared__ TaskPtrs tp;
    kernel_prologue();
    const uint32_t run = ld_u32_relaxed(a.epoch + blockIdx.x);
    const uint32_t target = run + 1u;                    // what a producer's semaphore reaches
    if (threadIdx.x == 0)
        give_up = 0;
    __syncthreads();
    const int i0 = a.start[blockIdx.x], i1 = a.start[blockIdx.x + 1];
    // the (step, extra-destination list) resolved into tp, and whether a task
    // has run since the last CTA barrier (all of these are uniform per CTA)
    int res_step = -1, res_x = -2;
    bool pending = false;
    // Skipping the barrier lets a CTA's warps drift apart across its chunks.
    // With short chunks (under 8 passes of the CTA) the barrier keeps them on
    // one contiguous chunk, which measured faster (two-shot plan, 8 KiB
    // chunks); with long chunks skipping it measured faster (one-shot plans).
    const bool may_skip = a.chunk >= (uint64_t)8 * blockDim.x * Elem<DT>::kPerVec;
    for (int i = i0; i < i1; ++i) {
        const int4 in = a.instr[i];
        // A task of the step and list already in tp needs no resolving (tp is
        // written only to resolve another).  Right after another task it also
        // needs no barrier: a step covers each chunk once, so it works on
        // chunks that the tasks run since the last barrier (the same step on
        // other chunks) neither read nor wrote.  Anything else (or any task,
        // with short chunks) first waits for every thread's part of those
        // tasks.
        const bool same_desc = in.x == kInstrTask && in.y == res_step && in.w == res_x;
        const bool same = may_skip && same_desc && pending;
        if (pending && !same) {
            __syncthreads();
            pending = false;
        }
        if (in.x == kInstrWait) {
            if (threadIdx.x == 0 && !give_up) {
                // bounded acquire-poll of the producer's semaphore
                const uint32_t *sem = a.sems + in.y;
                uint64_t deadline = 0;
                uint32_t tries = 0;
                for (;;) {
                    uint32_t v;
                    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(sem) : "memory");
                    if ((int32_t)(v - target) >= 0)
                        break;
                    if (++tries > 8)
                        __nanosleep(64);
                    if ((tries & 15u) == 15u) {
                        if (ld_u32_relaxed(a.c.abort) == target) {
                            give_up = 1;
                            break;
                        }
                        const uint64_t now = globaltimer_ns();
                        if (deadline == 0) {
                            deadline = now + a.c.timeout_ns;
                        } else if (now > deadline) {
                            record_error(a.c.status, AR_ERR_TIMEOUT);
                            st_u32_relaxed(a.c.abort, target);
                            give_up = 1;
                            break;
                        }
                    }
                }
            }
            __syncthreads();
        } else if (in.x == kInstrTask) {
            if (!give_up) {
                if (!same_desc) {
                    const PlanStep &st = a.steps[in.y];
                    const int nx = in.w >= 0 ? a.xdst[in.w] : 0;
                    if (threadIdx.x < (unsigned)st.nsrc)
                        tp.src[threadIdx.x] = buf_ptr(a, st.src[threadIdx.x]);
                    if (threadIdx.x < (unsigned)nx)
                        tp.xdst[threadIdx.x] =
                            const_cast<void *>(buf_ptr(a, a.xdst[in.w + 1 + threadIdx.x]));
                    if (threadIdx.x == 0) {
                        tp.dst = const_cast<void *>(buf_ptr(a, st.dst));
                        tp.kind = st.kind;
                        tp.nsrc = st.nsrc;
                        tp.nx = nx;
                    }
                    __syncthreads();
                    res_step = in.y;
                    res_x = in.w;
                }
                run_task<DT>(a, tp, (uint64_t)in.z);
                pending = true;
            }
        } else {
            // every thread's writes of the tasks before are done (the barrier
            // at the top of this iteration); make them visible GPU-wide, then
            // count the task complete
            if (threadIdx.x == 0 && !give_up) {
                __threadfence();
                asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(a.sems + in.y) : "memory");
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0)
        st_u32_relaxed(a.epoch + blockIdx.x, target);
}

template <int DT> static const void *plan_kernel() {
    return reinterpret_cast<const void *>(&k_plan<DT>);
}

static const void *plan_kernel_for(int dtype) {
    switch (dtype) {
    case AR_BF16: return plan_kernel<AR_BF16>();
    case AR_FP16: return plan_kernel<AR_FP16>();
    default: return plan_kernel<AR_FP32>();
    }
}

}  // namespace ar

using namespace ar;

// ---------------------------------------------------------------------------
// Host side: the compiler and the C ABI.
// ---------------------------------------------------------------------------

struct ar_plan {
    int R, dtype, G, nchunks, device;
    uint64_t N, chunk;
    size_t esz;
    int ntasks, nwaits, nsignals;
    void *dev;               // one allocation: steps | instr | start | sems | epoch | xdst
    PlanStep *steps;
    int4 *instr;
    int *start;
    int *xdst;               // extra destination lists of fused tasks
    uint32_t *sems;
    uint32_t *epoch;
    Ctl ctl;                 // the handle's status / abort words and timeout
};

namespace {

// CTAs per rank that fill the device's co-resident capacity, or at most
// max_per_sm CTAs per SM when that is not 0.
int plan_ctas_per_rank(int R, int dtype, int max_per_sm = 0) {
    int per_sm = 0, dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, plan_kernel_for(dtype),
                                                      kRegThreads, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (max_per_sm > 0 && per_sm > max_per_sm)
        per_sm = max_per_sm;
    int g = per_sm * sms / R;
    if (g > kEpochWords / R)
        g = kEpochWords / R;
    return g;
}

struct Task {
    int step, chunk, cta;
    std::vector<int> xdst;   // destinations gained by fusing later copies
    bool fused = false;      // this copy became an extra destination of another task
    std::vector<int> deps;   // producer tasks in other CTAs
    bool signals = false;
    int sem = -1;
};

uint64_t ceil_div_u(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

}  // namespace

// Largest plan, in tasks (one step on one chunk); keeps the host-side
// compilation and the instruction streams bounded.
constexpr uint64_t kMaxPlanTasks = 1u << 20;
// Built-in two-shot plans by default: chunk bytes of a rank buffer aimed at,
// and the most chunks per CTA that aim may lead to.
constexpr uint64_t kPlanChunkBytes = 8192;
constexpr uint64_t kPlanMaxChunksPerCta = 16;

static int compile_plan(ar_handle_t h, const ar_op *ops, int nops, int nchunks,
                        int ctas_per_rank, ar_plan_t *out) {
    ar_info info;
    if (!h || !ops || nops < 1 || nchunks < 1 || ctas_per_rank < 0 ||
        ar_get_info(h, &info) != AR_OK)
        return AR_ERR_INVALID;
    if (ctas_per_rank == 0) {
        // as many CTAs per rank as can be resident together
        ctas_per_rank = plan_ctas_per_rank(info.R, info.dtype);
        if (ctas_per_rank < 1)
            return AR_ERR_UNSUPPORTED;
    }
    const int R = info.R;
    for (int k = 0; k < nops; ++k) {
        const ar_op &o = ops[k];
        if ((o.kind != AR_OP_COPY && o.kind != AR_OP_REDUCE) || o.rank < 0 || o.rank >= R ||
            o.dst_buf < 0 || o.dst_buf > 1 || o.dst_rank < 0 || o.dst_rank >= R ||
            o.src_buf < 0 || o.src_buf > 1 || o.nsrc < 1 || o.nsrc > R ||
            (o.kind == AR_OP_COPY && o.nsrc != 1) || o.chunk_begin < 0 ||
            o.chunk_end > nchunks || o.chunk_begin > o.chunk_end)
            return AR_ERR_INVALID;
        for (int i = 0; i < o.nsrc; ++i)
            if (o.src_rank[i] < 0 || o.src_rank[i] >= R)
                return AR_ERR_INVALID;
    }
    uint64_t ntasks = 0;
    for (int k = 0; k < nops; ++k)
        ntasks += (uint64_t)(ops[k].chunk_end - ops[k].chunk_begin);
    if (ntasks > kMaxPlanTasks)
        return AR_ERR_UNSUPPORTED;
    int per_sm = 0, dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, plan_kernel_for(info.dtype),
                                                      kRegThreads, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ERR_CUDA;
    }
    const int G = ctas_per_rank;
    const int ctas = R * G;
    if (ctas > per_sm * sms || ctas > kEpochWords)
        return AR_ERR_UNSUPPORTED;                       // not all CTAs can be resident

    std::vector<PlanStep> steps(nops);
    for (int k = 0; k < nops; ++k) {
        const ar_op &o = ops[k];
        PlanStep &st = steps[k];
        st.kind = o.kind;
        st.dst = o.dst_buf * R + o.dst_rank;
        st.nsrc = o.nsrc;
        for (int i = 0; i < AR_MAX_RANKS; ++i)
            st.src[i] = i < o.nsrc ? o.src_buf * R + o.src_rank[i] : 0;
    }
    // tasks in program order
    std::vector<Task> tasks;
    tasks.reserve((size_t)ntasks);
    for (int k = 0; k < nops; ++k)
        for (int c = ops[k].chunk_begin; c < ops[k].chunk_end; ++c) {
            Task t;
            t.step = k;
            t.chunk = c;
            t.cta = ops[k].rank * G + c % G;
            tasks.push_back(t);
        }

    // fusion: copy u of region (S, c) into (E, c) joins t = the last writer
    // of (S, c) when no task at or after t has touched (E, c) and E is none
    // of t's own buffers
    using Region = std::pair<int, int>;                          // (buffer id, chunk)
    {
        std::map<Region, int> writer;       // last writer (a task that stays)
        std::map<Region, int> touched;      // last task reading or writing it
        for (int i = 0; i < (int)tasks.size(); ++i) {
            Task &u = tasks[i];
            const PlanStep &st = steps[u.step];
            const int c = u.chunk;
            if (st.kind == AR_OP_COPY && st.src[0] != st.dst) {
                auto w = writer.find({st.src[0], c});
                if (w != writer.end()) {
                    Task &t = tasks[w->second];
                    const PlanStep &ts = steps[t.step];
                    const int E = st.dst;
                    bool clash = E == ts.dst ||
                                 std::find(t.xdst.begin(), t.xdst.end(), E) != t.xdst.end() ||
                                 (int)t.xdst.size() >= kPlanMaxExtraDst;
                    for (int k = 0; k < ts.nsrc && !clash; ++k)
                        clash = ts.src[k] == E;
                    auto seen = touched.find({E, c});
                    if (!clash && (seen == touched.end() || seen->second < w->second)) {
                        t.xdst.push_back(E);
                        u.fused = true;
                        writer[{E, c}] = w->second;
                        touched[{E, c}] = w->second;
                        continue;
                    }
                }
            }
            for (int k = 0; k < st.nsrc; ++k)
                touched[{st.src[k], c}] = i;
            writer[{st.dst, c}] = i;
            touched[{st.dst, c}] = i;
        }
    }

    // dependencies between the tasks that stay: on the last writer of every
    // region read or written, and on the readers since of every region written
    std::vector<int> live;                                       // task indices that stay
    for (int i = 0; i < (int)tasks.size(); ++i)
        if (!tasks[i].fused)
            live.push_back(i);
    {
        std::map<Region, int> last_writer;
        std::map<Region, std::vector<int>> readers;               // since that write
        std::vector<int> dsts, deps;
        for (int id : live) {
            Task &t = tasks[id];
            const PlanStep &st = steps[t.step];
            const int c = t.chunk;
            dsts.assign(1, st.dst);
            dsts.insert(dsts.end(), t.xdst.begin(), t.xdst.end());
            deps.clear();
            for (int k = 0; k < st.nsrc; ++k) {
                auto w = last_writer.find({st.src[k], c});
                if (w != last_writer.end())
                    deps.push_back(w->second);
            }
            for (int d : dsts) {
                auto w = last_writer.find({d, c});
                if (w != last_writer.end())
                    deps.push_back(w->second);
                for (int rd : readers[{d, c}])
                    deps.push_back(rd);
            }
            std::sort(deps.begin(), deps.end());
            deps.erase(std::unique(deps.begin(), deps.end()), deps.end());
            for (int d : deps)
                if (tasks[d].cta != t.cta && d != id) {
                    t.deps.push_back(d);
                    tasks[d].signals = true;
                }
            for (int k = 0; k < st.nsrc; ++k)
                if (std::find(dsts.begin(), dsts.end(), st.src[k]) == dsts.end())
                    readers[{st.src[k], c}].push_back(id);
            for (int d : dsts) {
                last_writer[{d, c}] = id;
                readers[{d, c}].clear();
            }
        }
    }
    int nsems = 0, nwaits = 0;
    for (int id : live)
        if (tasks[id].signals)
            tasks[id].sem = nsems++;
    // one instruction stream per CTA, in program order; the extra
    // destination lists go to a table of their own, each distinct list once
    // (tasks of one step on different chunks usually share theirs, and the
    // interpreter keeps a resolved (step, list) across such tasks)
    std::vector<std::vector<int4>> prog(ctas);
    std::vector<int> xtable;
    std::map<std::vector<int>, int> xseen;
    for (int id : live) {
        const Task &t = tasks[id];
        for (int d : t.deps) {
            prog[t.cta].push_back(make_int4(kInstrWait, tasks[d].sem, 0, 0));
            ++nwaits;
        }
        int x = -1;
        if (!t.xdst.empty()) {
            const auto found = xseen.find(t.xdst);
            if (found != xseen.end()) {
                x = found->second;
            } else {
                x = (int)xtable.size();
                xtable.push_back((int)t.xdst.size());
                xtable.insert(xtable.end(), t.xdst.begin(), t.xdst.end());
                xseen.emplace(t.xdst, x);
            }
        }
        prog[t.cta].push_back(make_int4(kInstrTask, t.step, t.chunk, x));
        if (t.signals)
            prog[t.cta].push_back(make_int4(kInstrSignal, t.sem, 0, 0));
    }
    std::vector<int> start(ctas + 1, 0);
    std::vector<int4> flat;
    for (int b = 0; b < ctas; ++b) {
        start[b] = (int)flat.size();
        flat.insert(flat.end(), prog[b].begin(), prog[b].end());
    }
    start[ctas] = (int)flat.size();

    ar_plan *p = new (std::nothrow) ar_plan();
    if (!p)
        return AR_ERR_NOMEM;
    p->R = R;
    p->dtype = info.dtype;
    p->G = G;
    p->nchunks = nchunks;
    p->device = dev;
    p->N = info.N;
    p->esz = info.elem_size;
    const uint64_t per_vec = 16 / p->esz;
    p->chunk = ceil_div_u(ceil_div_u(p->N, (uint64_t)nchunks), per_vec) * per_vec;
    p->ntasks = (int)live.size();
    p->nwaits = nwaits;
    p->nsignals = nsems;
    const size_t b_steps = sizeof(PlanStep) * steps.size();
    const size_t b_instr = sizeof(int4) * (flat.size() + 1);
    const size_t b_start = sizeof(int) * start.size();
    const size_t b_sems = sizeof(uint32_t) * (nsems + 1);
    const size_t b_epoch = sizeof(uint32_t) * (ctas + 1);    // + the plan's abort word
    const size_t b_xdst = sizeof(int) * (xtable.size() + 1);
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t total =
        up(b_steps) + up(b_instr) + up(b_start) + up(b_sems) + up(b_epoch) + up(b_xdst);
    if (cudaMalloc(&p->dev, total) != cudaSuccess) {
        (void)cudaGetLastError();
        delete p;
        return AR_ERR_NOMEM;
    }
    uint8_t *base = static_cast<uint8_t *>(p->dev);
    p->steps = reinterpret_cast<PlanStep *>(base);
    p->instr = reinterpret_cast<int4 *>(base + up(b_steps));
    p->start = reinterpret_cast<int *>(base + up(b_steps) + up(b_instr));
    p->sems = reinterpret_cast<uint32_t *>(base + up(b_steps) + up(b_instr) + up(b_start));
    p->epoch = reinterpret_cast<uint32_t *>(base + up(b_steps) + up(b_instr) + up(b_start) +
                                            up(b_sems));
    p->xdst = reinterpret_cast<int *>(base + up(b_steps) + up(b_instr) + up(b_start) +
                                      up(b_sems) + up(b_epoch));
    if (cudaMemset(p->dev, 0, total) != cudaSuccess ||
        cudaMemcpy(p->steps, steps.data(), b_steps, cudaMemcpyHostToDevice) != cudaSuccess ||
        (flat.size() && cudaMemcpy(p->instr, flat.data(), sizeof(int4) * flat.size(),
                                   cudaMemcpyHostToDevice) != cudaSuccess) ||
        cudaMemcpy(p->start, start.data(), b_start, cudaMemcpyHostToDevice) != cudaSuccess ||
        (xtable.size() && cudaMemcpy(p->xdst, xtable.data(), sizeof(int) * xtable.size(),
                                     cudaMemcpyHostToDevice) != cudaSuccess) ||
        cudaDeviceSynchronize() != cudaSuccess) {
        (void)cudaGetLastError();
        cudaFree(p->dev);
        delete p;
        return AR_ERR_CUDA;
    }
    // status word and wait limit from the handle (ar_status reports plan
    // errors); an abort word of the plan's own, since plan runs and LL calls
    // name themselves with unrelated counters
    p->ctl = handle_ctl(h);
    p->ctl.abort = p->epoch + ctas;
    *out = p;
    return AR_OK;
}

extern "C" int ar_plan_compile(ar_handle_t h, const ar_op *ops, int nops, int nchunks,
                               int ctas_per_rank, ar_plan_t *out) {
    if (!out)
        return AR_ERR_INVALID;
    *out = nullptr;
    // host containers may throw; nothing that needs releasing exists before
    // the last of them is built
    try {
        return compile_plan(h, ops, nops, nchunks, ctas_per_rank, out);
    } catch (const std::bad_alloc &) {
        return AR_ERR_NOMEM;
    }
}

static int builtin_plan(ar_handle_t h, int algo, int chunks_per_rank, int ctas_per_rank,
                        ar_plan_t *out) {
    ar_info info;
    if (!out || !h || ar_get_info(h, &info) != AR_OK || chunks_per_rank < 0 ||
        ctas_per_rank < 0 || (algo != AR_ONE_SHOT && algo != AR_TWO_SHOT))
        return AR_ERR_INVALID;
    if (ctas_per_rank == 0) {
        // the resident capacity; for the two-shot from R = 16 two CTAs per
        // SM, which measured faster (bf16 R = 16 x 8M: 90.7 against 93.0 us;
        // binary32 R = 16 x 4M: 89.5 against 94.9; R = 32 x 4M: 92.8 against
        // 96.1) while at R = 8 the capacity was (x 16M: 86.9 against 98.2)
        const bool two_per_sm = algo == AR_TWO_SHOT && info.R >= 16;
        ctas_per_rank = plan_ctas_per_rank(info.R, info.dtype, two_per_sm ? 2 : 0);
    }
    if (ctas_per_rank < 1)
        return AR_ERR_UNSUPPORTED;
    if (chunks_per_rank == 0) {
        // one chunk per CTA; for the two-shot with R >= 8, chunks of about
        // kPlanChunkBytes of a rank buffer instead, at most kPlanMaxChunksPerCta
        // per CTA, adjacent chunks on adjacent CTAs (task c runs on CTA
        // c % ctas_per_rank).  With one long chunk per CTA, DRAM read past the
        // end of every CTA's chunk into data that the neighbouring CTA had
        // consumed long before (11% extra reads at R = 16 x 16 MiB); at about
        // 8 KiB the reads equal the inputs.  What is read past the ends grows
        // with the sources per task (R), while each task also starts with a
        // chain of dependent loads (instruction, step, pointers): the one-shot
        // plan (R tasks per chunk), R = 2 and R = 4 measured slower or mixed
        // with more chunks, R = 8, 16 and 32 4-10% faster.
        uint64_t m = 1;
        if (algo == AR_TWO_SHOT && info.R >= 8) {
            const uint64_t shard_bytes =
                ceil_div_u((uint64_t)info.N, (uint64_t)info.R) * (uint64_t)info.elem_size;
            m = (shard_bytes / (uint64_t)ctas_per_rank + kPlanChunkBytes / 2) / kPlanChunkBytes;
            if (m > kPlanMaxChunksPerCta)
                m = kPlanMaxChunksPerCta;
            if (m < 1)
                m = 1;
        }
        chunks_per_rank = (int)(m * (uint64_t)ctas_per_rank);
    }
    if ((uint64_t)chunks_per_rank * (uint64_t)info.R > kMaxPlanTasks)
        return AR_ERR_UNSUPPORTED;           // R * K chunks, at least as many tasks
    const int R = info.R, K = chunks_per_rank;
    std::vector<ar_op> ops;
    ar_op o = {};
    o.kind = AR_OP_REDUCE;
    o.src_buf = AR_BUF_IN;
    o.nsrc = R;
    for (int k = 0; k < R; ++k)
        o.src_rank[k] = k;
    o.dst_buf = AR_BUF_OUT;
    if (algo == AR_ONE_SHOT) {
        // every rank folds every input into its own output
        for (int r = 0; r < R; ++r) {
            o.rank = o.dst_rank = r;
            o.chunk_begin = 0;
            o.chunk_end = R * K;
            ops.push_back(o);
        }
    } else {
        // reduce-scatter: rank j folds shard j into out[j] ...
        for (int j = 0; j < R; ++j) {
            o.rank = o.dst_rank = j;
            o.chunk_begin = j * K;
            o.chunk_end = (j + 1) * K;
            ops.push_back(o);
        }
        // ... all-gather: rank r puts every other shard into its output
        ar_op c = {};
        c.kind = AR_OP_COPY;
        c.src_buf = AR_BUF_OUT;
        c.dst_buf = AR_BUF_OUT;
        c.nsrc = 1;
        for (int r = 0; r < R; ++r)
            for (int j = 0; j < R; ++j) {
                if (j == r)
                    continue;
                c.rank = c.dst_rank = r;
                c.src_rank[0] = j;
                c.chunk_begin = j * K;
                c.chunk_end = (j + 1) * K;
                ops.push_back(c);
            }
    }
    return ar_plan_compile(h, ops.data(), (int)ops.size(), R * K, ctas_per_rank, out);
}

extern "C" int ar_plan_builtin(ar_handle_t h, int algo, int chunks_per_rank, int ctas_per_rank,
                               ar_plan_t *out) {
    try {
        return builtin_plan(h, algo, chunks_per_rank, ctas_per_rank, out);
    } catch (const std::bad_alloc &) {
        return AR_ERR_NOMEM;
    }
}

extern "C" int ar_plan_execute(ar_plan_t p, const void *const in[], void *const out[],
                               cudaStream_t stream) {
    if (!p || !in || !out)
        return AR_ERR_INVALID;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device)
        return AR_ERR_INVALID;
    const size_t len = p->N * p->esz;
    uintptr_t all = 0;
    for (int r = 0; r < p->R; ++r) {
        if (!in[r] || !out[r] || ((uintptr_t)in[r] % p->esz) || ((uintptr_t)out[r] % p->esz))
            return AR_ERR_INVALID;
        all |= (uintptr_t)in[r] | (uintptr_t)out[r];
    }
    // the compiler reasoned about 2R distinct buffers: no overlaps at all
    for (int a = 0; a < 2 * p->R; ++a) {
        const uintptr_t x = a < p->R ? (uintptr_t)in[a] : (uintptr_t)out[a - p->R];
        for (int b = a + 1; b < 2 * p->R; ++b) {
            const uintptr_t y = b < p->R ? (uintptr_t)in[b] : (uintptr_t)out[b - p->R];
            if (x < y + len && y < x + len)
                return AR_ERR_INVALID;
        }
    }
    PlanArgs a;
    for (int r = 0; r < AR_MAX_RANKS; ++r) {
        a.p.in[r] = r < p->R ? in[r] : nullptr;
        a.p.out[r] = r < p->R ? out[r] : nullptr;
    }
    a.n = p->N;
    a.chunk = p->chunk;
    a.steps = p->steps;
    a.instr = p->instr;
    a.xdst = p->xdst;
    a.start = p->start;
    a.sems = p->sems;
    a.epoch = p->epoch;
    a.R = p->R;
    a.vec = (all & 15u) == 0;
    a.c = p->ctl;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p->R * p->G));
    cfg.blockDim = dim3(kRegThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&a};
    if (cudaLaunchKernelExC(&cfg, plan_kernel_for(p->dtype), args) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ERR_CUDA;
    }
    return AR_OK;
}

extern "C" int ar_plan_stats(ar_plan_t p, int *tasks, int *waits, int *signals) {
    if (!p)
        return AR_ERR_INVALID;
    if (tasks)
        *tasks = p->ntasks;
    if (waits)
        *waits = p->nwaits;
    if (signals)
        *signals = p->nsignals;
    return AR_OK;
}

extern "C" int ar_plan_destroy(ar_plan_t p) {
    if (!p)
        return AR_OK;
    int rc = AR_OK;
    DeviceScope on(p->device);
    if (!on.ok() || cudaDeviceSynchronize() != cudaSuccess || cudaFree(p->dev) != cudaSuccess)
        rc = AR_ERR_CUDA;
    delete p;
    return rc;
}
