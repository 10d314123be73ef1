// ar_allreduce_ll_static: the one-shot LL all-reduce without a handle and
// without any allocation.
//
// Some callers cannot allocate device memory at the point where they need
// the collective: an inference engine that reserves nearly all of the GPU's
// memory up front for its own pool and accounts for every byte (a side
// allocation would fail, or break its memory plan), or a hook on a
// latency-critical path that must not pay for cudaMalloc/cudaFree, which can
// synchronise the whole device.  ar_create allocates the packet scratch and
// the control words such callers cannot create; this entry point takes them
// from a fixed array compiled into the library instead.
//
// The array below is static device storage: every GPU that loads the library
// holds AR_NOALLOC_SCRATCH_BYTES of it (plus the control words) until the
// process exits.  All calls share it and it keeps the last call's contents,
// so calls whose kernels overlap on the GPU (different streams without an
// ordering between them, or different host threads) race on it.
#include <mutex>

#include "ar_internal.h"

namespace {

constexpr size_t kCtlBytes = 256;                                   // status, abort words
constexpr size_t kEpochBytes = sizeof(uint32_t) * ar::kEpochWords;
constexpr size_t kTotalBytes = kCtlBytes + kEpochBytes + AR_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// status | abort | epoch words | packet slots
static __device__ __align__(256) unsigned char g_noalloc_scratch[kTotalBytes];

struct DeviceState {
    bool ready;
    uint8_t *base;          // device address of g_noalloc_scratch on this device
    int num_sms;
    int cap[3];             // co-resident per-rank one-shot LL CTAs [dtype]
    int staged_cap[3];      // co-resident CTAs of the staged one-shot LL [dtype]
};

std::mutex g_setup_lock;
DeviceState g_state[kMaxDevices];

// Once per device, with that device current: resolve the array's device
// address (host code only sees a host-side stand-in under its name), zero
// the control and epoch words, and record the launch capacities.
int setup(int dev, DeviceState **out) {
    if (dev < 0 || dev >= kMaxDevices)
        return AR_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_lock);
    DeviceState &s = g_state[dev];
    if (!s.ready) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            (void)cudaGetLastError();
            return AR_ERR_CUDA;
        }
        if (cudaMemset(ptr, 0, kCtlBytes + kEpochBytes) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess ||
            cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess) {
            (void)cudaGetLastError();
            return AR_ERR_CUDA;
        }
        for (int dt = 0; dt < 3; ++dt) {
            int per_sm = 0, staged_per_sm = 0;
            if (ar::ll_occupancy(dt, false, &per_sm) != cudaSuccess ||
                ar::ll_staged_occupancy(dt, false, &staged_per_sm) != cudaSuccess) {
                (void)cudaGetLastError();
                return AR_ERR_CUDA;
            }
            s.cap[dt] = per_sm * s.num_sms;
            s.staged_cap[dt] = staged_per_sm * s.num_sms;
        }
        s.base = static_cast<uint8_t *>(ptr);
        s.ready = true;
    }
    *out = &s;
    return AR_OK;
}

bool overlap(uintptr_t a, uintptr_t b, size_t len) { return a < b + len && b < a + len; }

}  // namespace

extern "C" int ar_allreduce_ll_static(int R, size_t N, int dtype, const void *const in[],
                                      void *const out[], cudaStream_t stream) {
    if (R < 1 || R > AR_MAX_RANKS || N < 1 || !in || !out)
        return AR_ERR_INVALID;
    if (dtype != AR_BF16 && dtype != AR_FP16 && dtype != AR_FP32)
        return AR_ERR_INVALID;
    const size_t esz = ar::elem_size(dtype);
    if (N > ((size_t)1 << 40) / esz)
        return AR_ERR_INVALID;
    // R slots of ceil(N * esz / 4) packets rounded up to 4, 8 bytes each
    const uint64_t ppad = ((N * esz + 3) / 4 + 3) / 4 * 4;
    if ((uint64_t)R * ppad * sizeof(uint64_t) > AR_NOALLOC_SCRATCH_BYTES)
        return AR_ERR_UNSUPPORTED;              // message too large for the static scratch

    const size_t len = N * esz;
    uintptr_t all = 0;
    for (int r = 0; r < R; ++r) {
        if (!in[r] || !out[r])
            return AR_ERR_INVALID;
        if (((uintptr_t)in[r] % esz) != 0 || ((uintptr_t)out[r] % esz) != 0)
            return AR_ERR_INVALID;
        all |= (uintptr_t)in[r] | (uintptr_t)out[r];
    }
    for (int a = 0; a < R; ++a) {
        for (int b = a + 1; b < R; ++b)
            if (overlap((uintptr_t)out[a], (uintptr_t)out[b], len))
                return AR_ERR_INVALID;
        for (int b = 0; b < R; ++b)
            if (overlap((uintptr_t)out[a], (uintptr_t)in[b], len) &&
                !(a == b && out[a] == in[b]))
                return AR_ERR_INVALID;
    }

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return AR_ERR_CUDA;
    DeviceState *s = nullptr;
    const int rc = setup(dev, &s);
    if (rc != AR_OK)
        return rc;

    const bool vec = (all & 7u) == 0;
    ar::LlArgs a;
    for (int r = 0; r < AR_MAX_RANKS; ++r) {
        a.p.in[r] = r < R ? in[r] : nullptr;
        a.p.out[r] = r < R ? out[r] : nullptr;
    }
    a.n = N;
    a.shard = 0;                                 // one-shot: no shards
    a.slots = reinterpret_cast<uint64_t *>(s->base + kCtlBytes + kEpochBytes);
    a.ppad = ppad;
    a.R = R;
    a.c.status = reinterpret_cast<int *>(s->base);
    a.c.abort = reinterpret_cast<uint32_t *>(s->base + 4);
    a.c.epoch = reinterpret_cast<uint32_t *>(s->base + kCtlBytes);
    a.c.timeout_ns = 1000000000ull;
    a.c.drop_rank = -1;
    if (vec) {
        // 8-byte aligned: the staged kernel (CTAs serving all R ranks)
        int cap = s->staged_cap[dtype];
        if (cap > ar::kEpochWords)
            cap = ar::kEpochWords;
        if (cap < 1)
            return AR_ERR_UNSUPPORTED;
        const uint64_t ub = ar::kLlStagedThreads / R;
        uint64_t ctas = (N * esz / 8 + ub - 1) / ub;
        if (ctas < 1)
            ctas = 1;
        if (ctas > (uint64_t)cap)
            ctas = (uint64_t)cap;
        a.G = 0;
        if (ar::launch_ll_staged(a, dtype, false, (int)ctas, stream) != cudaSuccess) {
            (void)cudaGetLastError();
            return AR_ERR_CUDA;
        }
        return AR_OK;
    }
    // not 8-byte aligned: per-rank CTAs, one packet per unit
    int gmax = s->cap[dtype] / R;
    if (gmax > ar::kEpochWords / R)
        gmax = ar::kEpochWords / R;
    if (gmax < 1)
        return AR_ERR_UNSUPPORTED;
    const uint64_t work = (N * esz + 3) / 4;
    uint64_t G = (work + ar::kLlThreads - 1) / ar::kLlThreads;
    if (G < 1)
        G = 1;
    if (G > (uint64_t)gmax)
        G = (uint64_t)gmax;
    a.G = (int)G;
    if (ar::launch_ll(a, dtype, false, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ERR_CUDA;
    }
    return AR_OK;
}
