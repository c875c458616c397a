// smla_static.cu -- the allocation-free d_sink entry point.
//
// smla_bwd needs a caller-provided workspace, which means the caller must be
// able to allocate device memory. Some callers cannot: their device memory is
// wholly owned by another allocator (a framework's caching allocator, or a
// fixed arena reserved at start-up), or they run where allocation is not
// allowed at all. For them this file offers d_sink with its one scratch
// buffer (the per-(t, h) delta = rowsum(O * dO)) held in a file-scope device
// array instead of a workspace.
//
// The array is part of the library image: every GPU on which libsmla.so is
// loaded holds it (4 MiB) until the process exits. All calls share it, so two
// calls whose kernels overlap on the GPU race; serialize them (one stream, or
// events between streams). Every call overwrites the T * H entries it reads,
// so nothing needs clearing between calls.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "smla_internal.cuh"

namespace smla {
// Largest T * H the static scratch holds: 2^20 fp32 values (4 MiB).
constexpr int64_t kStaticDeltaMax = int64_t(1) << 20;
}  // namespace smla

static __device__ __align__(256) float g_static_delta[smla::kStaticDeltaMax];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
// Per device: the device address of g_static_delta and the id of the CUDA
// context it was looked up in. A device address belongs to one context: after
// cudaDeviceReset the device gets a new context (with a new id), the module is
// loaded again and the array may sit elsewhere, so the lookup is redone.
struct StaticAddr {
    unsigned long long ctx_id;
    float* addr;
};
StaticAddr g_static_delta_addr[kMaxDevices];

// The current context's unique id (never reused within a process), through
// the driver entry points; false if it cannot be read.
bool current_ctx_id(unsigned long long* id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    if (!get_current || !get_id) {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) !=
                cudaSuccess || qa != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
                cudaSuccess || qb != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return false;
        }
        get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
        get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// In host code `g_static_delta` names a host-side shadow, not device memory;
// the device address is looked up with the device current, once per device
// and context. Returns nullptr on failure.
float* static_delta_for(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned long long ctx = 0;
    if (!current_ctx_id(&ctx)) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    StaticAddr& e = g_static_delta_addr[dev];
    if (!e.addr || e.ctx_id != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_delta) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        e.addr = static_cast<float*>(p);
        e.ctx_id = ctx;
    }
    return e.addr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool disjoint(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return na == 0 || nb == 0 || a0 + na <= b0 || b0 + nb <= a0;
}

}  // namespace

extern "C" int smla_dsink_static(const uint16_t* dO, const uint16_t* o, const float* lse,
                                 const float* sink, float* d_sink, int32_t T, int32_t H,
                                 void* stream) {
    if (!sink || !d_sink) return SMLA_ERR_NULL;
    if (T < 0 || H < 16 || H > 128 || H % 16 != 0) return SMLA_ERR_SHAPE;
    if (int64_t(T) * H > smla::kStaticDeltaMax) return SMLA_ERR_SHAPE;
    if (T > 0 && (!dO || !o || !lse)) return SMLA_ERR_NULL;
    const void* ptrs[] = {dO, o, lse, sink, d_sink};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SMLA_ERR_ALIGN;
    const size_t thd = size_t(T) * H * smla::kD * 2, th4 = size_t(T) * H * 4, h4 = size_t(H) * 4;
    if (!disjoint(d_sink, h4, dO, thd) || !disjoint(d_sink, h4, o, thd) ||
        !disjoint(d_sink, h4, lse, th4) || !disjoint(d_sink, h4, sink, h4))
        return SMLA_ERR_OVERLAP;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return SMLA_ERR_CUDA; }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return SMLA_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return SMLA_ERR_ARCH;
    const void* dptrs[] = {dO, o, lse, sink, d_sink};
    if (const int rc = smla::check_device_ptrs(dptrs, 5)) return rc;
    float* delta = static_delta_for(dev);
    if (!delta) return SMLA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0)
        return cudaMemsetAsync(d_sink, 0, h4, s) == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
    if (smla::launch_delta(o, dO, delta, int64_t(T) * H, s) != cudaSuccess) return SMLA_ERR_CUDA;
    if (smla::launch_dsink(delta, lse, sink, d_sink, T, H, s) != cudaSuccess) return SMLA_ERR_CUDA;
    return SMLA_OK;
}
