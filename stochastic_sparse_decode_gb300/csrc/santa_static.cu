// santa_static.cu -- S2ANTA-prop decode for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory for a workspace: a plugin
// loaded into a host program that owns every device allocation through its own
// pool and hands plugins no allocator, or a C caller on a path where the
// implicit device synchronisation of cudaMalloc/cudaFree is not acceptable.
// santa_decode_prop_static_scratch serves them: its scratch is the file-scope
// array below, which every GPU that loads this library holds until the process
// exits.  The caller still passes and owns q, K, V, kv_indptr, U and out.
//
// The entry point runs the same kernels as santa_decode_prop, with this array
// as their workspace; it allocates nothing itself and calls no allocating
// routine.  All calls share the array and it keeps the last call's contents.
// The bytes a prop workspace needs zero-filled start zero (a __device__ array is
// zero when the module is loaded) and every call leaves them zero; everything
// else is written before it is read, so a call never depends on what an earlier
// call left behind.  Calls whose kernels overlap on the GPU (different streams,
// or threads that do not order their streams) race on the array.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "santa_decode.h"

namespace {

constexpr size_t kScratchBytes = SANTA_STATIC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char santa_static_scratch[kScratchBytes];

// The unique id of the current CUDA context (0 if none is current or the driver
// cannot say).  A device reset destroys the context the array was loaded in; the
// next one has a new id, and the array a possibly different address.
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device.  In host code the
// array's name only stands in for the symbol, so the address is looked up with
// cudaGetSymbolAddress -- once per device, with that device current -- and kept
// with the id of the context it belongs to; if the device was reset since, the
// context id differs and the address is looked up again.
int scratch_address(void **addr) {
    static std::mutex mu;
    static void *per_device[64] = {};
    static unsigned long long per_device_ctx[64] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SANTA_CUDA_ERROR;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = current_context_id();
    if (!per_device[dev] || ctx == 0 || ctx != per_device_ctx[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, santa_static_scratch) != cudaSuccess || !p) return SANTA_CUDA_ERROR;
        per_device[dev] = p;
        per_device_ctx[dev] = current_context_id();  // the lookup made the context current if none was
    }
    *addr = per_device[dev];
    return SANTA_OK;
}

}  // namespace

extern "C" int santa_decode_prop_static_scratch(const santa_problem *p, const void *q, const void *k, const void *v,
                                                const long long *kv_indptr, const float *U, float *out,
                                                const santa_debug *dbg, santa_stream_t stream) {
    size_t need = 0;
    const int st = santa_workspace_size(p, SANTA_MODE_PROP, &need);
    if (st != SANTA_OK) return st;
    if (need > kScratchBytes) return SANTA_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    const int st2 = scratch_address(&scratch);
    if (st2 != SANTA_OK) return st2;
    return santa_decode_prop(p, q, k, v, kv_indptr, U, out, scratch, kScratchBytes, dbg, stream);
}
