// santa_launch.h -- host-side glue between the C entry points and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "santa_common.cuh"

namespace santa {

// Records the timing event `ev` (if any) on `stream`.  Inside stream capture it
// becomes an event-record node of the graph, so a replayed graph is timed too.
inline void record_event(cudaEvent_t ev, cudaStream_t stream) {
    if (!ev) return;
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &st) == cudaSuccess && st == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal);
    else
        cudaEventRecord(ev, stream);
}

// Launches `kern` on `stream`; with `pdl` the kernel may start while the
// previous kernel in the stream drains (programmatic dependent launch).
// With cluster_x > 0 the grid's x dimension is cut into thread-block clusters of that size.
// With `cooperative` every CTA of the grid is resident at once (the launch fails
// rather than run a grid that cannot be).
template <typename... Exp, typename... Act>
cudaError_t launch_kernel(void (*kern)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                          int cluster_x, bool cooperative, Act &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = unsigned(cluster_x);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Act &&>(args)...);
}

// Raises a kernel's dynamic shared-memory limit (once per kernel and device).
template <typename K>
cudaError_t ensure_smem(K kern, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    struct Entry {
        const void *fn;
        int dev;
        size_t bytes;
    };
    static std::mutex mu;
    static Entry done[256];
    static int used = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const void *fn = reinterpret_cast<const void *>(kern);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (done[i].fn == fn && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    if (e == cudaSuccess && used < 256) done[used++] = Entry{fn, dev, bytes};
    return e;
}

struct Timing {
    cudaEvent_t begin = nullptr, end = nullptr;
};

// CTAs that share one prop head's thresholds (its splits): the most that the
// workspace has room for (kPropMaxSplit while the heads of a call number at most
// 32, fewer beyond; a function of the shape alone, so that santa_workspace_size
// needs no device) ...
inline int prop_split_bound(long long heads) {
    const long long n = heads > 0 ? 256 / heads : 1;
    return n < 1 ? 1 : n > kPropMaxSplit ? kPropMaxSplit : int(n);
}
// ... and, within that, as many as give every SM of the device one CTA.
inline int prop_nsplit(long long heads, int sms) {
    const long long n = heads > 0 ? sms / heads : 1;
    const int bound = prop_split_bound(heads);
    return n < 1 ? 1 : n > bound ? bound : int(n);
}

// Mode launchers (one translation unit each).  `dtype` is SANTA_F32/SANTA_BF16.
// kmap32: the K descriptor with boxes of 32 rows (the streaming pass-1 kernel).
// stages: kPass1 | kPass2 runs the streaming kernel and the pass-2 kernel in that
// order; with kFused as well, the one fused kernel instead when its shared memory
// fits (else the same two kernels).
enum { kPass1 = 1, kPass2 = 2, kFused = 4 };
cudaError_t launch_prop(const Params &p, int dtype, const CUtensorMap &kmap32, cudaStream_t stream, const Timing &tm,
                        int stages);
// S2ANTA-prop with the Bernoulli score stage: p.k is the feature-blocked K cache.
cudaError_t launch_prop_bernoulli(const Params &p, int dtype, cudaStream_t stream, const Timing &tm);
// Token-major K [rows][hkv][D] into the feature-blocked layout [ceil(rows/16)][hkv][D][16].
cudaError_t launch_feature_block(int dtype, const void *k, void *kfb, long long rows, int hkv, int D,
                                 cudaStream_t stream);
// kmap: the K descriptor with boxes of 32 rows (flash runs prop's streaming pass 1).
cudaError_t launch_flash(const Params &p, int dtype, const CUtensorMap &kmap, cudaStream_t stream, const Timing &tm);
cudaError_t launch_exact(const Params &p, int dtype, const CUtensorMap &kmap, const CUtensorMap &vmap,
                         cudaStream_t stream, const Timing &tm);

// Shared-memory needs, for validation on the host.
size_t prop_pass1_smem(int dtype, int D, int G, int smem_optin);
// The pass-2 kernel's split of a head's nch chunks on this device: *nsplit CTAs
// of *cps chunks each (whole tiles and whole warps), at most 8 per head, sized so
// that the grid fills about two CTAs per SM.
cudaError_t prop_pass2_split(int nch, int tile, long long heads, int *nsplit, int *cps);
size_t prop_pass2_smem(int D, int cps, int sampler, int S, bool paged);
size_t prop_fused_smem(int dtype, int D, int G, int sampler, int S, int smem_optin, int *nbuf);
size_t flash_sample_smem(int tile);
size_t exact_stream_smem(int dtype, int D, int G);
int exact_stream_warps(int dtype, int D, int G);

// CTAs of the exact streaming kernel: a multiple of Hkv (so a warp keeps one KV
// head), one per SM up to kExactCtaBound; the workspace is sized for the bound.
inline int exact_stream_cta_bound(int hkv) { return hkv > kExactCtaBound ? hkv : (kExactCtaBound / hkv) * hkv; }
inline int exact_stream_ctas(int hkv, int sms) {
    const int c = sms >= hkv ? (sms / hkv) * hkv : hkv;
    const int bound = exact_stream_cta_bound(hkv);
    return c < bound ? c : bound;
}

}  // namespace santa

// Expands the body (the variadic tail) with T (element type), D and G bound to the runtime
// (dtype, d, g); evaluates to cudaErrorNotSupported for combinations not built.
#define SANTA_DISPATCH(dtype, d, g, ...)                                        \
    [&]() -> cudaError_t {                                                       \
        if ((dtype) == SANTA_BF16) {                                             \
            using T = uint16_t;                                                  \
            SANTA_DISPATCH_DG(d, g, __VA_ARGS__)                                        \
        } else {                                                                 \
            using T = float;                                                     \
            SANTA_DISPATCH_DG(d, g, __VA_ARGS__)                                        \
        }                                                                        \
    }()
#define SANTA_DISPATCH_DG(d, g, ...)                                            \
    if ((d) == 128) {                                                            \
        constexpr int D = 128;                                                   \
        SANTA_DISPATCH_G(g, __VA_ARGS__)                                                \
    } else if ((d) == 64) {                                                      \
        constexpr int D = 64;                                                    \
        SANTA_DISPATCH_G(g, __VA_ARGS__)                                                \
    }                                                                            \
    return cudaErrorNotSupported;
#define SANTA_DISPATCH_G(g, ...)                                                \
    switch (g) {                                                                 \
        case 1: { constexpr int G = 1; __VA_ARGS__ }                                    \
        case 2: { constexpr int G = 2; __VA_ARGS__ }                                    \
        case 4: { constexpr int G = 4; __VA_ARGS__ }                                    \
        case 8: { constexpr int G = 8; __VA_ARGS__ }                                    \
        default: return cudaErrorNotSupported;                                   \
    }
