// santa_exact.cu -- launch of the exact split-KV decode: streaming kernel, then merge.
#include "santa_exact_stream.cuh"
#include "santa_launch.h"
#include "santa_merge.cuh"

namespace santa {

size_t exact_stream_smem(int dtype, int d, int g) {
    size_t bytes = 0;
    SANTA_DISPATCH(dtype, d, g, { bytes = ExactStreamGeom<T, D, G>::bytes(); return cudaSuccess; });
    return bytes;
}

int exact_stream_warps(int dtype, int d, int g) {
    int w = 0;
    SANTA_DISPATCH(dtype, d, g, { w = ExactStreamGeom<T, D, G>::kWarps; return cudaSuccess; });
    return w;
}

cudaError_t launch_exact(const Params &p, int dtype, const CUtensorMap &kmap, const CUtensorMap &vmap,
                         cudaStream_t stream, const Timing &tm) {
    int sms = 0;
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e0 != cudaSuccess) return e0;
    const int C = exact_stream_ctas(p.Hkv, sms);
    return SANTA_DISPATCH(dtype, p.D, p.G, {
        using EG = ExactStreamGeom<T, D, G>;
        auto k1 = exact_stream_kernel<T, D, G>;
        auto k2 = exact_stream_merge<D>;
        const size_t s1 = EG::bytes();
        cudaError_t e = ensure_smem(k1, s1);
        if (e != cudaSuccess) return e;
        record_event(tm.begin, stream);
        e = launch_kernel(k1, dim3(unsigned(C)), dim3(EG::kWarps * 32), s1, stream, false, 0, false, kmap, vmap, p);
        if (e != cudaSuccess) return e;
        record_event(tm.end, stream);
        return launch_kernel(k2, dim3(p.Hq, p.B), dim3(kExactMergeWarps * 32), 0, stream, false, 0, false, p, C, int(EG::kWarps));
    });
}

}  // namespace santa
