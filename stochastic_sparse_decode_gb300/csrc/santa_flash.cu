// santa_flash.cu -- launch of S2ANTA-flash: tile kernel then merge.
#include "santa_launch.h"
#include "santa_merge.cuh"
#include "santa_tile.cuh"

namespace santa {

size_t flash_tile_smem(int dtype, int d, int g, int tile) {
    size_t bytes = 0;
    SANTA_DISPATCH(dtype, d, g, { bytes = TileSmem<T, D, G>::bytes(tile); return cudaSuccess; });
    return bytes;
}

cudaError_t launch_flash(const Params &p, int dtype, const CUtensorMap &kmap, cudaStream_t stream, const Timing &tm) {
    return SANTA_DISPATCH(dtype, p.D, p.G, {
        auto k1 = tile_kernel<T, D, G>;
        auto k2 = merge_kernel<D>;
        const size_t s1 = TileSmem<T, D, G>::bytes(p.tile);
        cudaError_t e = ensure_smem(k1, s1);
        if (e != cudaSuccess) return e;
        record_event(tm.begin, stream);
        e = launch_kernel(k1, dim3(p.Hkv, p.Tmax, p.B), dim3(kTileWarps * 32), s1, stream, false, 0, false, kmap, p);
        if (e != cudaSuccess) return e;
        record_event(tm.end, stream);
        return launch_kernel(k2, dim3(p.Hq, p.B), dim3(kMergeThreads), 0, stream, true, 0, false, p);
    });
}

}  // namespace santa
