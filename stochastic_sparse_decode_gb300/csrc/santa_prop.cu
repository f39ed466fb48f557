// santa_prop.cu -- launch of S2ANTA-prop: pass 1 (tile kernel) then pass 2.
#include "santa_launch.h"
#include "santa_pass2.cuh"
#include "santa_tile.cuh"

namespace santa {

size_t prop_pass1_smem(int dtype, int d, int g, int tile) {
    size_t bytes = 0;
    SANTA_DISPATCH(dtype, d, g, { bytes = TileSmem<T, D, G, kProp>::bytes(tile); return cudaSuccess; });
    return bytes;
}

size_t prop_pass2_smem(int d, int tile) {
    return d == 128 ? Pass2Smem<uint16_t, 128>::bytes(kTilesPerSplit, tile)
                    : Pass2Smem<uint16_t, 64>::bytes(kTilesPerSplit, tile);
}

cudaError_t launch_prop(const Params &p, int dtype, const CUtensorMap &kmap, cudaStream_t stream, const Timing &tm) {
    return SANTA_DISPATCH(dtype, p.D, p.G, {
        auto k1 = tile_kernel<kProp, T, D, G>;
        auto k2 = prop_pass2_kernel<T, D>;
        const size_t s1 = TileSmem<T, D, G, kProp>::bytes(p.tile);
        const size_t s2 = Pass2Smem<T, D>::bytes(p.tiles_per_split, p.tile);
        cudaError_t e = ensure_smem(k1, s1);
        if (e == cudaSuccess) e = ensure_smem(k2, s2);
        if (e != cudaSuccess) return e;
        if (tm.begin) cudaEventRecord(tm.begin, stream);
        e = launch_kernel(k1, dim3(p.Tmax, p.Hkv, p.B), dim3(kTileWarps * 32), s1, stream, false, kmap, kmap, p);
        if (e != cudaSuccess) return e;
        if (tm.end) cudaEventRecord(tm.end, stream);
        return launch_kernel(k2, dim3(p.nsplit, p.Hq, p.B), dim3(kPass2Warps * 32), s2, stream, true, p);
    });
}

}  // namespace santa
