// santa_prop.cu -- launch of S2ANTA-prop: pass 1 (streaming or tile kernel) then pass 2.
#include "santa_launch.h"
#include "santa_pass2.cuh"
#include "santa_stream.cuh"
#include "santa_tile.cuh"

namespace santa {

size_t prop_pass1_smem(int dtype, int d, int g, int tile) {
    size_t bytes = 0;
    SANTA_DISPATCH(dtype, d, g, { bytes = TileSmem<T, D, G, kProp>::bytes(tile); return cudaSuccess; });
    return bytes;
}

size_t prop_pass2_smem(int d, int tile, int Tmax) {
    int nsplit, tps;
    prop_split(Tmax, &nsplit, &tps);
    return d == 128 ? Pass2Smem<uint16_t, 128>::bytes(tps, Tmax, tile) : Pass2Smem<uint16_t, 64>::bytes(tps, Tmax, tile);
}

// SM count and opt-in shared memory per block of the current device (cached).
static cudaError_t device_limits(int *sms, int *smem_optin) {
    static int cache_sms[64] = {}, cache_smem[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!cache_sms[dev]) {
        int a = 0, b = 0;
        e = cudaDeviceGetAttribute(&a, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&b, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        cache_smem[dev] = b;
        cache_sms[dev] = a;
    }
    *sms = cache_sms[dev];
    *smem_optin = cache_smem[dev];
    return cudaSuccess;
}

cudaError_t launch_prop(const Params &p, int dtype, const CUtensorMap &kmap64, const CUtensorMap &kmap32,
                        cudaStream_t stream, const Timing &tm) {
    int sms = 0, optin = 0;
    cudaError_t e0 = device_limits(&sms, &optin);
    if (e0 != cudaSuccess) return e0;
    return SANTA_DISPATCH(dtype, p.D, p.G, {
        auto k2 = prop_pass2_kernel<T, D>;
        const size_t s2 = Pass2Smem<T, D>::bytes(p.tiles_per_split, p.Tmax, p.tile);
        cudaError_t e = ensure_smem(k2, s2);
        if (e != cudaSuccess) return e;
        // Pass 1: the streaming kernel when a tile is one round of the CTA and a ring
        // of at least two tiles fits in shared memory; otherwise one CTA per tile.
        int ring = 0;
        const long long units = (long long)p.B * p.Tmax * p.Hkv;
        if (p.tile <= kRoundKeys && units < (1LL << 30))
            for (int r = 3; r >= 2 && !ring; --r)
                if (StreamSmem<T, D, G>::bytes(r) <= size_t(optin)) ring = r;
        if (tm.begin) cudaEventRecord(tm.begin, stream);
        if (ring) {
            auto k1 = prop_stream_kernel<T, D, G>;
            const size_t s1 = StreamSmem<T, D, G>::bytes(ring);
            e = ensure_smem(k1, s1);
            if (e != cudaSuccess) return e;
            // a multiple of Hkv keeps each CTA on one KV head (q reloads only when b changes)
            long long grid = sms >= p.Hkv ? (long long)(sms / p.Hkv) * p.Hkv : sms;
            if (grid > units) grid = units;
            e = launch_kernel(k1, dim3(unsigned(grid)), dim3(kStreamThreads), s1, stream, false, 0, kmap32, p, ring);
        } else {
            auto k1 = tile_kernel<kProp, T, D, G>;
            const size_t s1 = TileSmem<T, D, G, kProp>::bytes(p.tile);
            e = ensure_smem(k1, s1);
            if (e != cudaSuccess) return e;
            e = launch_kernel(k1, dim3(p.Hkv, p.Tmax, p.B), dim3(kTileWarps * 32), s1, stream, false, 0, kmap64, kmap64,
                              p);
        }
        if (e != cudaSuccess) return e;
        if (tm.end) cudaEventRecord(tm.end, stream);
        return launch_kernel(k2, dim3(p.nsplit, p.Hq, p.B), dim3(kPass2Warps * 32), s2, stream, true, p.nsplit, p);
    });
}

}  // namespace santa
