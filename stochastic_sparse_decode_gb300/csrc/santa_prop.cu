// santa_prop.cu -- launch of S2ANTA-prop: the streaming pass 1, then pass 2.
#include "santa_launch.h"
#include "santa_pass2.cuh"
#include "santa_stream.cuh"

namespace santa {

// Pass-1 shared memory with as many chunk buffers per warp as `smem_optin` allows
// (0 if not even one fits).
size_t prop_pass1_smem(int dtype, int d, int g, int smem_optin) {
    size_t bytes = 0;
    SANTA_DISPATCH(dtype, d, g, {
        using CG = ChunkGeom<T, D, G>;
        const int nbuf = CG::nbuf_for(size_t(smem_optin));
        bytes = nbuf ? CG::bytes(nbuf) : size_t(-1);
        return cudaSuccess;
    });
    return bytes;
}

size_t prop_pass2_smem(int d, int cps, int sampler, int S, bool paged) {
    const int nu = sampler_slots(sampler, S);
    return d == 128 ? Pass2Smem<uint16_t, 128>::bytes(cps, nu, paged) : Pass2Smem<uint16_t, 64>::bytes(cps, nu, paged);
}

template <typename T, int D>
static void *pass2_for(int sampler, bool paged) {
    if (paged) return sampler == kSys ? reinterpret_cast<void *>(prop_pass2_kernel<T, D, kSys, true>) : nullptr;
    switch (sampler) {
        case kSys: return reinterpret_cast<void *>(prop_pass2_kernel<T, D, kSys, false>);
        case kStrat: return reinterpret_cast<void *>(prop_pass2_kernel<T, D, kStrat, false>);
        case kIid: return reinterpret_cast<void *>(prop_pass2_kernel<T, D, kIid, false>);
        default: return nullptr;
    }
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

cudaError_t launch_prop(const Params &p, int dtype, const CUtensorMap &kmap32, cudaStream_t stream, const Timing &tm,
                        int stages) {
    int sms = 0, optin = 0;
    cudaError_t e0 = device_limits(&sms, &optin);
    if (e0 != cudaSuccess) return e0;
    return SANTA_DISPATCH(dtype, p.D, p.G, {
        using CG = ChunkGeom<T, D, G>;
        const int nbuf = CG::nbuf_for(size_t(optin));
        if (!nbuf) return cudaErrorNotSupported;
        auto k1 = p.page_table ? prop_stream_kernel<T, D, G, true> : prop_stream_kernel<T, D, G, false>;
        const size_t s1 = CG::bytes(nbuf);
        auto k2 = reinterpret_cast<void (*)(const Params)>(pass2_for<T, D>(p.sampler, p.page_table != nullptr));
        if (!k2) return cudaErrorInvalidValue;
        const size_t s2 = Pass2Smem<T, D>::bytes(p.chunks_per_split, sampler_slots(p.sampler, p.S), p.page_table);
        cudaError_t e = ensure_smem(k1, s1);
        if (e == cudaSuccess) e = ensure_smem(k2, s2);
        if (e != cudaSuccess) return e;
        // One CTA per SM, a multiple of Hkv CTAs so that every warp keeps one KV head;
        // no more CTAs than a warp each of chunks.
        const long long chunks = (long long)p.B * p.nch * p.Hkv;
        long long grid = sms >= p.Hkv ? (long long)(sms / p.Hkv) * p.Hkv : sms;
        if (grid > chunks) grid = chunks;
        if (stages & kPass1) record_event(tm.begin, stream);
        // Pass 1 may launch early (programmatic dependent launch): behind a previous
        // call's pass 2 it sets up while that kernel drains.  Pass 2 goes in plain
        // stream order -- launched early, its CTAs only wait on SMs pass 1 is using
        // (measured on GB300: 25.3 us per layer-step this way, 26.6 with neither
        // kernel early, 29.4 with both, 30.8 with only pass 2).
        if (stages & kPass1) {
            e = launch_kernel(k1, dim3(unsigned(grid)), dim3(kChunkWarps * 32), s1, stream, true, 0, kmap32, p, nbuf);
            if (e != cudaSuccess) return e;
            record_event(tm.end, stream);
        }
        if (!(stages & kPass2)) return cudaSuccess;
        return launch_kernel(k2, dim3(p.nsplit, p.Hq, p.B), dim3(kPass2Warps * 32), s2, stream, false, p.nsplit, p);
    });
}

}  // namespace santa
