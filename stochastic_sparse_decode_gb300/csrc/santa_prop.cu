// santa_prop.cu -- launch of S2ANTA-prop: the streaming pass 1 and the cluster
// pass 2 as two kernels, or the fused persistent kernel (pass 1 and the samplers
// in one grid).
#include "santa_launch.h"
#include "santa_pass2.cuh"
#include "santa_sampler.cuh"
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

// The fused kernel: the streaming layout with as many buffers per warp as fit,
// which the samplers then reuse; 0 if it does not fit.  *nbuf: the buffers per warp.
size_t prop_fused_smem(int dtype, int d, int g, int sampler, int S, int smem_optin, int *nbuf) {
    size_t bytes = 0;
    SANTA_DISPATCH(dtype, d, g, {
        using CG = ChunkGeom<T, D, G>;
        const int nb = CG::nbuf_for(size_t(smem_optin));
        const int nu = sampler_slots(sampler, S);
        const size_t need = nb ? fused_smem_bytes<T, D, G>(nb, nu) : size_t(-1);
        bytes = need <= size_t(smem_optin) ? need : 0;
        if (nbuf) *nbuf = nb;
        return cudaSuccess;
    });
    return bytes;
}

template <typename T, int D, int G>
static void *fused_for(int sampler, bool paged) {
    if (paged) return sampler == kSys ? reinterpret_cast<void *>(prop_fused_kernel<T, D, G, kSys, true>) : nullptr;
    switch (sampler) {
        case kSys: return reinterpret_cast<void *>(prop_fused_kernel<T, D, G, kSys, false>);
        case kStrat: return reinterpret_cast<void *>(prop_fused_kernel<T, D, G, kStrat, false>);
        case kIid: return reinterpret_cast<void *>(prop_fused_kernel<T, D, G, kIid, false>);
        default: return nullptr;
    }
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

cudaError_t prop_pass2_split(int nch, int tile, long long heads, int *nsplit, int *cps) {
    int sms = 0, optin = 0;
    if (device_limits(&sms, &optin) != cudaSuccess) {  // no device (host-side validation): GB300's count
        cudaGetLastError();
        sms = 152;
    }
    const int unit = (tile / 32) > kPass2Warps ? tile / 32 : kPass2Warps;
    int n = (nch + 127) / 128;
    const long long fill = heads > 0 ? (2LL * sms + heads - 1) / heads : 1;  // splits for two CTAs per SM
    if (n > fill) n = int(fill);
    const int n_smem = (nch + 8191) / 8192;  // at most 8192 chunks of C, N and exp(m - M) per CTA
    if (n < n_smem) n = n_smem;
    n = n < 1 ? 1 : (n > kP2MaxSplit ? kP2MaxSplit : n);
    int per = (nch + n - 1) / n;
    per = (per + unit - 1) / unit * unit;
    *nsplit = n;
    *cps = per < unit ? unit : per;
    return cudaSuccess;
}

cudaError_t launch_prop(const Params &p, int dtype, const CUtensorMap &kmap32, cudaStream_t stream, const Timing &tm,
                        int stages) {
    int sms = 0, optin = 0;
    cudaError_t e0 = device_limits(&sms, &optin);
    if (e0 != cudaSuccess) return e0;
    const bool paged = p.page_table != nullptr;
    return SANTA_DISPATCH(dtype, p.D, p.G, {
        using CG = ChunkGeom<T, D, G>;
        // One CTA per SM, a multiple of Hkv CTAs so that every warp keeps one KV head;
        // no more CTAs than a warp each of chunks.
        const long long chunks = (long long)p.B * p.nch * p.Hkv;
        long long grid = sms >= p.Hkv ? (long long)(sms / p.Hkv) * p.Hkv : sms;
        if (grid > chunks) grid = chunks;
        int nbf = 0;
        size_t sf = prop_fused_smem(dtype, D, G, p.sampler, p.S, optin, &nbf);
        Params ps = p;
        ps.nsplit = prop_nsplit((long long)p.B * p.Hq, sms);  // the fused kernel's splits of a head
        e0 = prop_pass2_split(p.nch, p.tile, (long long)p.B * p.Hq, &ps.p2_split, &ps.p2_cps);
        if (e0 != cudaSuccess) return e0;
        cudaError_t e = cudaSuccess;
        auto kf = reinterpret_cast<void (*)(const CUtensorMap, const Params, int)>(fused_for<T, D, G>(p.sampler, paged));
        if (!kf) return cudaErrorInvalidValue;
        const bool fused = (stages & kFused) && (stages & kPass1) && (stages & kPass2);
        if (fused && sf) {
            e = ensure_smem(kf, sf);
            if (e != cudaSuccess) return e;
            // the grid is sized so that every CTA is resident at once
            int per_sm = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kf, kChunkWarps * 32, sf);
            if (e != cudaSuccess) return e;
            if ((long long)per_sm * sms < grid) sf = 0;  // it could not be: two kernels
        }
        if (fused && sf) {
            // The fused kernel.  A sampler waits for records that other CTAs write, so
            // every CTA must run at once: the grid is one CTA per SM, which the device
            // holds at once whenever this kernel has it to itself.  (A cooperative
            // launch would guarantee it even beside other work, but measured 1.6 us
            // slower per call on GB300, as it gives up the early launch below.)  If
            // other work keeps an SM busy past a sampler's bounded wait, the wait gives
            // up with SANTA_ERR_TIMEOUT instead of hanging.  Launched early behind the
            // previous kernel (programmatic dependent launch), whose completion it
            // awaits before touching global memory.
            record_event(tm.begin, stream);
            e = launch_kernel(kf, dim3(unsigned(grid)), dim3(kChunkWarps * 32), sf, stream, true, 0, false, kmap32,
                              ps, nbf);
            if (e != cudaSuccess) return e;
            record_event(tm.end, stream);
            return cudaSuccess;
        }
        // Pass 1 may launch early (programmatic dependent launch): behind a previous
        // call's pass 2 it sets up while that kernel drains.  Pass 2 goes in plain
        // stream order: launched early, its CTAs would only wait on SMs pass 1 is
        // using (measured slower on GB300).
        if (stages & kPass1) {
            const int nbuf = CG::nbuf_for(size_t(optin));
            if (!nbuf) return cudaErrorNotSupported;
            auto k1 = paged ? prop_stream_kernel<T, D, G, true> : prop_stream_kernel<T, D, G, false>;
            const size_t s1 = CG::bytes(nbuf);
            e = ensure_smem(k1, s1);
            if (e != cudaSuccess) return e;
            record_event(tm.begin, stream);
            e = launch_kernel(k1, dim3(unsigned(grid)), dim3(kChunkWarps * 32), s1, stream, true, 0, false, kmap32, p,
                              nbuf);
            if (e != cudaSuccess) return e;
            record_event(tm.end, stream);
        }
        if (!(stages & kPass2)) return cudaSuccess;
        auto k2 = reinterpret_cast<void (*)(const Params)>(pass2_for<T, D>(p.sampler, paged));
        if (!k2) return cudaErrorInvalidValue;
        const size_t s2 = Pass2Smem<T, D>::bytes(ps.p2_cps, sampler_slots(p.sampler, p.S), paged);
        e = ensure_smem(k2, s2);
        if (e != cudaSuccess) return e;
        return launch_kernel(k2, dim3(unsigned(ps.p2_split), unsigned(p.Hq), unsigned(p.B)), dim3(kPass2Warps * 32),
                             s2, stream, false, ps.p2_split, false, ps);
    });
}

}  // namespace santa
