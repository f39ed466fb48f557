// santa_pass2.cuh -- S2ANTA-prop pass 2 (with the global reducer) and the
// flash / exact merge.
//
// prop pass 2 ("Stochastic Sparse Attention for Memory-Bound Inference", paper
// notes, Key design 2).  One CTA per (split, query head, sequence); a split
// owns `tiles_per_split` consecutive tiles.  Every CTA of a head first runs the
// reducer over that head's T_b tile records, in a fixed order, so all of them
// obtain bit-identical values:
//     M = max_t m_t,   w_t = z_t exp(m_t - M)   (Z_tile on a common scale),
//     C_t = w_0 + ... + w_t (inclusive),   Z = C_{T_b - 1}.
// The systematic thresholds are U + m/S, m = 0..S-1 (Key design 1), i.e. the
// points (U + m/S) Z on the unnormalised CDF.  The number of them below c is
//     N(c) = clamp(ceil(S c / Z - S U), 0, S),
// so tile t receives the thresholds m in [N(C_{t-1}), N(C_t)) -- its budget
// S_tile = N(C_t) - N(C_{t-1}), with N(C_{-1}) = 0 and N(C_{T_b - 1}) = S.
// N is evaluated by monotone float operations on non-decreasing C, so budgets
// are non-negative and add up to exactly S.  Tiles with S_tile = 0 read
// neither their stash nor V.  For the others one warp rebuilds the tile's
// in-tile prefix of the stashed e with the same scan pass 1 used (so its total
// equals z_t bit for bit), maps each threshold to the tile's own scale,
//     r_m = ((U + m/S) Z - C_{t-1}) / exp(m_t - M),
// takes the smallest key whose prefix exceeds r_m (clamped to the tile's keys
// of positive score), and adds V of that key.  The CTA sums its warps in warp
// order; with several splits, the last CTA to finish (a ticket counter, no
// waiting) sums the splits in split order.  out = sum / S: no multiply by a
// probability anywhere after the softmax.
//
// merge (flash, Key design 3; exact split-KV): per (query head, sequence)
//     flash: out = sum_t w_t o_t / Z   with o_t the tile's sample average,
//     exact: out = sum_t exp(m_t - M) o_t / Z   with o_t = sum_i e_i V_i,
// where Z = sum_t w_t.
#pragma once

#include "santa_common.cuh"
#include "santa_tile.cuh"

namespace santa {

// ---- block-wide helpers (every thread gets the result; fixed evaluation order)

template <int NW>
__device__ __forceinline__ float block_max(float v, float *scr) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max(v);
    __syncthreads();
    if (lane == 0) scr[warp] = v;
    __syncthreads();
    float r = scr[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) r = fmaxf(r, scr[w]);
    return r;
}

template <int NW>
__device__ __forceinline__ float block_sum(float v, float *scr) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) scr[warp] = v;
    __syncthreads();
    float r = scr[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) r += scr[w];
    return r;
}

// Inclusive scan over the block; *total is the sum of all values and equals,
// bit for bit, the inclusive value of the last thread.
template <int NW>
__device__ __forceinline__ float block_inclusive_scan(float v, float *scr, float *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_inclusive_scan(v, lane);
    __syncthreads();
    if (lane == 31) scr[warp] = v;
    __syncthreads();
    float off = 0.f, tot = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        if (w < warp) off += scr[w];
        if (w < NW - 1) tot += scr[w];
    }
    *total = scr[NW - 1] + tot;
    return v + off;
}

template <typename T, int D>
struct Pass2Smem {
    // [tps + 1] C, [tps] first, [tps] count, [8] scratch, [8] misc, [NW][tile] prefix, [NW][D] combine
    static __host__ __device__ size_t buf_off(int tps) {
        size_t o = size_t(tps + 1) * 4 + size_t(tps) * 8 + 64;
        return (o + 15) & ~size_t(15);
    }
    static __host__ __device__ size_t red_off(int tps, int tile) { return buf_off(tps) + size_t(kPass2Warps) * tile * 4; }
    static __host__ __device__ size_t bytes(int tps, int tile) { return red_off(tps, tile) + size_t(kPass2Warps) * D * 4; }
};

template <typename T, int D>
__global__ void __launch_bounds__(kPass2Warps * 32) prop_pass2_kernel(const Params p) {
    constexpr int kThreads = kPass2Warps * 32;
    constexpr int kE = D / 32;
    using Lay = Pass2Smem<T, D>;
    const int split = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = p.tile, tps = p.tiles_per_split;

    extern __shared__ __align__(128) unsigned char smem[];
    float *sC = reinterpret_cast<float *>(smem);    // C_{t_lo-1} .. C_{t_hi-1}
    int *s_first = reinterpret_cast<int *>(sC + tps + 1);
    int *s_cnt = s_first + tps;
    float *scr = reinterpret_cast<float *>(s_cnt + tps);  // [8]
    int *s_last = reinterpret_cast<int *>(scr + 8);
    float *buf = reinterpret_cast<float *>(smem + Lay::buf_off(tps));
    float *red = reinterpret_cast<float *>(smem + Lay::red_off(tps, tile));

    // Inputs the previous kernel does not write may be read before the dependency wait.
    long long start;
    const int L = seq_bounds(p, b, &start);
    const float u = load_offset(p, b, hq);
    pdl_wait();

    float *outp = p.out + (size_t(b) * p.Hq + hq) * D;
    const int Tb = (L + tile - 1) / tile;
    const int nsplit_b = (Tb + tps - 1) / tps;
    if (L == 0) {
        if (split == 0)
            for (int d = tid; d < D; d += kThreads) outp[d] = 0.f;
        return;
    }
    if (split >= nsplit_b) return;
    const int t_lo = split * tps, t_hi = min(Tb, t_lo + tps);
    const size_t rec0 = (size_t(b) * p.Hq + hq) * p.Tmax;

    // ---- reducer
    float mx = -INFINITY;
    for (int t = tid; t < Tb; t += kThreads) mx = fmaxf(mx, __ldcg(p.rec_m + rec0 + t));
    const float M = block_max<kPass2Warps>(mx, scr);
    float carry = 0.f;
    for (int c0 = 0; c0 < Tb; c0 += kThreads) {
        const int t = c0 + tid;
        const float w = (t < Tb) ? __ldcg(p.rec_z + rec0 + t) * expf(__ldcg(p.rec_m + rec0 + t) - M) : 0.f;
        float total;
        const float incl = block_inclusive_scan<kPass2Warps>(w, scr, &total) + carry;
        if (t >= t_lo - 1 && t < t_hi) sC[t - t_lo + 1] = incl;
        carry = total + carry;
    }
    const float Z = carry;
    if (t_lo == 0 && tid == 0) sC[0] = 0.f;
    __syncthreads();

    const float Sf = float(p.S);
    const float SU = Sf * u;
    auto N = [&](float c) -> int {
        const float x = ceilf(fmaf(Sf, c / Z, -SU));
        return int(fminf(fmaxf(x, 0.f), Sf));
    };
    for (int i = tid; i < t_hi - t_lo; i += kThreads) {
        const int t = t_lo + i;
        const int n_prev = (t == 0) ? 0 : N(sC[i]);
        const int n_cur = (t == Tb - 1) ? p.S : N(sC[i + 1]);
        s_first[i] = n_prev;
        s_cnt[i] = n_cur - n_prev;
        if (p.dbg_count) p.dbg_count[rec0 + t] = n_cur - n_prev;
    }
    __syncthreads();

    // ---- systematic search inside the tiles that got samples, and the V gather
    float acc[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) acc[e] = 0.f;
    float *wb = buf + warp * tile;
    const int kvh = hq / p.G;
    const size_t vstride = size_t(p.Hkv) * D;
    const T *vseq = static_cast<const T *>(p.v) + size_t(start) * vstride + size_t(kvh) * D;
    const float *sseq = p.stash + size_t(hq) * p.total_tokens + start;
    for (int i = warp; i < t_hi - t_lo; i += kPass2Warps) {
        const int cnt = s_cnt[i];
        if (cnt == 0) continue;
        const int t = t_lo + i, k0 = t * tile, len = min(tile, L - k0);
        TileScan sc;
        for (int i0 = 0; i0 < len; i0 += 32) {
            const int idx = i0 + lane;
            const float e = (idx < len) ? __ldcg(sseq + k0 + idx) : 0.f;
            const float P = sc.step(e, idx, lane);
            if (idx < len) wb[idx] = P;
        }
        sc.finish();
        __syncwarp();
        const float st = expf(__ldcg(p.rec_m + rec0 + t) - M);
        const float Cprev = sC[i];
        const int first = s_first[i];
        for (int s0 = 0; s0 < cnt; s0 += 32) {
            int j = 0;
            if (s0 + lane < cnt) {
                const int m = first + s0 + lane;
                const float thr = u + float(m) / Sf;
                j = cdf_search(wb, len, (thr * Z - Cprev) / st, sc.last_pos);
                if (p.dbg_idx) p.dbg_idx[(size_t(b) * p.Hq + hq) * p.S + m] = k0 + j;
            }
            gather_rows<T, D>(acc, vseq + size_t(k0) * vstride, vstride, j, min(32, cnt - s0), lane);
        }
        __syncwarp();
    }

    // ---- deterministic combine: warps in order, then splits in order
#pragma unroll
    for (int e = 0; e < kE; ++e) red[warp * D + lane * kE + e] = acc[e];
    __syncthreads();
    float cta = 0.f;
    if (tid < D) {
#pragma unroll
        for (int w = 0; w < kPass2Warps; ++w) cta += red[w * D + tid];
    }
    if (nsplit_b == 1) {
        if (tid < D) outp[tid] = cta / Sf;
        return;
    }
    float *part = p.partial + (size_t(b) * p.Hq + hq) * p.nsplit * D;
    if (tid < D) part[size_t(split) * D + tid] = cta;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(p.tickets + size_t(b) * p.Hq + hq, 1u);
        s_last[0] = (prev == unsigned(nsplit_b - 1));
    }
    __syncthreads();
    if (!s_last[0]) return;
    __threadfence();
    if (tid < D) {
        float s = 0.f;
        for (int k = 0; k < nsplit_b; ++k) s += __ldcg(part + size_t(k) * D + tid);
        outp[tid] = s / Sf;
    }
    if (tid == 0) p.tickets[size_t(b) * p.Hq + hq] = 0u;
}

template <int MODE, int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const Params p) {
    constexpr int kNW = kMergeThreads / 32;
    const int hq = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    __shared__ float s_coef[kMergeThreads];
    __shared__ float scr[kNW];

    long long start;
    const int L = seq_bounds(p, b, &start);
    pdl_wait();
    float *outp = p.out + (size_t(b) * p.Hq + hq) * D;
    if (L == 0) {
        if (tid < D) outp[tid] = 0.f;
        return;
    }
    const int Tb = (L + p.tile - 1) / p.tile;
    const size_t rec0 = (size_t(b) * p.Hq + hq) * p.Tmax;
    float mx = -INFINITY;
    for (int t = tid; t < Tb; t += kMergeThreads) mx = fmaxf(mx, __ldcg(p.rec_m + rec0 + t));
    const float M = block_max<kNW>(mx, scr);
    float num = 0.f, zpart = 0.f;
    for (int c0 = 0; c0 < Tb; c0 += kMergeThreads) {
        const int t = c0 + tid;
        float coef = 0.f;
        if (t < Tb) {
            const float s = expf(__ldcg(p.rec_m + rec0 + t) - M);
            const float w = __ldcg(p.rec_z + rec0 + t) * s;
            zpart += w;
            coef = (MODE == kFlash) ? w : s;
        }
        __syncthreads();
        s_coef[tid] = coef;
        __syncthreads();
        const int n = min(kMergeThreads, Tb - c0);
        if (tid < D)
            for (int k = 0; k < n; ++k) num = fmaf(s_coef[k], __ldcg(p.partial + (rec0 + c0 + k) * D + tid), num);
    }
    const float Z = block_sum<kNW>(zpart, scr);
    if (tid < D) outp[tid] = num / Z;
}

}  // namespace santa
