// santa_pass2.cuh -- S2ANTA-prop pass 2 (with the global reducer) and the
// flash / exact merge.
//
// prop pass 2 ("Stochastic Sparse Attention for Memory-Bound Inference", paper
// notes, Key design 2).  The tiles of one (query head, sequence) are split over
// the CTAs of one thread-block cluster (`nsplit` CTAs, `tiles_per_split` tiles
// each, two or more per warp).  Every CTA first runs the reducer over that
// head's T_b tile records, in a fixed order, so all of them obtain
// bit-identical values:
//     M = max_t m_t,   w_t = z_t exp(m_t - M)   (Z_tile on a common scale),
//     C_t = w_0 + ... + w_t (inclusive),   Z = C_{T_b - 1}.
// The systematic thresholds are U + m/S, m = 0..S-1 (Key design 1), i.e. the
// points (U + m/S) Z on the unnormalised CDF.  The number of them below c is
//     N(c) = clamp(ceil(S c / Z - S U), 0, S),
// so tile t receives the thresholds m in [N(C_{t-1}), N(C_t)) -- its budget
// S_tile = N(C_t) - N(C_{t-1}), with N(C_{-1}) = 0 and N(C_{T_b - 1}) = S.
// N is evaluated by monotone float operations on non-decreasing C, so budgets
// are non-negative and add up to exactly S.  Tiles with S_tile = 0 read
// neither their stash nor V.  For the others one warp scans the tile's stashed
// e into its in-tile prefix, maps each threshold to the tile's own scale,
//     r_m = ((U + m/S) Z - C_{t-1}) / exp(m_t - M),
// takes the smallest key whose prefix exceeds r_m (clamped to the tile's keys
// of positive score), and adds V of that key.  Each CTA sums its warps in warp
// order and stores the sum into the shared memory of cluster rank 0, which adds
// the CTAs in rank order after one cluster barrier.  out = sum / S: no multiply
// by a probability anywhere after the softmax.
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

// Pass-2 shared memory: [tps+1] C, [tps] first, [tps] count, [8] scratch,
// [Tmax] tile max, [Tmax] tile sum, [NW][2][tile] in-tile prefixes, [NW][D]
// warp sums, [8][D] the cluster's CTA sums (used in rank 0).
template <typename T, int D>
struct Pass2Smem {
    static __host__ __device__ size_t rec_off(int tps) { return (size_t(tps + 1) * 4 + size_t(tps) * 8 + 32 + 15) & ~size_t(15); }
    static __host__ __device__ size_t buf_off(int tps, int Tmax) {
        return (rec_off(tps) + size_t(Tmax) * 8 + 15) & ~size_t(15);
    }
    static __host__ __device__ size_t red_off(int tps, int Tmax, int tile) {
        return buf_off(tps, Tmax) + size_t(kPass2Warps) * 2 * tile * 4;
    }
    static __host__ __device__ size_t part_off(int tps, int Tmax, int tile) {
        return red_off(tps, Tmax, tile) + size_t(kPass2Warps) * D * 4;
    }
    static __host__ __device__ size_t bytes(int tps, int Tmax, int tile) {
        return part_off(tps, Tmax, tile) + size_t(kMaxSplit) * D * 4;
    }
};

template <typename T, int D>
__global__ void __launch_bounds__(kPass2Warps * 32, 2) prop_pass2_kernel(const Params p) {
    constexpr int kThreads = kPass2Warps * 32;
    constexpr int kE = D / 32;
    constexpr int kPre = 8;  // stash values per lane and tile read in one batch (first 256 keys)
    using Lay = Pass2Smem<T, D>;
    const int split = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;  // split == rank in the cluster
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = p.tile, tps = p.tiles_per_split, kpw = tps / kPass2Warps;

    extern __shared__ __align__(128) unsigned char smem[];
    float *sC = reinterpret_cast<float *>(smem);  // C_{t_lo-1} .. C_{t_hi-1}
    int *s_first = reinterpret_cast<int *>(sC + tps + 1);
    int *s_cnt = s_first + tps;
    float *scr = reinterpret_cast<float *>(s_cnt + tps);  // [8]
    float *s_m = reinterpret_cast<float *>(smem + Lay::rec_off(tps));
    float *s_z = s_m + p.Tmax;
    float *buf = reinterpret_cast<float *>(smem + Lay::buf_off(tps, p.Tmax));
    float *red = reinterpret_cast<float *>(smem + Lay::red_off(tps, p.Tmax, tile));
    float *part = reinterpret_cast<float *>(smem + Lay::part_off(tps, p.Tmax, tile));

    cluster_arrive();  // first half of the barrier that makes every CTA's shared memory addressable

    // Inputs the previous kernel does not write may be read before the dependency wait.
    long long start;
    const int L = seq_bounds(p, b, &start);
    const float u = load_offset(p, b, hq);
    pdl_wait();

    const int Tb = (L + tile - 1) / tile;
    const int t_lo = split * tps, t_hi = min(Tb, t_lo + tps);
    const bool active = t_lo < t_hi;  // CTA-uniform: this CTA owns at least one tile
    const size_t rec0 = (size_t(b) * p.Hq + hq) * p.Tmax;
    const float *sseq = p.stash + size_t(hq) * p.total_tokens + start;
    const float Sf = float(p.S);

    // Stash values of two of this warp's tiles (split-local indices i0, i0 + 8), one batch of loads.
    auto load_pair = [&](int i0, float (&ev)[2][kPre]) {
#pragma unroll
        for (int w2 = 0; w2 < 2; ++w2) {
            const int t = t_lo + i0 + kPass2Warps * w2;
            const int lent = (i0 + kPass2Warps * w2 < kpw * kPass2Warps && t < t_hi) ? min(tile, L - t * tile) : 0;
#pragma unroll
            for (int k = 0; k < kPre; ++k) {
                const int idx = lane + 32 * k;
                ev[w2][k] = idx < lent ? __ldcg(sseq + size_t(t) * tile + idx) : 0.f;
            }
        }
    };

    float acc[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) acc[e] = 0.f;

    if (active) {
        // ---- one round trip: the first pair of this warp's tiles (speculatively) and all tile records
        float ev[2][kPre];
        load_pair(warp, ev);
        for (int t0 = 0; t0 < Tb; t0 += 4 * kThreads) {
            float mm[4], zz[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int t = t0 + k * kThreads + tid;
                mm[k] = t < Tb ? __ldcg(p.rec_m + rec0 + t) : 0.f;
                zz[k] = t < Tb ? __ldcg(p.rec_z + rec0 + t) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int t = t0 + k * kThreads + tid;
                if (t < Tb) {
                    s_m[t] = mm[k];
                    s_z[t] = zz[k];
                }
            }
        }
        __syncthreads();

        // ---- reducer
        float mx = -INFINITY;
        for (int t = tid; t < Tb; t += kThreads) mx = fmaxf(mx, s_m[t]);
        const float M = block_max<kPass2Warps>(mx, scr);
        float carry = 0.f;
        for (int c0 = 0; c0 < Tb; c0 += kThreads) {
            const int t = c0 + tid;
            const float w = (t < Tb) ? s_z[t] * expf(s_m[t] - M) : 0.f;
            float total;
            const float incl = block_inclusive_scan<kPass2Warps>(w, scr, &total) + carry;
            if (t >= t_lo - 1 && t < t_hi) sC[t - t_lo + 1] = incl;
            carry = total + carry;
        }
        const float Z = carry;
        if (t_lo == 0 && tid == 0) sC[0] = 0.f;
        __syncthreads();

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

        // ---- this warp's tiles, two at a time: in-tile prefix, systematic search, V gather
        float *wb = buf + size_t(warp) * 2 * tile;
        const int kvh = hq / p.G;
        const size_t vstride = size_t(p.Hkv) * D;
        const T *vseq = static_cast<const T *>(p.v) + size_t(start) * vstride + size_t(kvh) * D;
        for (int kk = 0; kk < kpw; kk += 2) {
            const int i0 = warp + kPass2Warps * kk;
            if (kk > 0) load_pair(i0, ev);
            int cnt[2], first[2], k0[2], len[2], lastp[2];
            float st[2], Cprev[2];
#pragma unroll
            for (int w2 = 0; w2 < 2; ++w2) {
                const int i = i0 + kPass2Warps * w2;
                const int t = t_lo + i;
                const bool mine = (kk + w2 < kpw) && t < t_hi;
                cnt[w2] = mine ? s_cnt[i] : 0;
                first[w2] = mine ? s_first[i] : 0;
                k0[w2] = t * tile;
                len[w2] = mine ? min(tile, L - t * tile) : 0;
                lastp[w2] = -1;
                st[w2] = 1.f;
                Cprev[w2] = 0.f;
                if (cnt[w2] > 0) {
                    TileScan sc;
                    float *P = wb + w2 * tile;
#pragma unroll
                    for (int k = 0; k < kPre; ++k) {
                        const int idx = lane + 32 * k;
                        if (32 * k < len[w2]) {
                            const float v = sc.step(ev[w2][k], idx, lane);
                            if (idx < len[w2]) P[idx] = v;
                        }
                    }
                    for (int j0 = 32 * kPre; j0 < len[w2]; j0 += 32) {  // tiles longer than 256 keys
                        const int idx = j0 + lane;
                        const float e = idx < len[w2] ? __ldcg(sseq + k0[w2] + idx) : 0.f;
                        const float v = sc.step(e, idx, lane);
                        if (idx < len[w2]) P[idx] = v;
                    }
                    sc.finish();
                    lastp[w2] = sc.last_pos;
                    st[w2] = expf(s_m[t] - M);
                    Cprev[w2] = sC[i];
                }
            }
            __syncwarp();
            const int total = cnt[0] + cnt[1];
            for (int g0 = 0; g0 < total; g0 += 32) {
                const int g = g0 + lane;
                int j = 0;
                if (g < total) {
                    const bool second = g >= cnt[0];  // which of the two tiles holds sample g
                    const int m = second ? first[1] + (g - cnt[0]) : first[0] + g;
                    const float thr = u + float(m) / Sf;
                    const float r = (thr * Z - (second ? Cprev[1] : Cprev[0])) / (second ? st[1] : st[0]);
                    j = (second ? k0[1] : k0[0]) + cdf_search(wb + (second ? tile : 0), second ? len[1] : len[0], r,
                                                              second ? lastp[1] : lastp[0]);
                    if (p.dbg_idx) p.dbg_idx[(size_t(b) * p.Hq + hq) * p.S + m] = j;
                }
                gather_rows<T, D>(acc, vseq, vstride, j, min(32, total - g0), lane);
            }
            __syncwarp();
        }
    }

    // ---- deterministic combine: warps in order, then the cluster's CTAs in rank order
#pragma unroll
    for (int e = 0; e < kE; ++e) red[warp * D + lane * kE + e] = acc[e];
    __syncthreads();
    cluster_wait();  // every CTA of the cluster is running: rank 0's shared memory is addressable
    if (tid < D) {
        float cta = 0.f;
#pragma unroll
        for (int w = 0; w < kPass2Warps; ++w) cta += red[w * D + tid];
        st_cluster_f32(cluster_map(part + split * D + tid, 0), cta);
    }
    cluster_arrive();
    cluster_wait();
    if (split == 0 && tid < D) {
        float s = 0.f;
        for (int k = 0; k < int(gridDim.x); ++k) s += part[k * D + tid];
        p.out[(size_t(b) * p.Hq + hq) * D + tid] = L > 0 ? s / Sf : 0.f;
    }
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
