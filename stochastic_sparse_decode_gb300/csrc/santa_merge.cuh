// santa_merge.cuh -- block-wide reductions and the S2ANTA-flash merge.
//
// merge ("Stochastic Sparse Attention for Memory-Bound Inference", paper notes,
// Key design 3): per (query head, sequence)
//     out = sum_t w_t o_t / Z,   w_t = z_t exp(m_t - M),   Z = sum_t w_t,
// with o_t the tile's sample average and M the largest tile maximum.
#pragma once

#include "santa_common.cuh"

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

// The merge of one (sequence, query head): its kMergeThreads / 32 warps take the
// tiles t = warp, warp + warps, ... eight at a time (every load of a batch in flight
// at once), lane = a D/32 slice of the estimates.  A warp keeps its sums on the scale
// of the largest m_t it has seen (rescaling when a batch raises it), so no pass over
// the records precedes the loads; the warps' sums are then brought to the common
// maximum M and added in warp order: out = sum_t w_t o_t / sum_t w_t.
template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const Params p) {
    constexpr int kNW = kMergeThreads / 32;
    constexpr int kE = D / 32;
    constexpr int kB = 8;  // tiles per batch of a warp
    const int hq = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __shared__ float red[kNW][D];
    __shared__ float ms[kNW], zs[kNW];

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

    float acc[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) acc[e] = 0.f;
    float mw = -INFINITY, zw = 0.f;  // the warp's scale and sum of coefficients (the same in every lane)
    for (int t0 = warp; t0 < Tb; t0 += kB * kNW) {
        float m[kB], z[kB], o[kB][kE];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int t = t0 + u * kNW;
            m[u] = -INFINITY;
            z[u] = 0.f;
#pragma unroll
            for (int e = 0; e < kE; ++e) o[u][e] = 0.f;
            if (t < Tb) {
                m[u] = __ldcg(p.rec_m + rec0 + t);
                z[u] = __ldcg(p.rec_z + rec0 + t);
                const float *src = p.partial + (rec0 + t) * D + lane * kE;
#pragma unroll
                for (int e = 0; e < kE; ++e) o[u][e] = __ldcg(src + e);
            }
        }
        float mb = mw;
#pragma unroll
        for (int u = 0; u < kB; ++u) mb = fmaxf(mb, m[u]);
        if (mb > mw) {  // rescale what the warp holds to the batch's larger maximum
            const float sc = mw > -INFINITY ? expf(mw - mb) : 0.f;
            zw *= sc;
#pragma unroll
            for (int e = 0; e < kE; ++e) acc[e] *= sc;
            mw = mb;
        }
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const float cf = m[u] > -INFINITY ? z[u] * expf(m[u] - mw) : 0.f;
            zw += cf;
#pragma unroll
            for (int e = 0; e < kE; ++e) acc[e] = fmaf(cf, o[u][e], acc[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < kE; ++e) red[warp][lane * kE + e] = acc[e];
    if (lane == 0) {
        ms[warp] = mw;
        zs[warp] = zw;
    }
    __syncthreads();
    if (tid < D) {
        float M = ms[0];
#pragma unroll
        for (int w = 1; w < kNW; ++w) M = fmaxf(M, ms[w]);
        float num = 0.f, Z = 0.f;
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
            const float sc = ms[w] > -INFINITY ? expf(ms[w] - M) : 0.f;
            num = fmaf(red[w][tid], sc, num);
            Z = fmaf(zs[w], sc, Z);
        }
        outp[tid] = num / Z;
    }
}

}  // namespace santa
