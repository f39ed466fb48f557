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

template <int D>
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
            coef = __ldcg(p.rec_z + rec0 + t) * expf(__ldcg(p.rec_m + rec0 + t) - M);
            zpart += coef;
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
