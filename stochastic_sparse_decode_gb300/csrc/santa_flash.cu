// santa_flash.cu -- S2ANTA-flash: prop's streaming pass 1 (chunk records and the
// score stash), then the tiles' local sampling and V gather, then the merge.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (paper notes), Key
// design 3: every tile assumes it holds all of the mass and draws S_loc =
// ceil(S / T_b) systematic thresholds U_t + s/S_loc, U_t = U S / S_loc, on its own
// CDF; the chosen V rows are averaged into its estimate o_t, and the merge
// rescales the estimates by Z_tile / Z.  A tile is tile/32 of pass 1's 32-key
// chunks, so its scores need no second read of K:
//     m_t = max_c m_c,   z_t = sum_c z_c exp(m_c - m_t),
// and its unnormalised CDF is the running sum, in key order, of the stashed
// e_i = exp(x_i - m_c) times exp(m_c - m_t).  Threshold s is the smallest key whose
// running sum exceeds (U_t + s/S_loc) z_t (clamped to the tile's last key of
// positive score).
#include "santa_launch.h"
#include "santa_merge.cuh"
#include "santa_sampler.cuh"
#include "santa_stream.cuh"

namespace santa {

constexpr int kFlashWarps = 4;  // tiles per CTA of the sampling kernel, one per warp

size_t flash_sample_smem(int tile) { return size_t(kFlashWarps) * tile * 4; }

// One warp per (sequence, query head, tile): the tile's record and estimate.
// (eight CTAs per SM for bf16: the whole grid of the bench workload in one wave)
template <typename T, int D>
__global__ void __launch_bounds__(kFlashWarps * 32, sizeof(T) == 2 ? 8 : 4) flash_sample_kernel(const Params p) {
    extern __shared__ __align__(16) float fs_smem[];  // [warp][tile] running sums
    constexpr int kE = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kFlashWarps + warp, hq = blockIdx.y, b = blockIdx.z;
    float *pre = fs_smem + size_t(warp) * p.tile;
    long long start;
    const int L = seq_bounds(p, b, &start);
    const float u_raw = p.U[size_t(b) * p.Hq + hq];
    pdl_wait();
    const size_t head = size_t(b) * p.Hq + hq;
    if (t == 0 && lane == 0) p.cnt[head] = 0u;  // pass 1's publication count: unused here
    const int Tb = (L + p.tile - 1) / p.tile;
    if (t >= Tb) return;  // warps are independent: no CTA barrier below
    const int cpt = p.tile / kChunkRows, c0 = t * cpt;
    const int k0 = t * p.tile, len = min(p.tile, L - k0);
    const int nc = (len + kChunkRows - 1) / kChunkRows;

    // the tile's stash, global to shared memory in one round trip (keys past the
    // sequence's end read as 0), issued before the records are combined
    const float *st = p.stash + (head * p.nch + c0) * kChunkRows;
    for (int pi = lane; pi < nc * 8; pi += 32) {
        const int valid = min(max(len - 4 * pi, 0), 4);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(pre + 4 * pi)), "l"(st + 4 * pi),
                     "r"(4 * valid)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    float mc = -INFINITY, zc = 0.f;
    if (lane < nc) {
        const unsigned long long v = __ldcg(p.rec + head * p.nch + c0 + lane);
        if (v != 0ull) {
            mc = rec_m(v);
            zc = rec_z(v);
        } else {
            raise_flag(p, SANTA_ERR_WORKSPACE);  // a record pass 1 did not write
        }
    }
    const float mt = warp_max(mc);
    const float sc = (lane < nc && mc > -INFINITY) ? __expf(mc - mt) : 0.f;  // exp(m_c - m_t)
    const float zt = warp_sum(zc * sc);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();

    // running sums on the m_t scale, one chunk per step; the last key of positive score
    float carry = 0.f;
    int last = -1;
    for (int c = 0; c < nc; ++c) {
        const float e = pre[c * kChunkRows + lane] * __shfl_sync(kFull, sc, c);
        const float v = warp_inclusive_scan(e, lane) + carry;
        pre[c * kChunkRows + lane] = v;
        carry = __shfl_sync(kFull, v, 31);
        const unsigned pos = __ballot_sync(kFull, e > 0.f);
        if (pos) last = c * kChunkRows + 31 - __clz(pos);
    }
    __syncwarp();

    // S_loc thresholds, 32 at a time (lane = threshold), and their V rows
    const int S_loc = (p.S + Tb - 1) / Tb;
    const float Ut = checked_offset(p, u_raw) * float(p.S) / float(S_loc);
    const float inv = 1.0f / float(S_loc);
    const size_t vstride = size_t(p.Hkv) * D;
    const T *vseq = static_cast<const T *>(p.v) + size_t(start) * vstride + size_t(hq / p.G) * D;
    float acc[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) acc[e] = 0.f;
    for (int s0 = 0; s0 < S_loc; s0 += 32) {
        const int n = min(32, S_loc - s0);
        int j = 0;
        if (lane < n) {
            const float th = fmaf(float(s0 + lane), inv, Ut) * zt;
            j = k0 + cdf_search(pre, len, th, last);
            if (p.dbg_idx && s0 + lane < p.dbg_stride)
                p.dbg_idx[(head * p.Tmax + t) * p.dbg_stride + s0 + lane] = j;
        }
        gather_queue<T, D>(acc, vseq, vstride, j, n, lane);
    }
    float *o = p.partial + (head * p.Tmax + t) * D + lane * kE;
#pragma unroll
    for (int e = 0; e < kE; ++e) o[e] = acc[e] * inv;
    if (lane == 0) {
        p.rec_m[head * p.Tmax + t] = mt;
        p.rec_z[head * p.Tmax + t] = zt;
        if (p.dbg_tile_m) p.dbg_tile_m[head * p.Tmax + t] = mt;
        if (p.dbg_tile_z) p.dbg_tile_z[head * p.Tmax + t] = zt;
    }
}

cudaError_t launch_flash(const Params &p, int dtype, const CUtensorMap &kmap, cudaStream_t stream, const Timing &tm) {
    cudaError_t e = launch_prop(p, dtype, kmap, stream, tm, kPass1);  // the streaming pass 1
    if (e != cudaSuccess) return e;
    return SANTA_DISPATCH(dtype, p.D, p.G, {
        (void)sizeof(G);
        const unsigned tiles = unsigned((p.Tmax + kFlashWarps - 1) / kFlashWarps);
        cudaError_t e2 = launch_kernel(flash_sample_kernel<T, D>, dim3(tiles, unsigned(p.Hq), unsigned(p.B)),
                                       dim3(kFlashWarps * 32), flash_sample_smem(p.tile), stream, false, 0, false, p);
        if (e2 != cudaSuccess) return e2;
        return launch_kernel(merge_kernel<D>, dim3(p.Hq, p.B), dim3(kMergeThreads), 0, stream, true, 0, false, p);
    });
}

}  // namespace santa
