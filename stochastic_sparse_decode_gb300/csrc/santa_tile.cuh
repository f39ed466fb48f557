// santa_tile.cuh -- the split-KV tile kernel shared by the three modes.
//
// One CTA owns one (sequence b, KV head, tile t) and all G query heads of that
// KV head's GQA group, so each K row is read once for G heads.  The tile's K
// rows (and, for the exact mode, then its V rows) stream through a ring of
// kStages shared-memory slots filled by 3-D TMA copies of kChunk rows each;
// 4 warps compute the G dot products per key while later chunks are in flight.
//
// After the scores x = q.k / sqrt(d) of the tile are in shared memory, each
// head (one warp per head) forms the tile's max m_t and the exponentiated
// scores e_i = exp(x_i - m_t), and scans them once (TileScan) to get
// z_t = sum e_i -- the tile's partition sum Z_tile on the m_t scale
// ("Stochastic Sparse Attention for Memory-Bound Inference", paper notes,
// Key design 2: exponentiated scores plus one Z_tile per tile).  Then:
//
//   kProp   writes e to the score stash and (m_t, z_t) to the tile records;
//           the reducer and the sampling happen in pass 2.
//   kFlash  samples S_loc = ceil(S / T_b) systematic thresholds U_t + s/S_loc,
//           U_t = U S / S_loc, on the tile's own CDF (its prefix of e divided
//           by z_t), gather-averages the chosen V rows into the tile estimate
//           and writes it with (m_t, z_t) for the merge (Key design 3).
//   kExact  streams the tile's V rows and accumulates sum_i e_i V_i for the
//           log-sum-exp merge (exact split-KV decode).
#pragma once

#include "santa_common.cuh"

namespace santa {

template <typename T, int D>
struct TileGeom {
    static constexpr int kES = int(sizeof(T));
    static constexpr int kRowBytes = D * kES;        // 128, 256 or 512
    static constexpr int kVecs = kRowBytes / 16;     // 16-byte vectors per row
    static constexpr int kVecsPerLane = kVecs / 8;   // 8 lanes share one key
    static constexpr int kPairs = Vec16<T>::kPairs;  // float pairs per vector
    static constexpr int kChunkBytes = kChunk * kRowBytes;
};

// Shared-memory layout of a tile CTA (identical on host and device).
template <typename T, int D, int G, int MODE>
struct TileSmem {
    static constexpr size_t stage_off() { return 0; }
    static constexpr size_t xs_off() { return size_t(kStages) * TileGeom<T, D>::kChunkBytes; }
    static __host__ __device__ size_t bars_off(int tile) { return xs_off() + size_t(G) * tile * 4; }
    static __host__ __device__ size_t red_off(int tile) { return bars_off(tile) + kStages * 8 + 16; }
    static __host__ __device__ size_t bytes(int tile) {
        return red_off(tile) + (MODE == kExact ? size_t(kTileWarps) * G * D * 4 : 0);
    }
};

// Gather-average helper: adds V rows J (one per lane of `j`, the first n lanes)
// of one KV head to the lane's slice accumulator, 8 loads in flight at a time.
template <typename T, int D>
__device__ __forceinline__ void gather_rows(float (&acc)[D / 32], const T *vrow0, size_t row_stride, int j, int n,
                                            int lane) {
    constexpr int kE = D / 32;
    for (int r0 = 0; r0 < n; r0 += 8) {
        RowSlice<T, D> rows[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int jr = __shfl_sync(kFull, j, r0 + r);
            if (r0 + r < n) rows[r].load(vrow0 + size_t(jr) * row_stride, lane);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r)
            if (r0 + r < n) {
#pragma unroll
                for (int e = 0; e < kE; ++e) acc[e] += rows[r].v[e];
            }
    }
}

template <int MODE, typename T, int D, int G>
__global__ void __launch_bounds__(kTileWarps * 32)
    tile_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap, const Params p) {
    using Geo = TileGeom<T, D>;
    using Lay = TileSmem<T, D, G, MODE>;
    constexpr int kE = D / 32;
    const int t = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = p.tile;
    const int hq0 = kvh * G;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stage = smem + Lay::stage_off();
    float *xs = reinterpret_cast<float *>(smem + Lay::xs_off());
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::bars_off(tile));
    int *s_fail = reinterpret_cast<int *>(bars + kStages);

    // The dependent kernel (prop pass 2 / merge) may become resident as this grid drains;
    // it waits on pdl_wait() before touching anything written here.
    pdl_launch_dependents();

    if constexpr (MODE == kProp) {
        if (t == 0 && tid < G) p.tickets[size_t(b) * p.Hq + hq0 + tid] = 0u;
    }

    long long start;
    const int L = seq_bounds(p, b, &start);
    const int Tb = (L + tile - 1) / tile;
    if (t >= Tb) return;
    const int k0 = t * tile;
    const int len = min(tile, L - k0);
    const long long tok0 = start + k0;
    const int nk = (len + kChunk - 1) / kChunk;
    const int nchunks = (MODE == kExact) ? 2 * nk : nk;

    if (tid == 0) {
        prefetch_tensormap(&kmap);
        if (MODE == kExact) prefetch_tensormap(&vmap);
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        s_fail[0] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // Chunk c < nk is K rows [32c, 32c+32) of the tile; c >= nk (exact) the same rows of V.
    auto issue = [&](int c) {
        const int slot = c % kStages;
        const bool is_v = (MODE == kExact) && c >= nk;
        const int row = int(tok0) + (is_v ? c - nk : c) * kChunk;
        mbar_arrive_expect_tx(&bars[slot], Geo::kChunkBytes);
        tma_load_3d(stage + slot * Geo::kChunkBytes, is_v ? &vmap : &kmap, &bars[slot], 0, kvh, row);
    };
    int issued = 0;
    if (tid == 0) {
        issued = min(kStages, nchunks);
        for (int c = 0; c < issued; ++c) issue(c);
    }
    auto wait_chunk = [&](int c) {
        if (s_fail[0]) return;  // after a timeout nothing more is awaited
        if (!mbar_wait(&bars[c % kStages], (c / kStages) & 1)) s_fail[0] = 1;
    };
    auto release_chunk = [&](int c) {  // call after a __syncthreads: every warp is done with slot c
        if (tid == 0 && c + kStages < nchunks && !s_fail[0]) {
            fence_proxy_async_smem();
            issue(c + kStages);
            issued = c + kStages + 1;
        }
    };

    // q of the G heads: this lane's 16-byte vectors l8, l8 + 8, ... of the row, as float pairs.
    const int l8 = lane & 7, grp = lane >> 3;
    float2 qv[G][Geo::kVecsPerLane * Geo::kPairs];
    {
        const T *qb = static_cast<const T *>(p.q) + (size_t(b) * p.Hq + hq0) * D;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int i = 0; i < Geo::kVecsPerLane; ++i)
#pragma unroll
                for (int pp = 0; pp < Geo::kPairs; ++pp) {
                    const int e = (l8 + 8 * i) * (2 * Geo::kPairs) + 2 * pp;
                    qv[h][i * Geo::kPairs + pp] = make_float2(to_float<T>(qb[h * D + e]), to_float<T>(qb[h * D + e + 1]));
                }
    }

    // ---- scores: warp w takes keys 8w..8w+7 of each chunk, 8 lanes per key, two keys per pass
    for (int c = 0; c < nk; ++c) {
        wait_chunk(c);
        const unsigned char *base = stage + (c % kStages) * Geo::kChunkBytes;
        float dot[2][G];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const unsigned char *row = base + (warp * 8 + s * 4 + grp) * Geo::kRowBytes;
            float2 acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < Geo::kVecsPerLane; ++i) {
                const uint4 r = *reinterpret_cast<const uint4 *>(row + (l8 + 8 * i) * 16);
                float2 kv[Geo::kPairs];
                Vec16<T>::unpack(r, kv);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int pp = 0; pp < Geo::kPairs; ++pp)
                        acc[h] = __ffma2_rn(qv[h][i * Geo::kPairs + pp], kv[pp], acc[h]);
            }
#pragma unroll
            for (int h = 0; h < G; ++h) dot[s][h] = acc[h].x + acc[h].y;
        }
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float v = dot[s][h];
                v += __shfl_xor_sync(kFull, v, 4);
                v += __shfl_xor_sync(kFull, v, 2);
                v += __shfl_xor_sync(kFull, v, 1);
                dot[s][h] = v;
            }
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int kidx = c * kChunk + warp * 8 + s * 4 + grp;
            if (kidx < len) {
#pragma unroll
                for (int h = 0; h < G; ++h)
                    if (l8 == h) xs[h * tile + kidx] = dot[s][h] * p.scale;
            }
        }
        __syncthreads();
        release_chunk(c);
    }

    // ---- per-head tile statistics: m_t, e_i = exp(x_i - m_t), z_t (+ the flash sampler)
    for (int h = warp; h < G; h += kTileWarps) {
        float *xh = xs + h * tile;
        float m = -INFINITY;
        for (int i = lane; i < len; i += 32) m = fmaxf(m, xh[i]);
        m = warp_max(m);
        TileScan sc;
        float *srow = nullptr;
        if constexpr (MODE == kProp) srow = p.stash + size_t(hq0 + h) * p.total_tokens + tok0;
        for (int i0 = 0; i0 < len; i0 += 32) {
            const int i = i0 + lane;
            const float e = (i < len) ? __expf(xh[i] - m) : 0.f;
            const float P = sc.step(e, i, lane);
            if (i < len) {
                if constexpr (MODE == kProp) srow[i] = e;
                if constexpr (MODE == kExact) xh[i] = e;
                if constexpr (MODE == kFlash) xh[i] = P;
            }
        }
        sc.finish();
        const float z = sc.carry;
        const size_t rec = (size_t(b) * p.Hq + hq0 + h) * p.Tmax + t;
        if (lane == 0) {
            p.rec_m[rec] = m;
            p.rec_z[rec] = z;
            if (p.dbg_tile_m) p.dbg_tile_m[rec] = m;
            if (p.dbg_tile_z) p.dbg_tile_z[rec] = z;
        }
        if constexpr (MODE == kFlash) {
            __syncwarp();
            const int S_loc = (p.S + Tb - 1) / Tb;
            const float Ut = load_offset(p, b, hq0 + h) * float(p.S) / float(S_loc);
            const size_t vstride = size_t(p.Hkv) * D;
            const T *vrow0 = static_cast<const T *>(p.v) + size_t(tok0) * vstride + size_t(kvh) * D;
            float acc[kE];
#pragma unroll
            for (int e = 0; e < kE; ++e) acc[e] = 0.f;
            for (int s0 = 0; s0 < S_loc; s0 += 32) {
                const int s = s0 + lane;
                int j = 0;
                if (s < S_loc) {
                    const float thr = Ut + float(s) / float(S_loc);
                    j = cdf_search(xh, len, thr * z, sc.last_pos);
                    if (p.dbg_idx && s < p.dbg_stride) p.dbg_idx[rec * p.dbg_stride + s] = k0 + j;
                }
                gather_rows<T, D>(acc, vrow0, vstride, j, min(32, S_loc - s0), lane);
            }
            const float inv = 1.0f / float(S_loc);
#pragma unroll
            for (int e = 0; e < kE; ++e) p.partial[rec * D + lane * kE + e] = acc[e] * inv;
            if (p.dbg_count && lane == 0) p.dbg_count[rec] = S_loc;
        }
    }

    // ---- exact: stream the tile's V rows, o_t = sum_i e_i V_i per head
    if constexpr (MODE == kExact) {
        __syncthreads();  // e of every head is in xs
        float acc[G][kE];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < kE; ++e) acc[h][e] = 0.f;
        for (int c = nk; c < nchunks; ++c) {
            wait_chunk(c);
            const unsigned char *base = stage + (c % kStages) * Geo::kChunkBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int key = warp * 8 + kk;
                const int kidx = (c - nk) * kChunk + key;
                if (kidx < len) {
                    RowSlice<T, D> r;
                    r.load_shared(base + key * Geo::kRowBytes, lane);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float e = xs[h * tile + kidx];
#pragma unroll
                        for (int q = 0; q < kE; ++q) acc[h][q] = fmaf(e, r.v[q], acc[h][q]);
                    }
                }
            }
            __syncthreads();
            release_chunk(c);
        }
        float *red = reinterpret_cast<float *>(smem + Lay::red_off(tile));
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int q = 0; q < kE; ++q) red[(warp * G + h) * D + lane * kE + q] = acc[h][q];
        __syncthreads();
        for (int idx = tid; idx < G * D; idx += kTileWarps * 32) {
            const int h = idx / D, dd = idx % D;
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kTileWarps; ++w) s += red[(w * G + h) * D + dd];
            p.partial[((size_t(b) * p.Hq + hq0 + h) * p.Tmax + t) * D + dd] = s;
        }
    }

    // ---- a timed-out wait: flag it, and let copies still in flight land before exiting
    __syncthreads();
    if (tid == 0 && s_fail[0]) {
        raise_flag(p, SANTA_ERR_TIMEOUT);
        const long long t0 = clock64();
        for (int c = max(0, issued - kStages); c < issued; ++c)
            while (!mbar_try_wait(&bars[c % kStages], (c / kStages) & 1) && clock64() - t0 < kWaitCycles) {
            }
    }
}

}  // namespace santa
