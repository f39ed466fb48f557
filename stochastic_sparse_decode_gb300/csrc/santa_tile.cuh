// santa_tile.cuh -- the split-KV tile kernel of S2ANTA-flash, and geometry
// shared with the streaming kernels.
//
// One CTA owns one (sequence b, KV head, tile t) and all G query heads of that
// KV head's GQA group, so each K row is read once for G heads.  The CTA's four
// warps split the tile into 64-row chunks (chunk w of every 256-key round goes
// to warp w); each warp streams its chunks through its own shared-memory slots,
// filled by 3-D TMA boxes of 64 rows x 128 bytes with the 128-byte swizzle, and
// waits on its own mbarriers -- no CTA-wide barrier in the streaming loop.
//
// A lane owns whole keys (rows l and l + 32 of its warp's chunk), so a dot
// product never crosses lanes: for each 16-byte column vector j of the row the
// lane reads its two rows' vectors (the swizzle makes a column read by 32 lanes
// conflict-free), widens bf16 to fp32 and accumulates with packed fp32 FMA
// against q, which all lanes read from shared memory as a broadcast.
//
// With the scores x = q.k / sqrt(d) of the tile in shared memory, one warp per
// query head forms the tile's max m_t, the exponentiated scores
// e_i = exp(x_i - m_t) and their sum z_t -- the tile's partition sum Z_tile on
// the m_t scale ("Stochastic Sparse Attention for Memory-Bound Inference", paper
// notes, Key design 2: exponentiated scores plus one Z_tile per tile).  Then it
// samples S_loc = ceil(S / T_b) systematic thresholds U_t + s/S_loc,
// U_t = U S / S_loc, on the tile's own CDF (its prefix of e divided by z_t),
// gather-averages the chosen V rows into the tile estimate and writes it with
// (m_t, z_t) for the merge (Key design 3).
#pragma once

#include "santa_common.cuh"

namespace santa {

constexpr int kBoxBytes = kWarpRows * 128;           // one TMA box: 64 rows x 128 bytes
constexpr int kRoundKeys = kTileWarps * kWarpRows;   // keys per round of the CTA

template <typename T, int D>
struct TileGeom {
    static constexpr int kES = int(sizeof(T));
    static constexpr int kRowBytes = D * kES;        // 128, 256 or 512
    static constexpr int kBoxes = kRowBytes / 128;   // 128-byte column boxes per row
    static constexpr int kBoxElems = 128 / kES;      // elements per box row
    static constexpr int kEV = 16 / kES;             // elements per 16-byte vector
    static constexpr int kPairs = kEV / 2;           // float pairs per 16-byte vector
    static constexpr int kNJ = D / kEV;              // 16-byte vectors per row
    static constexpr int kChunkBytes = kBoxes * kBoxBytes;
};

// Byte offset of 16-byte vector j of row r (0..63) in a chunk: box j/8, and
// inside it the 128-byte swizzle (vector c of row r sits at c ^ (r mod 8)).
__device__ __forceinline__ uint32_t swz(int r, int j) {
    return uint32_t((j >> 3) * kBoxBytes + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

// Shared-memory layout of a tile CTA (identical on host and device).  Offsets
// are from a 1024-byte aligned base; `bytes` includes the alignment slack.
template <typename T, int D, int G>
struct TileSmem {
    static __host__ __device__ int nslot(int tile) { return tile > kRoundKeys ? 2 : 1; }
    static __host__ __device__ size_t q_off(int tile) {
        return size_t(kTileWarps) * nslot(tile) * TileGeom<T, D>::kChunkBytes;
    }
    static __host__ __device__ size_t xs_off(int tile) { return q_off(tile) + size_t(G) * D * 4; }
    static __host__ __device__ size_t es_off(int tile) { return xs_off(tile) + size_t(G) * tile * 4; }
    static __host__ __device__ size_t bars_off(int tile) { return es_off(tile); }
    static __host__ __device__ size_t red_off(int tile) { return bars_off(tile) + kTileWarps * 2 * 8 + 16; }
    static __host__ __device__ size_t bytes(int tile) {
        return 1024 + red_off(tile);
    }
};

// Gather-average helper: adds V rows J (one per lane of `j`, the first n lanes)
// of one KV head to the lane's slice accumulator, up to 16 loads in flight.
template <typename T, int D>
__device__ __forceinline__ void gather_rows(float (&acc)[D / 32], const T *vrow0, size_t row_stride, int j, int n,
                                            int lane) {
    constexpr int kE = D / 32;
    for (int r0 = 0; r0 < n; r0 += 16) {
        RowSlice<T, D> rows[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int jr = __shfl_sync(kFull, j, (r0 + r) & 31);
            if (r0 + r < n) rows[r].load(vrow0 + size_t(jr) * row_stride, lane);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r)
            if (r0 + r < n) {
#pragma unroll
                for (int e = 0; e < kE; ++e) acc[e] += rows[r].v[e];
            }
    }
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kTileWarps * 32) tile_kernel(const __grid_constant__ CUtensorMap kmap, const Params p) {
    using Geo = TileGeom<T, D>;
    using Lay = TileSmem<T, D, G>;
    constexpr int kE = D / 32;
    // KV head fastest: the Hkv CTAs of one tile are scheduled together and read
    // the same token rows, so each DRAM page is streamed by them at once.
    const int kvh = blockIdx.x, t = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = p.tile;
    const int hq0 = kvh * G;
    const int nslot = Lay::nslot(tile);

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~uintptr_t(1023));
    float *qs = reinterpret_cast<float *>(smem + Lay::q_off(tile));
    float *xs = reinterpret_cast<float *>(smem + Lay::xs_off(tile));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::bars_off(tile));
    int *s_fail = reinterpret_cast<int *>(bars + kTileWarps * 2);

    // The dependent kernel (prop pass 2 / merge) may become resident as this grid drains;
    // it waits on pdl_wait() before touching anything written here.
    pdl_launch_dependents();

    // q of the group's G heads: loads issued before the sequence bounds are known.
    constexpr int kQPerThread = (G * D + kTileWarps * 32 - 1) / (kTileWarps * 32);
    float qreg[kQPerThread];
    {
        const T *qb = static_cast<const T *>(p.q) + (size_t(b) * p.Hq + hq0) * D;
#pragma unroll
        for (int k = 0; k < kQPerThread; ++k) {
            const int i = tid + k * kTileWarps * 32;
            qreg[k] = i < G * D ? to_float<T>(qb[i]) : 0.f;
        }
    }

    long long start;
    const int L = seq_bounds(p, b, &start);
    const int Tb = (L + tile - 1) / tile;
    if (t >= Tb) return;
    const int k0 = t * tile;
    const int len = min(tile, L - k0);
    const long long tok0 = start + k0;

    // This warp's chunks: rounds r with keys 256 r + 64 warp < len.
    const int nr = len > kWarpRows * warp ? (len - kWarpRows * warp + kRoundKeys - 1) / kRoundKeys : 0;
    const int nch = nr;
    unsigned char *wslots = smem + size_t(warp) * nslot * Geo::kChunkBytes;
    uint64_t *wbars = bars + warp * 2;

    if (lane == 0) {
        for (int s = 0; s < nslot; ++s) mbar_init(&wbars[s], 1);
        fence_barrier_init();
    }
    if (tid == 0) s_fail[0] = 0;
    __syncthreads();

    auto issue = [&](int c) {  // lane 0 only
        const int slot = c % nslot;
        const int row = int(tok0) + c * kRoundKeys + warp * kWarpRows;
        unsigned char *dst = wslots + slot * Geo::kChunkBytes;
        mbar_arrive_expect_tx(&wbars[slot], Geo::kChunkBytes);
#pragma unroll
        for (int bx = 0; bx < Geo::kBoxes; ++bx)
            tma_load_3d(dst + bx * kBoxBytes, &kmap, &wbars[slot], bx * Geo::kBoxElems, kvh, row);
    };
    int issued = 0;
    if (lane == 0) {
        issued = min(nslot, nch);
        for (int c = 0; c < issued; ++c) issue(c);
    }
    auto wait_chunk = [&](int c) {
        if (s_fail[0]) return;  // after a timeout nothing more is awaited
        if (!mbar_wait(&wbars[c % nslot], (c / nslot) & 1)) s_fail[0] = 1;
    };
    auto release_chunk = [&](int c) {  // every lane of the warp is done with chunk c
        __syncwarp();
        if (lane == 0 && c + nslot < nch && !s_fail[0]) {
            fence_proxy_async_smem();
            issue(c + nslot);
            issued = c + nslot + 1;
        }
    };

    // q, widened to fp32, in shared memory for broadcast reads.
#pragma unroll
    for (int k = 0; k < kQPerThread; ++k) {
        const int i = tid + k * kTileWarps * 32;
        if (i < G * D) qs[i] = qreg[k];
    }
    __syncthreads();

    // ---- scores of this warp's keys: lane owns rows `lane` and `lane + 32` of each chunk
    for (int r = 0; r < nr; ++r) {
        wait_chunk(r);
        const unsigned char *base = wslots + (r % nslot) * Geo::kChunkBytes;
        float2 acc0[G], acc1[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            acc0[h] = make_float2(0.f, 0.f);
            acc1[h] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < Geo::kNJ; ++j) {
            const uint32_t o = swz(lane, j);
            const uint4 ra = *reinterpret_cast<const uint4 *>(base + o);
            const uint4 rb = *reinterpret_cast<const uint4 *>(base + o + 32 * 128);
            float2 ka[Geo::kPairs], kb[Geo::kPairs];
            Vec16<T>::unpack(ra, ka);
            Vec16<T>::unpack(rb, kb);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float4 *qh = reinterpret_cast<const float4 *>(qs + h * D + j * Geo::kEV);
#pragma unroll
                for (int i = 0; i < Geo::kPairs / 2; ++i) {
                    const float4 qq = qh[i];
                    const float2 q0 = make_float2(qq.x, qq.y), q1 = make_float2(qq.z, qq.w);
                    acc0[h] = __ffma2_rn(q0, ka[2 * i], acc0[h]);
                    acc1[h] = __ffma2_rn(q0, kb[2 * i], acc1[h]);
                    acc0[h] = __ffma2_rn(q1, ka[2 * i + 1], acc0[h]);
                    acc1[h] = __ffma2_rn(q1, kb[2 * i + 1], acc1[h]);
                }
            }
        }
        release_chunk(r);
        const int key0 = r * kRoundKeys + warp * kWarpRows + lane;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            if (key0 < len) xs[h * tile + key0] = (acc0[h].x + acc0[h].y) * p.scale;
            if (key0 + 32 < len) xs[h * tile + key0 + 32] = (acc1[h].x + acc1[h].y) * p.scale;
        }
    }
    __syncthreads();

    // ---- per-head tile statistics: m_t, the in-tile prefix of e_i = exp(x_i - m_t), z_t
    for (int h = warp; h < G; h += kTileWarps) {
        float *xh = xs + h * tile;
        float m = -INFINITY;
        for (int i = lane; i < len; i += 32) m = fmaxf(m, xh[i]);
        m = warp_max(m);
        TileScan sc;
        for (int i0 = 0; i0 < len; i0 += 32) {
            const int i = i0 + lane;
            const float e = (i < len) ? __expf(xh[i] - m) : 0.f;
            const float P = sc.step(e, i, lane);
            if (i < len) xh[i] = P;
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
        {  // the tile's local systematic sample
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

    // ---- a timed-out wait: flag it, and let copies still in flight land before exiting
    __syncthreads();
    if (lane == 0 && s_fail[0]) {
        if (warp == 0) raise_flag(p, SANTA_ERR_TIMEOUT);
        const long long t0 = clock64();
        for (int c = max(0, issued - nslot); c < issued; ++c)
            while (!mbar_try_wait(&wbars[c % nslot], (c / nslot) & 1) && clock64() - t0 < kWaitCycles) {
            }
    }
}

}  // namespace santa
