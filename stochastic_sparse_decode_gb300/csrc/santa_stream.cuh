// santa_stream.cuh -- S2ANTA-prop pass 1 as a persistent, streaming kernel.
//
// Pass 1 ("Stochastic Sparse Attention for Memory-Bound Inference", paper
// notes, Key design 2) reads the whole K cache once: per tile it computes the
// logits of the GQA group's query heads, stashes e = exp(x - m_t) and writes
// one record (m_t, z_t).  Launched as one CTA per SM, it streams:
//
//   * a "unit" is one (sequence, tile, KV head), numbered with the KV head
//     fastest; CTA c takes units c, c + C, c + 2C, ... (C CTAs, a multiple of
//     Hkv, so a CTA keeps one KV head and the CTAs move along the token rows
//     together);
//   * one producer warp walks the CTA's units and fills a ring of `ring` unit
//     slots, each split into 8 chunks of 32 rows, with 3-D TMA boxes
//     (32 rows x 128 bytes, 128-byte swizzle).  Every chunk has a "full" and an
//     "empty" mbarrier; the producer refills a slot as soon as its chunks have
//     been consumed, so loads never wait for the arithmetic.  A unit (or chunk)
//     without keys passes its barrier with a plain arrive, so the phase of
//     slot k % ring is (k / ring) & 1 for unit k.  The slot's descriptor names
//     the unit it holds, and a consumer waits for its unit to be published
//     before it waits on the chunk, so a group that runs ahead of the other
//     never mistakes the other group's phase for its own;
//   * 16 consumer warps form two groups of 8 that take alternate units; warp w
//     of a group owns chunk w, one key per lane: for each 16-byte column
//     vector of its row it widens bf16 to fp32 and accumulates, with packed
//     fp32 FMA, against q broadcast from shared memory.  Then one warp per
//     query head forms m_t, stashes e and writes (m_t, z_t).
//
// All waits -- including the consumer groups' barriers, which use mbarriers --
// are bounded; a timed-out wait raises SANTA_ERR_TIMEOUT and stops the producer.
#pragma once

#include "santa_common.cuh"
#include "santa_tile.cuh"

namespace santa {

constexpr int kStreamRows = 32;                              // rows per chunk (one per lane)
constexpr int kStreamChunks = kRoundKeys / kStreamRows;      // 8 chunks (= consumer warps) per unit
constexpr int kStreamGroups = 2;
constexpr int kStreamConsumers = kStreamGroups * kStreamChunks;  // 16 warps
constexpr int kStreamThreads = (kStreamConsumers + 1) * 32;      // + the producer warp
constexpr int kStreamBoxBytes = kStreamRows * 128;

struct UnitDesc {
    int b, t, kvh, len;
    long long start;
    int k;  // the unit this slot currently holds (-1: none yet)
    int pad;
};

template <typename T, int D, int G>
struct StreamSmem {
    using Geo = TileGeom<T, D>;
    static constexpr int kChunkBytes = Geo::kBoxes * kStreamBoxBytes;
    static __host__ __device__ size_t unit_bytes() { return size_t(kStreamChunks) * kChunkBytes; }
    static __host__ __device__ size_t q_off(int ring) { return size_t(ring) * unit_bytes(); }
    static __host__ __device__ size_t xs_off(int ring) { return q_off(ring) + size_t(kStreamGroups) * G * D * 4; }
    static __host__ __device__ size_t desc_off(int ring) {
        return xs_off(ring) + size_t(kStreamGroups) * G * kRoundKeys * 4;
    }
    static __host__ __device__ size_t bars_off(int ring) { return desc_off(ring) + size_t(ring) * sizeof(UnitDesc); }
    static __host__ __device__ size_t bytes(int ring) {
        return 1024 + bars_off(ring) + size_t(ring) * kStreamChunks * 2 * 8 + kStreamGroups * 8 + 16;
    }
};

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Barrier over the 8 warps of one consumer group, on an mbarrier (arrival count
// 8, one arrive per warp) so that the wait is bounded like every other wait.
// `phase` is the caller's running parity of that barrier.
__device__ __forceinline__ void group_sync(uint64_t *bar, uint32_t &phase, int *fail) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    if (!mbar_wait(bar, phase) && !fail[0]) fail[0] = 3;
    phase ^= 1u;
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kStreamThreads, 1)
    prop_stream_kernel(const __grid_constant__ CUtensorMap kmap, const Params p, int ring) {
    using Geo = TileGeom<T, D>;
    using Lay = StreamSmem<T, D, G>;
    constexpr int kCB = Lay::kChunkBytes;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = gridDim.x, c = blockIdx.x;
    const int U = p.B * p.Tmax * p.Hkv;  // fits in int: checked by the host
    const int K = U > c ? (U - c + C - 1) / C : 0;  // units of this CTA

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~uintptr_t(1023));
    UnitDesc *desc = reinterpret_cast<UnitDesc *>(smem + Lay::desc_off(ring));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::bars_off(ring));  // [ring][8]
    uint64_t *empty = full + ring * kStreamChunks;                              // [ring][8]
    uint64_t *gbar = empty + ring * kStreamChunks;                              // [2] group barriers
    int *s_fail = reinterpret_cast<int *>(gbar + kStreamGroups);  // 0, or where the first wait gave up

    pdl_launch_dependents();
    if (tid < ring * kStreamChunks) {
        mbar_init(&full[tid], 1);
        mbar_init(&empty[tid], 1);
    }
    if (tid < kStreamGroups) mbar_init(&gbar[tid], kStreamChunks);
    if (tid < ring) desc[tid].k = -1;
    if (tid == 0) {
        s_fail[0] = 0;
        prefetch_tensormap(&kmap);
    }
    fence_barrier_init();
    __syncthreads();

    if (warp == kStreamConsumers) {
        // ---------------- producer
        if (lane == 0) {
            int cb = -1, cL = 0;
            long long cstart = 0;
            for (int k = 0; k < K && !s_fail[0]; ++k) {  // after any timeout, stop issuing
                const int slot = k % ring;
                if (k >= ring) {  // every chunk of unit k - ring has been consumed
                    for (int w = 0; w < kStreamChunks && !s_fail[0]; ++w)
                        if (!mbar_wait(&empty[slot * kStreamChunks + w], ((k / ring) - 1) & 1)) s_fail[0] = 1;
                    if (s_fail[0]) break;
                }
                const int u = c + k * C;
                const int kvh = u % p.Hkv, r = u / p.Hkv, t = r % p.Tmax, b = r / p.Tmax;
                if (b != cb) {
                    cL = seq_bounds(p, b, &cstart);
                    cb = b;
                }
                const int len = t * p.tile < cL ? min(p.tile, cL - t * p.tile) : 0;
                desc[slot] = UnitDesc{b, t, kvh, len, cstart, k, 0};
                fence_proxy_async_smem();
                for (int w = 0; w < kStreamChunks; ++w) {
                    uint64_t *bar = &full[slot * kStreamChunks + w];
                    if (len > kStreamRows * w && !s_fail[0]) {
                        unsigned char *dst = smem + size_t(slot) * Lay::unit_bytes() + size_t(w) * kCB;
                        const int row = int(cstart) + t * p.tile + w * kStreamRows;
                        mbar_arrive_expect_tx(bar, kCB);
#pragma unroll
                        for (int bx = 0; bx < Geo::kBoxes; ++bx)
                            tma_load_3d(dst + bx * kStreamBoxBytes, &kmap, bar, bx * Geo::kBoxElems, kvh, row);
                    } else {
                        mbar_arrive(bar);
                    }
                }
            }
        }
    } else {
        // ---------------- consumers: group grp, chunk (warp) w
        const int grp = warp / kStreamChunks, w = warp % kStreamChunks;
        const int gtid = tid % (kStreamChunks * 32);
        float *qs = reinterpret_cast<float *>(smem + Lay::q_off(ring)) + grp * G * D;
        float *xs = reinterpret_cast<float *>(smem + Lay::xs_off(ring)) + grp * G * kRoundKeys;
        int qb = -1, qkvh = -1;  // whose q the group's buffer holds
        uint32_t gphase = 0;
        for (int k = grp; k < K; k += kStreamGroups) {
            const int slot = k % ring;
            const uint32_t par = (k / ring) & 1;
            // The two groups share the ring, so this warp may arrive here while the
            // slot still holds unit k - ring (the other group's).  A parity wait cannot
            // tell that phase from unit k's, so first wait until the producer has
            // published unit k in the slot -- it does so only after unit k - ring has
            // left it -- and only then wait for the chunk itself.
            if (!s_fail[0]) {
                const volatile int *slot_k = &desc[slot].k;
                const long long t0 = clock64();
                while (*slot_k != k) {
                    if (clock64() - t0 > kWaitCycles) {
                        s_fail[0] = 4;
                        break;
                    }
                    __nanosleep(64);
                }
            }
            if (!s_fail[0] && !mbar_wait(&full[slot * kStreamChunks + w], par)) s_fail[0] = 2;
            const UnitDesc du = desc[slot];
            const int hq0 = du.kvh * G;

            // scores of row `lane` of chunk w (then hand the chunk back to the producer)
            float2 acc[G][2];
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h][0] = acc[h][1] = make_float2(0.f, 0.f);
            const bool have = du.len > kStreamRows * w;
            if (du.len > 0 && (du.b != qb || du.kvh != qkvh)) {
                group_sync(&gbar[grp], gphase, s_fail);  // group-uniform branch: nobody still reads the old q
                const T *qsrc = static_cast<const T *>(p.q) + (size_t(du.b) * p.Hq + hq0) * D;
                for (int i = gtid; i < G * D; i += kStreamChunks * 32) qs[i] = to_float<T>(qsrc[i]);
                qb = du.b;
                qkvh = du.kvh;
                group_sync(&gbar[grp], gphase, s_fail);
            }
            if (have) {
                const unsigned char *base = smem + size_t(slot) * Lay::unit_bytes() + size_t(w) * kCB;
#pragma unroll
                for (int j = 0; j < Geo::kNJ; ++j) {
                    const uint32_t o =
                        uint32_t((j >> 3) * kStreamBoxBytes + lane * 128 + (((j & 7) ^ (lane & 7)) << 4));
                    const uint4 raw = *reinterpret_cast<const uint4 *>(base + o);
                    float2 kv[Geo::kPairs];
                    Vec16<T>::unpack(raw, kv);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float4 *qh = reinterpret_cast<const float4 *>(qs + h * D + j * Geo::kEV);
#pragma unroll
                        for (int i = 0; i < Geo::kPairs / 2; ++i) {
                            const float4 qq = qh[i];
                            acc[h][0] = __ffma2_rn(make_float2(qq.x, qq.y), kv[2 * i], acc[h][0]);
                            acc[h][1] = __ffma2_rn(make_float2(qq.z, qq.w), kv[2 * i + 1], acc[h][1]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot * kStreamChunks + w]);
            const int key = w * kStreamRows + lane;
            if (key < du.len) {
#pragma unroll
                for (int h = 0; h < G; ++h)
                    xs[h * kRoundKeys + key] = ((acc[h][0].x + acc[h][0].y) + (acc[h][1].x + acc[h][1].y)) * p.scale;
            }
            group_sync(&gbar[grp], gphase, s_fail);

            // tile statistics, one warp per query head: m_t, the stash of e, z_t
            if (du.len > 0) {
                for (int h = w; h < G; h += kStreamChunks) {
                    const float *xh = xs + h * kRoundKeys;
                    float m = -INFINITY;
                    for (int i = lane; i < du.len; i += 32) m = fmaxf(m, xh[i]);
                    m = warp_max(m);
                    float *srow = p.stash + size_t(hq0 + h) * p.total_tokens + du.start + size_t(du.t) * p.tile;
                    float zl = 0.f;
                    for (int i = lane; i < du.len; i += 32) {
                        const float e = __expf(xh[i] - m);
                        srow[i] = e;
                        zl += e;
                    }
                    const float z = warp_sum(zl);
                    if (lane == 0) {
                        const size_t rec = (size_t(du.b) * p.Hq + hq0 + h) * p.Tmax + du.t;
                        p.rec_m[rec] = m;
                        p.rec_z[rec] = z;
                        if (p.dbg_tile_m) p.dbg_tile_m[rec] = m;
                        if (p.dbg_tile_z) p.dbg_tile_z[rec] = z;
                    }
                }
            }
            group_sync(&gbar[grp], gphase, s_fail);  // xs is free for the group's next unit
        }
    }

    // ---- a timed-out wait: flag it, and let copies still in flight land before exiting
    __syncthreads();
    if (s_fail[0] && tid == 0) {
        // SANTA_ERR_TIMEOUT, plus where the first wait gave up: 1 producer (empty slot),
        // 2 consumer (full chunk), 3 group barrier, 4 consumer (slot not yet published)
        // -- in bits 8..11.
        raise_flag(p, SANTA_ERR_TIMEOUT | (unsigned(s_fail[0]) << 8));
        const long long t0 = clock64();
        for (int k = K > ring ? K - ring : 0; k < K; ++k)
            for (int w = 0; w < kStreamChunks; ++w)
                while (!mbar_try_wait(&full[(k % ring) * kStreamChunks + w], (k / ring) & 1) &&
                       clock64() - t0 < kWaitCycles) {
                }
    }
}

}  // namespace santa
