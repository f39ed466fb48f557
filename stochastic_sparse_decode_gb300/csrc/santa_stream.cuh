// santa_stream.cuh -- S2ANTA-prop pass 1 as a persistent, streaming kernel.
//
// Pass 1 ("Stochastic Sparse Attention for Memory-Bound Inference", paper
// notes, Key design 2) reads the whole K cache once, stashes the exponentiated
// scores and leaves one partition record per block of keys.  Here the block is
// a "chunk" of 32 consecutive keys of one sequence (a tile is tile/32 chunks):
// per chunk and query head the record is (m_c, z_c), m_c the chunk's largest
// logit and z_c = sum_i exp(x_i - m_c), and the stash holds e_i = exp(x_i - m_c).
// Pass 2 places the systematic thresholds on the CDF assembled from these
// records; because prop samples the one global CDF, the sample does not depend
// on how finely the records cut the keys, and chunk records let every warp
// finish its keys on its own.
//
// Launched as one CTA of kChunkWarps warps per SM (C CTAs, a multiple of Hkv).
// Chunks are numbered (sequence, chunk, KV head) with the KV head fastest; CTA
// c owns chunks c, c + C, c + 2C, ... (so all of them have one KV head and the
// CTAs move along the token rows together), and its warps claim them one at a
// time from a shared-memory counter, so the CTA's chunks, not a fixed share per
// warp, balance the work.  Each warp streams its claims through `nbuf`
// shared-memory buffers of its own, filled by 3-D TMA boxes (32 rows x 128
// bytes, 128-byte swizzle) that its lane 0 issues, one mbarrier per buffer: no
// warp ever waits for another.  A warp starts with one copy in flight and fills
// its other buffers when that copy lands, so every warp's first chunk is among
// the first bytes the memory system returns.
//
// Eight lanes share a key: lane l of a lane group holds q's slice of 16-byte
// column vectors l, l + 8, ... (the swizzle makes the eight reads of one row
// conflict-free), widens bf16 to fp32 and accumulates with packed fp32 FMA.
// A batch of 8/GH keys x GH heads gives 8 partial sums per lane, which three
// shuffle-and-add stages reduce-scatter over the lane group, so each lane ends
// with one full logit (each lane orders its heads and keys by its own index,
// so no stage needs a select).  The chunk's statistics are then warp shuffles over the
// lanes that hold the same head; e is stored straight to the stash.  With
// G * D / 8 > 64 (G = 8 at d = 128) the q slice does not fit in registers and
// the heads are taken GH at a time, re-reading the buffer.
//
// Launched with programmatic dependent launch: a CTA sets up its barriers while
// the previous kernel drains and waits for it before touching global memory.
// Every wait is bounded; a timed-out wait raises SANTA_ERR_TIMEOUT (location
// code 2 in bits 8..11), stops the warp, and lets its copies in flight land.
#pragma once

#include "santa_common.cuh"
#include "santa_tile.cuh"

namespace santa {

constexpr int kChunkRows = 32;                      // keys per chunk (one TMA box of rows)
constexpr int kChunkWarps = 12;                     // warps of a pass-1 CTA
constexpr int kChunkMaxBuf = 4;                     // buffers per warp, at most
constexpr int kChunkBoxBytes = kChunkRows * 128;    // one TMA box: 32 rows x 128 bytes

// What a buffer holds: chunk ch of sequence b (rows start + 32 ch ..), KV head, keys,
// and whether the chunk has records (its keys, or a page dropped for a bad id).
struct ChunkSlot {
    long long start;
    int b, ch, kvh, len, rec;
};

template <typename T, int D, int G>
struct ChunkGeom {
    using Geo = TileGeom<T, D>;
    static constexpr int kGH = (G * D / 8 <= 64) ? G : 64 / (D / 8);  // heads per pass over a chunk
    static constexpr int kPasses = G / kGH;
    static constexpr int kBytes = Geo::kBoxes * kChunkBoxBytes;       // one chunk of K rows
    static constexpr int kVPL = Geo::kNJ / 8;  // 16-byte vectors of a row per lane (8 lanes per key)
    static constexpr int kKB = 8 / kGH;        // keys per lane group in one reduction batch
    // shared memory: [kChunkWarps][nbuf] chunk buffers, [kChunkWarps][kChunkMaxBuf]
    // mbarriers, [kChunkWarps][kChunkMaxBuf] slot descriptors, the claim counter
    static __host__ __device__ size_t bars_off(int nbuf) { return size_t(kChunkWarps) * nbuf * kBytes; }
    static __host__ __device__ size_t slots_off(int nbuf) { return bars_off(nbuf) + size_t(kChunkWarps) * kChunkMaxBuf * 8; }
    static __host__ __device__ size_t next_off(int nbuf) {
        return slots_off(nbuf) + size_t(kChunkWarps) * kChunkMaxBuf * sizeof(ChunkSlot);
    }
    static __host__ __device__ size_t bytes(int nbuf) { return 1024 + next_off(nbuf) + 16; }
    // buffers per warp that fit in `optin` bytes of shared memory (0: none)
    static __host__ int nbuf_for(size_t optin) {
        for (int n = kChunkMaxBuf; n >= 1; --n)
            if (bytes(n) <= optin) return n;
        return 0;
    }
};

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One stage of a reduce-scatter over the 8 lanes of a lane group.  Slot s of
// lane l holds the partial sum of value s ^ l (each lane keeps its values in an
// order permuted by its own index), so for every stage the lane keeps slots
// [0, M) and hands slots [M, 2M) to its partner l ^ M, whose slot j + M holds
// the same value as this lane's slot j.  After the stages 4, 2, 1 slot 0 of
// lane l holds the full sum of value l.
template <int M>
__device__ __forceinline__ void reduce_scatter_stage(float (&v)[8]) {
#pragma unroll
    for (int j = 0; j < M; ++j) v[j] += __shfl_xor_sync(kFull, v[j + M], M);
}

// Max / sum over the lanes that hold the same head: lanes whose indices differ
// only in bits >= log2(GH).
template <int GH>
__device__ __forceinline__ float head_max(float v) {
#pragma unroll
    for (int o = GH; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
template <int GH>
__device__ __forceinline__ float head_sum(float v) {
#pragma unroll
    for (int o = GH; o < 32; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// This lane's slice of q for heads h0 .. h0 + GH - 1 of sequence b: 16-byte
// column vectors l8, l8 + 8, ... of each head, as float pairs; slot h holds
// head h0 + (h ^ hx) (the lane's head permutation of the reduce-scatter).
template <typename T, int D, int GH, int VPL, int PAIRS>
__device__ __forceinline__ void load_q_slice(const Params &p, int b, int hq0, int l8, int hx,
                                             float2 (&qreg)[GH][VPL * PAIRS]) {
    using Geo = TileGeom<T, D>;
    const T *qh = static_cast<const T *>(p.q) + (size_t(b) * p.Hq + hq0) * D;
#pragma unroll
    for (int h = 0; h < GH; ++h)
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(qh + (h ^ hx) * D + (l8 + 8 * i) * Geo::kEV));
            Vec16<T>::unpack(raw, &qreg[h][i * PAIRS]);
        }
}

// bf16 keys take their logits from the tensor cores: per chunk, the 32 keys
// are the A operand (two 16-key tiles, 16 dimensions per fragment, read from the
// swizzled buffer with ldmatrix) and q is the B operand (16 dimensions x 8
// heads, heads >= G zero), so a chunk costs 2 D/16 ldmatrix + mma pairs instead
// of G D / 8 packed FMAs per lane.  Products of bf16 values are exact in fp32;
// only the order of the fp32 additions differs from a plain dot product.
//
// The B fragments of q for heads hq0 .. hq0 + G - 1 of sequence b: lane
// (g = lane / 4, t = lane % 4) holds dimensions 16 ks + 2t, +1 and 16 ks + 2t + 8,
// +9 of head hq0 + g.
template <int D, int G>
__device__ __forceinline__ void load_q_frag(const Params &p, int b, int hq0, int lane, uint32_t (&qf)[D / 16][2]) {
    const int g = lane >> 2, t = lane & 3;
    const uint32_t *qh = reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(p.q) +
                                                            (size_t(b) * p.Hq + hq0 + min(g, G - 1)) * D);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        qf[ks][0] = g < G ? __ldg(qh + 8 * ks + t) : 0u;
        qf[ks][1] = g < G ? __ldg(qh + 8 * ks + 4 + t) : 0u;
    }
}

// Unscaled logits of the chunk in `base` (32 rows of D bf16 in boxes of 128-byte
// rows, 128-byte swizzle).  Lane (g, t) ends with c[mt][2 half + j] = q_{2t + j} .
// k_r for key r = 16 mt + 8 half + g.  The loads are all issued before the
// first product.
template <int D>
__device__ __forceinline__ void chunk_logits_mma(const unsigned char *base, const uint32_t (&qf)[D / 16][2], int lane,
                                                 float (&c)[2][4]) {
    constexpr int kKS = D / 16;
    const int rl = lane & 15, kx = lane >> 4;
    uint32_t a[2][kKS][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        const int r = mt * 16 + rl;  // lanes 0-7 / 8-15 / 16-23 / 24-31: matrices of rows 0-7, 8-15 at d 0-7, 8-15
#pragma unroll
        for (int ks = 0; ks < kKS; ++ks) {
            const int kv = 2 * ks + kx;  // 16-byte vector of the row: box kv / 8, swizzled slot (kv mod 8) ^ (r mod 8)
            ldmatrix_x4(a[mt][ks], base + (kv >> 3) * kChunkBoxBytes + r * 128 + (((kv & 7) ^ (r & 7)) << 4));
        }
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) c[mt][i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) mma_bf16_16816(c[mt], a[mt][ks], qf[ks]);
}

// Shared memory of the streaming warps, from a 1024-byte aligned base: [kChunkWarps][nbuf]
// chunk buffers, then per warp kChunkMaxBuf mbarriers and slot descriptors, then the
// CTA's claim counter.  Initialised by stream_setup, used by stream_chunks.
__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
    return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Barrier and counter initialisation of the streaming warps (warps 0 .. kChunkWarps - 1);
// the caller makes it visible with a CTA barrier before stream_chunks.
template <typename T, int D, int G>
__device__ __forceinline__ void stream_setup(const CUtensorMap &kmap, unsigned char *smem, int nbuf) {
    using CG = ChunkGeom<T, D, G>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < kChunkWarps && lane < nbuf)
        mbar_init(reinterpret_cast<uint64_t *>(smem + CG::bars_off(nbuf)) + warp * kChunkMaxBuf + lane, 1);
    if (threadIdx.x == 0) {
        *reinterpret_cast<int *>(smem + CG::next_off(nbuf)) = 0;
        prefetch_tensormap(&kmap);
    }
    fence_barrier_init();
}

// Stores the partition record (m_c, z_c) of one chunk and query head as one 64-bit
// word, z in the high half (a single store, so a reader sees both halves of one
// record or neither).  A written word is never 0 -- z >= 1 (the chunk's largest key
// contributes exp(0) = 1) or NaN, and a chunk dropped for a bad page id carries
// m = -inf -- so 0 means "not written yet".
__device__ __forceinline__ void store_record(unsigned long long *rec, float m, float z) {
    const unsigned long long v = (static_cast<unsigned long long>(__float_as_uint(z)) << 32) | __float_as_uint(m);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(rec), "l"(v) : "memory");
}

// Publishes n finished chunks of KV head kvh of sequence b to the samplers of the
// group's G query heads: a fence that makes the warp's stash and record stores
// visible (every lane's stores precede the publishing lanes' fences through the
// warp barrier), then count[b][h] += n for each head h of the group.  A warp
// publishes when it leaves a (sequence, KV head) and at the end of its walk, not
// per chunk: a fence waits for the warp's stores to land, which under a saturated
// memory system costs about a microsecond of the warp's time.
template <int G>
__device__ __forceinline__ void publish_chunks(const Params &p, int b, int kvh, int n, int lane) {
    __syncwarp();
    if (lane < G) {
        __threadfence();
        atomicAdd(p.cnt + size_t(b) * p.Hq + kvh * G + lane, unsigned(n));
    }
    __syncwarp();
}

// The streaming walk of pass 1, run by warps 0 .. kChunkWarps - 1 of a CTA whose
// shared memory `smem` (1024-byte aligned) holds the streaming layout, after
// stream_setup, a CTA barrier and the kernel's dependency wait.  Returns whether a
// wait for one of the warp's copies timed out (after a bounded wait for the rest).
// kPublish (the fused kernel, whose samplers read the records while others are still
// being written): publish the finished chunks, set the heads' finished-split
// counters to 0 and store each chunk's largest-key offset.  Pass 1 alone does none
// of the three: its reader starts after it ends, and a publication fence per
// (sequence, KV head) a warp leaves measured ~25 us slower at batch 16.
template <typename T, int D, int G, bool kPaged, bool kPublish>
__device__ __forceinline__ bool stream_chunks(const CUtensorMap &kmap, const Params &p, int nbuf, unsigned char *smem) {
    using Geo = TileGeom<T, D>;
    using CG = ChunkGeom<T, D, G>;
    constexpr int kGH = CG::kGH, kVPL = CG::kVPL, kKB = CG::kKB, kPairs = Geo::kPairs;
    constexpr int kBG = kGH >= 2 ? 2 : 1;  // batches whose partial sums are reduced together
    constexpr bool kMma = sizeof(T) == 2;  // bf16 keys: logits on the tensor cores
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g8 = lane >> 3, l8 = lane & 7;
    // the lane's permutation of its reduce-scatter slots (kk, h) -> (kk ^ kx, h ^ hx)
    const int hx = l8 & (kGH - 1), kx = l8 / kGH;
    const int C = gridDim.x, c = blockIdx.x;
    const long long X = (long long)p.B * p.nch * p.Hkv;  // chunks of the batch (with empty ones)
    const long long K_cta = X > c ? (X - c + C - 1) / C : 0;  // chunks c, c + C, ... of this CTA

    unsigned char *wbuf = smem + size_t(warp) * nbuf * CG::kBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + CG::bars_off(nbuf)) + warp * kChunkMaxBuf;
    ChunkSlot *slots = reinterpret_cast<ChunkSlot *>(smem + CG::slots_off(nbuf)) + warp * kChunkMaxBuf;
    int *s_next = reinterpret_cast<int *>(smem + CG::next_off(nbuf));

    // lane 0's cache of the last sequence's bounds
    int lb = -1, lL = 0;
    long long lstart = 0;
    const bool one_kvh = C % p.Hkv == 0;  // every chunk of the CTA has KV head c % Hkv
    int n_issued = 0, n_done = 0;
    bool more = true;  // warp-uniform: the CTA's walk still has chunks to claim
    // Claims the next chunk of the CTA's walk and starts its copy into buffer
    // n_issued % nbuf; a chunk without keys completes the buffer's phase with a
    // plain arrive.  Warp-uniform.
    auto claim = [&]() {
        int i = 0;
        if (lane == 0) i = atomicAdd(s_next, 1);
        i = __shfl_sync(kFull, i, 0);
        if (i >= K_cta) {
            more = false;
            return;
        }
        if (lane == 0) {
            int kvh;
            long long r;  // b * nch + ch
            if (one_kvh) {
                kvh = c % p.Hkv;
                r = c / p.Hkv + (long long)i * (C / p.Hkv);
            } else {
                const long long x = c + (long long)i * C;
                kvh = int(x % p.Hkv);
                r = x / p.Hkv;
            }
            int b, ch;
            if (r < 0x7fffffffLL) {
                b = int(unsigned(r) / unsigned(p.nch));
                ch = int(r) - b * p.nch;
            } else {
                b = int(r / p.nch);
                ch = int(r - (long long)b * p.nch);
            }
            if (b != lb) {
                lL = seq_bounds<kPaged>(p, b, &lstart);
                lb = b;
            }
            int len = min(kChunkRows, lL - ch * kChunkRows);
            int rec = len > 0 ? 1 : 0;
            // the group's finished-split counters start this call at 0 (published with
            // the chunk, before any split of the head can count itself in)
            if (kPublish && ch == 0)
                for (int h = 0; h < G; ++h) p.done[size_t(b) * p.Hq + kvh * G + h] = 0u;
            long long row = lstart + ch * kChunkRows;
            if (kPaged && len > 0) {
                row = key_row<kPaged>(p, b, lstart, ch * kChunkRows);  // a chunk never straddles pages
                if (row < 0) {  // bad page id (flagged): the chunk carries no mass
                    for (int h = 0; h < G; ++h)
                        store_record(p.rec + (size_t(b) * p.Hq + kvh * G + h) * p.nch + ch, -INFINITY, 0.f);
                    len = 0;
                    rec = 1;
                }
            }
            const int slot = n_issued % nbuf;
            slots[slot] = ChunkSlot{lstart, b, ch, kvh, len, rec};
            uint64_t *bar = &bars[slot];
            if (len > 0) {
                unsigned char *dst = wbuf + size_t(slot) * CG::kBytes;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, CG::kBytes);
#pragma unroll
                for (int bx = 0; bx < Geo::kBoxes; ++bx)
                    tma_load_3d_hint(dst + bx * kChunkBoxBytes, &kmap, bar, bx * Geo::kBoxElems, kvh, int(row),
                                     l2_evict_first());
            } else {
                mbar_arrive(bar);
            }
        }
        ++n_issued;
    };
    claim();  // one copy per warp at first
    __syncwarp();

    // q of the first chunk is loaded while its keys are in flight
    float2 qreg[kGH][kVPL * kPairs];
    uint32_t qf[D / 16][2];
    int qb = -1, qkvh = -1;  // whose q the registers hold (one pass only)
    if ((kMma || CG::kPasses == 1) && n_issued > 0) {
        qb = slots[0].b;
        qkvh = slots[0].kvh;
        if constexpr (kMma)
            load_q_frag<D, G>(p, qb, qkvh * G, lane, qf);
        else
            load_q_slice<T, D, kGH, kVPL, kPairs>(p, qb, qkvh * G, l8, hx, qreg);
    }

    bool failed = false;
    // Chunks of the current (sequence, KV head) whose records are stored but not yet
    // published (warp-uniform).  Called once a chunk is finished: publishes them when
    // the next chunk in flight belongs to another (sequence, KV head), or none is.
    int pend = 0;
    auto finished = [&](const ChunkSlot &cs) {
        if constexpr (!kPublish) return;  // pass 1 alone: its reader starts after it ends
        pend += cs.rec;
        __syncwarp();  // lane 0's slot descriptors of the chunks claimed since
        const bool last = n_done + 1 >= n_issued || slots[(n_done + 1) % nbuf].b != cs.b ||
                          slots[(n_done + 1) % nbuf].kvh != cs.kvh;
        if (pend > 0 && last) {
            publish_chunks<G>(p, cs.b, cs.kvh, pend, lane);
            pend = 0;
        }
    };
    while (n_done < n_issued) {
        const int slot = n_done % nbuf;
        if (!mbar_wait(&bars[slot], (n_done / nbuf) & 1)) {
            failed = true;
            break;
        }
        if (n_done == 0)  // the first copy has landed: fill the other buffers
            while (more && n_issued < nbuf) claim();
        const ChunkSlot cs = slots[slot];
        const int len = cs.len, b = cs.b, kvh = cs.kvh, ch = cs.ch;
        if (len <= 0) {  // nothing to read: pass the buffer on
            if (more) claim();
            finished(cs);
            ++n_done;
            continue;
        }
        const unsigned char *base = wbuf + size_t(slot) * CG::kBytes;
        if constexpr (kMma) {
            if (b != qb || kvh != qkvh) {
                load_q_frag<D, G>(p, b, kvh * G, lane, qf);
                qb = b;
                qkvh = kvh;
            }
            float c[2][4];
            chunk_logits_mma<D>(base, qf, lane, c);
            // Every lane is done with the buffer: refill it with the next claim.
            __syncwarp();
            if (more) claim();

            // Lane (g, t) holds heads 2t + j of keys 8k + g (k = 2 mt + half).  The
            // chunk's statistics per head are shuffles over the lanes of one t.
            const int g = lane >> 2, t = lane & 3;
            float xv[2][4], m[2], z[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    xv[j][k] = 8 * k + g < len ? c[k >> 1][(k & 1) * 2 + j] * p.scale : -INFINITY;
                m[j] = fmaxf(fmaxf(xv[j][0], xv[j][1]), fmaxf(xv[j][2], xv[j][3]));
            }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1)
#pragma unroll
                for (int j = 0; j < 2; ++j) m[j] = fmaxf(m[j], __shfl_xor_sync(kFull, m[j], o));
            int am[2];  // the chunk's first key of largest logit, per head
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                z[j] = 0.f;
                am[j] = kChunkRows;
#pragma unroll
                for (int k = 3; k >= 0; --k) {
                    if (xv[j][k] == m[j]) am[j] = 8 * k + g;
                    xv[j][k] = __expf(xv[j][k] - m[j]);  // 0 for keys past the end
                    z[j] += xv[j][k];
                }
            }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    z[j] += __shfl_xor_sync(kFull, z[j], o);
                    am[j] = min(am[j], __shfl_xor_sync(kFull, am[j], o));
                }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int h = 2 * t + j;
                if (h < G) {
                    const int hq = kvh * G + h;
                    float *srow = p.stash + ((size_t(b) * p.Hq + hq) * p.nch + ch) * kChunkRows;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (8 * k + g < len) srow[8 * k + g] = xv[j][k];
                }
            }
            if (g == 0) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (2 * t + j < G) {
                        const size_t hq = size_t(b) * p.Hq + kvh * G + 2 * t + j;
                        store_record(p.rec + hq * p.nch + ch, m[j], z[j]);
                        if constexpr (kPublish) p.amax[hq * p.nch4 + ch] = static_cast<unsigned char>(am[j]);
                    }
            }
            finished(cs);
            ++n_done;
            continue;
        }
#pragma unroll
        for (int hp = 0; hp < CG::kPasses; ++hp) {
            if (CG::kPasses > 1 || b != qb || kvh != qkvh) {
                load_q_slice<T, D, kGH, kVPL, kPairs>(p, b, kvh * G + hp * kGH, l8, hx, qreg);
                qb = b;
                qkvh = kvh;
            }
            float x[kGH];  // logit of this lane's key of batch bt, head l8 % GH of the pass
#pragma unroll
            for (int bg = 0; bg < kGH; bg += kBG) {  // kBG batches of kKB keys per lane group
                float v[kBG][8];
#pragma unroll
                for (int bb = 0; bb < kBG; ++bb)
#pragma unroll
                    for (int kk = 0; kk < kKB; ++kk) {
                        const int r = (bg + bb) * 4 * kKB + g8 * kKB + (kk ^ kx);  // row of slot (kk, .)
                        float2 acc[kGH];
#pragma unroll
                        for (int h = 0; h < kGH; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
                        for (int i = 0; i < kVPL; ++i) {
                            // 16-byte vector l8 + 8i of row r: box i, swizzled position l8 ^ (r mod 8)
                            const uint4 raw = *reinterpret_cast<const uint4 *>(base + i * kChunkBoxBytes + r * 128 +
                                                                               ((l8 ^ (r & 7)) << 4));
                            float2 kv[kPairs];
                            Vec16<T>::unpack(raw, kv);
#pragma unroll
                            for (int h = 0; h < kGH; ++h)
#pragma unroll
                                for (int pp = 0; pp < kPairs; ++pp)
                                    acc[h] = __ffma2_rn(qreg[h][i * kPairs + pp], kv[pp], acc[h]);
                        }
#pragma unroll
                        for (int h = 0; h < kGH; ++h) v[bb][kk * kGH + h] = acc[h].x + acc[h].y;
                    }
                // lane l8 of the group ends with value l8 of each batch: key l8 / GH, head l8 % GH
#pragma unroll
                for (int bb = 0; bb < kBG; ++bb) reduce_scatter_stage<4>(v[bb]);
#pragma unroll
                for (int bb = 0; bb < kBG; ++bb) reduce_scatter_stage<2>(v[bb]);
#pragma unroll
                for (int bb = 0; bb < kBG; ++bb) reduce_scatter_stage<1>(v[bb]);
#pragma unroll
                for (int bb = 0; bb < kBG; ++bb) {
                    const int key = (bg + bb) * 4 * kKB + g8 * kKB + l8 / kGH;
                    x[bg + bb] = key < len ? v[bb][0] * p.scale : -INFINITY;
                }
            }
            if (hp == CG::kPasses - 1) {
                // Every lane is done with the buffer: refill it with the next claim.
                __syncwarp();
                if (more) claim();
            }

            // chunk statistics of the pass's heads; e to the stash, (m_c, z_c) to the records
            const int hq = kvh * G + hp * kGH + l8 % kGH;
            float m = x[0];
#pragma unroll
            for (int bt = 1; bt < kGH; ++bt) m = fmaxf(m, x[bt]);
            m = head_max<kGH>(m);
            float *srow = p.stash + ((size_t(b) * p.Hq + hq) * p.nch + ch) * kChunkRows;
            float z = 0.f;
            int am = kChunkRows;  // the chunk's first key of largest logit
#pragma unroll
            for (int bt = 0; bt < kGH; ++bt) {
                const int key = bt * 4 * kKB + g8 * kKB + l8 / kGH;
                if (key < len) {
                    if (x[bt] == m) am = min(am, key);
                    const float e = __expf(x[bt] - m);
                    srow[key] = e;
                    z += e;
                }
            }
            z = head_sum<kGH>(z);
#pragma unroll
            for (int o = kGH; o < 32; o <<= 1) am = min(am, __shfl_xor_sync(kFull, am, o));
            if (lane < kGH) {  // g8 = 0, l8 = lane: head `lane` of the pass
                store_record(p.rec + (size_t(b) * p.Hq + hq) * p.nch + ch, m, z);
                if constexpr (kPublish) p.amax[(size_t(b) * p.Hq + hq) * p.nch4 + ch] = static_cast<unsigned char>(am);
            }
        }
        finished(cs);
        ++n_done;
    }

    if (failed) {
        // SANTA_ERR_TIMEOUT with location code 2 (a chunk copy never completed);
        // wait, bounded, for this warp's copies still in flight before exiting.
        if (lane == 0) {
            raise_flag(p, SANTA_ERR_TIMEOUT | (2u << 8));
            const long long t0 = clock64();
            for (int k = n_done; k < n_issued; ++k)
                while (!mbar_try_wait(&bars[k % nbuf], (k / nbuf) & 1) && clock64() - t0 < kWaitCycles) {
                }
        }
        __syncwarp();
    } else if (lane < nbuf) {
        mbar_inval(&bars[lane]);  // every copy has landed: the shared memory may be reused
    }
    return failed;  // warp-uniform
}

// Pass 1 alone (santa_prop_pass1 and the two-kernel prop path): one CTA of
// kChunkWarps streaming warps per SM.  Launched with programmatic dependent launch:
// a CTA sets up its barriers while the previous kernel drains and waits for it
// before touching global memory.
template <typename T, int D, int G, bool kPaged>
__global__ void __launch_bounds__(kChunkWarps * 32, 1)
    prop_stream_kernel(const __grid_constant__ CUtensorMap kmap, const Params p, int nbuf) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align1024(smem_raw);
    stream_setup<T, D, G>(kmap, smem, nbuf);
    __syncthreads();
    // Nothing above touches global memory; the previous kernel in the stream (which
    // may produce q, K or read this call's workspace) must be complete below.
    pdl_wait();
    pdl_launch_dependents();
    stream_chunks<T, D, G, kPaged, false>(kmap, p, nbuf, smem);
}

}  // namespace santa
