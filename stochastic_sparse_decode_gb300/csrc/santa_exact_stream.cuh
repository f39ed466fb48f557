// santa_exact_stream.cuh -- exact split-KV decode attention as a streaming kernel.
//
// The dense comparison point of the paper notes ("Stochastic Sparse Attention
// for Memory-Bound Inference", Related work: FlashDecoding): out = sum_i A_i V_i,
// reading all of K and V.  The kernel streams like prop's pass 1: one CTA of
// kChunkWarps warps per SM, chunks of 32 keys numbered (sequence, chunk, KV head)
// with the KV head fastest, and warp W = w C + c taking chunks W, W + P, W + 2P,
// ... (P = C kChunkWarps) -- a fixed walk, so that which partial results exist is
// a function of the problem alone.  Each warp owns one K and one V buffer,
// filled by TMA (32 rows x 128 bytes, 128-byte swizzle) under one mbarrier each:
// the next chunk's K is requested as soon as the logits of the current one are
// formed, its V as soon as the current V has been accumulated.
//
// Per chunk the logits come from the same d-split dot products as prop (eight
// lanes per key, q slice in registers, reduce-scatter by shuffles).  The warp
// keeps, per query head of the group, an online softmax state (M, Z, O): with
// the chunk's maximum m_c, M' = max(M, m_c), e_i = exp(x_i - M'),
// Z' = Z exp(M - M') + sum e_i and O' = O exp(M - M') + sum e_i V_i.  A lane owns
// D/32 output elements of every head; e_i goes through shared memory as a
// broadcast.  When the walk moves to another sequence, and at the end, the warp
// writes its (M, Z, O) for the sequence it leaves; exact_stream_merge combines
// a head's partials by the log-sum-exp rule.
#pragma once

#include "santa_common.cuh"
#include "santa_merge.cuh"
#include "santa_stream.cuh"
#include "santa_tile.cuh"

namespace santa {

template <typename T, int D, int G>
struct ExactStreamGeom {
    using CG = ChunkGeom<T, D, G>;
    static constexpr int kBytes = CG::kBytes;                   // one chunk of K (or V) rows
    static constexpr int kWarps = kBytes > 8192 ? 6 : kChunkWarps;  // fp32 d = 128: 16 KiB chunks
    // shared memory: [kWarps][2] buffers (K, V), [kWarps][2] mbarriers,
    // [kWarps][32][G] exponentiated scores
    static __host__ __device__ size_t bars_off() { return size_t(kWarps) * 2 * kBytes; }
    static __host__ __device__ size_t es_off() { return bars_off() + size_t(kWarps) * 2 * 8; }
    static __host__ __device__ size_t bytes() { return 1024 + es_off() + size_t(kWarps) * 32 * G * 4; }
};

// Where warp W's n-th chunk x = W + n P lies: KV head, sequence, chunk of it.
__device__ __forceinline__ void exact_walk(const Params &p, long long x, int *kvh, int *b, int *ch) {
    *kvh = int(x % p.Hkv);
    const long long r = x / p.Hkv;
    *b = int(r / p.nch);
    *ch = int(r - (long long)*b * p.nch);
}

// Does the walk of warp W (stride P, n_mine chunks) touch sequence b?  Every warp
// writes one partial for each sequence it touches, and only for those.
__host__ __device__ __forceinline__ bool exact_touches(long long W, long long P, long long X, long long per_seq, int b) {
    const long long lo = (long long)b * per_seq, hi = lo + per_seq;
    const long long n0 = lo > W ? (lo - W + P - 1) / P : 0;
    const long long x = W + n0 * P;
    return x < hi && x < X;
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(ExactStreamGeom<T, D, G>::kWarps * 32, 1)
    exact_stream_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const Params p) {
    using Geo = TileGeom<T, D>;
    using CG = ChunkGeom<T, D, G>;
    using EG = ExactStreamGeom<T, D, G>;
    constexpr int kGH = CG::kGH, kVPL = CG::kVPL, kKB = CG::kKB, kPairs = Geo::kPairs;
    constexpr int kBG = kGH >= 2 ? 2 : 1;
    constexpr int kE = D / 32;                          // output elements per lane and head
    constexpr int kLaneBytes = kE * int(sizeof(T));     // 4, 8 or 16
    constexpr bool kMma = sizeof(T) == 2;               // bf16 keys: logits on the tensor cores
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g8 = lane >> 3, l8 = lane & 7;
    const int hx = l8 & (kGH - 1), kx = l8 / kGH;
    const long long X = (long long)p.B * p.nch * p.Hkv;
    const long long P = (long long)gridDim.x * EG::kWarps;
    const long long W = (long long)warp * gridDim.x + blockIdx.x;
    const int n_mine = W < X ? int((X - W + P - 1) / P) : 0;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~uintptr_t(1023));
    unsigned char *kbuf = smem + size_t(warp) * 2 * EG::kBytes;
    unsigned char *vbuf = kbuf + EG::kBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + EG::bars_off()) + warp * 2;  // [0] K, [1] V
    float *es = reinterpret_cast<float *>(smem + EG::es_off()) + warp * 32 * G;       // [key][head]

    if (lane < 2) mbar_init(&bars[lane], 1);
    if (threadIdx.x == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    fence_barrier_init();
    __syncwarp();

    struct Cur {
        int kvh, b, ch, len;
        long long start;
    };
    int lb = -1, lL = 0;  // sequence-bounds cache (every lane keeps its own copy)
    long long lstart = 0;
    auto locate = [&](int n, Cur &cu) {
        exact_walk(p, W + n * P, &cu.kvh, &cu.b, &cu.ch);
        if (cu.b != lb) {
            lL = seq_bounds(p, cu.b, &lstart);
            lb = cu.b;
        }
        cu.start = lstart;
        cu.len = min(kChunkRows, lL - cu.ch * kChunkRows);
    };
    // lane 0: start the copy of the K (which = 0) or V (1) rows of chunk cu; a chunk
    // without keys completes the buffer's phase with a plain arrive
    auto issue = [&](int which, const Cur &cu) {
        if (lane != 0) return;
        uint64_t *bar = &bars[which];
        if (cu.len > 0) {
            unsigned char *dst = which ? vbuf : kbuf;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, EG::kBytes);
#pragma unroll
            for (int bx = 0; bx < Geo::kBoxes; ++bx)
                tma_load_3d(dst + bx * kChunkBoxBytes, which ? &vmap : &kmap, bar, bx * Geo::kBoxElems, cu.kvh,
                            int(cu.start) + cu.ch * kChunkRows);
        } else {
            mbar_arrive(bar);
        }
    };

    // online softmax state of the group's heads for sequence sb
    float Ms[G], Zs[G], O[G][kE];
    // bf16, tensor-core layout: lane (g, t) owns heads 2t, 2t + 1 (Mown: their M)
    // and holds O^T in m16n8 tiles: Ot[m] = O[2t, 2t + 1][16 m + g] and [.. + 8]
    float Mown[2], Ot[kMma ? D / 16 : 1][4];
    int sb = -1;
    auto reset = [&]() {
        Mown[0] = Mown[1] = -INFINITY;
#pragma unroll
        for (int m = 0; m < (kMma ? D / 16 : 1); ++m) Ot[m][0] = Ot[m][1] = Ot[m][2] = Ot[m][3] = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            Ms[h] = -INFINITY;
            Zs[h] = 0.f;
#pragma unroll
            for (int e = 0; e < kE; ++e) O[h][e] = 0.f;
        }
    };
    auto flush = [&]() {  // this warp's partial of sequence sb (its KV head is c mod Hkv)
        if (sb < 0) return;
        const size_t slot = (size_t(sb) * P + W) * G;
        if constexpr (kMma) {
            const int g = lane >> 2, t = lane & 3;
#pragma unroll
            for (int j = 0; j < 2; ++j)
                if (2 * t + j < G) {
                    float *o = p.partial + (slot + 2 * t + j) * D + g;
#pragma unroll
                    for (int m = 0; m < D / 16; ++m) {
                        o[16 * m] = Ot[m][j];
                        o[16 * m + 8] = Ot[m][2 + j];
                    }
                }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            if constexpr (!kMma) {
                float *o = p.partial + (slot + h) * D + lane * kE;
#pragma unroll
                for (int e = 0; e < kE; ++e) o[e] = O[h][e];
            }
            if (lane == 0) reinterpret_cast<float2 *>(p.rec_m)[slot + h] = make_float2(Ms[h], Zs[h]);
        }
    };
    reset();

    Cur cur{}, nxt{};
    if (n_mine > 0) {
        locate(0, cur);
        issue(0, cur);
        issue(1, cur);
    }
    float2 qreg[kGH][kVPL * kPairs];
    uint32_t qf[D / 16][2];
    int qb = -1, qkvh = -1;
    uint32_t phK = 0, phV = 0;
    bool failed = false;
    int n = 0;
    for (; n < n_mine; ++n) {
        const bool has_next = n + 1 < n_mine;
        if (has_next) locate(n + 1, nxt);
        if (cur.b != sb) {
            flush();
            reset();
            sb = cur.b;
        }
        const int len = cur.len;
        // ---- logits of the chunk (the K buffer)
        if (!mbar_wait(&bars[0], phK)) {
            failed = true;
            break;
        }
        phK ^= 1u;
        float x[CG::kPasses][kGH];
        float c[2][4];  // bf16: the chunk's logits from the tensor cores (layout of chunk_logits_mma)
        if constexpr (kMma) {
            if (len > 0) {
                if (cur.b != qb || cur.kvh != qkvh) {
                    load_q_frag<D, G>(p, cur.b, cur.kvh * G, lane, qf);
                    qb = cur.b;
                    qkvh = cur.kvh;
                }
                chunk_logits_mma<D>(kbuf, qf, lane, c);
            }
        } else if (len > 0) {
#pragma unroll
            for (int hp = 0; hp < CG::kPasses; ++hp) {
                if (CG::kPasses > 1 || cur.b != qb || cur.kvh != qkvh) {
                    load_q_slice<T, D, kGH, kVPL, kPairs>(p, cur.b, cur.kvh * G + hp * kGH, l8, hx, qreg);
                    qb = cur.b;
                    qkvh = cur.kvh;
                }
#pragma unroll
                for (int bg = 0; bg < kGH; bg += kBG) {
                    float v[kBG][8];
#pragma unroll
                    for (int bb = 0; bb < kBG; ++bb)
#pragma unroll
                        for (int kk = 0; kk < kKB; ++kk) {
                            const int r = (bg + bb) * 4 * kKB + g8 * kKB + (kk ^ kx);
                            float2 acc[kGH];
#pragma unroll
                            for (int h = 0; h < kGH; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
                            for (int i = 0; i < kVPL; ++i) {
                                const uint4 raw = *reinterpret_cast<const uint4 *>(kbuf + i * kChunkBoxBytes + r * 128 +
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
#pragma unroll
                    for (int bb = 0; bb < kBG; ++bb) reduce_scatter_stage<4>(v[bb]);
#pragma unroll
                    for (int bb = 0; bb < kBG; ++bb) reduce_scatter_stage<2>(v[bb]);
#pragma unroll
                    for (int bb = 0; bb < kBG; ++bb) reduce_scatter_stage<1>(v[bb]);
#pragma unroll
                    for (int bb = 0; bb < kBG; ++bb) {
                        const int key = (bg + bb) * 4 * kKB + g8 * kKB + l8 / kGH;
                        x[hp][bg + bb] = key < len ? v[bb][0] * p.scale : -INFINITY;
                    }
                }
            }
        }
        __syncwarp();
        if (has_next) issue(0, nxt);  // the K buffer is free

        // ---- online softmax update; e to the warp's score array
        if constexpr (kMma) {
          if (len > 0) {
            // lane (g, t) holds heads 2t + j of keys 8k + g; a head's statistics are
            // shuffles over the lanes of one t, then broadcast from lane t of group 0
            const int g = lane >> 2, t = lane & 3;
            float xv[2][4], m2[2], z2[2], Mn[G], zc[G], mine[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    xv[j][k] = 8 * k + g < len ? c[k >> 1][(k & 1) * 2 + j] * p.scale : -INFINITY;
                m2[j] = fmaxf(fmaxf(xv[j][0], xv[j][1]), fmaxf(xv[j][2], xv[j][3]));
            }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1)
#pragma unroll
                for (int j = 0; j < 2; ++j) m2[j] = fmaxf(m2[j], __shfl_xor_sync(kFull, m2[j], o));
#pragma unroll
            for (int h = 0; h < G; ++h) Mn[h] = fmaxf(Ms[h], __shfl_sync(kFull, m2[h & 1], h >> 1));
            float sco[2];  // rescale of the lane's own heads
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float mold = Mown[j];
                Mown[j] = fmaxf(Mown[j], m2[j]);  // = Mn[2t + j]
                sco[j] = __expf(mold - Mown[j]);  // 0 while the state is empty
                mine[j] = Mown[j];
                z2[j] = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float e = __expf(xv[j][k] - mine[j]);  // 0 for keys past the end
                    if (2 * t + j < G) es[(8 * k + g) * G + 2 * t + j] = e;
                    z2[j] += e;
                }
            }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1)
#pragma unroll
                for (int j = 0; j < 2; ++j) z2[j] += __shfl_xor_sync(kFull, z2[j], o);
#pragma unroll
            for (int h = 0; h < G; ++h) zc[h] = __shfl_sync(kFull, z2[h & 1], h >> 1);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float sc = __expf(Ms[h] - Mn[h]);  // 0 while the state is empty
                Zs[h] = fmaf(Zs[h], sc, zc[h]);
                Ms[h] = Mn[h];
            }
#pragma unroll
            for (int m = 0; m < D / 16; ++m) {
                Ot[m][0] *= sco[0];
                Ot[m][1] *= sco[1];
                Ot[m][2] *= sco[0];
                Ot[m][3] *= sco[1];
            }
          }
        } else if (len > 0) {
            float Mn[G], zc[G];
#pragma unroll
            for (int hp = 0; hp < CG::kPasses; ++hp) {
                float mh = x[hp][0];
#pragma unroll
                for (int bt = 1; bt < kGH; ++bt) mh = fmaxf(mh, x[hp][bt]);
                mh = head_max<kGH>(mh);  // lane l of lane group 0 holds head hp * GH + l
#pragma unroll
                for (int j = 0; j < kGH; ++j) {
                    const int h = hp * kGH + j;
                    Mn[h] = fmaxf(Ms[h], __shfl_sync(kFull, mh, j));
                }
                float mine = Mn[hp * kGH];  // M' of this lane's head
#pragma unroll
                for (int j = 1; j < kGH; ++j) mine = (l8 % kGH) == j ? Mn[hp * kGH + j] : mine;
                float zl = 0.f;
#pragma unroll
                for (int bt = 0; bt < kGH; ++bt) {
                    const int key = bt * 4 * kKB + g8 * kKB + l8 / kGH;
                    const float e = key < len ? __expf(x[hp][bt] - mine) : 0.f;
                    es[key * G + hp * kGH + l8 % kGH] = e;
                    zl += e;
                }
                zl = head_sum<kGH>(zl);
#pragma unroll
                for (int j = 0; j < kGH; ++j) zc[hp * kGH + j] = __shfl_sync(kFull, zl, j);
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float sc = __expf(Ms[h] - Mn[h]);  // 0 while the state is empty
                Zs[h] = fmaf(Zs[h], sc, zc[h]);
                Ms[h] = Mn[h];
#pragma unroll
                for (int e = 0; e < kE; ++e) O[h][e] *= sc;
            }
        }
        __syncwarp();

        // ---- O += sum_i e_i V_i (the V buffer)
        if (!mbar_wait(&bars[1], phV)) {
            failed = true;
            break;
        }
        phV ^= 1u;
        if constexpr (kMma) {
            // O^T += V^T P^T on the tensor cores: A = V^T (16 dims x 16 keys, read
            // transposed from the swizzled V buffer), B = P^T (16 keys x 8 heads,
            // heads >= G zero) from the score array, split into bf16 high and low
            // parts so that e keeps ~16 bits.  Keys past the chunk's end have e = 0.
            if (len > 0) {
                const int g = lane >> 2, t = lane & 3, mq = lane >> 3, mi = lane & 7;
                uint32_t bh[2][2], bl[2][2];
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int key = 16 * ks + 8 * hf + 2 * t;
                        const float e0 = g < G ? es[key * G + g] : 0.f;
                        const float e1 = g < G ? es[(key + 1) * G + g] : 0.f;
                        bf16_split2(e0, e1, &bh[ks][hf], &bl[ks][hf]);
                    }
#pragma unroll
                for (int m = 0; m < D / 16; ++m)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        // matrix mq: keys 16 ks + 8 (mq / 2) + row, dims 16 m + 8 (mq % 2) ..
                        const int key = 16 * ks + 8 * (mq >> 1) + mi;
                        const int dv = 2 * m + (mq & 1);  // 16-byte vector of the row
                        uint32_t a[4];
                        ldmatrix_x4_trans(a, vbuf + (dv >> 3) * kChunkBoxBytes + key * 128 +
                                                 (((dv & 7) ^ (key & 7)) << 4));
                        mma_bf16_16816(Ot[m], a, bh[ks]);
                        mma_bf16_16816(Ot[m], a, bl[ks]);
                    }
            }
        } else if (len > 0) {
            // this lane's D/32 elements of a row: box, 16-byte vector and offset in it
            const int lb0 = lane * kLaneBytes;
            const unsigned char *vlane = vbuf + (lb0 >> 7) * kChunkBoxBytes + (lb0 & 15);
            const int vec = (lb0 & 127) >> 4;
            for (int r0 = 0; r0 < len; r0 += 8) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {  // row r0 + j, swizzled position vec ^ j
                    const int r = r0 + j;
                    if (r < len) {
                        const unsigned char *row = vlane + r * 128 + ((vec ^ j) << 4);
                        float vv[kE];
                        if constexpr (kLaneBytes == 4) {
                            const uint32_t w = *reinterpret_cast<const uint32_t *>(row);
                            vv[0] = bf16_lo(w);
                            vv[1] = bf16_hi(w);
                        } else if constexpr (kLaneBytes == 8) {
                            const uint2 w = *reinterpret_cast<const uint2 *>(row);
                            if constexpr (sizeof(T) == 2) {
                                vv[0] = bf16_lo(w.x);
                                vv[1] = bf16_hi(w.x);
                                vv[2] = bf16_lo(w.y);
                                vv[3] = bf16_hi(w.y);
                            } else {
                                vv[0] = __uint_as_float(w.x);
                                vv[1] = __uint_as_float(w.y);
                            }
                        } else {
                            const uint4 w = *reinterpret_cast<const uint4 *>(row);
                            vv[0] = __uint_as_float(w.x);
                            vv[1] = __uint_as_float(w.y);
                            vv[2] = __uint_as_float(w.z);
                            vv[3] = __uint_as_float(w.w);
                        }
                        float eh[G];  // the row's scores for the group's heads (a broadcast)
                        if constexpr (G % 4 == 0) {
#pragma unroll
                            for (int h4 = 0; h4 < G; h4 += 4) {
                                const float4 e4 = *reinterpret_cast<const float4 *>(es + r * G + h4);
                                eh[h4] = e4.x;
                                eh[h4 + 1] = e4.y;
                                eh[h4 + 2] = e4.z;
                                eh[h4 + 3] = e4.w;
                            }
                        } else {
#pragma unroll
                            for (int h = 0; h < G; ++h) eh[h] = es[r * G + h];
                        }
#pragma unroll
                        for (int h = 0; h < G; ++h)
#pragma unroll
                            for (int e = 0; e < kE; e += 2) {
                                const float2 o = __ffma2_rn(make_float2(eh[h], eh[h]), make_float2(vv[e], vv[e + 1]),
                                                            make_float2(O[h][e], O[h][e + 1]));
                                O[h][e] = o.x;
                                O[h][e + 1] = o.y;
                            }
                    }
                }
            }
        }
        __syncwarp();
        if (has_next) issue(1, nxt);  // the V buffer is free
        cur = nxt;
    }
    if (!failed) {
        flush();
    } else {
        // SANTA_ERR_TIMEOUT, location code 2; wait, bounded, for the copies in flight
        if (lane == 0) {
            raise_flag(p, SANTA_ERR_TIMEOUT | (2u << 8));
            const long long t0 = clock64();
            while (!mbar_try_wait(&bars[0], phK) && clock64() - t0 < kWaitCycles) {
            }
            while (!mbar_try_wait(&bars[1], phV) && clock64() - t0 < kWaitCycles) {
            }
        }
        __syncwarp();
    }
}

// Log-sum-exp merge of one (query head, sequence): the partials (M_w, Z_w, O_w) of
// the warps whose walk touched the sequence (W = w C + c with c = kvh mod Hkv),
// in a fixed order: out = sum_w exp(M_w - M) O_w / sum_w exp(M_w - M) Z_w.
// One CTA of 16 warps per head: the coefficients of all candidates first (one
// round trip for the (M, Z) pairs), then warp k sums candidates k, k + 16, ...
// with all its partial rows in flight at once, then the warps in order.
constexpr int kExactMergeWarps = 16;
constexpr int kExactMergeMax = kExactCtaBound * 12;  // candidates: warps per CTA x CTAs of one KV head

template <int D>
__global__ void __launch_bounds__(kExactMergeWarps * 32) exact_stream_merge(const Params p, int C, int warps) {
    constexpr int kE = D / 32;
    constexpr int kT = kExactMergeWarps * 32;
    const int hq = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = hq / p.G, h = hq % p.G;
    __shared__ float s_coef[kExactMergeMax];
    __shared__ int s_w[kExactMergeMax];
    __shared__ float red[kExactMergeWarps][D];
    __shared__ float scr[kExactMergeWarps];

    long long start;
    const int L = seq_bounds(p, b, &start);
    float *outp = p.out + (size_t(b) * p.Hq + hq) * D;
    if (L == 0) {
        if (tid < D) outp[tid] = 0.f;
        return;
    }
    const long long P = (long long)C * warps;
    const long long X = (long long)p.B * p.nch * p.Hkv, per_seq = (long long)p.nch * p.Hkv;
    const int per_w = C / p.Hkv;  // CTAs of this KV head
    const int ncand = min(warps * per_w, kExactMergeMax);
    const float2 *mz = reinterpret_cast<const float2 *>(p.rec_m);
    const size_t base = size_t(b) * P;

    // (M_w, Z_w) of every candidate; M, then the coefficients exp(M_w - M)
    float mw[kExactMergeMax / kT + 1], zw[kExactMergeMax / kT + 1];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k * kT < kExactMergeMax; ++k) {
        const int i = tid + k * kT;
        mw[k] = -INFINITY;
        zw[k] = 0.f;
        if (i < ncand) {
            const long long Wi = (long long)(i / per_w) * C + kvh + (long long)(i % per_w) * p.Hkv;
            s_w[i] = int(Wi);
            if (exact_touches(Wi, P, X, per_seq, b)) {
                const float2 v = __ldcg(&mz[(base + Wi) * p.G + h]);
                mw[k] = v.x;
                zw[k] = v.y;
            }
        }
        mx = fmaxf(mx, mw[k]);
    }
    const float M = block_max<kExactMergeWarps>(mx, scr);
    float zpart = 0.f;
#pragma unroll
    for (int k = 0; k * kT < kExactMergeMax; ++k) {
        const int i = tid + k * kT;
        if (i < ncand) {
            const float cf = mw[k] > -INFINITY ? expf(mw[k] - M) : 0.f;
            s_coef[i] = cf;
            zpart = fmaf(zw[k], cf, zpart);
        }
    }
    const float Z = block_sum<kExactMergeWarps>(zpart, scr);  // its barriers also publish s_coef / s_w

    float acc[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) acc[e] = 0.f;
    for (int i0 = warp; i0 < ncand; i0 += 8 * kExactMergeWarps) {
        float v[8][kE], cf[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * kExactMergeWarps;
            cf[u] = i < ncand ? s_coef[i] : 0.f;
            if (cf[u] != 0.f) {
                const float *src = p.partial + ((base + s_w[i]) * p.G + h) * D + lane * kE;
#pragma unroll
                for (int e = 0; e < kE; ++e) v[u][e] = __ldcg(src + e);
            } else {
#pragma unroll
                for (int e = 0; e < kE; ++e) v[u][e] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int e = 0; e < kE; ++e) acc[e] = fmaf(cf[u], v[u][e], acc[e]);
    }
#pragma unroll
    for (int e = 0; e < kE; ++e) red[warp][lane * kE + e] = acc[e];
    __syncthreads();
    if (tid < D) {
        float num = 0.f;
#pragma unroll
        for (int w = 0; w < kExactMergeWarps; ++w) num += red[w][tid];
        outp[tid] = num / Z;
    }
}

}  // namespace santa
