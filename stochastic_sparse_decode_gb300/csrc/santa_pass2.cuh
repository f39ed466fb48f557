// santa_pass2.cuh -- S2ANTA-prop pass 2 as a kernel of its own (after the
// streaming pass 1), with the global reducer.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (paper notes, Key
// design 2), on the 32-key chunk records of pass 1.  The chunks of one (query
// head, sequence) are split over the CTAs of one thread-block cluster (p2_split
// CTAs of p2_cps chunks, whole tiles and whole warps each).  Every CTA first runs
// the reducer over all of that head's chunk records, in a fixed order, so all of
// them obtain bit-identical values:
//     M = max_c m_c,   w_c = z_c exp(m_c - M)   (the chunks' mass on one scale),
//     C_c = w_0 + ... + w_c (inclusive),   Z = C_{N_b - 1}.
// The systematic thresholds are U + m/S, m = 0..S-1 (Key design 1), i.e. the
// points (U + m/S) Z on the unnormalised CDF.  The number of them below c is
//     N(c) = clamp(ceil(S c / Z - S U), 0, S),
// so chunk c receives the thresholds m in [N(C_{c-1}), N(C_c)), with
// N(C_{-1}) = 0 and N(C_{N_b - 1}) = S.  The masses w_c are summed as 64-bit
// fixed-point integers, so C is exact whatever the order of the additions:
// non-decreasing, identical in every CTA, budgets never negative and adding up
// to exactly S.  Chunks with no threshold read neither their stash nor V (a
// warp's first 16 chunks are read speculatively, in the round trip of the
// records).  A warp takes its chunks 16 at a time: it scans the 32 stashed e
// of each into its in-chunk prefix, then gives every lane one threshold of the
// batch, maps it to its chunk's own scale,
//     r_m = ((U + m/S) Z - C_{c-1}) / exp(m_c - M),
// takes the smallest key whose prefix exceeds r_m (clamped to the chunk's keys
// of positive score), and queues that key (the stratified and i.i.d. samplers of
// Key design 1 only change the thresholds: (m + u_m)/S, or the sorted u_s); the
// queue is flushed by gathering up to 32 V rows at a time.  Each CTA sums its
// warps in warp order and stores the sum into the shared memory of cluster rank
// 0, which adds the CTAs in rank order after one cluster barrier.  out = sum / S:
// no multiply by a probability anywhere after the softmax.  Rank 0 then sets the
// head's chunk records and published-chunk count back to zero, as the workspace
// contract asks.  A tile's budget S_tile (a debug output, with its Z_tile and
// m_t) is the sum over its chunks.
//
// Every index derived from workspace data is clamped: a count below zero or a
// sample number at or above S (possible only on a workspace that pass 1 did not
// fill) is clamped and raises SANTA_ERR_WORKSPACE.
#pragma once

#include "santa_common.cuh"
#include "santa_sampler.cuh"
#include "santa_tile.cuh"

namespace santa {

constexpr int kPass2Warps = 8;  // warps of a pass-2 CTA
constexpr int kP2MaxSplit = 8;  // CTAs per head at most = the cluster size (portable)

// Inclusive prefix sum of 64-bit integers across the warp (exact, so any order of
// additions gives the same, non-decreasing result).
__device__ __forceinline__ unsigned long long warp_inclusive_scan_u64(unsigned long long v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long u = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += u;
    }
    return v;
}
__device__ __forceinline__ int warp_inclusive_scan_int(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

constexpr int kP2Rec = 4;     // chunk records per thread per reducer block
constexpr int kP2Batch = 16;  // chunks of a warp taken together (stash read, prefixes, searches)
// Pass-2 shared memory (prop): [cps+1] C (fixed point, C_{c_lo-1} .. C_{c_hi-1}),
// [cps+1] threshold counts N of the same, [cps] exp(m_c - M), [48] 64-bit
// scratch, per warp [16][32] stash batch / in-chunk prefixes, [16] cumulative
// sample counts, [16] last positive key, [32] queued keys, [8][D] warp sums,
// [8][D] the cluster's CTA sums (used in rank 0).
template <typename T, int D>
struct Pass2Smem {
    static __host__ __device__ size_t n_off(int cps) { return size_t(cps + 1) * 8; }
    static __host__ __device__ size_t st_off(int cps) { return n_off(cps) + size_t(cps + 1) * 4; }
    static __host__ __device__ size_t scr_off(int cps) { return (st_off(cps) + size_t(cps) * 4 + 15) & ~size_t(15); }
    static __host__ __device__ size_t ev_off(int cps) { return scr_off(cps) + 48 * 8; }
    static __host__ __device__ size_t cum_off(int cps) { return ev_off(cps) + size_t(kPass2Warps) * kP2Batch * 32 * 4; }
    static __host__ __device__ size_t last_off(int cps) { return cum_off(cps) + size_t(kPass2Warps) * kP2Batch * 4; }
    static __host__ __device__ size_t wl_off(int cps) { return last_off(cps) + size_t(kPass2Warps) * kP2Batch * 4; }
    static __host__ __device__ size_t red_off(int cps) { return wl_off(cps) + size_t(kPass2Warps) * 32 * 4; }
    static __host__ __device__ size_t part_off(int cps) { return red_off(cps) + size_t(kPass2Warps) * D * 4; }
    static __host__ __device__ size_t u_off(int cps) { return part_off(cps) + size_t(kP2MaxSplit) * D * 4; }
    // nu: the head's uniforms (stratified / i.i.d. samplers), padded to a power of two; 0 otherwise
    static __host__ __device__ size_t pg_off(int cps, int nu) { return u_off(cps) + size_t(nu) * 4; }
    // paged cache: the page ids of a CTA's keys (page_size >= 32, so at most cps + 1 of them)
    static __host__ __device__ size_t bytes(int cps, int nu, bool paged = false) {
        return pg_off(cps, nu) + (paged ? size_t(cps + 2) * 4 : 0);
    }
};

// Ascending sort of a[0, n) into out[0, n) by rank, in one pass: element i goes to
// #{k : a[k] < a[i]} + #{k < i : a[k] == a[i]}, a distinct slot for every i.  Ends
// with a block barrier.
template <int NT>
__device__ __forceinline__ void block_rank_sort(const float *a, float *out, int n) {
    for (int i = threadIdx.x; i < n; i += NT) {
        const float x = a[i];
        int r = 0;
        for (int k = 0; k < n; ++k) {
            const float y = a[k];
            r += (y < x || (y == x && k < i)) ? 1 : 0;
        }
        out[r] = x;
    }
    __syncthreads();
}

// Ascending bitonic sort of a[0, n) in shared memory by the whole block (n a power of two).
template <int NT>
__device__ __forceinline__ void block_bitonic_sort(float *a, int n) {
    for (int k = 2; k <= n; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += NT) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const float x = a[i], y = a[ixj];
                    if ((x > y) == ((i & k) == 0)) {
                        a[i] = y;
                        a[ixj] = x;
                    }
                }
            }
            __syncthreads();
        }
}

template <typename T, int D, int SAMPLER, bool kPaged>
__global__ void __launch_bounds__(kPass2Warps * 32, 2) prop_pass2_kernel(const Params p) {
    constexpr int kThreads = kPass2Warps * 32;
    constexpr int kE = D / 32;
    constexpr int kBlk = kThreads * kP2Rec;
    using Lay = Pass2Smem<T, D>;
    using u64 = unsigned long long;
    const int split = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;  // split == rank in the cluster
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cps = p.p2_cps, kper = cps / kPass2Warps;

    extern __shared__ __align__(128) unsigned char smem[];
    u64 *sC = reinterpret_cast<u64 *>(smem);                        // C of chunks c_lo-1 .. c_hi-1
    int *sN = reinterpret_cast<int *>(smem + Lay::n_off(cps));       // N of the same
    float *s_st = reinterpret_cast<float *>(smem + Lay::st_off(cps));
    u64 *scr = reinterpret_cast<u64 *>(smem + Lay::scr_off(cps));
    float *scrf = reinterpret_cast<float *>(scr + 32);               // [8] warp maxima
    float *wev = reinterpret_cast<float *>(smem + Lay::ev_off(cps)) + warp * kP2Batch * 32;
    int *wcum = reinterpret_cast<int *>(smem + Lay::cum_off(cps)) + warp * kP2Batch;
    int *wlast = reinterpret_cast<int *>(smem + Lay::last_off(cps)) + warp * kP2Batch;
    int *wl = reinterpret_cast<int *>(smem + Lay::wl_off(cps)) + warp * 32;
    float *red = reinterpret_cast<float *>(smem + Lay::red_off(cps));
    float *part = reinterpret_cast<float *>(smem + Lay::part_off(cps));
    float *s_u = reinterpret_cast<float *>(smem + Lay::u_off(cps));  // stratified / i.i.d. uniforms
    // paged cache: this CTA's page ids (systematic sampler only: no uniforms before them)
    int *s_pg = reinterpret_cast<int *>(smem + Lay::pg_off(cps, 0));

    pdl_launch_dependents();  // the next call's pass 1 may start its prologue on free SMs
    cluster_arrive();         // first half of the barrier that makes every CTA's shared memory addressable

    // One round trip for everything the reducer and the first batch need: the first
    // block of chunk records, speculatively the stash of this warp's first 16 chunks
    // (the stash is laid out per (sequence, head) with a stride of nch * 32, so no
    // address waits for another load), the sequence bounds and the offset.  Values
    // past the sequence's end are masked once its length is known.
    const size_t rec0 = (size_t(b) * p.Hq + hq) * p.nch;
    const size_t head = size_t(b) * p.Hq + hq;
    const float *sseq = p.stash + head * size_t(p.nch) * kChunkRows;
    const int cw0 = split * cps + warp * kper;  // this warp's first chunk
    float mr[kP2Rec], zr[kP2Rec];
    unsigned unwritten = 0;  // bit k: record k of the thread's block read as 0
    auto load_block = [&](int base, int lim) {
        unwritten = 0;
#pragma unroll
        for (int k = 0; k < kP2Rec; ++k) {
            const int c = base + tid * kP2Rec + k;
            const u64 v = c < lim ? __ldcg(p.rec + rec0 + c) : 0ull;
            // 0: a record pass 1 did not write (no mass; flagged once the length is known)
            mr[k] = v ? rec_m(v) : -INFINITY;
            zr[k] = v ? rec_z(v) : 0.f;
            if (v == 0ull) unwritten |= 1u << k;
        }
    };
    load_block(0, p.nch);
    float ev[kP2Batch];
#pragma unroll
    for (int k = 0; k < kP2Batch; ++k) {
        const int c = cw0 + k;
        const int key = c * kChunkRows + lane;
        ev[k] = (k < kper && key < p.nch * kChunkRows) ? __ldcg(sseq + key) : 0.f;
    }
    // Inputs the previous kernel does not write may be read before the dependency wait
    // (pass 1 lets this kernel start only once its own predecessor is complete).  All
    // loads are issued before any of them is checked: one round trip, not two.
    long long ind0, ind1;
    raw_bounds<kPaged>(p, b, &ind0, &ind1);
    const float u_raw = SAMPLER == kSys ? p.U[size_t(b) * p.Hq + hq] : 0.f;
    // paged cache: the page ids of this CTA's keys, kept in shared memory
    int pg_lo = 0;
    if constexpr (kPaged) {
        const int key_lo = split * cps * kChunkRows;
        pg_lo = key_lo / p.page_size;
        const int npg = min(p.max_pages, (key_lo + cps * kChunkRows - 1) / p.page_size + 1) - pg_lo;
        for (int i = tid; i < npg; i += kThreads) s_pg[i] = __ldg(p.page_table + size_t(b) * p.max_pages + pg_lo + i);
    }
    long long start;
    const int L = checked_bounds(p, ind0, ind1, &start);
    const float u = SAMPLER == kSys ? checked_offset(p, u_raw) : 0.f;
    if constexpr (SAMPLER != kSys) {
        // the head's S uniforms, each checked into [0, 1); the i.i.d. ones sorted
        int nu = 1;
        while (nu < p.S) nu <<= 1;
        const float *ug = p.u_samples + (size_t(b) * p.Hq + hq) * p.S;
        for (int i = tid; i < nu; i += kThreads) {
            float x = INFINITY;  // padding sorts last
            if (i < p.S) {
                x = __ldg(ug + i);
                if (!(x >= 0.f && x < 1.f)) {
                    raise_flag(p, SANTA_ERR_OFFSET);
                    x = x >= 1.f ? nextafterf(1.f, 0.f) : 0.f;
                }
            }
            s_u[i] = x;
        }
        __syncthreads();
        if constexpr (SAMPLER == kIid) {
            if (nu <= kRankSortMax) {
                block_rank_sort<kThreads>(s_u, s_u + nu, nu);
                s_u += nu;  // the sorted copy
            } else {
                block_bitonic_sort<kThreads>(s_u, nu);
            }
        }
    }
    pdl_wait();

    const int Nb = (L + kChunkRows - 1) / kChunkRows;
    const int c_lo = split * cps, c_hi = min(Nb, c_lo + cps);
    const bool active = c_lo < c_hi;  // CTA-uniform: this CTA owns at least one chunk
    const int cw1 = min(c_hi, cw0 + kper);  // end of this warp's chunks

    float acc[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) acc[e] = 0.f;

    if (active) {
        // ---- mask what the speculative loads read past the sequence's end
        bool hole = false;  // a record of the sequence that pass 1 did not write
#pragma unroll
        for (int k = 0; k < kP2Rec; ++k)
            if (tid * kP2Rec + k >= Nb) {
                mr[k] = -INFINITY;
                zr[k] = 0.f;
            } else if ((unwritten >> k) & 1u) {
                hole = true;
            }
#pragma unroll
        for (int k = 0; k < kP2Batch; ++k) {
            const int c = cw0 + k;
            wev[k * 32 + lane] = (c < cw1 && c * kChunkRows + lane < L) ? ev[k] : 0.f;
        }

        // ---- reducer: M; then C (fixed point, exact sums) and Z
        float mx = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3]));
        for (int base = kBlk; base < Nb; base += kBlk)
            for (int k = 0; k < kP2Rec; ++k) {
                const int c = base + tid * kP2Rec + k;
                if (c < Nb) {
                    const u64 v = __ldcg(p.rec + rec0 + c);
                    if (v != 0ull) mx = fmaxf(mx, rec_m(v));
                }
            }
        mx = warp_max(mx);
        if (lane == 0) scrf[warp] = mx;
        __syncthreads();
        float M = scrf[0];
#pragma unroll
        for (int w = 1; w < kPass2Warps; ++w) M = fmaxf(M, scrf[w]);

        // threshold counts N(c): the number of the sampler's thresholds below the
        // normalised CDF value cn = C / Z (each form is monotone in cn)
        const float Sf = float(p.S), SU = Sf * u;
        auto thresholds_below = [&](float cn) -> int {
            if constexpr (SAMPLER == kSys) {  // U + m/S < cn  <=>  m < S cn - S U
                return int(fminf(fmaxf(ceilf(fmaf(Sf, cn, -SU)), 0.f), Sf));
            } else if constexpr (SAMPLER == kStrat) {  // (m + u_m)/S < cn: all m < floor(S cn), maybe one more
                const float y = Sf * cn;
                const int k = int(fminf(fmaxf(floorf(y), 0.f), Sf));
                return k + ((k < p.S && s_u[k] < y - float(k)) ? 1 : 0);
            } else {  // sorted u_s < cn
                int lo = 0, hi = p.S;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (s_u[mid] < cn)
                        lo = mid + 1;
                    else
                        hi = mid;
                }
                return lo;
            }
        };
        // C (and, when the head's records fit one block, N at once: Z is that block's sum)
        const bool one_block = Nb <= kBlk;
        u64 carry = 0;
        for (int base = 0, it = 0; base < Nb; base += kBlk, ++it) {
            if (base > 0) {
                load_block(base, Nb);
                hole |= unwritten != 0;
            }
            u64 pl[kP2Rec];  // this thread's chunks: local inclusive prefix
            u64 run = 0;
#pragma unroll
            for (int k = 0; k < kP2Rec; ++k) {
                const int c = base + tid * kP2Rec + k;
                const float st = __expf(mr[k] - M);
                if (c >= c_lo && c < c_hi) s_st[c - c_lo] = st;
                run += c < Nb ? (u64)__float2ll_rn(zr[k] * st * kMassScale) : 0ull;
                pl[k] = run;
            }
            const u64 incl = warp_inclusive_scan_u64(run, lane);
            u64 *wsum = scr + (it & 1) * 8;  // alternate slots: no barrier needed before reuse
            if (lane == 31) wsum[warp] = incl;
            __syncthreads();
            u64 woff = 0, btot = 0;
#pragma unroll
            for (int w = 0; w < kPass2Warps; ++w) {
                const u64 t = wsum[w];
                if (w < warp) woff += t;
                btot += t;
            }
            const u64 excl = carry + woff + (incl - run);
            const float rZb = 1.0f / __ull2float_rn(btot);
#pragma unroll
            for (int k = 0; k < kP2Rec; ++k) {
                const int c = base + tid * kP2Rec + k;
                if (c >= c_lo - 1 && c < c_hi) {
                    const u64 Cc = excl + pl[k];
                    sC[c - c_lo + 1] = Cc;
                    if (one_block) sN[c - c_lo + 1] = c == Nb - 1 ? p.S : thresholds_below(__ull2float_rn(Cc) * rZb);
                }
            }
            carry += btot;
        }
        const u64 Z = carry;  // = C_{N_b - 1}
        if (hole) raise_flag(p, SANTA_ERR_WORKSPACE);
        if (c_lo == 0 && tid == 0) {
            sC[0] = 0ull;
            sN[0] = 0;
        }
        __syncthreads();
        const float fZ = __ull2float_rn(Z);
        if (!one_block) {  // N(C_{c-1}) for c = c_lo .. c_hi
            for (int i = tid; i <= c_hi - c_lo; i += kThreads) {
                const int c = c_lo + i - 1;
                int n;
                if (c < 0)
                    n = 0;
                else if (c == Nb - 1)
                    n = p.S;
                else
                    n = thresholds_below(__ull2float_rn(sC[i]) / fZ);
                sN[i] = n;
            }
            __syncthreads();
        }

        // ---- debug: per tile of this CTA, m_t, Z_tile (on the m_t scale) and S_tile
        if (p.dbg_tile_m || p.dbg_tile_z || p.dbg_count) {
            const int cpt = p.tile / kChunkRows;
            for (int t = c_lo / cpt + tid; t * cpt < c_hi; t += kThreads) {
                const int ca = t * cpt, cb = min(c_hi, ca + cpt);
                float tm = -INFINITY, tz = 0.f;
                for (int c = ca; c < cb; ++c) {
                    const u64 v = __ldcg(p.rec + rec0 + c);
                    if (v != 0ull) tm = fmaxf(tm, rec_m(v));
                }
                for (int c = ca; c < cb; ++c) {
                    const u64 v = __ldcg(p.rec + rec0 + c);
                    if (v != 0ull) tz += rec_z(v) * expf(rec_m(v) - tm);
                }
                const size_t rt = (size_t(b) * p.Hq + hq) * p.Tmax + t;
                if (p.dbg_tile_m) p.dbg_tile_m[rt] = tm;
                if (p.dbg_tile_z) p.dbg_tile_z[rt] = tz;
                if (p.dbg_count) p.dbg_count[rt] = sN[cb - c_lo] - sN[ca - c_lo];
            }
        }

        // ---- this warp's chunks, 16 at a time: in-chunk prefixes, the batch's
        // thresholds one per lane (systematic search), queued V gathers
        const int kvh = hq / p.G;
        const size_t vstride = size_t(p.Hkv) * D;
        const T *vseq = static_cast<const T *>(p.v) + size_t(start) * vstride + size_t(kvh) * D;
        const float Zf = fZ / kMassScale, invS = 1.0f / Sf;  // Z on the mass scale
        int nq = 0;  // keys queued in wl
        auto flush = [&]() {
            __syncwarp();
            const int j = wl[lane];
            gather_rows<T, D>(acc, vseq, vstride, j, nq, lane);
            nq = 0;
            __syncwarp();
        };
        for (int c0 = cw0; c0 < cw1; c0 += kP2Batch) {
            const int kend = min(kP2Batch, cw1 - c0);
            // samples of the batch's chunks: lane k < kend holds chunk k's count
            // N is non-decreasing whenever the records are what pass 1 writes; on any other
            // workspace a count could come out negative: clamp it and flag the workspace.
            int my_cnt = lane < kend ? sN[c0 - c_lo + lane + 1] - sN[c0 - c_lo + lane] : 0;
            if (my_cnt < 0) {
                raise_flag(p, SANTA_ERR_WORKSPACE);
                my_cnt = 0;
            }
            if (c0 > cw0) {  // later batches: read only the chunks that hold a threshold
#pragma unroll
                for (int k = 0; k < kP2Batch; ++k) {
                    const int c = c0 + k;
                    const int key = c * kChunkRows + lane;
                    const bool need = __shfl_sync(kFull, my_cnt, k) > 0;
                    wev[k * 32 + lane] = (need && key < L) ? __ldcg(sseq + key) : 0.f;
                }
            }
            const int cum = warp_inclusive_scan_int(my_cnt, lane);
            const int total = __shfl_sync(kFull, cum, 31);
            if (total == 0) continue;
            if (lane < kP2Batch) wcum[lane] = cum;
            // in-chunk prefixes of all chunks of the batch: 16 independent scans,
            // all loads first so that their latencies overlap, written back in place
            float ev[kP2Batch];
#pragma unroll
            for (int k = 0; k < kP2Batch; ++k) ev[k] = wev[k * 32 + lane];
            unsigned last_pos = 0;  // lane k: last positive key of chunk k
#pragma unroll
            for (int k = 0; k < kP2Batch; ++k) {
                const unsigned pos = __ballot_sync(kFull, ev[k] > 0.f);
                if (lane == k) last_pos = pos;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1)
#pragma unroll
                for (int k = 0; k < kP2Batch; ++k) {
                    const float t = __shfl_up_sync(kFull, ev[k], o);
                    if (lane >= o) ev[k] += t;
                }
#pragma unroll
            for (int k = 0; k < kP2Batch; ++k) wev[k * 32 + lane] = ev[k];
            if (lane < kP2Batch) wlast[lane] = last_pos ? 31 - __clz(last_pos) : -1;
            __syncwarp();
            for (int g0 = 0; g0 < total; g0 += 32) {
                const int nn = min(32, total - g0);
                if (nq + nn > 32) flush();
                const int g = g0 + lane;
                if (g < total) {
                    int k = 0;  // chunk of the batch that holds sample g: first k with cum[k] > g
#pragma unroll
                    for (int s = kP2Batch / 2; s > 0; s >>= 1)
                        if (wcum[k + s - 1] <= g) k += s;
                    const int c = c0 + k, i = c - c_lo;
                    int m = sN[i] + g - (k > 0 ? wcum[k - 1] : 0);
                    if (m >= p.S) {  // only on a workspace pass 1 did not fill (flagged)
                        raise_flag(p, SANTA_ERR_WORKSPACE);
                        m = p.S - 1;
                    }
                    float thr;  // threshold m of the sampler
                    if constexpr (SAMPLER == kSys)
                        thr = fmaf(float(m), invS, u);
                    else if constexpr (SAMPLER == kStrat)
                        thr = (float(m) + s_u[m]) * invS;
                    else
                        thr = s_u[m];
                    const float r = fmaf(thr, Zf, -__ull2float_rn(sC[i]) / kMassScale) / s_st[i];
                    const int len = min(kChunkRows, L - c * kChunkRows);
                    const int j = c * kChunkRows + cdf_search(wev + k * 32, len, r, wlast[k]);
                    int row = j;  // row of V relative to vseq
                    if constexpr (kPaged) {
                        const int pg = s_pg[j / p.page_size - pg_lo];
                        if (pg < 0 || pg >= p.num_pages) {  // bad page id: flagged, row 0 read instead
                            raise_flag(p, SANTA_ERR_INDPTR);
                            row = 0;
                        } else {
                            row = pg * p.page_size + j % p.page_size;
                        }
                    }
                    wl[nq + lane] = row;
                    if (p.dbg_idx) p.dbg_idx[(size_t(b) * p.Hq + hq) * p.S + m] = j;
                }
                nq += nn;
            }
            __syncwarp();
        }
        if (nq > 0) flush();
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
    if (split == 0) {
        if (tid < D) {
            float s = 0.f;
            for (int k = 0; k < int(gridDim.x); ++k) s += part[k * D + tid];
            p.out[head * D + tid] = L > 0 ? s / float(p.S) : 0.f;
        }
        // every CTA of the cluster is past its reads of the records: set them and the
        // head's published-chunk count back to 0 for the next call
        for (int c = tid; c < Nb; c += kThreads) p.rec[rec0 + c] = 0ull;
        if (tid == 0) p.cnt[head] = 0u;
    }
}


}  // namespace santa
