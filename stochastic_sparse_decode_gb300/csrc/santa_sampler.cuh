// santa_sampler.cuh -- the S2ANTA-prop sampler of one (sequence, query head), and
// the fused prop kernel that runs it (pass 1, then the samplers, in one persistent
// grid).
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (paper notes, Key
// design 2): pass 1 leaves exponentiated scores and one partition record per
// block of keys; a reducer forms Z from the records and places the systematic
// thresholds U + m/S (Key design 1) on the global CDF, a block's budget being the
// number of thresholds in its CDF interval; pass 2 searches the stashed in-block
// CDF for each threshold and averages the chosen V rows.  Here a block is a
// 32-key chunk, and nsplit CTAs of kSampWarps warps serve one head (its splits):
// each runs steps 1-3 on all of the head's records, and then samples its own
// share of the S thresholds:
//
//   1. records.  The head's chunk records, one 64-bit word (m_c, z_c) each, are
//      read into registers, kSampReg consecutive chunks per thread (kSampBlock
//      chunks at a time).  In the fused kernel the sampler polls them, and the
//      head's count of chunks published by pass 1, until every chunk is in: the
//      wait and the read are the same round trips.
//   2. reducer.  M = max_c m_c; the masses w_c = z_c exp(m_c - M) as 64-bit
//      fixed-point integers (w 2^40), so the inclusive prefix C_c is exact and
//      order-independent: non-decreasing, and the same in every launch mode.
//      Z = C_{N_b - 1}.  Chunk c holds the thresholds m in [N(C_{c-1}), N(C_c)),
//      N(c) = clamp(ceil(S c / Z - S U), 0, S), N(C_{-1}) = 0, N(C_{N_b - 1}) = S
//      (the stratified and i.i.d. samplers only change N and the threshold values).
//   3. list.  The chunks that hold a threshold are listed, kSampList at a time;
//      the list's thresholds are shared evenly among the warps, 32 at a time (one
//      per lane): a warp loads the stashed scores of the chunks its thresholds fall
//      in, in one round trip (cp.async into shared memory), scans them into
//      in-chunk prefixes, then each lane takes its threshold:
//      r_m = (t_m Z - C_{c-1}) / exp(m_c - M) on the chunk's own scale, the
//      smallest key whose prefix exceeds r_m (clamped to the chunk's keys of
//      positive score); the 32 lanes' V rows are then gathered together.
//   4. the split's sum = the sum of its warps' sums, in warp order; the split that
//      finishes last adds the splits' sums in split order (a counter in the
//      workspace, no wait): out = total / S.  It then sets the head's record words
//      and published-chunk count back to 0 for the next call.
//
// The work of one head is a chain of dependent steps, so it is spread over all
// warps of the CTA: a few chunks per thread in the reducer, a few list entries per
// warp, and every V row of a warp in flight at once.
//
// Every index derived from workspace data is clamped: a count below zero or a
// sample number at or above S (possible only on a workspace that pass 1 did not
// fill) is clamped and raises SANTA_ERR_WORKSPACE.
#pragma once

#include "santa_common.cuh"
#include "santa_stream.cuh"
#include "santa_tile.cuh"

namespace santa {

constexpr int kSampWarps = kChunkWarps;                 // the sampler: every warp of a CTA
constexpr int kSampThreads = kSampWarps * 32;
constexpr int kSampReg = 4;                             // chunk records per thread and block
constexpr int kSampBlock = kSampThreads * kSampReg;     // chunks per block of the reducer
constexpr int kSampList = kSampThreads;                 // listed chunks per round
// Row stride of a warp's in-chunk prefixes, in floats: 36 = 9 x 16 bytes keeps every
// row 16-byte aligned for cp.async and staggers the rows over the shared-memory
// banks (4 k mod 32), so the lanes' binary searches in different rows collide at
// most four to a bank.
constexpr int kEvStride = 36;
// The reducer's masses are summed as integers: w 2^40 rounded.  The largest chunk
// mass is <= 32 (a chunk's maximum key has e = 1 at the global maximum) and a
// sequence has at most 2^17 chunks here, so a sum stays below 2^62; the absolute
// error, <= 2^-41 per chunk, is below 2^-24 of Z >= 1.
constexpr float kMassScale = 1099511627776.0f;  // 2^40
constexpr int kRankSortMax = 512;               // i.i.d. uniforms up to this many are sorted by rank

// Shared-memory floats for the uniforms of a stratified / i.i.d. call: S rounded up
// to a power of two (the i.i.d. sampler sorts them; a rank sort needs a second
// array), 0 for the systematic sampler.
__host__ __device__ inline int sampler_slots(int sampler, int S) {
    if (sampler == kSys) return 0;
    int n = 1;
    while (n < S) n <<= 1;
    return (sampler == kIid && n <= kRankSortMax) ? 2 * n : n;
}

// Sampler shared memory (offsets from a 16-byte aligned base): the list of
// sampled chunks (C_{c-1}, chunk, first threshold, count, 1 / exp(m_c - M)), per
// warp 32 x kEvStride in-chunk prefixes, the last positive key and page id of each
// of those 32 chunks, per warp the D-float sums, scratch, and the uniforms.
template <int D>
struct SampSmem {
    static constexpr size_t kCp = 0;                                       // float [kSampList]
    static constexpr size_t kC = kCp + size_t(kSampList) * 4;              // int
    static constexpr size_t kN0 = kC + size_t(kSampList) * 4;              // int
    static constexpr size_t kCnt = kN0 + size_t(kSampList) * 4;            // int
    static constexpr size_t kIst = kCnt + size_t(kSampList) * 4;           // float
    static constexpr size_t kEv = kIst + size_t(kSampList) * 4;            // float [warps][32][kEvStride]
    static constexpr size_t kLast = kEv + size_t(kSampWarps) * 32 * kEvStride * 4;  // int [warps][32]
    static constexpr size_t kPg = kLast + size_t(kSampWarps) * 32 * 4;     // int [warps][32]
    static constexpr size_t kRed = kPg + size_t(kSampWarps) * 32 * 4;      // float [warps][D]
    static constexpr size_t kScr = kRed + size_t(kSampWarps) * D * 4;      // u64 [2][warps]
    static constexpr size_t kScrF = kScr + size_t(2) * kSampWarps * 8;     // float [warps]
    static constexpr size_t kScrI = kScrF + size_t(kSampWarps) * 4;        // int [2][warps] + 1
    static constexpr size_t kU = (kScrI + size_t(2 * kSampWarps + 1) * 4 + 15) & ~size_t(15);  // float [nu]
    static __host__ __device__ size_t bytes(int nu) { return kU + size_t(nu) * 4; }
};

// ---- small helpers

// Barrier of the sampler's threads (named barrier 1).
__device__ __forceinline__ void samp_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSampThreads) : "memory"); }
// The same barrier, returning whether any sampler thread passed `pred`.
__device__ __forceinline__ bool samp_sync_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "n"(kSampThreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
// 16-byte asynchronous copy global -> shared (L2 only); bytes past src_bytes are zero-filled.
__device__ __forceinline__ void cp_async_16(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ float rec_m(unsigned long long v) { return __uint_as_float(uint32_t(v)); }
__device__ __forceinline__ float rec_z(unsigned long long v) { return __uint_as_float(uint32_t(v >> 32)); }

// Exclusive prefix over the sampler's threads of an integer; *total is the sum of
// all.  `scr` holds two alternating sets of per-warp totals (parity).
template <typename I>
__device__ __forceinline__ I samp_exclusive(I v, I *scr, int parity, I *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    I incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const I u = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += u;
    }
    I *ws = scr + kSampWarps * parity;
    if (lane == 31) ws[warp] = incl;
    samp_sync();
    I off = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kSampWarps; ++w) {
        const I t = ws[w];
        if (w < warp) off += t;
        tot += t;
    }
    *total = tot;
    return off + incl - v;
}

// Ascending sort of a[0, n) into out[0, n) by rank, in one pass (element i goes to
// #{k : a[k] < a[i]} + #{k < i : a[k] == a[i]}).  Ends with a sampler barrier.
__device__ __forceinline__ void samp_rank_sort(const float *a, float *out, int n, int tid) {
    for (int i = tid; i < n; i += kSampThreads) {
        const float x = a[i];
        int r = 0;
        for (int k = 0; k < n; ++k) {
            const float y = a[k];
            r += (y < x || (y == x && k < i)) ? 1 : 0;
        }
        out[r] = x;
    }
    samp_sync();
}

// Ascending bitonic sort of a[0, n) (n a power of two) by the sampler's threads.
__device__ __forceinline__ void samp_bitonic_sort(float *a, int n, int tid) {
    for (int k = 2; k <= n; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < n; i += kSampThreads) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const float x = a[i], y = a[ixj];
                    if ((x > y) == ((i & k) == 0)) {
                        a[i] = y;
                        a[ixj] = x;
                    }
                }
            }
            samp_sync();
        }
}

// Adds V rows (one index per lane of `j`, the first n lanes) of one KV head to the
// lane's slice accumulator (D/32 consecutive elements at lane D/32), rows added in
// lane order.  The raw slices of up to 16 rows are in flight at once, held
// undecoded (32 rows for slices of up to 8 bytes measured no faster and spilled).
template <typename T, int D>
__device__ __forceinline__ void gather_queue(float (&acc)[D / 32], const T *vrow0, size_t row_stride, int j, int n,
                                             int lane) {
    constexpr int kE = D / 32;
    constexpr int kBytes = kE * int(sizeof(T));  // 4, 8 or 16
    constexpr int kWords = kBytes / 4;
    constexpr int kFlight = 16;
    for (int r0 = 0; r0 < n; r0 += kFlight) {
        uint32_t raw[kFlight][kWords];
#pragma unroll
        for (int r = 0; r < kFlight; ++r) {
            const int jr = __shfl_sync(kFull, j, (r0 + r) & 31);
            if (r0 + r < n) {
                const unsigned char *src = reinterpret_cast<const unsigned char *>(vrow0 + size_t(jr) * row_stride) +
                                           lane * kBytes;
                if constexpr (kWords == 1) {
                    raw[r][0] = __ldg(reinterpret_cast<const unsigned int *>(src));
                } else if constexpr (kWords == 2) {
                    const uint2 w = __ldg(reinterpret_cast<const uint2 *>(src));
                    raw[r][0] = w.x;
                    raw[r][1] = w.y;
                } else {
                    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(src));
                    raw[r][0] = w.x;
                    raw[r][1] = w.y;
                    raw[r][2] = w.z;
                    raw[r][3] = w.w;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kFlight; ++r)
            if (r0 + r < n) {
                RowSlice<T, D> row;
                row.unpack_words(raw[r]);
#pragma unroll
                for (int e = 0; e < kE; ++e) acc[e] += row.v[e];
            }
    }
}

// Threshold counts and values of the three samplers of Key design 1.
template <int SAMPLER>
struct Thresholds {
    int S;
    float Sf, SU, invS, u;
    const float *su;  // stratified: u_m; i.i.d.: the sorted u
    // Number of thresholds below the normalised CDF value cn (monotone in cn).
    __device__ __forceinline__ int below(float cn) const {
        if constexpr (SAMPLER == kSys) {  // U + m/S < cn  <=>  m < S cn - S U
            return int(fminf(fmaxf(ceilf(fmaf(Sf, cn, -SU)), 0.f), Sf));
        } else if constexpr (SAMPLER == kStrat) {  // (m + u_m)/S < cn: all m < floor(S cn), maybe one more
            const float y = Sf * cn;
            const int k = int(fminf(fmaxf(floorf(y), 0.f), Sf));
            return k + ((k < S && su[k] < y - float(k)) ? 1 : 0);
        } else {  // sorted u_s < cn
            int lo = 0, hi = S;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (su[mid] < cn)
                    lo = mid + 1;
                else
                    hi = mid;
            }
            return lo;
        }
    }
    // Threshold m, in [0, 1).
    __device__ __forceinline__ float value(int m) const {
        if constexpr (SAMPLER == kSys)
            return fmaf(float(m), invS, u);
        else if constexpr (SAMPLER == kStrat)
            return (float(m) + su[m]) * invS;
        else
            return su[m];
    }
};

// ---- the sampler of one head
//
// Run by the kSampThreads threads of a CTA (tid = threadIdx.x, all warps, converged),
// after the CTA's own streaming: it polls for the chunks that pass 1 (other CTAs)
// has not finished yet.  *give_up: set after a wait timed out (the grid's later
// heads are not waited for).
template <typename T, int D, int SAMPLER, bool kPaged>
__device__ void sample_head(const Params &p, int b, int hq, int split, unsigned char *sm, int tid, bool *give_up) {
    using L = SampSmem<D>;
    using u64 = unsigned long long;
    constexpr int kE = D / 32;
    const int warp = tid >> 5, lane = tid & 31;
    float *l_cp = reinterpret_cast<float *>(sm + L::kCp);
    int *l_c = reinterpret_cast<int *>(sm + L::kC);
    int *l_n0 = reinterpret_cast<int *>(sm + L::kN0);
    int *l_cnt = reinterpret_cast<int *>(sm + L::kCnt);
    float *l_ist = reinterpret_cast<float *>(sm + L::kIst);
    float *wev = reinterpret_cast<float *>(sm + L::kEv) + warp * 32 * kEvStride;
    int *wlast = reinterpret_cast<int *>(sm + L::kLast) + warp * 32;
    int *wpg = reinterpret_cast<int *>(sm + L::kPg) + warp * 32;
    float *red = reinterpret_cast<float *>(sm + L::kRed);
    u64 *scr64 = reinterpret_cast<u64 *>(sm + L::kScr);
    float *scrf = reinterpret_cast<float *>(sm + L::kScrF);
    int *scri = reinterpret_cast<int *>(sm + L::kScrI);
    float *s_u = reinterpret_cast<float *>(sm + L::kU);

    const size_t head = size_t(b) * p.Hq + hq;
    float *outp = p.out + head * D;
    long long start;
    long long ind0, ind1;
    raw_bounds<kPaged>(p, b, &ind0, &ind1);
    const int Lb = checked_bounds(p, ind0, ind1, &start);
    const int Nb = (Lb + kChunkRows - 1) / kChunkRows;
    // this split's thresholds: [s_lo, s_hi)
    const int s_lo = int((long long)p.S * split / p.nsplit), s_hi = int((long long)p.S * (split + 1) / p.nsplit);

    // the thresholds' parameters (uniforms checked into range; the i.i.d. ones sorted)
    Thresholds<SAMPLER> th;
    th.S = p.S;
    th.Sf = float(p.S);
    th.invS = 1.0f / th.Sf;
    th.u = SAMPLER == kSys ? checked_offset(p, p.U[head]) : 0.f;
    th.SU = th.Sf * th.u;
    th.su = s_u;
    if constexpr (SAMPLER != kSys) {
        int nu = 1;
        while (nu < p.S) nu <<= 1;
        const float *ug = p.u_samples + head * p.S;
        for (int i = tid; i < nu; i += kSampThreads) {
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
        samp_sync();
        if constexpr (SAMPLER == kIid) {
            if (nu <= kRankSortMax) {
                samp_rank_sort(s_u, s_u + nu, nu, tid);
                th.su = s_u + nu;
            } else {
                samp_bitonic_sort(s_u, nu, tid);
            }
        }
    }

    // a workspace poisoned by an earlier timeout holds records nobody will reset
    bool stop = *give_up;
    if (tid == 0) scri[2 * kSampWarps] = stop ? 0 : int(*reinterpret_cast<volatile unsigned int *>(p.hdr));
    samp_sync();
    if (scri[2 * kSampWarps] != 0) {
        if (tid == 0) raise_flag(p, SANTA_ERR_WORKSPACE);
        stop = true;
    }
    if (Nb == 0 || stop) {
        samp_sync();  // the scratch is reused by the next head
        if (tid < D) outp[tid] = 0.f;
        return;
    }

    unsigned long long *recs = p.rec + head * p.nch;
    const int nblk = (Nb + kSampBlock - 1) / kSampBlock;
    // wait_cycles < 0 (a test of the timeout path): wait |wait_cycles| for one chunk
    // more than the head has, a publication that never comes
    const long long limit = p.wait_cycles > 0 ? p.wait_cycles : p.wait_cycles < 0 ? -p.wait_cycles : kWaitCycles;
    const unsigned target = unsigned(Nb) + (p.wait_cycles < 0 ? 1u : 0u);

    // ---- 1. records (and, in the fused kernel, the wait for them); M
    // A head is complete when every chunk record is written and pass 1 has published
    // all N_b chunks to it (its counter): the publication's fence makes the stash
    // visible too.  Both are polled in the same round trips.
    const unsigned int *cntp = p.cnt + head;
    u64 r[kSampReg];
    float mx = -INFINITY;
    bool timed_out = false, empty_rec = false;
    for (int blk = 0; blk < nblk; ++blk) {
        const int c0 = blk * kSampBlock + tid * kSampReg;
        int missing = 0;
#pragma unroll
        for (int i = 0; i < kSampReg; ++i) {
            r[i] = c0 + i < Nb ? ld_relaxed_u64(recs + c0 + i) : 0ull;
            missing += (c0 + i < Nb && r[i] == 0ull) ? 1 : 0;
        }
        unsigned pub = ld_relaxed_u32(cntp);
        const long long t0 = clock64();
        while (missing > 0 || pub < target) {
            if (clock64() - t0 > limit) {
                timed_out = true;
                break;
            }
            __nanosleep(missing > 1 ? 128 : 32);
            missing = 0;
#pragma unroll
            for (int i = 0; i < kSampReg; ++i)
                if (c0 + i < Nb && r[i] == 0ull) {
                    r[i] = ld_relaxed_u64(recs + c0 + i);
                    missing += r[i] == 0ull ? 1 : 0;
                }
            pub = ld_relaxed_u32(cntp);
        }
        empty_rec |= missing > 0 || pub != unsigned(Nb);
#pragma unroll
        for (int i = 0; i < kSampReg; ++i)
            if (c0 + i < Nb && r[i] != 0ull) mx = fmaxf(mx, rec_m(r[i]));
    }
    // Acquire side of the publication: the stash written before it is visible to
    // every load below (each thread fences after its own observation of the counter,
    // and the barrier below orders that before every thread's later loads).
    __threadfence();
    // the largest-logit offsets of this thread's chunks (one word: four bytes), for
    // the prefetch below
    const int ca0 = (nblk - 1) * kSampBlock + tid * kSampReg;
    const unsigned amx = (nblk == 1 && ca0 < Nb && !kPaged)
                             ? __ldcg(reinterpret_cast<const unsigned *>(p.amax + head * p.nch4 + ca0))
                             : 0u;
    // One barrier for M, a wait that timed out and a record pass 1 did not write.
    mx = warp_max(mx);
    const bool w_to = __any_sync(kFull, timed_out), w_em = __any_sync(kFull, empty_rec);
    if (lane == 0) {
        scrf[warp] = mx;
        scri[warp] = (w_to ? 1 : 0) | (w_em ? 2 : 0);
    }
    samp_sync();
    float M = scrf[0];
    int wflags = scri[0];
#pragma unroll
    for (int w = 1; w < kSampWarps; ++w) {
        M = fmaxf(M, scrf[w]);
        wflags |= scri[w];
    }
    if (wflags & 1) {
        // SANTA_ERR_TIMEOUT with location code 3 (a sampler waiting for its head's
        // scores); the records of this call will never be reset: poison the workspace
        if (tid == 0) {
            raise_flag(p, SANTA_ERR_TIMEOUT | (3u << 8));
            atomicExch(p.hdr, 1u);
        }
        *give_up = true;
        if (tid < D) outp[tid] = 0.f;
        samp_sync();  // the scratch is reused by the next head
        return;
    }
    // a record pass 1 did not write (no mass), or a count that disagrees
    if (tid == 0 && (wflags & 2)) raise_flag(p, SANTA_ERR_WORKSPACE);
    // V rows that the gather will most likely read, fetched into L2 while the list is
    // formed: the largest key of every chunk that may hold a sample (each split of the
    // head takes every nsplit-th chunk).  A chunk's share of the mass is at most
    // 32 exp(m_c - M) (Z >= 1), below 1e-4 when m_c < M - 13, so those are skipped.
    // (Only when the head's records fit one block; a prefetch changes no result.)
    auto prefetch_v = [&]() {
        if (nblk != 1 || kPaged) return;
        const unsigned char *vb = static_cast<const unsigned char *>(p.v) +
                                  ((size_t(start) * p.Hkv + hq / p.G) * D) * sizeof(T);
#pragma unroll
        for (int i = 0; i < kSampReg; ++i) {
            const int c = ca0 + i;
            if (c < Nb && c % p.nsplit == split && r[i] != 0ull && rec_m(r[i]) >= M - 13.f) {
                const int key = c * kChunkRows + int((amx >> (8 * i)) & 31u);
                if (key < Lb) {
                    const unsigned char *row = vb + size_t(key) * p.Hkv * D * sizeof(T);
#pragma unroll
                    for (int off = 0; off < D * int(sizeof(T)); off += 128)
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
                }
            }
        }
    };

    // masses of the thread's chunks of block blk (records in r), inclusive local prefix
    auto masses = [&](int blk, u64 (&pl)[kSampReg]) {
        const int c0 = blk * kSampBlock + tid * kSampReg;
        u64 run = 0;
#pragma unroll
        for (int i = 0; i < kSampReg; ++i) {
            if (c0 + i < Nb && r[i] != 0ull)
                run += (u64)__float2ll_rn(rec_z(r[i]) * __expf(rec_m(r[i]) - M) * kMassScale);
            pl[i] = run;
        }
        return run;
    };
    auto reload = [&](int blk) {
        const int c0 = blk * kSampBlock + tid * kSampReg;
#pragma unroll
        for (int i = 0; i < kSampReg; ++i) r[i] = c0 + i < Nb ? __ldcg(recs + c0 + i) : 0ull;
    };

    // ---- 2. Z (one extra pass over the records when they span several blocks)
    u64 pl[kSampReg];
    u64 Z = 0;
    int par = 0;
    if (nblk > 1) {
        for (int blk = 0; blk < nblk; ++blk) {
            reload(blk);
            u64 bt;
            samp_exclusive<u64>(masses(blk, pl), scr64, par, &bt);
            par ^= 1;
            Z += bt;
        }
    }
    const int cpt = p.tile / kChunkRows;  // chunks per tile (debug outputs)
    const bool dbg_tiles = p.dbg_tile_m || p.dbg_tile_z || p.dbg_count;
    const T *vseq = static_cast<const T *>(p.v) + (kPaged ? size_t(0) : size_t(start) * p.Hkv * D) + size_t(hq / p.G) * D;
    const size_t vstride = size_t(p.Hkv) * D;
    const float *sseq = p.stash + head * size_t(p.nch) * kChunkRows;

    float acc[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) acc[e] = 0.f;

    // ---- 3. per block: C, N, counts; the list of chunks with samples, kSampList per round
    u64 carry = 0;
    float Zf = 0.f, rZ = 0.f;
    for (int blk = 0; blk < nblk; ++blk) {
        if (nblk > 1) reload(blk);
        const int c0 = blk * kSampBlock + tid * kSampReg;
        u64 bt;
        const u64 base = carry + samp_exclusive<u64>(masses(blk, pl), scr64, par, &bt);
        par ^= 1;
        if (nblk == 1) Z = bt;
        prefetch_v();
        const float fZ = __ull2float_rn(Z);
        Zf = fZ / kMassScale;
        rZ = 1.0f / fZ;
        // per chunk: 1 / exp(m_c - M), C_{c-1} as a float, and N(C_c); the counts are the
        // differences of N.  N is non-decreasing on any workspace pass 1 filled; on any
        // other it is made so here (a count that would be negative is 0, flagged), which
        // keeps every sample number below S.
        float ist[kSampReg], cpf[kSampReg];
        int nN[kSampReg];
        const int nfirst = c0 == 0 ? 0 : th.below(__ull2float_rn(base) * rZ);
        int nprev = nfirst, nsel = 0;
        bool clamped = false;
#pragma unroll
        for (int i = 0; i < kSampReg; ++i) {
            const int c = c0 + i;
            ist[i] = (c < Nb && r[i] != 0ull) ? __expf(M - rec_m(r[i])) : 0.f;
            cpf[i] = __ull2float_rn(base + (i > 0 ? pl[i - 1] : 0ull));
            int n = nprev;
            if (c < Nb) n = c == Nb - 1 ? p.S : th.below(__ull2float_rn(base + pl[i]) * rZ);
            if (n < nprev) {
                clamped = true;
                n = nprev;
            }
            nsel += n > nprev ? 1 : 0;
            nN[i] = n;
            nprev = n;
        }
        if (clamped) raise_flag(p, SANTA_ERR_WORKSPACE);

        // debug: m_t, Z_tile (on the m_t scale) and S_tile of the tiles of this block,
        // from the records (still in place) and the N values, staged in shared memory
        // (the list area is free until the list is built below)
        if (dbg_tiles && split == 0) {
            int *sN = reinterpret_cast<int *>(sm + L::kEv);  // kSampBlock + 1 ints fit in the prefix buffers
#pragma unroll
            for (int i = 0; i < kSampReg; ++i) sN[tid * kSampReg + i + 1] = nN[i];
            if (tid == 0) sN[0] = nfirst;
            samp_sync();
            const int cb = blk * kSampBlock;  // a block is a whole number of tiles
            const int nt = (min(Nb - cb, kSampBlock) + cpt - 1) / cpt;
            for (int t = tid; t < nt; t += kSampThreads) {
                const int ca = cb + t * cpt, ce = min(Nb, ca + cpt);
                float tm = -INFINITY, tz = 0.f;
                for (int c = ca; c < ce; ++c) {
                    const unsigned long long v = __ldcg(recs + c);
                    if (v != 0ull) tm = fmaxf(tm, rec_m(v));
                }
                for (int c = ca; c < ce; ++c) {
                    const unsigned long long v = __ldcg(recs + c);
                    if (v != 0ull) tz += rec_z(v) * expf(rec_m(v) - tm);
                }
                const size_t rt = head * p.Tmax + ca / cpt;
                if (p.dbg_tile_m) p.dbg_tile_m[rt] = tm;
                if (p.dbg_tile_z) p.dbg_tile_z[rt] = tz;
                if (p.dbg_count) p.dbg_count[rt] = sN[ce - cb] - sN[ca - cb];
            }
            samp_sync();
        }
        int ntot;
        const int off = samp_exclusive<int>(nsel, scri, par, &ntot);
        par ^= 1;
        for (int r0 = 0; r0 < ntot; r0 += kSampList) {
            // this round's list entries
            int e = off;
#pragma unroll
            for (int i = 0; i < kSampReg; ++i) {
                const int n0 = i > 0 ? nN[i - 1] : nfirst;
                if (nN[i] > n0) {
                    if (e >= r0 && e < r0 + kSampList) {
                        const int s = e - r0;
                        l_c[s] = c0 + i;
                        l_n0[s] = n0;
                        l_cnt[s] = nN[i] - n0;
                        l_ist[s] = ist[i];
                        l_cp[s] = cpf[i];
                    }
                    ++e;
                }
            }
            samp_sync();
            const int nl = min(kSampList, ntot - r0);
            // The round's samples are the thresholds [l_n0[0], l_n0[nl-1] + l_cnt[nl-1])
            // (each entry holds l_cnt of them from l_n0 on); this split takes those in
            // [s_lo, s_hi), every warp an even share of them, 32 at a time: lane = one
            // threshold, its entry found by a binary search over l_n0.
            const int m_first = max(l_n0[0], s_lo), m_end = min(l_n0[nl - 1] + l_cnt[nl - 1], s_hi);
            const int per = max(0, m_end - m_first + kSampWarps - 1) / kSampWarps;
            const int ws0 = m_first + warp * per, ws1 = min(ws0 + per, m_end);
            for (int g0 = ws0; g0 < ws1; g0 += 32) {
                const int nn = min(32, ws1 - g0);
                const int g = g0 + min(lane, nn - 1);  // lanes past nn repeat the last sample
                int lo = 0, hi = nl - 1;  // the last entry whose first threshold is <= g
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (l_n0[mid] <= g)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                // the warp's entries: ea .. ea + ne - 1, at most one per sample
                const int ea = __shfl_sync(kFull, lo, 0);
                int ne = __shfl_sync(kFull, lo, nn - 1) - ea + 1;
                if (ne < 1 || ne > 32) {  // only on a workspace pass 1 did not fill (flagged)
                    raise_flag(p, SANTA_ERR_WORKSPACE);
                    ne = ne < 1 ? 1 : 32;
                }
                // Their stashed scores into the warp's rows, global to shared memory without
                // a register on the way (cp.async); 16 bytes per copy, lane l copies pieces l, l + 32, ... of the
                // ne x 8 pieces; keys past the sequence's end read as 0.
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int pi = lane + 32 * j, k = pi >> 3, q = pi & 7;
                    if (k < ne) {
                        const int ck = l_c[ea + k];
                        const int valid = min(max(Lb - ck * kChunkRows - 4 * q, 0), 4);
                        cp_async_16(wev + k * kEvStride + 4 * q, sseq + size_t(ck) * kChunkRows + 4 * q, 4 * valid);
                    }
                }
                if constexpr (kPaged) {
                    if (lane < ne) {
                        const int ck = l_c[ea + lane];
                        int pg = __ldg(p.page_table + size_t(b) * p.max_pages + (ck * kChunkRows) / p.page_size);
                        if (pg < 0 || pg >= p.num_pages) {  // bad page id: flagged, row 0 read instead
                            raise_flag(p, SANTA_ERR_INDPTR);
                            pg = -1;
                        }
                        wpg[lane] = pg;
                    }
                }
                cp_async_wait_all();
                __syncwarp();
                // in-chunk inclusive prefixes, eight chunks at a time, written back in place
                unsigned lastbits = 0;  // lane k: positive keys of entry ea + k
                for (int k0 = 0; k0 < ne; k0 += 8) {
                    float ev[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) ev[k] = wev[(k0 + k) * kEvStride + lane];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const unsigned pos = __ballot_sync(kFull, ev[k] > 0.f);
                        if (lane == k0 + k) lastbits = pos;
                    }
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1)
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float t = __shfl_up_sync(kFull, ev[k], o);
                            if (lane >= o) ev[k] += t;
                        }
#pragma unroll
                    for (int k = 0; k < 8; ++k) wev[(k0 + k) * kEvStride + lane] = ev[k];
                }
                wlast[lane] = lastbits ? 31 - __clz(lastbits) : -1;
                __syncwarp();
                int row = 0;  // row of V relative to vseq
                if (lane < nn) {
                    int k = lo - ea;
                    if (k < 0 || k >= ne) {  // only on a workspace pass 1 did not fill (flagged)
                        raise_flag(p, SANTA_ERR_WORKSPACE);
                        k = k < 0 ? 0 : ne - 1;
                    }
                    const int ek = ea + k;
                    int m = g;
                    if (m >= p.S || m < 0) {  // only on a workspace pass 1 did not fill (flagged)
                        raise_flag(p, SANTA_ERR_WORKSPACE);
                        m = m < 0 ? 0 : p.S - 1;
                    }
                    const float rr = fmaf(th.value(m), Zf, -l_cp[ek] / kMassScale) * l_ist[ek];
                    const int c = l_c[ek];
                    const int len = min(kChunkRows, Lb - c * kChunkRows);
                    const int j = c * kChunkRows + cdf_search(wev + k * kEvStride, len, rr, wlast[k]);
                    row = j;
                    if constexpr (kPaged) {
                        const int pg = wpg[k];
                        row = pg < 0 ? 0 : pg * p.page_size + j % p.page_size;
                    }
                    if (p.dbg_idx) p.dbg_idx[head * p.S + m] = j;
                }
                gather_queue<T, D>(acc, vseq, vstride, row, nn, lane);
                __syncwarp();  // the prefixes are rewritten by the next 32
            }
            samp_sync();  // the list is rewritten by the next round
        }
        carry += bt;
    }

    // ---- 4. the warps' sums in warp order: the split's sum.  One split: out = sum / S.
    // Several: each stores its sum, then counts itself in (after a fence) on the
    // head's counter, which pass 1 set to 0; the split that counts last adds the
    // splits' sums in split order, out = total / S.  The last one also sets the
    // head's records and published-chunk count back to 0 for the next call (every
    // split has read them by then).
#pragma unroll
    for (int e = 0; e < kE; ++e) red[warp * D + lane * kE + e] = acc[e];
    samp_sync();
    float sum = 0.f;
    if (tid < D) {
#pragma unroll
        for (int w = 0; w < kSampWarps; ++w) sum += red[w * D + tid];
    }
    const int ns = p.nsplit;
    bool last = true;
    if (ns > 1) {
        if (tid < D) p.part[(head * ns + split) * D + tid] = sum;
        __threadfence();
        samp_sync();
        if (tid == 0) {
            const unsigned before = atomicAdd(p.done + head, 1u);
            // before >= ns: a counter pass 1 did not set (a workspace it did not fill);
            // each split then writes its own sum, flagged
            scri[2 * kSampWarps] = before < unsigned(ns) ? (before == unsigned(ns - 1) ? 1 : 0) : 2;
            if (before >= unsigned(ns)) raise_flag(p, SANTA_ERR_WORKSPACE);
        }
        samp_sync();
        const int verdict = scri[2 * kSampWarps];
        last = verdict == 1;
        if (verdict == 2 && tid < D) outp[tid] = sum / float(p.S);
        if (last) {
            __threadfence();  // acquire: the other splits' sums
            if (tid < D) {
                float tot = 0.f;
                for (int k = 0; k < ns; ++k) tot += __ldcg(p.part + (head * ns + k) * D + tid);
                sum = tot;
            }
        }
    }
    if (last) {
        if (tid < D) outp[tid] = sum / float(p.S);
        if (tid == 0) p.cnt[head] = 0u;
        for (int c = tid; c < Nb; c += kSampThreads) recs[c] = 0ull;
    }
    samp_sync();  // red and the scratch are reused by the next head
}

// ---- kernels

// Shared memory of the fused kernel: the streaming layout, which the samplers then
// reuse from its start once the CTA's stream is done (its chunk buffers are idle and
// its mbarriers invalidated).
template <typename T, int D, int G>
__host__ __device__ inline size_t fused_smem_bytes(int nbuf, int nu) {
    const size_t s1 = ChunkGeom<T, D, G>::bytes(nbuf);
    const size_t s2 = 1024 + SampSmem<D>::bytes((nu + 3) & ~3);
    return s1 > s2 ? s1 : s2;
}

// Fused S2ANTA-prop: one persistent CTA of kChunkWarps warps per SM.  The warps first
// stream their CTA's share of K (pass 1, as prop_stream_kernel), then serve as the
// sampler of the items blockIdx.x, blockIdx.x + gridDim.x, ... (item = head x
// nsplit + split), each as soon as its head's records are complete.  Every CTA must
// be resident at once: a sampler waits on records that the streaming warps of other
// CTAs write (a bounded wait), and no streaming warp ever waits on a sampler.
template <typename T, int D, int G, int SAMPLER, bool kPaged>
__global__ void __launch_bounds__(kChunkWarps * 32, 1)
    prop_fused_kernel(const __grid_constant__ CUtensorMap kmap, const Params p, int nbuf) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align1024(smem_raw);
    // a flag in the spare bytes after the streaming layout's claim counter
    volatile int *s_failed = reinterpret_cast<volatile int *>(smem + ChunkGeom<T, D, G>::next_off(nbuf) + 8);
    stream_setup<T, D, G>(kmap, smem, nbuf);
    if (threadIdx.x == 0) *s_failed = 0;
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();
    const bool failed = stream_chunks<T, D, G, kPaged, true>(kmap, p, nbuf, smem);
    if (failed && (threadIdx.x & 31) == 0) *s_failed = 1;
    __syncthreads();  // the CTA's stream is done: its chunk buffers are the samplers' now
    // a warp whose copy timed out may have left a copy in flight into the buffers:
    // then this CTA samples nothing (its heads read as zeros, the timeout is flagged)
    bool give_up = *s_failed != 0;
    const long long items = (long long)p.B * p.Hq * p.nsplit;
    for (long long it = blockIdx.x; it < items; it += gridDim.x) {
        const long long head = it / p.nsplit;
        if (give_up) {
            if (threadIdx.x < D) p.out[size_t(head) * D + threadIdx.x] = 0.f;
            continue;
        }
        sample_head<T, D, SAMPLER, kPaged>(p, int(head / p.Hq), int(head % p.Hq), int(it % p.nsplit), smem,
                                           int(threadIdx.x), &give_up);
    }
}

}  // namespace santa
