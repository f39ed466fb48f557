// santa_common.cuh -- device helpers shared by the decode kernels (sm_103a).
//
// PTX wrappers for the asynchronous-copy machinery (mbarrier, TMA tensor loads,
// programmatic dependent launch), warp/block scans and reductions, bf16
// unpacking, and the parameter block every kernel receives.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "santa_decode.h"

namespace santa {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMergeThreads = 256;
constexpr int kExactCtaBound = 160;  // exact: streaming CTAs at most (the workspace is sized for it)
constexpr long long kWaitCycles = 1LL << 31;  // ~1 s: bound on any wait for a copy
constexpr int kPropMaxSplit = 8;  // prop: CTAs sharing one head's thresholds, at most
constexpr int kMaxBernoulliDraws = 64;  // Bernoulli score stage: draws per feature, at most

enum Mode { kProp = 0, kFlash = 1, kExact = 2 };
// Thresholds of the prop sampler ("Stochastic Sparse Attention for Memory-Bound
// Inference", paper notes, Key design 1): systematic U + m/S, stratified
// (m + u_m)/S, or i.i.d. u_s (taken in increasing order).
enum Sampler { kSys = 0, kStrat = 1, kIid = 2 };
constexpr int kMaxSamplerS = 16384;  // stratified / i.i.d.: the head's S uniforms sit in shared memory

// Everything a kernel needs; built by the host entry points.
struct Params {
    int B, Hq, Hkv, G, D, tile, S, Tmax, max_len;
    int nch;  // prop: 32-key chunks per sequence slot, ceil(max_len / 32)
    long long total_tokens;
    float scale;  // 1/sqrt(d)
    const void *q, *k, *v;
    const long long *kv_indptr;
    const float *U;          // prop (systematic) / flash: offsets [B][Hq] in [0, 1/S)
    const float *u_samples;  // prop stratified / i.i.d.: uniforms [B][Hq][S] in [0, 1)
    float *out;
    // workspace
    float *rec_m, *rec_z;  // flash: [B][Hq][Tmax] tile max logit and partition sum;
                           // exact: rec_m holds float2 (M, Z) per (sequence, warp, head)
    unsigned long long *rec;  // prop: [B][Hq][nch] chunk records, (m_c, z_c) as one 64-bit
                              // word, z in the high half; 0 = not written (see store_record)
    unsigned int *cnt;        // prop: [B][Hq] chunks published to the head's sampler (publish_chunks)
    unsigned char *amax;      // prop: [B][Hq][nch4] offset of each chunk's first key of largest logit
    int nch4;                 // prop: nch rounded up to a multiple of 4 (the row stride of amax)
    int nsplit;               // prop, fused kernel: CTAs per head, each taking an equal share of the S thresholds
    int p2_split, p2_cps;     // prop pass 2 kernel: CTAs (one cluster) per head, chunks per CTA
    // prop, Bernoulli score stage: uniforms [B][Hq or Hkv][draws][D], per-group
    // effective queries [B][Hq][D] and kept features [B][Hkv][D] in list order, and
    // the list lengths [B][Hkv] (also copied to dbg_feat when given)
    const float *bern_u;
    int draws, group_mean;
    float *tq_c;
    unsigned char *tq_list;
    int *tq_cnt, *dbg_feat;
    float *part;              // prop: [B][Hq][nsplit][D] the splits' sums of V rows (nsplit > 1)
    unsigned int *done;       // prop: [B][Hq] splits of the head that have stored their sum
    unsigned int *hdr;        // prop: workspace header word; nonzero = poisoned by a timeout
    long long wait_cycles;    // bound on a sampler's wait for its records (0: kWaitCycles)
    float *stash;          // prop: [B][Hq][nch * 32] exp(x - m_c), key i of sequence b at i
                           // (rows padded to whole chunks: a chunk's scores are one 128-byte line)
    float *partial;        // flash: [B][Hq][Tmax][D] tile estimates;
                           // exact: [sequence slot][warp][head][D] unnormalised sums
    int sampler;                   // prop: kSys, kStrat or kIid
    // optional debug outputs
    float *dbg_tile_m, *dbg_tile_z;
    int *dbg_count, *dbg_idx;
    int dbg_stride;
    unsigned int *err;
    // paged KV cache (prop): key i of sequence b is row
    // page_table[b * max_pages + i / page_size] * page_size + i % page_size of the
    // K / V pools, and its length is kv_lens[b]; null page_table: contiguous
    // cache addressed by kv_indptr
    const int *page_table, *kv_lens;
    int page_size, max_pages;
    long long num_pages;
};

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Ends an mbarrier's life, so that its shared memory may serve another purpose.
__device__ __forceinline__ void mbar_inval(uint64_t *bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Makes initialised barriers visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier shared-memory accesses before later async-proxy writes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// As mbar_try_wait, but the thread may sleep up to `hint_ns` waiting for the
// phase (it wakes as soon as the phase completes): waiting warps do not spin
// through issue slots that working warps on the same scheduler need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// Waits for phase `parity` of `bar` to complete; gives up after kWaitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait_sleep(bar, parity, 1u << 20)) {
        if (clock64() - t0 > kWaitCycles) return false;
    }
    return true;
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}
// L2 policy for data that is read once: its lines are the first evicted, so that a
// streamed K or V cache does not push out what the kernel reads again (records,
// stash, code).
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// tma_load_3d with an L2 cache policy (l2_evict_first).
__device__ __forceinline__ void tma_load_3d_hint(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                                 int c2, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Distributed shared memory of a thread-block cluster: the address of `p` (a
// shared-memory location of this CTA) in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_map(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Hardware cluster barrier, split in its two halves (every thread of every CTA
// of the cluster executes both, outside divergent code).
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Four 8x8 matrices of 16-bit elements from shared memory; lanes 8j .. 8j + 7
// give the row addresses of matrix j, and register j receives its fragment.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&a)[4], const void *row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                 : "r"(smem_addr(row))
                 : "memory");
}

// The same with each 8x8 matrix transposed on the way: lane (g, t) receives the
// elements (rows 2t, 2t + 1; column g) of matrix j in register j.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&a)[4], const void *row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                 : "r"(smem_addr(row))
                 : "memory");
}

// Two floats as a bf16 pair (x in the low half), each rounded to nearest even,
// and the pair of what the rounding left out, also as bf16 (x = hi + lo to
// about 2^-16 relative).
__device__ __forceinline__ void bf16_split2(float x, float y, uint32_t *hi, uint32_t *lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x - __low2float(h), y - __high2float(h));
    *hi = *reinterpret_cast<const uint32_t *>(&h);
    *lo = *reinterpret_cast<const uint32_t *>(&l);
}

// d += A B on the tensor cores: A 16x16 bf16 (row-major fragment), B 16x8 bf16
// (column-major fragment), d 16x8 fp32.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now; and, in that kernel, wait until this one's memory is visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ element types

// K/V/q storage: bf16 is carried as its 16-bit pattern.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T>
__device__ __forceinline__ float to_float(T x);
template <>
__device__ __forceinline__ float to_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_float<uint16_t>(uint16_t x) { return __uint_as_float(uint32_t(x) << 16); }

// A 16-byte vector of elements as float pairs (4 pairs of bf16, 2 pairs of fp32).
template <typename T>
struct Vec16;
template <>
struct Vec16<uint16_t> {
    static constexpr int kPairs = 4;
    __device__ __forceinline__ static void unpack(const uint4 &r, float2 *o) {
        o[0] = make_float2(bf16_lo(r.x), bf16_hi(r.x));
        o[1] = make_float2(bf16_lo(r.y), bf16_hi(r.y));
        o[2] = make_float2(bf16_lo(r.z), bf16_hi(r.z));
        o[3] = make_float2(bf16_lo(r.w), bf16_hi(r.w));
    }
};
template <>
struct Vec16<float> {
    static constexpr int kPairs = 2;
    __device__ __forceinline__ static void unpack(const uint4 &r, float2 *o) {
        o[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
        o[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
    }
};

// A lane's slice of one V row: D/32 consecutive elements at element lane*D/32.
template <typename T, int D>
struct RowSlice {
    static constexpr int kElems = D / 32;
    static constexpr int kBytes = kElems * int(sizeof(T));  // 4, 8 or 16
    float v[kElems];
    __device__ __forceinline__ void load(const T *row, int lane) {
        const unsigned char *p = reinterpret_cast<const unsigned char *>(row) + lane * kBytes;
        if constexpr (kBytes == 4) {
            uint32_t w = __ldg(reinterpret_cast<const unsigned int *>(p));
            unpack_words(&w);
        } else if constexpr (kBytes == 8) {
            uint2 w = __ldg(reinterpret_cast<const uint2 *>(p));
            uint32_t a[2] = {w.x, w.y};
            unpack_words(a);
        } else {
            uint4 w = __ldg(reinterpret_cast<const uint4 *>(p));
            uint32_t a[4] = {w.x, w.y, w.z, w.w};
            unpack_words(a);
        }
    }
    __device__ __forceinline__ void load_shared(const unsigned char *row, int lane) {
        const unsigned char *p = row + lane * kBytes;
        if constexpr (kBytes == 4) {
            uint32_t w = *reinterpret_cast<const uint32_t *>(p);
            unpack_words(&w);
        } else if constexpr (kBytes == 8) {
            uint2 w = *reinterpret_cast<const uint2 *>(p);
            uint32_t a[2] = {w.x, w.y};
            unpack_words(a);
        } else {
            uint4 w = *reinterpret_cast<const uint4 *>(p);
            uint32_t a[4] = {w.x, w.y, w.z, w.w};
            unpack_words(a);
        }
    }
    __device__ __forceinline__ void unpack_words(const uint32_t *w) {
        if constexpr (sizeof(T) == 2) {
#pragma unroll
            for (int i = 0; i < kElems / 2; ++i) {
                v[2 * i] = bf16_lo(w[i]);
                v[2 * i + 1] = bf16_hi(w[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < kElems; ++i) v[i] = __uint_as_float(w[i]);
        }
    }
};

// ------------------------------------------------------------------ reductions / scans

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
// Inclusive prefix sum across the warp (Hillis-Steele, fixed order).
__device__ __forceinline__ float warp_inclusive_scan(float v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// Chunked inclusive scan of exp-scores over one tile by one warp: element i of
// the tile sits at lane i % 32 of step i / 32, and each step adds the previous
// step's total.  Both the producer of the stash and its reader run exactly this
// sequence of additions, so they obtain bit-identical prefixes.
struct TileScan {
    float carry = 0.f;
    int last_pos = -1;  // last index with a positive score
    __device__ __forceinline__ float step(float e, int idx, int lane) {
        const float v = warp_inclusive_scan(e, lane) + carry;
        carry = __shfl_sync(kFull, v, 31);
        if (e > 0.f) last_pos = idx;
        return v;
    }
    __device__ __forceinline__ void finish() { last_pos = warp_max_int(last_pos); }
};

// Smallest i in [0, len) with P[i] > target (P non-decreasing), else last_pos.
// Negative or NaN targets count as 0, so a zero-mass key is never returned.
// (last_pos < 0 only if every score of the tile is NaN; key 0 keeps the read in bounds.)
__device__ __forceinline__ int cdf_search(const float *P, int len, float target, int last_pos) {
    if (last_pos < 0) return 0;
    if (!(target > 0.f)) target = 0.f;
    int lo = 0, hi = len;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (P[mid] > target)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo < last_pos ? lo : last_pos;
}

// ------------------------------------------------------------------ validation

__device__ __forceinline__ void raise_flag(const Params &p, unsigned bit) {
    if (p.err) atomicOr(p.err, bit);
}

// Start and length of a sequence from its kv_indptr entries s = kv_indptr[b],
// e = kv_indptr[b + 1]; an inconsistent pair gives an empty sequence and raises
// SANTA_ERR_INDPTR.
__device__ __forceinline__ int checked_bounds(const Params &p, long long s, long long e, long long *start) {
    if (s < 0 || e < s || e > p.total_tokens || e - s > (long long)p.max_len) {
        raise_flag(p, SANTA_ERR_INDPTR);
        *start = 0;
        return 0;
    }
    *start = s;
    return int(e - s);
}
// The raw bounds of sequence b: (kv_indptr[b], kv_indptr[b + 1]), or (0, kv_lens[b])
// for a paged cache (whose length must also fit its page-table row).
template <bool kPaged = false>
__device__ __forceinline__ void raw_bounds(const Params &p, int b, long long *s, long long *e) {
    if constexpr (kPaged) {
        const long long L = p.kv_lens[b];
        *s = 0;
        *e = L <= (long long)p.max_pages * p.page_size ? L : -1;  // -1: rejected below
    } else {
        *s = p.kv_indptr[b];
        *e = p.kv_indptr[b + 1];
    }
}
template <bool kPaged = false>
__device__ __forceinline__ int seq_bounds(const Params &p, int b, long long *start) {
    long long s, e;
    raw_bounds<kPaged>(p, b, &s, &e);
    return checked_bounds(p, s, e, start);
}

// Row of the K / V cache that holds key i of sequence b (start: the sequence's
// first row, contiguous layout).  A page id outside [0, num_pages) raises
// SANTA_ERR_INDPTR and gives -1.
template <bool kPaged>
__device__ __forceinline__ long long key_row(const Params &p, int b, long long start, int i) {
    if constexpr (!kPaged) return start + i;
    const int pg = __ldg(p.page_table + (size_t)b * p.max_pages + i / p.page_size);
    if (pg < 0 || pg >= p.num_pages) {
        raise_flag(p, SANTA_ERR_INDPTR);
        return -1;
    }
    return (long long)pg * p.page_size + i % p.page_size;
}

// An offset U clamped into [0, 1/S) (SANTA_ERR_OFFSET if it was not).
__device__ __forceinline__ float checked_offset(const Params &p, float u) {
    if (!(u >= 0.f) || double(u) * double(p.S) >= 1.0) {
        raise_flag(p, SANTA_ERR_OFFSET);
        u = (u >= 0.f) ? nextafterf(1.0f / float(p.S), 0.f) : 0.f;
        while (double(u) * double(p.S) >= 1.0) u = nextafterf(u, 0.f);
    }
    return u;
}
__device__ __forceinline__ float load_offset(const Params &p, int b, int h) {
    return checked_offset(p, p.U[size_t(b) * p.Hq + h]);
}

}  // namespace santa
