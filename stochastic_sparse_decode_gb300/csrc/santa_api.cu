// santa_api.cu -- the C entry points declared in santa_decode.h: argument
// validation, workspace layout, TMA descriptors for the K/V cache, launches.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "santa_launch.h"

using namespace santa;

namespace {

constexpr long long kMaxTokens = (1LL << 31) - 4096;  // TMA row coordinates are int32
constexpr int kMaxS = 1 << 20;
constexpr int kMaxPropLen = 1 << 22;  // 2^17 chunks of 32 keys

__global__ void zero_out_kernel(float *out, size_t n) {
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x)
        out[i] = 0.f;
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Layout {
    int Tmax = 0, nch = 0;
    size_t rec_m = 0, rec_z = 0, stash = 0, partial = 0, total = 0;
    // prop: counters, packed chunk records, split counters, chunk argmax offsets, the
    // splits' sums; bytes that start at zero
    size_t cnt = 0, rec = 0, done = 0, amax = 0, part = 0, clear = 0;
    // prop, Bernoulli score stage: effective queries, kept-feature lists, list lengths
    size_t tq_c = 0, tq_list = 0, tq_cnt = 0;
};

int check_problem(const santa_problem *p, int mode) {
    if (!p) return SANTA_INVALID_ARG;
    if (mode < SANTA_MODE_PROP || mode > SANTA_MODE_EXACT) return SANTA_INVALID_ARG;
    if (p->batch < 0 || p->batch > 65535) return SANTA_INVALID_ARG;
    if (p->num_q_heads < 1 || p->num_q_heads > 65535 || p->num_kv_heads < 1 || p->num_kv_heads > 65535)
        return SANTA_INVALID_ARG;
    if (p->num_q_heads % p->num_kv_heads != 0) return SANTA_INVALID_ARG;
    const int G = p->num_q_heads / p->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return SANTA_UNSUPPORTED;
    if (p->head_dim != 64 && p->head_dim != 128) return SANTA_UNSUPPORTED;
    if (p->dtype != SANTA_F32 && p->dtype != SANTA_BF16) return SANTA_UNSUPPORTED;
    if (!is_pow2(p->tile) || p->tile < 32 || p->tile > 1024) return SANTA_INVALID_ARG;
    if (mode != SANTA_MODE_EXACT && (p->S < 1 || p->S > kMaxS)) return SANTA_INVALID_ARG;
    // prop's fixed-point masses hold at most 2^17 chunks of 32 keys per sequence
    if (mode == SANTA_MODE_PROP && p->max_len > kMaxPropLen) return SANTA_UNSUPPORTED;
    if (p->max_len < 0 || p->total_tokens < 0 || p->total_tokens > kMaxTokens) return SANTA_INVALID_ARG;
    if ((p->max_len + p->tile - 1) / p->tile > 65535) return SANTA_INVALID_ARG;  // tiles are a grid dimension
    return SANTA_OK;
}

// Workspace regions of one call, each 256-byte aligned.  Sizes are computed in
// double first so that absurd shapes are rejected instead of wrapping around.
//   prop:        a 256-byte header (its first word: nonzero = poisoned by a timeout),
//                per (sequence, query head) the count of chunks pass 1 has published,
//                the chunk records [B][Hq][nch] as 64-bit words (m, z), nch =
//                ceil(max_len / 32), per head the count of its splits that are done
//                (set to 0 by pass 1), the score stash [B][Hq][nch * 32], per chunk the offset of its
//                largest key [B][Hq][nch rounded up to 4] (bytes), and the splits'
//                sums [B][Hq][prop_split_bound][d], and for the Bernoulli score stage
//                the effective queries [B][Hq][d] float, the kept features [B][Hkv][d]
//                bytes and their counts [B][Hkv]; the header, counters and records
//                must be zero before the first call (`clear` bytes from the start) and
//                every call leaves them so;
//   flash:       the regions of prop up to the chunk offsets (its pass 1 is prop's
//                streaming pass; nothing needs to start at zero), then the tile records
//                rec_m, rec_z [B][Hq][Tmax] and the tile estimates [B][Hq][Tmax][d];
//   exact:       per (sequence, streaming warp, head of the group) the partial state
//                (M, Z) as rec_m [B][P][G][2] and O as [B][P][G][d], P the warps of
//                the streaming kernel's largest grid.
int make_layout(const santa_problem *p, int mode, Layout *L) {
    const int Tmax = (p->max_len + p->tile - 1) / p->tile;
    const int nch = (p->max_len + 31) / 32;
    const bool prop = mode == SANTA_MODE_PROP;
    const double B = p->batch, Hq = p->num_q_heads, D = p->head_dim;
    if (mode == SANTA_MODE_EXACT) {
        const int G = p->num_q_heads / p->num_kv_heads;
        const int warps = exact_stream_warps(p->dtype, p->head_dim, G);
        if (warps <= 0) return SANTA_UNSUPPORTED;
        const double P = double(exact_stream_cta_bound(p->num_kv_heads)) * warps;
        if (B * P * G * (D + 2) * 4 > 1e15) return SANTA_INVALID_ARG;
        const size_t n = size_t(p->batch) * size_t(P) * G;
        L->Tmax = Tmax;
        L->nch = nch;
        L->rec_m = 0;
        L->rec_z = align256(n * 8);
        L->partial = L->rec_z;
        L->total = L->partial + align256(n * p->head_dim * 4);
        return SANTA_OK;
    }
    const double nrec = B * Hq * (prop ? nch : Tmax);
    const double nchunk = B * Hq * nch;  // prop and flash both run the streaming pass 1
    double est = nchunk * (8 + 32 * 4 + 1) + B * Hq * 8;
    if (prop)
        est += B * Hq * (kPropMaxSplit * D * 4 + D * 4) + B * p->num_kv_heads * (D + 4);
    else
        est += nrec * (D + 2) * 4;
    if (est > 1e15) return SANTA_INVALID_ARG;

    const size_t n_chunk = size_t(p->batch) * p->num_q_heads * size_t(nch);
    const size_t n_tile = size_t(p->batch) * p->num_q_heads * size_t(Tmax);
    size_t off = 0;
    L->Tmax = Tmax;
    L->nch = nch;
    // the streaming pass 1's outputs (prop and flash)
    off = 256;  // header
    L->cnt = off;
    off += align256(size_t(p->batch) * p->num_q_heads * 4);
    L->rec = off;
    off += align256(n_chunk * 8);
    L->clear = prop ? off : 0;  // only prop's samplers need the bytes before here zero
    L->done = off;
    off += align256(size_t(p->batch) * p->num_q_heads * 4);
    L->stash = off;
    off += align256(n_chunk * 32 * 4);
    L->amax = off;
    off += align256(size_t(p->batch) * p->num_q_heads * size_t((nch + 3) & ~3));
    if (prop) {
        L->part = off;
        const long long heads = (long long)p->batch * p->num_q_heads;
        off += align256(size_t(heads) * prop_split_bound(heads) * p->head_dim * 4);
        const size_t groups = size_t(p->batch) * p->num_kv_heads;
        L->tq_c = off;
        off += align256(size_t(heads) * p->head_dim * 4);
        L->tq_list = off;
        off += align256(groups * p->head_dim);
        L->tq_cnt = off;
        off += align256(groups * 4);
    } else {  // flash: per tile (m_t, z_t) and the tile estimates
        L->rec_m = off;
        off += align256(n_tile * 4);
        L->rec_z = off;
        off += align256(n_tile * 4);
        L->partial = off;
        off += align256(n_tile * p->head_dim * 4);
    }
    L->total = off > 256 ? off : 256;
    return SANTA_OK;
}

int smem_check(const santa_problem *p, int mode, int sampler, bool paged) {
    constexpr size_t kOptin = 227 * 1024;  // shared memory a block may opt in to on sm_103
    const int G = p->num_q_heads / p->num_kv_heads;
    size_t need = 0;
    if (mode == SANTA_MODE_PROP) {
        need = prop_pass1_smem(p->dtype, p->head_dim, G, int(kOptin));
        int nsplit = 0, cps = 0;
        if (prop_pass2_split((p->max_len + 31) / 32, p->tile, (long long)p->batch * p->num_q_heads, &nsplit, &cps) !=
            cudaSuccess)
            return SANTA_CUDA_ERROR;
        const size_t s2 = prop_pass2_smem(p->head_dim, cps, sampler, p->S, paged);
        if (s2 > need) need = s2;
    } else if (mode == SANTA_MODE_FLASH) {
        need = prop_pass1_smem(p->dtype, p->head_dim, G, int(kOptin));
        if (flash_sample_smem(p->tile) > need) need = flash_sample_smem(p->tile);
    } else {
        need = exact_stream_smem(p->dtype, p->head_dim, G);
    }
    return need <= kOptin ? SANTA_OK : SANTA_UNSUPPORTED;
}

// ---- TMA descriptors of a [total_tokens][Hkv][d] cache: boxes of 128 bytes of one
// KV head's row x box_rows rows, with the 128-byte swizzle the kernels expect

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

struct MapKey {
    const void *base;
    int dtype, d, hkv, dev, box_rows;
    long long rows;
    bool operator==(const MapKey &o) const {
        return base == o.base && dtype == o.dtype && d == o.d && hkv == o.hkv && dev == o.dev &&
               box_rows == o.box_rows && rows == o.rows;
    }
};

bool kv_map(CUtensorMap *map, const void *base, int dtype, int d, int hkv, long long rows, int box_rows) {
    static std::mutex mu;
    static MapKey keys[32];
    static CUtensorMap maps[32];
    static int used = 0, next = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const MapKey key{base, dtype, d, hkv, dev, box_rows, rows};
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (keys[i] == key) {
            *map = maps[i];
            return true;
        }
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    const int es = dtype == SANTA_BF16 ? 2 : 4;
    const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(hkv), cuuint64_t(rows)};
    const cuuint64_t strides[2] = {cuuint64_t(d) * es, cuuint64_t(hkv) * d * es};
    const cuuint32_t box[3] = {cuuint32_t(128 / es), 1u, cuuint32_t(box_rows)};
    const cuuint32_t estride[3] = {1u, 1u, 1u};
    CUtensorMap m;
    const CUresult r = enc(&m, dtype == SANTA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                           3, const_cast<void *>(base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    keys[next] = key;
    maps[next] = m;
    next = (next + 1) % 32;
    if (used < 32) ++used;
    *map = m;
    return true;
}

// `sampler` (prop only): kSys with offsets U [B][Hq], or kStrat / kIid with uniforms U [B][Hq][S].
// `stages` (prop only): which of the two passes to run; the other modes run whole.
// Pass 1 alone needs q, k and kv_indptr; pass 2 alone needs v, kv_indptr, U and out.
// `pages` (prop only): a paged cache; k and v are then the page pools and kv_indptr is unused.
// `bern` (prop only): the Bernoulli score stage; k is then the feature-blocked K cache.
struct Bern {
    const float *u;
    int draws, group_mean;
};
int run(int mode, int sampler, const santa_problem *p, const void *q, const void *k, const void *v,
        const long long *kv_indptr, const float *U, float *out, void *workspace, size_t workspace_bytes,
        const santa_debug *dbg, santa_stream_t stream_, int stages = kPass1 | kPass2,
        const santa_pages *pages = nullptr, const Bern *bern = nullptr) {
    int st = check_problem(p, mode);
    if (st != SANTA_OK) return st;
    if (sampler != kSys && p->S > kMaxSamplerS) return SANTA_UNSUPPORTED;
    if (pages) {
        if (mode != SANTA_MODE_PROP || pages->page_size <= 0 || pages->page_size % 32 != 0 || pages->max_pages <= 0 ||
            pages->num_pages <= 0 || pages->num_pages > kMaxTokens / pages->page_size ||
            pages->num_pages * pages->page_size != p->total_tokens ||
            (long long)p->max_len > (long long)pages->max_pages * pages->page_size)
            return SANTA_INVALID_ARG;
    }
    if (bern && (mode != SANTA_MODE_PROP || sampler != kSys || pages || stages != (kPass1 | kPass2) || !bern->u ||
                 !aligned(bern->u, 4) || bern->draws < 1 || bern->draws > kMaxBernoulliDraws))
        return SANTA_INVALID_ARG;
    if (p->batch == 0) return SANTA_OK;
    const bool p1 = stages & kPass1, p2 = stages & kPass2;
    if (pages && (!pages->page_table || !pages->kv_lens || !aligned(pages->page_table, 4) ||
                  !aligned(pages->kv_lens, 4)))
        return SANTA_INVALID_ARG;
    if ((p1 && (!q || !k)) || (p2 && (!v || !out)) || (!kv_indptr && !pages) || !workspace)
        return SANTA_INVALID_ARG;
    if (p2 && mode != SANTA_MODE_EXACT && !U) return SANTA_INVALID_ARG;
    if ((q && !aligned(q, 16)) || (k && !aligned(k, 16)) || (v && !aligned(v, 16)) || (out && !aligned(out, 16)) ||
        (kv_indptr && !aligned(kv_indptr, 8)) || !aligned(workspace, 256) || (U && !aligned(U, 4)))
        return SANTA_INVALID_ARG;
    if (dbg && dbg->sample_stride < 0) return SANTA_INVALID_ARG;
    Layout L;
    st = make_layout(p, mode, &L);
    if (st != SANTA_OK) return st;
    if (workspace_bytes < L.total) return SANTA_WORKSPACE_TOO_SMALL;
    st = smem_check(p, mode, sampler, pages != nullptr);
    if (st != SANTA_OK) return st;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const size_t n_out = size_t(p->batch) * p->num_q_heads * p->head_dim;
    if (L.Tmax == 0 || p->total_tokens == 0) {  // no sequence can hold a key
        if (!p2) return SANTA_OK;
        const unsigned blocks = unsigned((n_out + 255) / 256 < 1024 ? (n_out + 255) / 256 : 1024);
        zero_out_kernel<<<blocks, 256, 0, stream>>>(out, n_out);
        return cudaGetLastError() == cudaSuccess ? SANTA_OK : SANTA_CUDA_ERROR;
    }

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    Params prm = {};
    prm.B = p->batch;
    prm.Hq = p->num_q_heads;
    prm.Hkv = p->num_kv_heads;
    prm.G = p->num_q_heads / p->num_kv_heads;
    prm.D = p->head_dim;
    prm.tile = p->tile;
    prm.S = mode == SANTA_MODE_EXACT ? 1 : p->S;
    prm.Tmax = L.Tmax;
    prm.nch = L.nch;
    prm.max_len = p->max_len;
    prm.total_tokens = p->total_tokens;
    prm.scale = float(1.0 / std::sqrt(double(p->head_dim)));
    prm.q = q;
    prm.k = k;
    prm.v = v;
    prm.kv_indptr = pages ? nullptr : kv_indptr;
    if (pages) {
        prm.page_table = pages->page_table;
        prm.kv_lens = pages->kv_lens;
        prm.page_size = pages->page_size;
        prm.max_pages = pages->max_pages;
        prm.num_pages = pages->num_pages;
    }
    prm.U = sampler == kSys ? U : nullptr;
    prm.u_samples = sampler == kSys ? nullptr : U;
    prm.sampler = sampler;
    prm.out = out;
    if (mode == SANTA_MODE_PROP || mode == SANTA_MODE_FLASH) {  // the streaming pass 1's outputs
        prm.hdr = reinterpret_cast<unsigned int *>(ws);
        prm.rec = reinterpret_cast<unsigned long long *>(ws + L.rec);
        prm.cnt = reinterpret_cast<unsigned int *>(ws + L.cnt);
        prm.stash = reinterpret_cast<float *>(ws + L.stash);
        prm.amax = ws + L.amax;
        prm.done = reinterpret_cast<unsigned int *>(ws + L.done);
        prm.nch4 = (L.nch + 3) & ~3;
        prm.nsplit = 1;  // set by the launcher
    }
    if (mode == SANTA_MODE_PROP) {
        prm.part = reinterpret_cast<float *>(ws + L.part);
    } else {
        prm.rec_m = reinterpret_cast<float *>(ws + L.rec_m);
        prm.rec_z = reinterpret_cast<float *>(ws + L.rec_z);
        prm.partial = reinterpret_cast<float *>(ws + L.partial);
    }
    Timing tm;
    if (dbg) {
        prm.dbg_tile_m = dbg->tile_m;
        prm.dbg_tile_z = dbg->tile_z;
        prm.dbg_count = dbg->tile_count;
        prm.dbg_idx = dbg->sample_idx;
        prm.dbg_stride = dbg->sample_stride;
        prm.err = dbg->error_flags;
        prm.wait_cycles = dbg->wait_cycles;
        tm.begin = reinterpret_cast<cudaEvent_t>(dbg->main_begin);
        tm.end = reinterpret_cast<cudaEvent_t>(dbg->main_end);
    }

    CUtensorMap kmap, vmap;
    cudaError_t e;
    if (bern) {
        prm.bern_u = bern->u;
        prm.draws = bern->draws;
        prm.group_mean = bern->group_mean ? 1 : 0;
        prm.tq_c = reinterpret_cast<float *>(ws + L.tq_c);
        prm.tq_list = ws + L.tq_list;
        prm.tq_cnt = reinterpret_cast<int *>(ws + L.tq_cnt);
        prm.dbg_feat = dbg ? dbg->features_read : nullptr;
        e = launch_prop_bernoulli(prm, p->dtype, stream, tm);
    } else if (mode == SANTA_MODE_PROP) {
        if (p1 && !kv_map(&kmap, k, p->dtype, p->head_dim, p->num_kv_heads, p->total_tokens, 32))
            return SANTA_CUDA_ERROR;
        e = launch_prop(prm, p->dtype, kmap, stream, tm, stages);
    } else if (mode == SANTA_MODE_FLASH) {
        if (!kv_map(&kmap, k, p->dtype, p->head_dim, p->num_kv_heads, p->total_tokens, 32))
            return SANTA_CUDA_ERROR;
        e = launch_flash(prm, p->dtype, kmap, stream, tm);
    } else {
        if (!kv_map(&kmap, k, p->dtype, p->head_dim, p->num_kv_heads, p->total_tokens, 32) ||
            !kv_map(&vmap, v, p->dtype, p->head_dim, p->num_kv_heads, p->total_tokens, 32))
            return SANTA_CUDA_ERROR;
        e = launch_exact(prm, p->dtype, kmap, vmap, stream, tm);
    }
    if (e == cudaErrorNotSupported) return SANTA_UNSUPPORTED;
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return SANTA_CUDA_ERROR;
    return SANTA_OK;
}

}  // namespace

extern "C" {

int santa_workspace_size(const santa_problem *p, int mode, size_t *bytes) {
    if (!bytes) return SANTA_INVALID_ARG;
    const int st = check_problem(p, mode);
    if (st != SANTA_OK) return st;
    Layout L;
    const int s2 = make_layout(p, mode, &L);
    if (s2 != SANTA_OK) return s2;
    *bytes = L.total;
    return SANTA_OK;
}

int santa_workspace_init(const santa_problem *p, int mode, void *workspace, size_t workspace_bytes,
                         santa_stream_t stream) {
    const int st = check_problem(p, mode);
    if (st != SANTA_OK) return st;
    Layout L;
    const int s2 = make_layout(p, mode, &L);
    if (s2 != SANTA_OK) return s2;
    if (!workspace || !aligned(workspace, 256)) return SANTA_INVALID_ARG;
    if (workspace_bytes < L.total) return SANTA_WORKSPACE_TOO_SMALL;
    if (L.clear == 0) return SANTA_OK;
    return cudaMemsetAsync(workspace, 0, L.clear, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SANTA_OK
               : SANTA_CUDA_ERROR;
}

int santa_decode_prop(const santa_problem *p, const void *q, const void *k, const void *v, const long long *kv_indptr,
                      const float *U, float *out, void *workspace, size_t workspace_bytes, const santa_debug *dbg,
                      santa_stream_t stream) {
    return run(SANTA_MODE_PROP, kSys, p, q, k, v, kv_indptr, U, out, workspace, workspace_bytes, dbg, stream);
}

int santa_decode_prop_fused(const santa_problem *p, const void *q, const void *k, const void *v,
                            const long long *kv_indptr, const float *U, float *out, void *workspace,
                            size_t workspace_bytes, const santa_debug *dbg, santa_stream_t stream) {
    return run(SANTA_MODE_PROP, kSys, p, q, k, v, kv_indptr, U, out, workspace, workspace_bytes, dbg, stream,
               kPass1 | kPass2 | kFused);
}

int santa_decode_prop_bernoulli(const santa_problem *p, const void *q, const void *k_fb, const void *v,
                                const long long *kv_indptr, const float *U, const float *bern_u, int draws,
                                int group_mean, float *out, void *workspace, size_t workspace_bytes,
                                const santa_debug *dbg, santa_stream_t stream) {
    const Bern bern{bern_u, draws, group_mean};
    return run(SANTA_MODE_PROP, kSys, p, q, k_fb, v, kv_indptr, U, out, workspace, workspace_bytes, dbg, stream,
               kPass1 | kPass2, nullptr, &bern);
}

int santa_k_feature_blocked_size(const santa_problem *p, size_t *bytes) {
    if (!bytes) return SANTA_INVALID_ARG;
    const int st = check_problem(p, SANTA_MODE_PROP);
    if (st != SANTA_OK) return st;
    const size_t esz = p->dtype == SANTA_BF16 ? 2 : 4;
    *bytes = size_t((p->total_tokens + 63) / 64) * p->num_kv_heads * p->head_dim * 64 * esz;
    return SANTA_OK;
}

int santa_k_feature_blocked(const santa_problem *p, const void *k, void *k_fb, size_t k_fb_bytes,
                            santa_stream_t stream) {
    size_t need = 0;
    const int st = santa_k_feature_blocked_size(p, &need);
    if (st != SANTA_OK) return st;
    if (need == 0) return SANTA_OK;
    if (!k || !k_fb || !aligned(k, 16) || !aligned(k_fb, 16)) return SANTA_INVALID_ARG;
    if (k_fb_bytes < need) return SANTA_WORKSPACE_TOO_SMALL;
    const cudaError_t e = launch_feature_block(p->dtype, k, k_fb, p->total_tokens, p->num_kv_heads, p->head_dim,
                                               reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SANTA_OK : SANTA_CUDA_ERROR;
}

int santa_prop_pass1(const santa_problem *p, const void *q, const void *k, const long long *kv_indptr,
                     void *workspace, size_t workspace_bytes, const santa_debug *dbg, santa_stream_t stream) {
    return run(SANTA_MODE_PROP, kSys, p, q, k, nullptr, kv_indptr, nullptr, nullptr, workspace, workspace_bytes, dbg,
               stream, kPass1);
}

int santa_prop_pass2(const santa_problem *p, const void *v, const long long *kv_indptr, const float *U, float *out,
                     void *workspace, size_t workspace_bytes, const santa_debug *dbg, santa_stream_t stream) {
    return run(SANTA_MODE_PROP, kSys, p, nullptr, nullptr, v, kv_indptr, U, out, workspace, workspace_bytes, dbg,
               stream, kPass2);
}

int santa_decode_prop_paged(const santa_problem *p, const santa_pages *pages, const void *q, const void *k_pool,
                            const void *v_pool, const float *U, float *out, void *workspace, size_t workspace_bytes,
                            const santa_debug *dbg, santa_stream_t stream) {
    if (!pages) return SANTA_INVALID_ARG;
    return run(SANTA_MODE_PROP, kSys, p, q, k_pool, v_pool, nullptr, U, out, workspace, workspace_bytes, dbg, stream,
               kPass1 | kPass2, pages);
}

int santa_decode_prop_strat(const santa_problem *p, const void *q, const void *k, const void *v,
                            const long long *kv_indptr, const float *u, float *out, void *workspace,
                            size_t workspace_bytes, const santa_debug *dbg, santa_stream_t stream) {
    return run(SANTA_MODE_PROP, kStrat, p, q, k, v, kv_indptr, u, out, workspace, workspace_bytes, dbg, stream);
}

int santa_decode_prop_iid(const santa_problem *p, const void *q, const void *k, const void *v,
                          const long long *kv_indptr, const float *u, float *out, void *workspace,
                          size_t workspace_bytes, const santa_debug *dbg, santa_stream_t stream) {
    return run(SANTA_MODE_PROP, kIid, p, q, k, v, kv_indptr, u, out, workspace, workspace_bytes, dbg, stream);
}

int santa_decode_flash(const santa_problem *p, const void *q, const void *k, const void *v, const long long *kv_indptr,
                       const float *U, float *out, void *workspace, size_t workspace_bytes, const santa_debug *dbg,
                       santa_stream_t stream) {
    return run(SANTA_MODE_FLASH, kSys, p, q, k, v, kv_indptr, U, out, workspace, workspace_bytes, dbg, stream);
}

int exact_decode(const santa_problem *p, const void *q, const void *k, const void *v, const long long *kv_indptr,
                 float *out, void *workspace, size_t workspace_bytes, const santa_debug *dbg, santa_stream_t stream) {
    return run(SANTA_MODE_EXACT, kSys, p, q, k, v, kv_indptr, nullptr, out, workspace, workspace_bytes, dbg, stream);
}

int santa_read_device_error(unsigned int *error_flags, santa_stream_t stream_, unsigned int *flags) {
    if (!error_flags || !flags) return SANTA_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    unsigned int h = 0;
    if (cudaMemcpyAsync(&h, error_flags, sizeof(h), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemsetAsync(error_flags, 0, sizeof(h), stream) != cudaSuccess || cudaStreamSynchronize(stream) != cudaSuccess)
        return SANTA_CUDA_ERROR;
    *flags = h;
    return h ? SANTA_DEVICE_CHECK : SANTA_OK;
}

const char *santa_status_string(int status) {
    switch (status) {
        case SANTA_OK: return "ok";
        case SANTA_INVALID_ARG: return "invalid argument";
        case SANTA_UNSUPPORTED: return "unsupported head_dim, GQA group or dtype";
        case SANTA_WORKSPACE_TOO_SMALL: return "workspace too small";
        case SANTA_CUDA_ERROR: return "CUDA error";
        case SANTA_DEVICE_CHECK: return "device check flagged an input";
        default: return "unknown status";
    }
}

}  // extern "C"
