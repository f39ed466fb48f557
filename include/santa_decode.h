/*
 * santa_decode.h -- C ABI of the GB300 (sm_103a) stochastic sparse decode-attention library.
 *
 * One decode step of attention for a batch of sequences with a GQA-shared,
 * token-major K/V cache, in three modes:
 *
 *   santa_decode_prop   S2ANTA-prop: a split-KV pass computes the logits
 *                       x = q.k / sqrt(d) of every key, stashes the
 *                       exponentiated scores and one partition sum per block
 *                       of keys (a 32-key chunk; a tile is tile/32 of them);
 *                       a reducer forms Z from them and places the S
 *                       systematic thresholds U + m/S on the global CDF, so a
 *                       block's budget is the number of thresholds in its CDF
 *                       interval (0 for low-mass blocks, which read no V);
 *                       a second pass searches the stashed in-block CDF for
 *                       each threshold and averages the chosen V rows:
 *                       out = (1/S) sum_m V[J_m].  The sample is the one
 *                       systematic sample of the global CDF, whatever the
 *                       block size; a tile's S_tile is the sum over its blocks.
 *                       ("Stochastic Sparse Attention for Memory-Bound
 *                       Inference", paper notes, Key designs 1 and 2.)
 *   santa_decode_flash  S2ANTA-flash: every tile draws S_loc = ceil(S / T_b)
 *                       systematic samples from its own scores as if it held
 *                       all the mass; a merge rescales the tile estimates by
 *                       Z_tile / Z.  (Same notes, Key design 3.)
 *   exact_decode        exact split-KV decode attention, sum_i A_i V_i: every
 *                       warp streams a fixed stretch of K and V rows with an
 *                       online softmax, and a log-sum-exp merge combines the
 *                       warps a sequence spans (the dense comparison point;
 *                       same notes, Related work: FlashDecoding).
 *
 * The logit scale is 1/sqrt(d) ("Double-P: Hierarchical Top-P Sparse Attention
 * for Long-Context LLMs", paper review, Stage 1, Eq. 3).  A temperature is
 * folded into q by the caller.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Shapes: B = batch, Hq query heads, Hkv KV heads (Hq % Hkv == 0; query head h
 * reads KV head h / (Hq / Hkv)), d = head_dim, L_b = length of sequence b,
 * T_b = ceil(L_b / tile) tiles, Tmax = ceil(max_len / tile).
 *
 * Layouts (all row-major, contiguous, device memory, 16-byte aligned):
 *   q          [B][Hq][d]                 dtype
 *   k, v       [total_tokens][Hkv][d]     dtype; sequence b owns rows
 *                                         kv_indptr[b] .. kv_indptr[b+1]-1
 *   kv_indptr  [B+1]   int64              non-decreasing, kv_indptr[B] <= total_tokens,
 *                                         every L_b <= max_len
 *   U          [B][Hq] float32            sampling offsets, each in [0, 1/S)
 *   out        [B][Hq][d] float32         written entirely by every call
 *
 * Ownership: every buffer belongs to the caller.  The library allocates no
 * device memory on the call path; its scratch lives in `workspace` (device,
 * 256-byte aligned, at least santa_workspace_size() bytes).  The flash and exact
 * workspaces carry no state from one call to the next.  A prop workspace must be
 * zero-filled once before its first use (santa_workspace_init, or memory that is
 * allocated zeroed): its first bytes hold the chunk records through which the
 * samplers learn that pass 1 has finished a chunk, and every call leaves them
 * zero again.  Calls are asynchronous on `stream`; results are valid once the
 * stream has reached the call's end.  Two calls may run concurrently only with
 * distinct workspaces and outputs.
 *
 * Errors: host-side validation returns a status before anything is enqueued
 * (nothing is written).  Inconsistent device data (a bad kv_indptr entry, an
 * offset outside [0, 1/S)) cannot be seen from the host: the kernels treat such
 * a sequence as empty (zeros out) or clamp the offset, and OR a bit into
 * dbg->error_flags when that pointer is given.  No kernel traps.
 */
#ifndef SANTA_DECODE_H
#define SANTA_DECODE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA stream and event handles, declared without the CUDA headers
 * (layout-compatible with cudaStream_t / cudaEvent_t). */
typedef struct CUstream_st *santa_stream_t;
typedef struct CUevent_st *santa_event_t;

/* Status codes. */
enum {
    SANTA_OK = 0,
    SANTA_INVALID_ARG = 1,          /* a null pointer, a bad size or a misaligned buffer */
    SANTA_UNSUPPORTED = 2,          /* head_dim, GQA group or dtype not built */
    SANTA_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < santa_workspace_size() */
    SANTA_CUDA_ERROR = 4,           /* a CUDA launch or runtime call failed */
    SANTA_DEVICE_CHECK = 5          /* santa_read_device_error found a flag set */
};

/* Element types of q, k and v (out is always float32). */
enum { SANTA_F32 = 0, SANTA_BF16 = 1 };

/* Modes, for santa_workspace_size. */
enum { SANTA_MODE_PROP = 0, SANTA_MODE_FLASH = 1, SANTA_MODE_EXACT = 2 };

/* Bits of the device error word (dbg->error_flags). */
enum {
    SANTA_ERR_INDPTR = 1u,   /* kv_indptr entry out of order / range: sequence treated as empty */
    SANTA_ERR_OFFSET = 2u,   /* U outside [0, 1/S) or NaN: clamped into range */
    SANTA_ERR_TIMEOUT = 4u,  /* a bounded wait gave up (an asynchronous copy, or a
                                sampler waiting for the scores of its head) */
    SANTA_ERR_WORKSPACE = 8u /* the workspace held records no pass 1 of this problem
                                wrote: the affected values were clamped into range */
};

typedef struct {
    int batch;               /* B >= 0 (B = 0 is a no-op) */
    int num_q_heads;         /* Hq >= 1 */
    int num_kv_heads;        /* Hkv >= 1, Hq / Hkv in {1, 2, 4, 8} */
    int head_dim;            /* d in {64, 128} */
    long long total_tokens;  /* rows of the K/V cache, >= kv_indptr[B] */
    int max_len;             /* upper bound on every L_b (sizes the grid and workspace) */
    int tile;                /* keys per tile: a power of two in [32, 1024] */
    int S;                   /* samples per (sequence, query head), 1 <= S <= 2^20;
                                ignored by exact_decode */
    int dtype;               /* SANTA_F32 or SANTA_BF16 */
} santa_problem;

/* Optional outputs for inspection and timing; every pointer may be NULL.
 * Entries for tiles t >= T_b of a sequence are left untouched. */
typedef struct {
    float *tile_m;           /* [B][Hq][Tmax] max logit of each tile */
    float *tile_z;           /* [B][Hq][Tmax] sum of exp(x - tile_m) over the tile */
    int *tile_count;         /* [B][Hq][Tmax] prop: S_tile; flash: S_loc of the tile
                                (prop writes tile_m, tile_z and tile_count in pass 2,
                                from its 32-key chunk records) */
    int *sample_idx;         /* prop:  [B][Hq][S], key index within the sequence of
                                       sample m (thresholds in increasing order);
                                flash: [B][Hq][Tmax][sample_stride], the first
                                       min(S_loc, sample_stride) samples of each tile */
    int sample_stride;       /* flash only: row length of sample_idx */
    unsigned int *error_flags;   /* device word; kernels OR SANTA_ERR_* bits into it */
    santa_event_t main_begin;    /* recorded on `stream` right before / after the */
    santa_event_t main_end;      /* mode's dominant kernel (prop: pass 1, or the fused
                                    kernel of santa_decode_prop_fused; flash tile;
                                    exact stream), for timing that kernel alone */
    long long wait_cycles;       /* > 0: bound, in SM clock cycles, on a fused prop sampler's
                                    wait for its head's scores (0: about 1 s); a wait
                                    that runs out raises SANTA_ERR_TIMEOUT.  < 0, a
                                    test of that path: each sampler waits |wait_cycles|
                                    for one chunk more than its head has, which never
                                    comes, and gives up */
    int *features_read;          /* santa_decode_prop_bernoulli: [B][Hkv], the number of
                                    features of d that some draw of the group kept
                                    (the K features pass 1 read for that group) */
} santa_debug;

/*
 * Bytes of workspace `mode` needs for problem *p.  Host only; enqueues nothing.
 * Returns SANTA_OK, SANTA_INVALID_ARG or SANTA_UNSUPPORTED.
 */
int santa_workspace_size(const santa_problem *p, int mode, size_t *bytes);

/*
 * Makes `workspace` ready for the first call of `mode` on problem *p: enqueues on
 * `stream` a zero fill of the bytes that must start at zero (for prop, the
 * header and the chunk records; nothing for the other modes).  Needed once per
 * workspace -- every prop call leaves those bytes zero again -- and again after
 * a call raised SANTA_ERR_TIMEOUT (which leaves the workspace poisoned: later
 * calls write zeros and raise SANTA_ERR_WORKSPACE until it is re-initialised).
 * Returns SANTA_OK, SANTA_INVALID_ARG, SANTA_WORKSPACE_TOO_SMALL or
 * SANTA_CUDA_ERROR.
 */
int santa_workspace_init(const santa_problem *p, int mode, void *workspace, size_t workspace_bytes,
                         santa_stream_t stream);

/*
 * S2ANTA-prop decode (paper notes, Key designs 1-2).
 * q, k, v, kv_indptr, U, out, workspace: device pointers as described above.
 * Two kernels on `stream`.  Pass 1 streams K, one CTA per SM: scores, the
 * exponentiated-score stash and one record (m, z) per 32-key chunk.  Pass 2
 * runs per head on a cluster of up to 8 CTAs: the reducer over the
 * ceil(L_b / 32) chunk records (M, exact fixed-point CDF, per-chunk budgets),
 * the per-chunk systematic search, the V gather, and a combine in a fixed
 * order (the result is deterministic); it then sets the head's records back
 * to zero.
 * Workspace (santa_workspace_size bytes, 256-byte aligned regions): a 256-byte
 * header, per head a published-chunk counter, the chunk records
 * [B][Hq][ceil(max_len / 32)] as 64-bit words, per head a finished-split
 * counter (the fused kernel's), the score stash [B][Hq][32 ceil(max_len / 32)]
 * float32, a byte per chunk and the fused kernel's per-split float32 sums;
 * zero-filled once before first use (see santa_workspace_init).  Supported up
 * to max_len = 2^22 keys (longer is SANTA_UNSUPPORTED).  Returns a status; see
 * the conventions above.
 */
int santa_decode_prop(const santa_problem *p, const void *q, const void *k, const void *v,
                      const long long *kv_indptr, const float *U, float *out,
                      void *workspace, size_t workspace_bytes, const santa_debug *dbg,
                      santa_stream_t stream);

/*
 * S2ANTA-prop in one persistent kernel: the same arguments, workspace and
 * results (to rounding: the V sums are added in another order) as
 * santa_decode_prop.  One CTA per SM, all resident at once: its warps first
 * stream K (pass 1), then serve as pass 2, a head starting as soon as every
 * chunk record of it is written (each CTA polls the records, with a bounded
 * wait: SANTA_ERR_TIMEOUT, see santa_debug.wait_cycles).  When there are SMs
 * to spare, a head's S thresholds are shared by up to 8 CTAs (its splits)
 * whose sums the last one to finish adds in split order.  When the fused
 * kernel's shared memory does not fit (stratified or i.i.d. samplers with
 * large S) the two kernels of santa_decode_prop run instead.  On GB300 at 32k
 * keys this form takes longer than the two kernels: the samplers' chain of
 * dependent steps after the last record outlasts the second launch it saves.
 */
int santa_decode_prop_fused(const santa_problem *p, const void *q, const void *k, const void *v,
                            const long long *kv_indptr, const float *U, float *out,
                            void *workspace, size_t workspace_bytes, const santa_debug *dbg,
                            santa_stream_t stream);

/*
 * S2ANTA-prop with the Bernoulli ternary score stage (paper notes, Key design 4;
 * mean group query: the ablation table).  Instead of q . k, pass 1 computes an
 * unbiased estimate of it and reads only the K features that the draws keep:
 *   per head (group_mean = 0): p_i = |q_i| / max_j |q_j|; draw b keeps feature i
 *     when bern_u[b][i] < p_i, as the ternary entry sign(q_i); the estimate is
 *     max|q| * (mean over the draws of the ternary query) . k;
 *   mean group query (group_mean = 1): one set of draws per KV group from the
 *     mean of its G queries, p_i = |mean_i| / max_j |mean_j|; head g weights a
 *     kept feature by q_gi / p_i (times the fraction of draws that kept it).
 * The probabilities and the draw decisions are computed in single precision.  A
 * group reads the union of the features any of its draws kept.
 *   k_fb    the K cache in the feature-blocked layout of santa_k_feature_blocked
 *           (64 keys of one feature per 128-byte line for bf16), device
 *   bern_u  float32 uniforms in [0, 1), device: [B][Hq][draws][d] per head, or
 *           [B][Hkv][draws][d] for the mean group query
 *   draws   1 .. 64 draws averaged per feature
 * Every other argument, the workspace and the errors are those of
 * santa_decode_prop (the same pass 2 runs on pass 1's records); dbg->
 * features_read, when set, receives the kept-feature count of every group.
 * Returns SANTA_INVALID_ARG for draws out of range or a missing bern_u.
 */
int santa_decode_prop_bernoulli(const santa_problem *p, const void *q, const void *k_fb, const void *v,
                                const long long *kv_indptr, const float *U, const float *bern_u, int draws,
                                int group_mean, float *out, void *workspace, size_t workspace_bytes,
                                const santa_debug *dbg, santa_stream_t stream);

/*
 * The feature-blocked K layout of santa_decode_prop_bernoulli:
 * K_fb[ceil(total_tokens / 64)][Hkv][d][64], element (row r, head h, feature f)
 * at [r / 64][h][f][r % 64]; rows past total_tokens are zero.  *bytes receives
 * its size; santa_k_feature_blocked writes it from the token-major cache k
 * ([total_tokens][Hkv][d]) on `stream` (both device pointers, 16-byte aligned;
 * the caller owns both).  A serving system would append keys in this layout
 * directly; the conversion is for callers holding a token-major cache.
 * Return SANTA_OK, SANTA_INVALID_ARG, SANTA_WORKSPACE_TOO_SMALL (k_fb_bytes too
 * small) or SANTA_CUDA_ERROR.
 */
int santa_k_feature_blocked_size(const santa_problem *p, size_t *bytes);
int santa_k_feature_blocked(const santa_problem *p, const void *k, void *k_fb, size_t k_fb_bytes,
                            santa_stream_t stream);

/*
 * The two passes of santa_decode_prop as separate calls (same notes, Key design
 * 2: pass 1 reads all of K, pass 2 samples from what pass 1 left), for callers
 * that schedule them apart or time them one by one.  santa_prop_pass1 followed
 * by santa_prop_pass2 on the same problem, kv_indptr and workspace, in stream
 * order, gives bit for bit what santa_decode_prop gives.
 *
 *   santa_prop_pass1  reads q, K and kv_indptr; writes the chunk records and the
 *                     score stash into `workspace` (layout of santa_decode_prop);
 *                     of dbg it uses error_flags, main_begin and main_end.
 *   santa_prop_pass2  reads the workspace as santa_prop_pass1 left it for the
 *                     same problem, V, kv_indptr and the offsets U; writes out
 *                     and dbg's tile and sample outputs, and sets the chunk
 *                     records and counters back to zero (the workspace is then
 *                     ready for any prop call).  It follows santa_prop_pass1 on the same problem
 *                     and workspace in stream order.  On any other workspace the
 *                     records are whatever it holds: every index derived from them
 *                     is clamped into range (no out-of-bounds access), a record
 *                     that reads zero counts as a chunk without mass, `out` stays
 *                     finite, and SANTA_ERR_WORKSPACE is raised where a clamp fired.
 *
 * Arguments, ownership and errors are those of santa_decode_prop; a pass takes
 * only the pointers it reads.
 */
int santa_prop_pass1(const santa_problem *p, const void *q, const void *k, const long long *kv_indptr,
                     void *workspace, size_t workspace_bytes, const santa_debug *dbg, santa_stream_t stream);
int santa_prop_pass2(const santa_problem *p, const void *v, const long long *kv_indptr, const float *U, float *out,
                     void *workspace, size_t workspace_bytes, const santa_debug *dbg, santa_stream_t stream);

/*
 * A paged K / V cache (page-table indirection, as serving systems keep it).
 * The pools hold num_pages pages of page_size keys: K and V are
 * [num_pages * page_size][num_kv_heads][head_dim] in the problem's dtype, that
 * is the contiguous layout with total_tokens = num_pages * page_size rows.  Key
 * i of sequence b is row page_table[b * max_pages + i / page_size] * page_size
 * + i % page_size; sequence b holds kv_lens[b] keys.
 */
typedef struct {
    const int *page_table;   /* device [B][max_pages] int32 page ids */
    const int *kv_lens;      /* device [B] int32 sequence lengths, each <= max_len */
    int page_size;           /* keys per page, a positive multiple of 32 */
    int max_pages;           /* row length of page_table; max_len <= max_pages * page_size */
    long long num_pages;     /* pages in each pool; num_pages * page_size == total_tokens */
} santa_pages;

/*
 * S2ANTA-prop decode (same notes, Key designs 1-2) on a paged cache; the pages
 * themselves only claim compatibility with paged serving (Overall framework).
 * Same arguments as santa_decode_prop with k_pool / v_pool for k / v and the
 * page table for kv_indptr; workspace: santa_workspace_size with
 * SANTA_MODE_PROP.  A page size that is not a multiple of 32, a pool size that
 * disagrees with total_tokens or a max_len beyond a page-table row is
 * SANTA_INVALID_ARG.  On the device, a length outside [0, max_len] makes the
 * sequence empty and a page id outside [0, num_pages) drops that page's keys
 * (pass 1) or reads row 0 (pass 2); both raise SANTA_ERR_INDPTR.  A chunk of 32
 * keys never straddles two pages, so the results equal those of
 * santa_decode_prop on the same keys laid out contiguously, bit for bit.
 */
int santa_decode_prop_paged(const santa_problem *p, const santa_pages *pages, const void *q, const void *k_pool,
                            const void *v_pool, const float *U, float *out, void *workspace, size_t workspace_bytes,
                            const santa_debug *dbg, santa_stream_t stream);

/*
 * The prop pipeline with the two other samplers of the same notes (Key design 1):
 *
 *   santa_decode_prop_strat   S2ANTA-strat: threshold m is (m + u_m) / S, one
 *                             uniform draw inside each stratum [m/S, (m+1)/S);
 *   santa_decode_prop_iid     SANTA: S independent draws, threshold s is u_s;
 *                             the samples are taken in increasing order of u.
 *
 * u: device [B][Hq][S] float32, each in [0, 1) (a value outside is clamped into
 * it and raises SANTA_ERR_OFFSET).  out = (1/S) sum V[J], as for prop.  Every
 * other argument, layout, workspace (santa_workspace_size with SANTA_MODE_PROP),
 * ownership and error are those of santa_decode_prop; dbg->sample_idx holds, per
 * (b, h), the key chosen for threshold m (strat) or for the m-th smallest u (iid).
 * Supported for S <= 16384 (the head's uniforms are kept in shared memory; a
 * larger S is SANTA_UNSUPPORTED).
 */
int santa_decode_prop_strat(const santa_problem *p, const void *q, const void *k, const void *v,
                            const long long *kv_indptr, const float *u, float *out,
                            void *workspace, size_t workspace_bytes, const santa_debug *dbg,
                            santa_stream_t stream);
int santa_decode_prop_iid(const santa_problem *p, const void *q, const void *k, const void *v,
                          const long long *kv_indptr, const float *u, float *out,
                          void *workspace, size_t workspace_bytes, const santa_debug *dbg,
                          santa_stream_t stream);

/*
 * S2ANTA-flash decode (paper notes, Key design 3): S_loc = ceil(S / T_b)
 * samples per tile with the shared offset U * S / S_loc, then a merge with
 * weights Z_tile / Z.  Same arguments as santa_decode_prop.
 */
int santa_decode_flash(const santa_problem *p, const void *q, const void *k, const void *v,
                       const long long *kv_indptr, const float *U, float *out,
                       void *workspace, size_t workspace_bytes, const santa_debug *dbg,
                       santa_stream_t stream);

/*
 * Exact split-KV decode: out = sum_i softmax(x)_i V_i, reading all of K and V.
 * Same arguments as santa_decode_prop without U (p->S and p->tile are ignored;
 * of dbg only error_flags, main_begin and main_end are used).  Workspace: per
 * (sequence slot, warp, query head) a float2 (M, Z) and a D-float partial sum,
 * for at most 160 rounded to a multiple of num_kv_heads streaming CTAs.
 */
int exact_decode(const santa_problem *p, const void *q, const void *k, const void *v,
                 const long long *kv_indptr, float *out,
                 void *workspace, size_t workspace_bytes, const santa_debug *dbg,
                 santa_stream_t stream);

/* Size of the library's built-in scratch array (see santa_decode_prop_static_scratch). */
#define SANTA_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * santa_decode_prop without a workspace argument, for callers that cannot
 * allocate device memory: e.g. a plugin inside a host program that owns every
 * device allocation through its own pool and gives plugins no allocator, or a
 * C caller on a path where cudaMalloc's implicit synchronisation is not allowed.
 * (This entry point has no counterpart in the paper; it is a packaging choice.)
 *
 * The scratch is a file-scope device array of SANTA_STATIC_SCRATCH_BYTES (16 MiB)
 * that every GPU loading this library holds until the process exits.  Problems
 * whose prop workspace (santa_workspace_size with SANTA_MODE_PROP) exceeds that
 * size are rejected with SANTA_WORKSPACE_TOO_SMALL before anything is enqueued;
 * roughly, batch * num_q_heads * max_len must stay below about 4 million.  The other
 * arguments, their layouts, ownership and errors are those of santa_decode_prop.
 * Nothing is allocated: not by this call, and not by any routine it calls.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.  (After a device reset the address is looked up again.)
 * Every call shares the one array, which keeps the last call's contents.  The
 * part of it that a prop workspace needs zero-filled (santa_workspace_init)
 * starts zero -- device arrays are zero when the library's code is loaded -- and
 * every call leaves it zero again; the rest is written before it is read, so
 * results never depend on an earlier call.  One exception: a call that raises
 * SANTA_ERR_TIMEOUT (a wait that gave up after about a second) poisons the array,
 * and later calls write zeros and raise SANTA_ERR_WORKSPACE until the process
 * exits.  Calls whose kernels overlap on the GPU (unordered streams or threads)
 * race on the array: order them.
 */
int santa_decode_prop_static_scratch(const santa_problem *p, const void *q, const void *k, const void *v,
                                     const long long *kv_indptr, const float *U, float *out,
                                     const santa_debug *dbg, santa_stream_t stream);

/*
 * Waits for `stream`, copies the device error word to *flags and clears it.
 * Returns SANTA_OK if it was zero, SANTA_DEVICE_CHECK if a bit was set,
 * SANTA_INVALID_ARG / SANTA_CUDA_ERROR otherwise.
 */
int santa_read_device_error(unsigned int *error_flags, santa_stream_t stream, unsigned int *flags);

/* A static, human-readable name for a status code. */
const char *santa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SANTA_DECODE_H */
