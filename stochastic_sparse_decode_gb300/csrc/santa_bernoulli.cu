// santa_bernoulli.cu -- S2ANTA-prop with the Bernoulli ternary score stage.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (paper notes), Key
// design 4: the query, scaled into [-1, 1] by its largest magnitude, gives each
// feature a Bernoulli probability; a draw keeps feature i as sign(q_i) (else 0),
// and max|q| times that ternary query dotted with a key estimates q . k without
// bias.  Only the features some draw keeps are read from K.  The ablation table's
// mean group query draws one feature set per GQA group from the mean of its
// queries, so that the group's heads share the features read; head g then weights
// a kept feature by q_gi / p_i, which keeps its estimate unbiased.
//
// Three kernels on the stream:
//   1. bernoulli_query_kernel, one CTA per (KV head, sequence), one thread per
//      feature: the draw probabilities in single precision (as the caller's
//      queries and uniforms are), the draws (u < p), the effective queries
//      c_g = estimate weights, and the group's list of features kept by any draw,
//      compacted in feature order, with c stored in list order.
//   2. fb_pass1_kernel, pass 1 on a feature-blocked K cache: K_fb[row / 64][kvh]
//      [feature][row % 64], so the 64 keys of one feature are one 128-byte line
//      (bf16) and a feature no draw kept costs no DRAM traffic.  (With 16 keys per
//      32-byte sector the saving vanished: GB300's DRAM traffic, measured, comes
//      in lines, and a line of 4 features almost always holds a kept one.)  One
//      warp per 64 keys, two chunks: x_g = scale * sum over the list of c_g,j k_j,
//      then each chunk's record (m, z) and exp(x - m) into the stash, exactly the
//      outputs of the token-major pass 1.
//   3. the cluster pass 2 of santa_decode_prop, unchanged.
#include "santa_launch.h"
#include "santa_stream.cuh"

namespace santa {

constexpr int kFbWarps = 8;   // warps of a feature-blocked pass-1 CTA
constexpr int kFbBatch = 32;  // features whose loads a warp issues together

// Effective queries and the kept-feature list of one (KV head, sequence).
template <typename T, int G>
__global__ void __launch_bounds__(128) bernoulli_query_kernel(const Params p) {
    const int kvh = blockIdx.x, b = blockIdx.y, i = threadIdx.x, D = p.D;
    const int lane = i & 31, warp = i >> 5;
    __shared__ float s_red[4];
    __shared__ int s_cnt[4];
    const size_t hq0 = size_t(b) * p.Hq + size_t(kvh) * G;
    const T *q = static_cast<const T *>(p.q) + hq0 * D;
    float qv[G];
#pragma unroll
    for (int g = 0; g < G; ++g) qv[g] = i < D ? to_float<T>(q[size_t(g) * D + i]) : 0.f;

    // the largest magnitude over the features: per head, or of the group's mean
    auto block_max_abs = [&](float a) {
        a = warp_max(a);
        __syncthreads();
        if (lane == 0) s_red[warp] = a;
        __syncthreads();
        float m = s_red[0];
        for (int w = 1; w < D / 32; ++w) m = fmaxf(m, s_red[w]);
        return m;
    };
    const float invB = 1.0f / float(p.draws);
    int hits[G];
    float c[G];
    bool kept = false;
    if (p.group_mean) {
        float s = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) s += qv[g];
        const float mean = s / float(G);
        const float mx = block_max_abs(fabsf(mean));
        const float pr = mx > 0.f ? fabsf(mean) / mx : 0.f;
        int n = 0;
        if (pr > 0.f && i < D) {
            const float *u = p.bern_u + (size_t(b) * p.Hkv + kvh) * p.draws * D + i;
            for (int d = 0; d < p.draws; ++d) n += __ldg(u + size_t(d) * D) < pr ? 1 : 0;
        }
        kept = n > 0;
#pragma unroll
        for (int g = 0; g < G; ++g) c[g] = n > 0 ? qv[g] / pr * (float(n) * invB) : 0.f;
        (void)hits;
    } else {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float mx = block_max_abs(fabsf(qv[g]));
            int n = 0;
            if (mx > 0.f && i < D) {
                const float pr = fabsf(qv[g]) / mx;
                const float *u = p.bern_u + ((hq0 + g) * p.draws) * D + i;
                for (int d = 0; d < p.draws; ++d) n += __ldg(u + size_t(d) * D) < pr ? 1 : 0;
            }
            hits[g] = n;
            const float sgn = qv[g] > 0.f ? 1.f : (qv[g] < 0.f ? -1.f : 0.f);
            c[g] = mx * sgn * (float(n) * invB);
            kept |= n > 0;
        }
    }
    // compaction in feature order: this thread's slot among the kept features
    const unsigned bal = __ballot_sync(kFull, kept && i < D);
    if (lane == 0) s_cnt[warp] = __popc(bal);
    __syncthreads();
    int off = 0, total = 0;
    for (int w = 0; w < D / 32; ++w) {
        if (w < warp) off += s_cnt[w];
        total += s_cnt[w];
    }
    off += __popc(bal & ((1u << lane) - 1u));
    const size_t grp = size_t(b) * p.Hkv + kvh;
    if (kept && i < D) {
        p.tq_list[grp * D + off] = static_cast<unsigned char>(i);
#pragma unroll
        for (int g = 0; g < G; ++g) p.tq_c[(hq0 + g) * D + off] = c[g];
    }
    if (i == 0) {
        p.tq_cnt[grp] = total;
        if (p.dbg_feat) p.dbg_feat[grp] = total;
    }
}

// Pass 1 on the feature-blocked cache: warps walk (sequence, chunk pair, KV head)
// units with a stride of the grid's warp count; a warp stages its group's list and
// effective queries in shared memory when its (sequence, KV head) changes.  A unit
// is 64 keys, chunks 2cp and 2cp + 1: lane l holds keys 64cp + l and 64cp + 32 + l,
// so that for one feature the warp's two loads cover the feature's 128-byte line
// of 64 keys (for bf16; a key block that starts mid-line touches two lines).
template <typename T, int D, int G>
__global__ void __launch_bounds__(kFbWarps * 32, 3) fb_pass1_kernel(const Params p) {
    __shared__ int s_list[kFbWarps][D];
    __shared__ float s_c[kFbWarps][G][D];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int npair = (p.nch + 1) / 2;
    const long long units = (long long)p.B * npair * p.Hkv;
    const long long stride = (long long)gridDim.x * kFbWarps;
    int cur_b = -1, cur_kvh = -1, nsel = 0, L = 0;
    long long start = 0;
    const T *kfb = static_cast<const T *>(p.k);
    pdl_wait();
    pdl_launch_dependents();
    for (long long u = (long long)blockIdx.x * kFbWarps + warp; u < units; u += stride) {
        const int kvh = int(u % p.Hkv);
        const long long r = u / p.Hkv;
        const int b = int(r / npair), cp = int(r % npair);
        if (b != cur_b || kvh != cur_kvh) {
            __syncwarp();
            if (b != cur_b) L = seq_bounds(p, b, &start);
            cur_b = b;
            cur_kvh = kvh;
            const size_t grp = size_t(b) * p.Hkv + kvh;
            nsel = min(max(p.tq_cnt[grp], 0), D);
            for (int j = lane; j < nsel; j += 32) {
                s_list[warp][j] = p.tq_list[grp * D + j];
#pragma unroll
                for (int g = 0; g < G; ++g)
                    s_c[warp][g][j] = p.tq_c[(size_t(b) * p.Hq + size_t(kvh) * G + g) * D + j];
            }
            __syncwarp();
        }
        const int key0 = cp * 2 * kChunkRows;
        if (key0 >= L) continue;  // past the sequence: no record
        const int ka = key0 + lane, kb = ka + kChunkRows;
        const bool va = ka < L, vb = kb < L;
        const long long ra = start + (va ? ka : key0), rb = start + (vb ? kb : key0);
        const T *pa = kfb + ((size_t(ra >> 6) * p.Hkv + kvh) * D) * 64 + (ra & 63);
        const T *pb = kfb + ((size_t(rb >> 6) * p.Hkv + kvh) * D) * 64 + (rb & 63);
        float xa[G], xb[G];
#pragma unroll
        for (int g = 0; g < G; ++g) xa[g] = xb[g] = 0.f;
        // kFbBatch / 2 features at a time: kFbBatch independent loads of the warp in flight
        constexpr int kF = kFbBatch / 2;
        int j = 0;
        for (; j + kF <= nsel; j += kF) {
            T ea[kF], eb[kF];
#pragma unroll
            for (int t = 0; t < kF; ++t) {
                const int off = s_list[warp][j + t] * 64;
                ea[t] = __ldg(pa + off);
                eb[t] = __ldg(pb + off);
            }
#pragma unroll
            for (int t = 0; t < kF; ++t) {
                const float fa = to_float<T>(ea[t]), fb = to_float<T>(eb[t]);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float c = s_c[warp][g][j + t];
                    xa[g] = fmaf(c, fa, xa[g]);
                    xb[g] = fmaf(c, fb, xb[g]);
                }
            }
        }
        for (; j < nsel; ++j) {
            const int off = s_list[warp][j] * 64;
            const float fa = to_float<T>(__ldg(pa + off)), fb = to_float<T>(__ldg(pb + off));
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float c = s_c[warp][g][j];
                xa[g] = fmaf(c, fa, xa[g]);
                xb[g] = fmaf(c, fb, xb[g]);
            }
        }
        // the two chunks' records and stash rows
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int ch = 2 * cp + half;
            if (ch * kChunkRows >= L) break;
            const bool valid = half ? vb : va;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float xs = valid ? (half ? xb[g] : xa[g]) * p.scale : -INFINITY;
                const float m = warp_max(xs);
                const float e = valid ? __expf(xs - m) : 0.f;
                const float z = warp_sum(e);
                const size_t hq = size_t(b) * p.Hq + size_t(kvh) * G + g;
                p.stash[(hq * p.nch + ch) * kChunkRows + lane] = e;
                if (lane == 0) store_record(p.rec + hq * p.nch + ch, m, z);
            }
        }
    }
}

// Token-major [rows][Hkv][D] to feature-blocked [ceil(rows / 64)][Hkv][D][64]
// (rows past the end are zero).
template <typename T>
__global__ void feature_block_kernel(const T *k, T *kfb, long long rows, int hkv, int D) {
    const long long blocks = (rows + 63) / 64;
    const long long n = blocks * hkv * D * 64;
    for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < n; o += (long long)gridDim.x * blockDim.x) {
        const int pos = int(o & 63);
        const long long rest = o >> 6;
        const int f = int(rest % D);
        const long long bh = rest / D;
        const int h = int(bh % hkv);
        const long long blk = bh / hkv;
        const long long row = blk * 64 + pos;
        kfb[o] = row < rows ? k[(row * hkv + h) * D + f] : T(0);
    }
}

cudaError_t launch_feature_block(int dtype, const void *k, void *kfb, long long rows, int hkv, int D,
                                 cudaStream_t stream) {
    const long long n = (rows + 63) / 64 * hkv * D * 64;
    const unsigned blocks = unsigned(n / 256 + 1 < 4096 ? n / 256 + 1 : 4096);
    if (dtype == SANTA_BF16)
        feature_block_kernel<uint16_t><<<blocks, 256, 0, stream>>>(static_cast<const uint16_t *>(k),
                                                                   static_cast<uint16_t *>(kfb), rows, hkv, D);
    else
        feature_block_kernel<float><<<blocks, 256, 0, stream>>>(static_cast<const float *>(k),
                                                                static_cast<float *>(kfb), rows, hkv, D);
    return cudaGetLastError();
}

cudaError_t launch_prop_bernoulli(const Params &p, int dtype, cudaStream_t stream, const Timing &tm) {
    int sms = 0;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = SANTA_DISPATCH(dtype, p.D, p.G, {
        bernoulli_query_kernel<T, G><<<dim3(unsigned(p.Hkv), unsigned(p.B)), 128, 0, stream>>>(p);
        cudaError_t e1 = cudaGetLastError();
        if (e1 != cudaSuccess) return e1;
        // three CTAs of 8 warps per SM, each warp with up to kFbBatch loads in flight
        const long long units = (long long)p.B * ((p.nch + 1) / 2) * p.Hkv;
        long long grid = (long long)sms * 3;
        if (grid > (units + kFbWarps - 1) / kFbWarps) grid = (units + kFbWarps - 1) / kFbWarps;
        if (grid < 1) grid = 1;
        record_event(tm.begin, stream);
        e1 = launch_kernel(fb_pass1_kernel<T, D, G>, dim3(unsigned(grid)), dim3(kFbWarps * 32), 0, stream, true, 0,
                           false, p);
        if (e1 != cudaSuccess) return e1;
        record_event(tm.end, stream);
        return cudaSuccess;
    });
    if (e != cudaSuccess) return e;
    CUtensorMap unused = {};
    return launch_prop(p, dtype, unused, stream, Timing{}, kPass2);
}

}  // namespace santa
