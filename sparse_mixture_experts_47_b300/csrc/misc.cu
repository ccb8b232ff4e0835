// Gather of token rows into the grouped layout, weighted combine, load
// statistics and the grouped-GEMM tile table.
//
// Sources: "Mixture of Experts" (waylandz.com ch. 30) §30.6.1 (weighted
// accumulation of expert outputs, aux loss), §30.4.5 (routed + shared
// output), §30.2.6 (load-balancing loss); "Mixture of Experts (MoE) memo"
// (iwashi.co), auxiliary loss section (f = routed share, p = mean router
// probability, aux = E sum f p); "混合エキスパートモデル（MoE）実践"
// (deepseekmodel.com), expert-parallel dispatch/combine (x[order // k],
// index_add_ back to token order).
#include "block_ops.cuh"
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace moe {

// Fixed-order tree reduction of one double per thread over a 256-thread block;
// the result is valid in thread 0.
__device__ double block_sum_256(double v, double *red) {
    red[threadIdx.x] = v;
    __syncthreads();
#pragma unroll
    for (int off = 128; off >= 1; off >>= 1) {
        if (threadIdx.x < off) red[threadIdx.x] += red[threadIdx.x + off];
        __syncthreads();
    }
    return red[0];
}

// p_e = (sum over blocks b of p_partial[b][e]) / T (block_p_finalize): one
// CTA of 1024 threads per 32 consecutive experts.
__global__ void __launch_bounds__(1024) p_finalize_kernel(const float *p_partial, int nblk, int E,
                                                          int T, float *p) {
    block_p_finalize(p_partial, nblk, E, T, p, blockIdx.x * 32);
}

cudaError_t launch_p_finalize(const float *p_partial, int nblk, int E, int T, float *p,
                              cudaStream_t st) {
    p_finalize_kernel<<<(E + 31) / 32, 1024, 0, st>>>(p_partial, nblk, E, T, p);
    note_launch();
    return cudaGetLastError();
}

// Column partial sums of a stored probs [T, E]: block b sums rows
// [32 b, 32 b + 32) per expert, in row order.
__global__ void prob_partials_kernel(const float *probs, int T, int E, float *p_partial) {
    const int t0 = blockIdx.x * 32;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float s = 0.f;
        for (int t = t0; t < t0 + 32 && t < T; ++t) s += probs[(size_t)t * E + e];
        p_partial[(size_t)blockIdx.x * E + e] = s;
    }
}

cudaError_t launch_prob_partials(const float *probs, int T, int E, float *p_partial,
                                 cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    prob_partials_kernel<<<(T + 31) / 32, 256, 0, st>>>(probs, T, E, p_partial);
    note_launch();
    return cudaGetLastError();
}

// Load statistics and observability outputs (block_load_stats) in one CTA of
// n threads, n the power of two >= E (32 to 1024).
__global__ void __launch_bounds__(1024) stats_finalize_kernel(const int32_t *counts,
                                                              const float *p, int T, int E,
                                                              int k, float *f, float *p_out,
                                                              float *aux, float *load,
                                                              ObsArgs o) {
    __shared__ StatsSmem sm;
    const int e = threadIdx.x;
    const int c = (e < E && counts) ? counts[e] : 0;
    block_load_stats(sm, blockDim.x, c, p, T, E, k, f, p_out, aux, load, o);
}

cudaError_t launch_stats_finalize(const int32_t *counts, const float *p, int T, int E, int k,
                                  float *f, float *p_out, float *aux, float *load,
                                  cudaStream_t st, const ObsArgs &o) {
    int n = 32;
    while (n < E && n < 1024) n *= 2;
    stats_finalize_kernel<<<1, n, 0, st>>>(counts, p, T, E, k, f, p_out, aux, load, o);
    note_launch();
    return cudaGetLastError();
}

// Per-block sums of the tokens' gate entropies -sum_e p ln p from stored
// probabilities [T, E] (terms with p = 0 contribute 0): 32 tokens per block,
// warp w owns tokens 4w..4w+3, fixed reduction order.
__global__ void __launch_bounds__(256) entropy_partials_kernel(const float *probs, int T, int E,
                                                               float *ent_partial) {
    __shared__ float st_h[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r = 0; r < 4; ++r) {
        const int tt = 4 * warp + r, t = blockIdx.x * 32 + tt;
        float h = 0.f;
        if (t < T)
            for (int e = lane; e < E; e += 32) {
                const float pv = probs[(size_t)t * E + e];
                if (pv > 0.f) h -= pv * logf(pv);
            }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) h += __shfl_xor_sync(0xffffffffu, h, off);
        if (lane == 0) st_h[tt] = h;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int tt = 0; tt < 32; ++tt) tot += st_h[tt];
        ent_partial[blockIdx.x] = tot;
    }
}

cudaError_t launch_entropy_partials(const float *probs, int T, int E, float *ent_partial,
                                    cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    entropy_partials_kernel<<<(T + 31) / 32, 256, 0, st>>>(probs, T, E, ent_partial);
    note_launch();
    return cudaGetLastError();
}

// Element i of the expert outputs (planes added in plane order).
__device__ __forceinline__ float expert_out_at(const ExpertOut &o, long long i) {
    float v = o.p[i];
    for (int sp = 1; sp < o.planes; ++sp) v += o.p[sp * o.plane + i];
    return v;
}
// Elements 4i .. 4i+3 of the expert outputs.
__device__ __forceinline__ float4 expert_out4(const ExpertOut &o, long long i) {
    const float4 *P = reinterpret_cast<const float4 *>(o.p);
    float4 v = P[i];
    for (int sp = 1; sp < o.planes; ++sp) {
        const float4 q = P[sp * (o.plane / 4) + i];
        v.x += q.x; v.y += q.y; v.z += q.z; v.w += q.w;
    }
    return v;
}

// Per sorted row r < *rows_end of the expert outputs: sum, sum of squares
// (fp64) and max |o|.  One warp per row; lane-strided partial sums, fixed
// butterfly.
__global__ void __launch_bounds__(256) row_stats_kernel(ExpertOut o, int d,
                                                        const int32_t *rows_end,
                                                        long long max_rows, double *rs) {
    const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= max_rows || r >= *rows_end) return;
    double s1 = 0.0, s2 = 0.0;
    float mx = 0.f;
    for (int c = lane; c < d; c += 32) {
        const float v = expert_out_at(o, r * d + c);
        s1 += v;
        s2 += (double)v * v;
        mx = fmaxf(mx, fabsf(v));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, off);
        s2 += __shfl_xor_sync(0xffffffffu, s2, off);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    if (lane == 0) {
        rs[3 * r] = s1;
        rs[3 * r + 1] = s2;
        rs[3 * r + 2] = mx;
    }
}

// Per expert e over its rows [offsets[e], offsets[e+1]) of row_stats: mean,
// population standard deviation and max |o| over all n_e * d elements.
__global__ void __launch_bounds__(256) expert_scale_kernel(const double *rs,
                                                           const int32_t *offsets, int d,
                                                           float *mean, float *std_,
                                                           float *maxabs) {
    __shared__ double red[256];
    __shared__ float redm[256];
    const int e = blockIdx.x;
    const int a = offsets[e], b = offsets[e + 1];
    double s1 = 0.0, s2 = 0.0;
    float mx = 0.f;
    for (int r = a + threadIdx.x; r < b; r += 256) {
        s1 += rs[3 * (size_t)r];
        s2 += rs[3 * (size_t)r + 1];
        mx = fmaxf(mx, (float)rs[3 * (size_t)r + 2]);
    }
    s1 = block_sum_256(s1, red);
    __syncthreads();
    s2 = block_sum_256(s2, red);
    redm[threadIdx.x] = mx;
    __syncthreads();
    for (int off = 128; off >= 1; off >>= 1) {
        if (threadIdx.x < off) redm[threadIdx.x] = fmaxf(redm[threadIdx.x], redm[threadIdx.x + off]);
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double n = (double)(b - a) * (double)d;
        const double mu = n > 0 ? s1 / n : 0.0;
        const double var = n > 0 ? fmax(s2 / n - mu * mu, 0.0) : 0.0;
        if (mean) mean[e] = (float)mu;
        if (std_) std_[e] = (float)sqrt(var);
        if (maxabs) maxabs[e] = redm[0];
    }
}

cudaError_t launch_expert_scale(const ExpertOut &o, int d, const int32_t *offsets, int E,
                                long long max_rows, double *rs, float *mean, float *std_,
                                float *maxabs, cudaStream_t st) {
    if (max_rows > 0) {
        row_stats_kernel<<<(unsigned)((max_rows + 7) / 8), 256, 0, st>>>(o, d, offsets + E,
                                                                         max_rows, rs);
        note_launch();
    }
    expert_scale_kernel<<<E, 256, 0, st>>>(rs, offsets, d, mean, std_, maxabs);
    note_launch();
    return cudaGetLastError();
}

// xs[s] = x[perm[s] / k] for s < offsets_end[0]; one warp per row,
// 16-byte vectors.
__global__ void gather_rows_kernel(const uint4 *x, int vec_per_row, const int32_t *perm,
                                   const int32_t *offsets_end, int k, long long max_rows,
                                   uint4 *xs) {
    const long long s = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= max_rows || s >= *offsets_end) return;
    const long long t = perm[s] / k;
    const uint4 *src = x + t * vec_per_row;
    uint4 *dst = xs + s * vec_per_row;
    // up to eight 16-byte loads in flight per lane before the stores; the
    // grouped rows are written once and read by the up projection, so they
    // are stored evict-first and leave L2 to x, which each token's k rows
    // re-read
    for (int i0 = 0; i0 < vec_per_row; i0 += 256) {
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = i0 + lane + 32 * q;
            if (i < vec_per_row) v[q] = src[i];
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = i0 + lane + 32 * q;
            if (i < vec_per_row) __stcs(dst + i, v[q]);
        }
    }
}

cudaError_t launch_gather_rows(const void *x, int elem_bytes, int d, const int32_t *perm,
                               const int32_t *offsets_end, int k, long long max_rows, void *xs,
                               cudaStream_t st) {
    if (max_rows == 0) return cudaSuccess;
    const int vpr = d * elem_bytes / 16;
    gather_rows_kernel<<<(unsigned)((max_rows + 7) / 8), 256, 0, st>>>(
        static_cast<const uint4 *>(x), vpr, perm, offsets_end, k, max_rows,
        static_cast<uint4 *>(xs));
    note_launch();
    return cudaGetLastError();
}

// Token-major form of the same copy (token choice, slots known by inv): one
// warp per token reads its row of x once and writes it to the rows of its
// kept slots.  x is read from HBM once instead of k times through L2, which
// misses once x outgrows L2 (the 896-expert layer: 134 MB of x, k = 8).
__global__ void scatter_rows_kernel(const uint4 *x, int vec_per_row, const int32_t *inv, int k,
                                    long long T, uint4 *xs) {
    const long long t = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    // rows of the token's slots (k <= 16), spread to every lane while the
    // whole warp is converged
    const int my_row = lane < k ? inv[t * k + lane] : -1;
    int rows[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) rows[j] = __shfl_sync(0xffffffffu, my_row, j);
    const uint4 *src = x + t * vec_per_row;
    // up to 8 16-byte loads per lane in flight before the stores (a row of
    // 1024 bf16 is 4 per lane)
    for (int i0 = 0; i0 < vec_per_row; i0 += 256) {
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int i = i0 + lane + 32 * q;
            if (i < vec_per_row) v[q] = src[i];
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j >= k || rows[j] < 0) continue;
            uint4 *dst = xs + (long long)rows[j] * vec_per_row;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int i = i0 + lane + 32 * q;
                if (i < vec_per_row) __stcs(dst + i, v[q]);
            }
        }
    }
}

cudaError_t launch_scatter_rows(const void *x, int elem_bytes, int d, const int32_t *inv, int k,
                                long long T, void *xs, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int vpr = d * elem_bytes / 16;
    scatter_rows_kernel<<<(unsigned)((T + 7) / 8), 256, 0, st>>>(
        static_cast<const uint4 *>(x), vpr, inv, k, T, static_cast<uint4 *>(xs));
    note_launch();
    return cudaGetLastError();
}

// y[t] = sum_j [inv >= 0] w[t,j] o[inv[t,j]] (j in order) + s[t], where
// o = sum of the out_sorted planes and s = sum of the shared planes, each in
// plane order.
__device__ __forceinline__ float4 sum_planes4(const float4 *p, int planes, long long plane4,
                                              long long i) {
    float4 o = p[i];
    for (int s = 1; s < planes; ++s) {
        const float4 q = p[s * plane4 + i];
        o.x += q.x; o.y += q.y; o.z += q.z; o.w += q.w;
    }
    return o;
}

template <typename TO>
__device__ __forceinline__ void store_y4(TO *y, long long i, float4 acc) {
    if constexpr (sizeof(TO) == 4) {
        reinterpret_cast<float4 *>(y)[i] = acc;
    } else {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&lo);
        u.y = *reinterpret_cast<uint32_t *>(&hi);
        reinterpret_cast<uint2 *>(y)[i] = u;
    }
}

// One warp per (token, chunk of U * 32 float4 columns): lane l holds columns
// c0 + l + 32 u (u < U) of the token's output, loads the U vectors of a slot
// together and adds the slots in j order (then the shared expert): the same
// arithmetic per element for every chunk width.  U follows the grid: 8
// vectors per lane when the batch fills the GPU, fewer when few tokens must
// spread their columns over more warps (DeepSeek T = 128: 14 chunks of 128
// columns per token instead of one CTA per token on 128 of 148 SMs).  One
// CTA per token took 28 us for Switch's 8192 tokens of 4 KB of output each.
template <typename TO, int U>
__global__ void __launch_bounds__(256) combine_kernel(ExpertOut out_sorted, const int32_t *inv,
                                                      const float *w, ExpertOut sh, int T, int k,
                                                      int d4, int chunks, TO *y) {
    const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= (long long)T * chunks) return;
    const long long t = gw / chunks;
    const int c0 = (int)(gw - t * chunks) * (U * 32) + lane;
    // slot rows and weights (k <= 16), spread to every lane
    const int my_row = lane < k ? inv[t * k + lane] : -1;
    const float my_w = lane < k ? w[t * k + lane] : 0.f;
    float4 acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int s = __shfl_sync(0xffffffffu, my_row, j);
        const float wj = __shfl_sync(0xffffffffu, my_w, j);
        if (s < 0) continue;
        float4 o[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + 32 * u;
            o[u] = c < d4 ? expert_out4(out_sorted, (long long)s * d4 + c)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            acc[u].x = fmaf(wj, o[u].x, acc[u].x); acc[u].y = fmaf(wj, o[u].y, acc[u].y);
            acc[u].z = fmaf(wj, o[u].z, acc[u].z); acc[u].w = fmaf(wj, o[u].w, acc[u].w);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c >= d4) break;
        if (sh.p) {
            const float4 sv = expert_out4(sh, t * d4 + c);
            acc[u].x += sv.x; acc[u].y += sv.y; acc[u].z += sv.z; acc[u].w += sv.w;
        }
        store_y4(y, t * d4 + c, acc[u]);
    }
}

// One CTA per token (with more than 2 slots and enough tokens to fill the GPU):
// its slots' rows and weights are read once into shared memory, each thread
// takes one column vector at a time and adds the slots in j order.  At k = 8
// this kept more loads in flight than a warp per column chunk (DeepSeek
// T = 8192 0.345 against 0.40 ms, the 896-expert layer 0.343 against 0.38).
template <typename TO, int kCombineU>
__global__ void combine_token_kernel(ExpertOut out_sorted, const int32_t *inv, const float *w,
                               ExpertOut sh, int k, int d4, TO *y) {
    __shared__ int srow[16];
    __shared__ float sw[16];
    const long long t = blockIdx.x;
    if (threadIdx.x < k) {
        srow[threadIdx.x] = inv[t * k + threadIdx.x];
        sw[threadIdx.x] = w[t * k + threadIdx.x];
    }
    __syncthreads();
    for (int c0 = threadIdx.x; c0 < d4; c0 += kCombineU * blockDim.x) {
        float4 acc[kCombineU];
#pragma unroll
        for (int u = 0; u < kCombineU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int s = srow[j];
            if (s < 0) continue;
            const float wj = sw[j];
            float4 o[kCombineU];
#pragma unroll
            for (int u = 0; u < kCombineU; ++u) {
                const int c = c0 + u * blockDim.x;
                o[u] = c < d4 ? expert_out4(out_sorted, (long long)s * d4 + c)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kCombineU; ++u) {
                acc[u].x = fmaf(wj, o[u].x, acc[u].x); acc[u].y = fmaf(wj, o[u].y, acc[u].y);
                acc[u].z = fmaf(wj, o[u].z, acc[u].z); acc[u].w = fmaf(wj, o[u].w, acc[u].w);
            }
        }
#pragma unroll
        for (int u = 0; u < kCombineU; ++u) {
            const int c = c0 + u * blockDim.x;
            if (c >= d4) break;
            if (sh.p) {
                const float4 sv = expert_out4(sh, t * d4 + c);
                acc[u].x += sv.x; acc[u].y += sv.y; acc[u].z += sv.z; acc[u].w += sv.w;
            }
            store_y4(y, t * d4 + c, acc[u]);
        }
    }
}

template <typename TO, int U>
static void launch_combine_u(const ExpertOut &o, const int32_t *inv, const float *w,
                             const ExpertOut &sh, int T, int k, int d4, TO *y, cudaStream_t st) {
    const int chunks = (d4 + U * 32 - 1) / (U * 32);
    const long long warps = (long long)T * chunks;
    combine_kernel<TO, U><<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(o, inv, w, sh, T, k, d4,
                                                                        chunks, y);
}

template <typename TO>
static void launch_combine_t(const ExpertOut &o, const int32_t *inv, const float *w,
                             const ExpertOut &sh, int T, int k, int d4, TO *y, cudaStream_t st) {
    // the widest chunk that still gives every SM about 32 warps; with more
    // than 2 slots at most 2 vectors per lane
    constexpr long long kWantWarps = 148 * 32;
    auto warps = [&](int u) { return (long long)T * ((d4 + u * 32 - 1) / (u * 32)); };
    if (k <= 2 && warps(8) >= kWantWarps) launch_combine_u<TO, 8>(o, inv, w, sh, T, k, d4, y, st);
    else if (k <= 2 && warps(4) >= kWantWarps)
        launch_combine_u<TO, 4>(o, inv, w, sh, T, k, d4, y, st);
    else if (warps(2) >= kWantWarps) launch_combine_u<TO, 2>(o, inv, w, sh, T, k, d4, y, st);
    else launch_combine_u<TO, 1>(o, inv, w, sh, T, k, d4, y, st);
}

cudaError_t launch_combine(const ExpertOut &o, const int32_t *inv, const float *w,
                           const ExpertOut &sh, int T, int k, int d, int out_dtype, void *y,
                           cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int d4 = d / 4;
    if (k > 2 && T >= 148 * 8) {
        const int threads = d4 >= 256 ? 256 : ((d4 + 31) / 32) * 32;
        if (out_dtype == MOE_DTYPE_FP32)
            combine_token_kernel<float, 1><<<T, threads, 0, st>>>(o, inv, w, sh, k, d4,
                                                                   static_cast<float *>(y));
        else
            combine_token_kernel<__nv_bfloat16, 1><<<T, threads, 0, st>>>(
                o, inv, w, sh, k, d4, static_cast<__nv_bfloat16 *>(y));
    } else if (out_dtype == MOE_DTYPE_FP32) {
        launch_combine_t(o, inv, w, sh, T, k, d4, static_cast<float *>(y), st);
    } else {
        launch_combine_t(o, inv, w, sh, T, k, d4, static_cast<__nv_bfloat16 *>(y), st);
    }
    note_launch();
    return cudaGetLastError();
}

// Combine over a per-token row list (expert choice): y[t] = sum over
// i in [tok_start[t], tok_start[t+1]) of row_w[r_i] o[r_i] (list order) +
// s[t], o and s summed over their planes in plane order.
template <typename TO>
__global__ void combine_rows_kernel(ExpertOut out_sorted, const int32_t *tok_start,
                                    const int32_t *tok_rows, const float *row_w, ExpertOut sh,
                                    int d4, TO *y) {
    const long long t = blockIdx.x;
    const int a = tok_start[t], b = tok_start[t + 1];
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = a; i < b; ++i) {
            const int r = tok_rows[i];
            const float wr = row_w[r];
            const float4 o = expert_out4(out_sorted, (long long)r * d4 + c);
            acc.x = fmaf(wr, o.x, acc.x); acc.y = fmaf(wr, o.y, acc.y);
            acc.z = fmaf(wr, o.z, acc.z); acc.w = fmaf(wr, o.w, acc.w);
        }
        if (sh.p) {
            const float4 sv = expert_out4(sh, t * d4 + c);
            acc.x += sv.x; acc.y += sv.y; acc.z += sv.z; acc.w += sv.w;
        }
        if constexpr (sizeof(TO) == 4) {
            reinterpret_cast<float4 *>(y)[t * d4 + c] = acc;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t *>(&lo);
            u.y = *reinterpret_cast<uint32_t *>(&hi);
            reinterpret_cast<uint2 *>(y)[t * d4 + c] = u;
        }
    }
}

cudaError_t launch_combine_rows(const ExpertOut &o, const int32_t *tok_start,
                                const int32_t *tok_rows, const float *row_w, const ExpertOut &sh,
                                int T, int d, int out_dtype, void *y, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int d4 = d / 4;
    const int threads = d4 >= 256 ? 256 : ((d4 + 31) / 32) * 32;
    if (out_dtype == MOE_DTYPE_FP32)
        combine_rows_kernel<float><<<T, threads, 0, st>>>(o, tok_start, tok_rows, row_w, sh, d4,
                                                          static_cast<float *>(y));
    else
        combine_rows_kernel<__nv_bfloat16><<<T, threads, 0, st>>>(
            o, tok_start, tok_rows, row_w, sh, d4, static_cast<__nv_bfloat16 *>(y));
    note_launch();
    return cudaGetLastError();
}

// Per-slot result of the plain capacity rule: the slot's expert and gate
// weight, or -1 and 0 when it was dropped.
__global__ void slot_outputs_kernel(const int32_t *idx, const float *w, const int32_t *inv,
                                    long long n, int32_t *slot_expert, float *slot_w) {
    for (long long f = blockIdx.x * (long long)blockDim.x + threadIdx.x; f < n;
         f += (long long)gridDim.x * blockDim.x) {
        const bool kept = inv[f] >= 0;
        if (slot_expert) slot_expert[f] = kept ? idx[f] : -1;
        if (slot_w) slot_w[f] = kept ? w[f] : 0.f;
    }
}

cudaError_t launch_slot_outputs(const int32_t *idx, const float *w, const int32_t *inv,
                                long long n, int32_t *slot_expert, float *slot_w,
                                cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int grid = (int)std::min<long long>((n + 255) / 256, 148 * 8);
    slot_outputs_kernel<<<grid, 256, 0, st>>>(idx, w, inv, n, slot_expert, slot_w);
    note_launch();
    return cudaGetLastError();
}

// Activation of split up-projection partial sums: one thread per 8 features
// of one row; the splits are added in order.
template <bool SWIGLU>
__global__ void split_activation_kernel(const float *P, int splits, long long plane, int N,
                                        const int32_t *rows_end, long long max_rows,
                                        __nv_bfloat16 *h) {
    const int n8 = N / 8;
    const long long ldp = SWIGLU ? 2ll * N : (long long)N;
    const long long rows = min((long long)*rows_end, max_rows);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < rows * n8;
         i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / n8;
        const int f = (int)(i - r * n8) * 8;
        float a[8], b[8];
        const float *p = P + r * ldp + f;
#pragma unroll
        for (int q = 0; q < 8; ++q) { a[q] = p[q]; b[q] = SWIGLU ? p[N + q] : 0.f; }
        for (int s = 1; s < splits; ++s) {
            const float *ps = p + s * plane;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                a[q] += ps[q];
                if (SWIGLU) b[q] += ps[N + q];
            }
        }
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = SWIGLU ? silu(a[q]) * b[q] : fmaxf(a[q], 0.f);
        uint4 u;
        uint32_t *wv = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            __nv_bfloat162 pr = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
            wv[q] = *reinterpret_cast<uint32_t *>(&pr);
        }
        *reinterpret_cast<uint4 *>(h + r * N + f) = u;
    }
}

cudaError_t launch_split_activation(const float *P, int splits, long long plane, int N,
                                    int swiglu, const int32_t *rows_end, long long max_rows,
                                    __nv_bfloat16 *h, cudaStream_t st) {
    if (max_rows == 0) return cudaSuccess;
    const long long work = max_rows * (N / 8);
    const int grid = (int)std::min<long long>((work + 255) / 256, 148 * 8);
    if (swiglu)
        split_activation_kernel<true><<<grid, 256, 0, st>>>(P, splits, plane, N, rows_end,
                                                            max_rows, h);
    else
        split_activation_kernel<false><<<grid, 256, 0, st>>>(P, splits, plane, N, rows_end,
                                                             max_rows, h);
    note_launch();
    return cudaGetLastError();
}

// out[r] = sum_s P_s[r] for rows r < *rows_end (fp32, split order).
__global__ void sum_planes_kernel(const float4 *P, int splits, long long plane4, int d4,
                                  const int32_t *rows_end, long long max_rows, float4 *out) {
    const long long rows = min((long long)*rows_end, max_rows);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < rows * d4;
         i += (long long)gridDim.x * blockDim.x)
        out[i] = sum_planes4(P, splits, plane4, i);
}

cudaError_t launch_sum_planes(const float *P, int splits, long long plane, int d,
                              const int32_t *rows_end, long long max_rows, float *out,
                              cudaStream_t st) {
    if (max_rows == 0) return cudaSuccess;
    const long long work = max_rows * (d / 4);
    const int grid = (int)std::min<long long>((work + 255) / 256, 148 * 8);
    sum_planes_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const float4 *>(P), splits,
                                            plane / 4, d / 4, rows_end, max_rows,
                                            reinterpret_cast<float4 *>(out));
    note_launch();
    return cudaGetLastError();
}

// Tile table of a grouped GEMM with BM-row tiles (block_build_tiles).
__global__ void __launch_bounds__(1024) build_tiles_kernel(const int32_t *offsets, int E,
                                                           int BM, int32_t *tile_e,
                                                           int32_t *tile_m0, int32_t *tile_start,
                                                           int32_t *n_tiles) {
    block_build_tiles(offsets, E, BM, tile_e, tile_m0, tile_start, n_tiles);
}

cudaError_t launch_build_tiles(const int32_t *offsets, int E, int BM, int32_t *tile_e,
                               int32_t *tile_m0, int32_t *tile_start, int32_t *n_tiles,
                               cudaStream_t st) {
    build_tiles_kernel<<<1, 1024, 0, st>>>(offsets, E, BM, tile_e, tile_m0, tile_start, n_tiles);
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
