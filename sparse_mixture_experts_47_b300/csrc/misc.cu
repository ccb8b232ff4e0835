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
#include "common.cuh"
#include "kernels.h"

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

// p_e = (sum over blocks b of p_partial[b][e]) / T in fp64: one CTA per expert,
// thread i sums blocks i, i+256, ... in order, then a fixed tree.
__global__ void __launch_bounds__(256) p_finalize_kernel(const float *p_partial, int nblk, int E,
                                                         int T, float *p) {
    __shared__ double red[256];
    const int e = blockIdx.x;
    double s = 0.0;
    for (int b = threadIdx.x; b < nblk; b += 256) s += (double)p_partial[(size_t)b * E + e];
    s = block_sum_256(s, red);
    if (threadIdx.x == 0) p[e] = T > 0 ? (float)(s / (double)T) : 0.f;
}

cudaError_t launch_p_finalize(const float *p_partial, int nblk, int E, int T, float *p,
                              cudaStream_t st) {
    p_finalize_kernel<<<E, 256, 0, st>>>(p_partial, nblk, E, T, p);
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

// f_e = count_e / (T k); aux = E * sum_e f_e p_e (fp64, fixed tree order);
// load = max_e count_e / (T k / E).  One CTA of 1024 threads, E <= 1024.
__global__ void __launch_bounds__(1024) stats_finalize_kernel(const int32_t *counts,
                                                              const float *p, int T, int E,
                                                              int k, float *f, float *p_out,
                                                              float *aux, float *load) {
    __shared__ double red[1024];
    __shared__ int redmax[1024];
    const int e = threadIdx.x;
    const double tk = (double)T * (double)k;
    double fp = 0.0;
    int c = 0;
    if (e < E) {
        c = counts[e];
        const double fe = tk > 0 ? (double)c / tk : 0.0;
        if (f) f[e] = (float)fe;
        if (p_out && p_out != p) p_out[e] = p[e];
        fp = fe * (double)p[e];
    }
    red[e] = fp;
    redmax[e] = c;
    __syncthreads();
#pragma unroll
    for (int off = 512; off >= 1; off >>= 1) {
        if (e < off) {
            red[e] += red[e + off];
            redmax[e] = max(redmax[e], redmax[e + off]);
        }
        __syncthreads();
    }
    if (e == 0) {
        if (aux) *aux = (float)((double)E * red[0]);
        if (load) *load = tk > 0 ? (float)((double)redmax[0] / (tk / (double)E)) : 0.f;
    }
}

cudaError_t launch_stats_finalize(const int32_t *counts, const float *p, int T, int E, int k,
                                  float *f, float *p_out, float *aux, float *load,
                                  cudaStream_t st) {
    stats_finalize_kernel<<<1, 1024, 0, st>>>(counts, p, T, E, k, f, p_out, aux, load);
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
    for (int i = lane; i < vec_per_row; i += 32) dst[i] = src[i];
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

// y[t] = sum_j [inv >= 0] w[t,j] out_sorted[inv[t,j]] (j in order) + shared[t].
template <typename TO>
__global__ void combine_kernel(const float4 *out_sorted, const int32_t *inv, const float *w,
                               const float4 *shared_out, int k, int d4, TO *y) {
    const long long t = blockIdx.x;
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int s = inv[t * k + j];
            if (s < 0) continue;
            const float wj = w[t * k + j];
            const float4 o = out_sorted[(long long)s * d4 + c];
            acc.x = fmaf(wj, o.x, acc.x); acc.y = fmaf(wj, o.y, acc.y);
            acc.z = fmaf(wj, o.z, acc.z); acc.w = fmaf(wj, o.w, acc.w);
        }
        if (shared_out) {
            const float4 sv = shared_out[t * d4 + c];
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

cudaError_t launch_combine(const float *out_sorted, const int32_t *inv, const float *w,
                           const float *shared_out, int T, int k, int d, int out_dtype, void *y,
                           cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int d4 = d / 4;
    const int threads = d4 >= 256 ? 256 : ((d4 + 31) / 32) * 32;
    if (out_dtype == MOE_DTYPE_FP32)
        combine_kernel<float><<<T, threads, 0, st>>>(
            reinterpret_cast<const float4 *>(out_sorted), inv, w,
            reinterpret_cast<const float4 *>(shared_out), k, d4, static_cast<float *>(y));
    else
        combine_kernel<__nv_bfloat16><<<T, threads, 0, st>>>(
            reinterpret_cast<const float4 *>(out_sorted), inv, w,
            reinterpret_cast<const float4 *>(shared_out), k, d4,
            static_cast<__nv_bfloat16 *>(y));
    note_launch();
    return cudaGetLastError();
}

// Tile table of a grouped GEMM with BM-row tiles: expert e owns
// ceil((offsets[e+1]-offsets[e]) / BM) tiles starting at row offsets[e];
// tile_start[e] is the index of its first tile (tile_start[E] = total).
__global__ void __launch_bounds__(1024) build_tiles_kernel(const int32_t *offsets, int E,
                                                           int BM, int32_t *tile_e,
                                                           int32_t *tile_m0, int32_t *tile_start,
                                                           int32_t *n_tiles) {
    __shared__ int warp_tot[32];
    __shared__ int carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int e0 = 0; e0 < E; e0 += 1024) {
        const int e = e0 + threadIdx.x;
        int mt = 0;
        if (e < E) mt = (offsets[e + 1] - offsets[e] + BM - 1) / BM;
        int incl = mt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int wt = warp_tot[lane];
            int wi = wt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, wi, off);
                if (lane >= off) wi += o;
            }
            warp_tot[lane] = wi - wt;
        }
        __syncthreads();
        const int start = carry + warp_tot[warp] + incl - mt;
        if (e < E && tile_start) tile_start[e] = start;
        for (int i = 0; i < mt; ++i) {
            tile_e[start + i] = e;
            if (tile_m0) tile_m0[start + i] = offsets[e] + i * BM;
        }
        __syncthreads();
        if (threadIdx.x == 1023) carry = start + mt;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        *n_tiles = carry;
        if (tile_start) tile_start[E] = carry;
    }
}

cudaError_t launch_build_tiles(const int32_t *offsets, int E, int BM, int32_t *tile_e,
                               int32_t *tile_m0, int32_t *tile_start, int32_t *n_tiles,
                               cudaStream_t st) {
    build_tiles_kernel<<<1, 1024, 0, st>>>(offsets, E, BM, tile_e, tile_m0, tile_start, n_tiles);
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
