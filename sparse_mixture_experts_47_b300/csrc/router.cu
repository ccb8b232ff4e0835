// Router of the token-choice MoE layer: linear (x W_r^T + logit_bias),
// softmax over experts, top-k of (score + selection bias), renormalisation.
//
// Sources: "Mixture of Experts" (waylandz.com LLM book, ch. 30) §30.2.3,
// steps 1-4; "混合エキスパートモデル（MoE）実践" (deepseekmodel.com):
// TopKRouter (renormalise after top-k, no router bias) and BiasBalancedRouter
// (bias added to the probabilities for selection only, weights from the
// unbiased probabilities); "Mixture of Experts (MoE) memo" (iwashi.co),
// "Kimi K3 → Quantile Balancing" (bias read off each expert's score
// distribution so that the target share of tokens lands in the top-k).
//
// The logits are fp32 FFMA on CUDA cores (x widened from bf16/fp32, W_r fp32);
// softmax with max subtraction and expf; exactly equal selection scores go to
// the lower expert index.  Every reduction has a fixed order, so results are
// bitwise reproducible.
#include "common.cuh"
#include "kernels.h"

#include <math_constants.h>

#include <algorithm>

namespace moe {

// --------------------------------------------------------------------------
// Small E (<= 32): one warp holds TPW = 32/EP tokens x EP (padded) experts.
// Lanes split d into 16-byte vectors, accumulate all TPW*EP = 32 partial
// logits, and a reduce-scatter butterfly leaves lane L with the full logit
// of (token L / EP, expert L % EP).  W_r is staged through shared memory in
// 32 KB chunks of d.
// --------------------------------------------------------------------------
template <typename TX, int EP>
__global__ void __launch_bounds__(256) router_small_kernel(RouterArgs a) {
    constexpr int VN = Vec<TX>::N;
    constexpr int TPW = 32 / EP;
    constexpr int R = 32 / EP;            // vectors per lane per chunk
    constexpr int DC = 32 * VN * R;       // chunk of d held in shared memory
    extern __shared__ __align__(16) float smem[];
    float *wsm = smem;                    // [EP][DC]
    float *part = smem + EP * DC;         // [8 warps][32 lanes]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tok0 = (blockIdx.x * 8 + warp) * TPW;
    const TX *x = static_cast<const TX *>(a.x);

    float acc[TPW][EP];
#pragma unroll
    for (int t = 0; t < TPW; ++t)
#pragma unroll
        for (int e = 0; e < EP; ++e) acc[t][e] = 0.f;

    for (int c0 = 0; c0 < a.d; c0 += DC) {
        const int clen = min(DC, a.d - c0);
        __syncthreads();
        for (int i = threadIdx.x * 4; i < EP * DC; i += 256 * 4) {
            const int e = i / DC, c = i % DC;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < a.E && c < clen)
                v = *reinterpret_cast<const float4 *>(a.w_r + (size_t)e * a.d + c0 + c);
            *reinterpret_cast<float4 *>(wsm + i) = v;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int c = (r * 32 + lane) * VN;
            if (c < clen) {
                float xv[TPW][VN];
#pragma unroll
                for (int t = 0; t < TPW; ++t) {
                    if (tok0 + t < a.T) {
                        load16_f32(x + (size_t)(tok0 + t) * a.d + c0 + c, xv[t]);
                    } else {
#pragma unroll
                        for (int i = 0; i < VN; ++i) xv[t][i] = 0.f;
                    }
                }
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    if (e < a.E) {
                        float wv[VN];
#pragma unroll
                        for (int i = 0; i < VN; i += 4) {
                            float4 q = *reinterpret_cast<const float4 *>(wsm + e * DC + c + i);
                            wv[i] = q.x; wv[i + 1] = q.y; wv[i + 2] = q.z; wv[i + 3] = q.w;
                        }
#pragma unroll
                        for (int t = 0; t < TPW; ++t)
#pragma unroll
                            for (int i = 0; i < VN; ++i) acc[t][e] = fmaf(xv[t][i], wv[i], acc[t][e]);
                    }
                }
            }
        }
    }

    // Reduce-scatter: afterwards v[0] of lane L holds the sum over lanes of
    // the flattened accumulator entry L.
    float v[32];
#pragma unroll
    for (int t = 0; t < TPW; ++t)
#pragma unroll
        for (int e = 0; e < EP; ++e) v[t * EP + e] = acc[t][e];
#pragma unroll
    for (int off = 16, n = 32; off >= 1; off >>= 1, n >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }

    const int ge = lane % EP;               // expert of this lane
    const int t = tok0 + lane / EP;          // token of this lane
    const bool ve = ge < a.E, vt = t < a.T;
    float logit = v[0];
    if (ve && a.logit_bias) logit += a.logit_bias[ge];
    if (!ve) logit = -CUDART_INF_F;

    float m = logit;
#pragma unroll
    for (int off = EP / 2; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float ex = ve ? expf(logit - m) : 0.f;
    float s = ex;
#pragma unroll
    for (int off = EP / 2; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    const float prob = ex / s;

    if (vt && ve) {
        if (a.probs) a.probs[(size_t)t * a.E + ge] = prob;
        if (a.probsT) a.probsT[(size_t)ge * a.T + t] = prob;
    }

    if (a.do_select) {
        float sel = -CUDART_INF_F;
        if (ve) sel = (a.select_space == MOE_SELECT_PROBS ? prob : logit) +
                      (a.select_bias ? a.select_bias[ge] : 0.f);
        float psum = 0.f, my_p = 0.f;
        int my_e = 0;
        for (int j = 0; j < a.k; ++j) {
            float bv = sel;
            int bi = ge;
#pragma unroll
            for (int off = EP / 2; off >= 1; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            const float pw = __shfl_sync(0xffffffffu, prob, (lane & ~(EP - 1)) + bi);
            psum += pw;
            if (ge == j) { my_e = bi; my_p = pw; }
            if (ge == bi) sel = -CUDART_INF_F;
        }
        if (vt && ge < a.k) {
            a.idx[(size_t)t * a.k + ge] = my_e;
            a.w[(size_t)t * a.k + ge] = my_p / psum;
        }
    }

    // Per-block partial sums of the probabilities, fixed order.
    part[warp * 32 + lane] = (vt && ve) ? prob : 0.f;
    __syncthreads();
    if (a.p_partial && threadIdx.x < a.E) {
        const int e = threadIdx.x;
        float sum = 0.f;
        for (int w = 0; w < 8; ++w)
            for (int g = 0; g < TPW; ++g) sum += part[w * 32 + g * EP + e];
        a.p_partial[(size_t)blockIdx.x * a.E + e] = sum;
    }
}

// --------------------------------------------------------------------------
// Any E: a CTA computes the [32 tokens x E] logit tile as a SIMT fp32 GEMM
// (4 tokens x 4 experts per thread, d in steps of 32 through shared memory),
// keeps it in shared memory, then each warp runs softmax and top-k for 4
// tokens with lanes striding over the experts.
// --------------------------------------------------------------------------
constexpr int kTB = 32, kEC = 128, kDK = 32;

__host__ __device__ inline size_t router_tiled_smem(int E) {
    return sizeof(float) * ((size_t)kTB * E + kDK * kTB + kDK * (kEC + 4) + 2 * kTB);
}

__device__ __forceinline__ void load4_f32(const float *p, float *v) {
    float4 a = *reinterpret_cast<const float4 *>(p);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void load4_f32(const __nv_bfloat16 *p, float *v) {
    uint2 a = *reinterpret_cast<const uint2 *>(p);
    v[0] = __uint_as_float(a.x << 16); v[1] = __uint_as_float(a.x & 0xffff0000u);
    v[2] = __uint_as_float(a.y << 16); v[3] = __uint_as_float(a.y & 0xffff0000u);
}

// Softmax, load-statistics partial sums, optional probs/probsT and top-k with
// renormalisation for a tile of kTB tokens whose logits (logit offset included)
// are in shared memory lg[kTB][E].  256 threads; warp w owns tokens 4w..4w+3.
__device__ void router_rows_epilogue(const RouterArgs &a, float *lg, float *st_m, float *st_s,
                                     int t0) {
    const int E = a.E;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Softmax statistics per token (warp per 4 tokens), optional probs rows.
    for (int r = 0; r < 4; ++r) {
        const int tt = 4 * warp + r, t = t0 + tt;
        const float *row = lg + tt * E;
        float m = -CUDART_INF_F;
        for (int e = lane; e < E; e += 32) m = fmaxf(m, row[e]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        float s = 0.f;
        for (int e = lane; e < E; e += 32) s += expf(row[e] - m);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) { st_m[tt] = m; st_s[tt] = s; }
        if (t < a.T && a.probs)
            for (int e = lane; e < E; e += 32) a.probs[(size_t)t * E + e] = expf(row[e] - m) / s;
    }
    __syncthreads();

    // Column pass: per-block partial sums of probs (fixed token order) and
    // the expert-major copy used by quantile balancing.
    for (int e = tid; e < E; e += 256) {
        float sum = 0.f;
        for (int tt = 0; tt < kTB && t0 + tt < a.T; ++tt) {
            const float p = expf(lg[tt * E + e] - st_m[tt]) / st_s[tt];
            sum += p;
            if (a.probsT) a.probsT[(size_t)e * a.T + t0 + tt] = p;
        }
        if (a.p_partial) a.p_partial[(size_t)blockIdx.x * E + e] = sum;
    }
    if (!a.do_select) return;
    __syncthreads();

    // Top-k per token; a taken expert's logit is overwritten with -inf.
    for (int r = 0; r < 4; ++r) {
        const int tt = 4 * warp + r, t = t0 + tt;
        if (t >= a.T) break;
        float *row = lg + tt * E;
        const float m = st_m[tt], s = st_s[tt];
        float psum = 0.f, my_p = 0.f;
        int my_e = 0;
        for (int j = 0; j < a.k; ++j) {
            float bv = -CUDART_INF_F;
            int bi = 0x7fffffff;
            for (int e = lane; e < E; e += 32) {
                const float l = row[e];
                if (l == -CUDART_INF_F) continue;
                const float sc = (a.select_space == MOE_SELECT_PROBS ? expf(l - m) / s : l) +
                                 (a.select_bias ? a.select_bias[e] : 0.f);
                if (sc > bv) { bv = sc; bi = e; }
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            const float pw = expf(row[bi] - m) / s;
            psum += pw;
            if (lane == j) { my_e = bi; my_p = pw; }
            __syncwarp();
            if (lane == 0) row[bi] = -CUDART_INF_F;
            __syncwarp();
        }
        if (lane < a.k) {
            a.idx[(size_t)t * a.k + lane] = my_e;
            a.w[(size_t)t * a.k + lane] = my_p / psum;
        }
    }
}

template <typename TX>
__global__ void __launch_bounds__(256) router_tiled_kernel(RouterArgs a) {
    extern __shared__ __align__(16) float smem[];
    const int E = a.E, d = a.d;
    float *lg = smem;                         // [kTB][E]
    float *xs = lg + kTB * E;                 // [kDK][kTB]
    float *wsh = xs + kDK * kTB;              // [kDK][kEC + 4]
    float *st_m = wsh + kDK * (kEC + 4);      // [kTB]
    float *st_s = st_m + kTB;                 // [kTB]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * kTB;
    const TX *x = static_cast<const TX *>(a.x);

    for (int e0 = 0; e0 < E; e0 += kEC) {
        float acc[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[r][i] = 0.f;
        for (int k0 = 0; k0 < d; k0 += kDK) {
            __syncthreads();
            {
                const int tt = tid >> 3, kk = (tid & 7) * 4, t = t0 + tt;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (t < a.T && k0 + kk < d) load4_f32(x + (size_t)t * d + k0 + kk, v);
#pragma unroll
                for (int i = 0; i < 4; ++i) xs[(kk + i) * kTB + tt] = v[i];
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int id = tid + q * 256, ee = id >> 3, kk = (id & 7) * 4, e = e0 + ee;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (e < E && k0 + kk < d) load4_f32(a.w_r + (size_t)e * d + k0 + kk, v);
#pragma unroll
                for (int i = 0; i < 4; ++i) wsh[(kk + i) * (kEC + 4) + ee] = v[i];
            }
            __syncthreads();
#pragma unroll 8
            for (int kk = 0; kk < kDK; ++kk) {
                const float4 xv = *reinterpret_cast<const float4 *>(xs + kk * kTB + 4 * warp);
                const float xr[4] = {xv.x, xv.y, xv.z, xv.w};
                float wv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) wv[i] = wsh[kk * (kEC + 4) + lane + 32 * i];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[r][i] = fmaf(xr[r], wv[i], acc[r][i]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = e0 + lane + 32 * i;
            if (e < E) {
                const float lb = a.logit_bias ? a.logit_bias[e] : 0.f;
#pragma unroll
                for (int r = 0; r < 4; ++r) lg[(4 * warp + r) * E + e] = acc[r][i] + lb;
            }
        }
    }
    __syncthreads();
    router_rows_epilogue(a, lg, st_m, st_s, t0);
}

// --------------------------------------------------------------------------
// Tensor-core router support.  W_r (fp32) is split exactly into three bf16
// parts, w = hi + mid + lo (8 + 8 + 8 significant bits, residual at most
// 2^-24 |w|), laid out as one [E, 3*dp] bf16 matrix (dp = d rounded up to 64,
// zero padded), so that x W_r^T = x [hi|mid|lo]^T over a 3*dp reduction with
// x's column taken mod dp.  bf16 x bf16 products are exact in fp32.
// --------------------------------------------------------------------------
__global__ void split_router_weight_kernel(const float *w_r, int E, int d, int dp,
                                           __nv_bfloat16 *out) {
    const long long n = (long long)E * dp;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int e = (int)(i / dp), c = (int)(i % dp);
        const float w = c < d ? w_r[(size_t)e * d + c] : 0.f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
        __nv_bfloat16 *row = out + (size_t)e * 3 * dp;
        row[c] = hi;
        row[dp + c] = mid;
        row[2 * dp + c] = lo;
    }
}

// Logits = sum of S partial products (fixed order) + logit offset, then the
// same per-token epilogue as the SIMT router.
__global__ void __launch_bounds__(256) router_from_logits_kernel(RouterArgs a,
                                                                 const float *part, int S) {
    extern __shared__ __align__(16) float smem[];
    const int E = a.E;
    float *lg = smem;
    float *st_m = lg + kTB * E;
    float *st_s = st_m + kTB;
    const int t0 = blockIdx.x * kTB;
    const size_t plane = (size_t)a.T * E;
    for (int i = threadIdx.x; i < kTB * E; i += blockDim.x) {
        const int tt = i / E, e = i - tt * E, t = t0 + tt;
        float v = 0.f;
        if (t < a.T) {
            const size_t o = (size_t)t * E + e;
            for (int sp = 0; sp < S; ++sp) v += part[sp * plane + o];
            if (a.logit_bias) v += a.logit_bias[e];
        }
        lg[i] = v;
    }
    __syncthreads();
    router_rows_epilogue(a, lg, st_m, st_s, t0);
}

// --------------------------------------------------------------------------
// Top-k from stored expert-major probabilities probsT [E, T] with a bias
// (second pass of quantile balancing).  32 tokens per CTA, the [E x 32]
// tile transposed through shared memory.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(256) select_from_probsT_kernel(
        const float *probsT, const float *bias, int T, int E, int k,
        int32_t *idx, float *w) {
    extern __shared__ __align__(16) float tile[];   // [E][33]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * 32;
    for (int i = tid; i < E * 32; i += 256) {
        const int e = i >> 5, tt = i & 31, t = t0 + tt;
        tile[e * 33 + tt] = t < T ? probsT[(size_t)e * T + t] : 0.f;
    }
    __syncthreads();
    for (int r = 0; r < 4; ++r) {
        const int tt = 4 * warp + r, t = t0 + tt;
        if (t >= T) break;
        float psum = 0.f, my_p = 0.f;
        int my_e = 0;
        for (int j = 0; j < k; ++j) {
            float bv = -CUDART_INF_F;
            int bi = 0x7fffffff;
            for (int e = lane; e < E; e += 32) {
                const float p = tile[e * 33 + tt];
                if (p < 0.f) continue;                        // taken
                const float sc = p + (bias ? bias[e] : 0.f);
                if (sc > bv) { bv = sc; bi = e; }
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            const float pw = tile[bi * 33 + tt];
            psum += pw;
            if (lane == j) { my_e = bi; my_p = pw; }
            __syncwarp();
            if (lane == 0) tile[bi * 33 + tt] = -1.f;
            __syncwarp();
        }
        if (lane < k) {
            if (idx) idx[(size_t)t * k + lane] = my_e;
            if (w) w[(size_t)t * k + lane] = my_p / psum;
        }
    }
}

// --------------------------------------------------------------------------
// Quantile bias: b_e = -(v_lo + frac (v_hi - v_lo)) with v_lo, v_hi the
// order statistics of rank lo and lo+1 of column e (linear interpolation,
// h = (T-1) q, lo = floor h, frac = h - lo).  One CTA per expert; exact
// order statistics by a 4-pass radix select on the fp32 bit patterns
// (probabilities are >= 0, so bit order equals value order).
// --------------------------------------------------------------------------
__device__ float radix_select_col(const float *col, int T, long long r, unsigned *hist,
                                  unsigned *sh) {
    unsigned prefix = 0, mask = 0;
    const int tid = threadIdx.x, lane = tid & 31;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        const int n = (T + blockDim.x - 1) / blockDim.x * blockDim.x;
        for (int i = tid; i < n; i += blockDim.x) {
            unsigned bin = 256;
            if (i < T) {
                const unsigned b = __float_as_uint(col[i]);
                if ((b & mask) == prefix) bin = (b >> shift) & 255u;
            }
            const unsigned peers = __match_any_sync(0xffffffffu, bin);
            if (bin < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
        }
        __syncthreads();
        if (tid == 0) {
            unsigned long long cum = 0;
            unsigned bin = 0;
            for (; bin < 255; ++bin) {
                if (cum + hist[bin] > (unsigned long long)r) break;
                cum += hist[bin];
            }
            sh[0] = bin;
            sh[1] = (unsigned)(r - (long long)cum);
        }
        __syncthreads();
        prefix |= sh[0] << shift;
        mask |= 255u << shift;
        r = sh[1];
        __syncthreads();
    }
    return __uint_as_float(prefix);
}

__global__ void __launch_bounds__(512) quantile_bias_kernel(const float *probsT, int T,
                                                            long long lo, float frac,
                                                            float *bias_out) {
    __shared__ unsigned hist[256];
    __shared__ unsigned sh[2];
    const float *col = probsT + (size_t)blockIdx.x * T;
    const float v_lo = radix_select_col(col, T, lo, hist, sh);
    const float v_hi = (lo + 1 < T) ? radix_select_col(col, T, lo + 1, hist, sh) : v_lo;
    if (threadIdx.x == 0) bias_out[blockIdx.x] = -(v_lo + frac * (v_hi - v_lo));
}

// --------------------------------------------------------------------------
// Host launchers
// --------------------------------------------------------------------------
template <typename TX, int EP>
static cudaError_t launch_small(const RouterArgs &a, cudaStream_t st) {
    constexpr int TPW = 32 / EP, R = 32 / EP, DC = 32 * Vec<TX>::N * R;
    const size_t smem = sizeof(float) * (EP * DC + 256);
    auto kern = router_small_kernel<TX, EP>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int tok_per_cta = 8 * TPW;
    const int grid = (a.T + tok_per_cta - 1) / tok_per_cta;
    kern<<<grid, 256, smem, st>>>(a);
    note_launch();
    return cudaGetLastError();
}

int router_blocks(int T, int E) {
    if (E <= 8) return (T + 31) / 32;
    if (E <= 16) return (T + 15) / 16;
    if (E <= 32) return (T + 7) / 8;
    return (T + kTB - 1) / kTB;
}

size_t router_smem_bytes(int E, int dtype) {
    if (E <= 32) return 0;
    (void)dtype;
    return router_tiled_smem(E);
}

template <typename TX>
static cudaError_t launch_router_t(const RouterArgs &a, cudaStream_t st) {
    if (a.E <= 8) return launch_small<TX, 8>(a, st);
    if (a.E <= 16) return launch_small<TX, 16>(a, st);
    if (a.E <= 32) return launch_small<TX, 32>(a, st);
    const size_t smem = router_tiled_smem(a.E);
    auto kern = router_tiled_kernel<TX>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<(a.T + kTB - 1) / kTB, 256, smem, st>>>(a);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_router(const RouterArgs &a, int dtype, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    return dtype == MOE_DTYPE_FP32 ? launch_router_t<float>(a, st)
                                   : launch_router_t<__nv_bfloat16>(a, st);
}

cudaError_t launch_split_router_weight(const float *w_r, int E, int d, int dp,
                                       __nv_bfloat16 *out, cudaStream_t st) {
    const long long n = (long long)E * dp;
    const int grid = (int)std::min<long long>((n + 255) / 256, 148 * 8);
    split_router_weight_kernel<<<grid, 256, 0, st>>>(w_r, E, d, dp, out);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_router_from_logits(const RouterArgs &a, const float *part, int S,
                                      cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * ((size_t)kTB * a.E + 2 * kTB);
    cudaError_t err = cudaFuncSetAttribute(router_from_logits_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    router_from_logits_kernel<<<(a.T + kTB - 1) / kTB, 256, smem, st>>>(a, part, S);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_select_from_probsT(const float *probsT, const float *bias, int T, int E,
                                      int k, int32_t *idx, float *w, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * (size_t)E * 33;
    cudaError_t err = cudaFuncSetAttribute(select_from_probsT_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    select_from_probsT_kernel<<<(T + 31) / 32, 256, smem, st>>>(probsT, bias, T, E, k, idx, w);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_quantile_bias(const float *probsT, int T, int E, long long lo, float frac,
                                 float *bias_out, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    quantile_bias_kernel<<<E, 512, 0, st>>>(probsT, T, lo, frac, bias_out);
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
