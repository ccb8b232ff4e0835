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
// Up to 32 experts (and for fp32 layers) the logits are fp32 FFMA on CUDA
// cores (x widened from bf16/fp32, W_r fp32); above that a bf16 layer takes
// them from the grouped tensor-core GEMM over a two-part bf16 split of W_r
// (split_router_weight_kernel here, the GEMM in gemm_tcgen05.cu), and the
// softmax kernel adds its planes.  Softmax with max subtraction and expf;
// exactly equal selection scores go to the lower expert index.  Every
// reduction has a fixed order, so results are bitwise reproducible.  With
// quantile balancing the bias comes from order statistics of each expert's
// column (quantile_tail_kernel / quantile_bias_kernel) and a second pass
// selects (select_rows_kernel).
#include "common.cuh"
#include "kernels.h"

#include <math_constants.h>

#include <algorithm>

namespace moe {

// --------------------------------------------------------------------------
// Small E (<= 32): partial logits of one slice of d (kRouterSlice columns)
// for a tile of tokens; the softmax kernel adds the slices in order.  A warp
// holds TPW = 32/EP tokens x EP (padded) experts; lanes split the slice into
// 16-byte vectors, accumulate all TPW*EP = 32 partial logits, and a
// reduce-scatter butterfly leaves lane L with the slice's logit of
// (token L / EP, expert L % EP).  The W_r slice is staged in shared memory
// once per CTA; the CTAs of a slice then stride over the token groups, so
// W_r is read from L2 about three times per SM instead of once per 8 x TPW
// tokens.  Each token's arithmetic is the same whatever the batch size and
// grid, so a token's routing does not depend on the batch it comes in.
// --------------------------------------------------------------------------
// The values of 16 bytes of x, widened to fp32.
template <typename TX> __device__ __forceinline__ void widen16(const uint4 &u, float *v);
template <> __device__ __forceinline__ void widen16<float>(const uint4 &u, float *v) {
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
}
template <> __device__ __forceinline__ void widen16<__nv_bfloat16>(const uint4 &u, float *v) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <typename TX, int EP>
__global__ void __launch_bounds__(256) router_partial_kernel(RouterArgs a, float *part) {
    constexpr int VN = Vec<TX>::N;
    constexpr int TPW = 32 / EP;
    constexpr int DS = kRouterSlice;
    extern __shared__ __align__(16) float wsm[];   // [EP][DS]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = blockIdx.y * DS, clen = min(DS, a.d - c0);
    const TX *x = static_cast<const TX *>(a.x);

    for (int i = threadIdx.x * 4; i < EP * DS; i += 256 * 4) {
        const int e = i / DS, c = i % DS;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < a.E && c < clen)
            v = *reinterpret_cast<const float4 *>(a.w_r + (size_t)e * a.d + c0 + c);
        *reinterpret_cast<float4 *>(wsm + i) = v;
    }
    __syncthreads();

    // A token group's x (TPW tokens x this lane's NJ 16-byte vectors) is
    // loaded raw, and the next group's is in flight while this one is used.
    constexpr int NJ = DS / (32 * VN);
    const int tok_step = gridDim.x * 8 * TPW;
    auto load_group = [&](int tk, uint4 (&r)[NJ][TPW]) {
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
            for (int t = 0; t < TPW; ++t) {
                const int c = (j * 32 + lane) * VN;
                r[j][t] = (c < clen && tk + t < a.T)
                              ? *reinterpret_cast<const uint4 *>(x + (size_t)(tk + t) * a.d + c0 + c)
                              : make_uint4(0u, 0u, 0u, 0u);
            }
    };
    uint4 cur[NJ][TPW], nxt[NJ][TPW];
    int tok0 = (blockIdx.x * 8 + warp) * TPW;
    if (tok0 < a.T) load_group(tok0, cur);
#pragma unroll 1
    for (; tok0 < a.T; tok0 += tok_step) {
        if (tok0 + tok_step < a.T) load_group(tok0 + tok_step, nxt);
        float acc[TPW][EP];
#pragma unroll
        for (int t = 0; t < TPW; ++t)
#pragma unroll
            for (int e = 0; e < EP; ++e) acc[t][e] = 0.f;

#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int c = (j * 32 + lane) * VN;
            if (c < clen) {
                float xv[TPW][VN];
#pragma unroll
                for (int t = 0; t < TPW; ++t) widen16<TX>(cur[j][t], xv[t]);
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    if (e < a.E) {
                        float wv[VN];
#pragma unroll
                        for (int i = 0; i < VN; i += 4) {
                            const float4 q = *reinterpret_cast<const float4 *>(wsm + e * DS + c + i);
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
        const int ge = lane % EP;
        const int t = tok0 + lane / EP;
        if (ge < a.E && t < a.T)
            part[(size_t)blockIdx.y * a.T * a.E + (size_t)t * a.E + ge] = v[0];
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
            for (int t = 0; t < TPW; ++t) cur[j][t] = nxt[j][t];
    }
}

// --------------------------------------------------------------------------
// E <= 8: the same partial logits with each lane's W_r columns in registers.
// A slice is 32 lanes x VN columns (one 16-byte vector of x per token and
// lane); lane l holds W_r[e][c .. c+VN) for all 8 (padded) experts, so the
// FMAs read no shared memory (staging W_r in shared memory and reading it
// back for every 4 tokens made the kernel bound by shared-memory bandwidth).
// A warp takes TPW = 4 tokens at a time, the next 4 tokens' x in flight;
// per (token, expert) the lane's VN products are summed in column order, the
// same reduce-scatter butterfly leaves lane L with (token L / 8, expert
// L % 8), and the softmax kernel adds the slices in order: fixed by d alone.
// --------------------------------------------------------------------------
template <typename TX>
__global__ void __launch_bounds__(256, 2) router_partial_w8_kernel(RouterArgs a, float *part) {
    constexpr int VN = Vec<TX>::N;
    constexpr int EP = 8, TPW = 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = (blockIdx.y * 32 + lane) * VN;     // this lane's first column
    const bool cv = c < a.d;                         // d is a multiple of VN
    const TX *x = static_cast<const TX *>(a.x);

    float wr[EP][VN];
#pragma unroll
    for (int e = 0; e < EP; ++e)
#pragma unroll
        for (int i = 0; i < VN; i += 4) {
            float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < a.E && cv)
                q = *reinterpret_cast<const float4 *>(a.w_r + (size_t)e * a.d + c + i);
            wr[e][i] = q.x; wr[e][i + 1] = q.y; wr[e][i + 2] = q.z; wr[e][i + 3] = q.w;
        }

    const int tok_step = gridDim.x * 8 * TPW;
    auto load_group = [&](int tk, uint4 (&r)[TPW]) {
#pragma unroll
        for (int t = 0; t < TPW; ++t)
            r[t] = (cv && tk + t < a.T)
                       ? *reinterpret_cast<const uint4 *>(x + (size_t)(tk + t) * a.d + c)
                       : make_uint4(0u, 0u, 0u, 0u);
    };
    uint4 cur[TPW], nxt[TPW];
    int tok0 = (blockIdx.x * 8 + warp) * TPW;
    if (tok0 < a.T) load_group(tok0, cur);
#pragma unroll 1
    for (; tok0 < a.T; tok0 += tok_step) {
        if (tok0 + tok_step < a.T) load_group(tok0 + tok_step, nxt);
        float v[32];
#pragma unroll
        for (int t = 0; t < TPW; ++t) {
            float xv[VN];
            widen16<TX>(cur[t], xv);
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < VN; ++i) s = fmaf(xv[i], wr[e][i], s);
                v[t * EP + e] = s;
            }
        }
        // Reduce-scatter: afterwards v[0] of lane L holds the sum over lanes
        // of the flattened entry L.
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
        const int ge = lane % EP;
        const int t = tok0 + lane / EP;
        if (ge < a.E && t < a.T)
            part[(size_t)blockIdx.y * a.T * a.E + (size_t)t * a.E + ge] = v[0];
#pragma unroll
        for (int t2 = 0; t2 < TPW; ++t2) cur[t2] = nxt[t2];
    }
}

// --------------------------------------------------------------------------
// Small E (<= 32), second step: softmax, top-k and renormalisation with one
// lane per (token, expert): a warp holds TPW = 32/EP tokens, the slice sums
// are added in slice order (+ logit offset), the softmax and the top-k run
// as butterflies over the EP lanes of a token.  Also the per-block partial
// sums of the probabilities and of the gate entropy, and the candidates
// ranked after the top k (for redirected overflow).
// --------------------------------------------------------------------------
template <int EP>
__global__ void __launch_bounds__(256) router_small_epilogue_kernel(RouterArgs a,
                                                                    const float *part,
                                                                    int S) {
    constexpr int TPW = 32 / EP;
    __shared__ float red[256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ge = lane % EP;                               // expert of this lane
    const int t = (blockIdx.x * 8 + warp) * TPW + lane / EP; // token of this lane
    const bool ve = ge < a.E, vt = t < a.T;
    float logit = -CUDART_INF_F;
    if (ve && vt) {
        const size_t plane = (size_t)a.T * a.E, o = (size_t)t * a.E + ge;
        float v = 0.f;
        for (int sp = 0; sp < S; ++sp) v += part[sp * plane + o];
        if (a.logit_bias) v += a.logit_bias[ge];
        logit = v;
    } else if (ve) {
        logit = 0.f;                                        // padding token, not stored
    }
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
        for (int j = 0; j < a.k + a.n_cand; ++j) {
            float bv = sel;
            int bi = ge;
#pragma unroll
            for (int off = EP / 2; off >= 1; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            const float pw = __shfl_sync(0xffffffffu, prob, (lane & ~(EP - 1)) + bi);
            if (j < a.k) psum += pw;
            if (ge == j) { my_e = bi; my_p = pw; }
            if (ge == bi) sel = -CUDART_INF_F;
        }
        if (vt && ge < a.k) {
            a.idx[(size_t)t * a.k + ge] = my_e;
            a.w[(size_t)t * a.k + ge] = my_p / psum;
        } else if (vt && ge < a.k + a.n_cand) {
            a.cand_idx[(size_t)t * a.n_cand + ge - a.k] = my_e;
            a.cand_w[(size_t)t * a.n_cand + ge - a.k] = my_p / psum;
        }
    }

    // Per-block partial sums of the probabilities, fixed order.
    red[threadIdx.x] = (vt && ve) ? prob : 0.f;
    __syncthreads();
    if (a.p_partial && threadIdx.x < a.E) {
        const int e = threadIdx.x;
        float sum = 0.f;
        for (int w = 0; w < 8; ++w)
            for (int g = 0; g < TPW; ++g) sum += red[w * 32 + g * EP + e];
        a.p_partial[(size_t)blockIdx.x * a.E + e] = sum;
        // a batch of one block: the mean probability directly, as
        // p_finalize_kernel computes it from one partial row
        if (a.p_direct) a.p_direct[e] = (float)((double)sum / (double)a.T);
    }
    // Per-block sum of the tokens' gate entropies -sum_e p ln p, with
    // ln p = (logit - max) - ln(sum): fixed butterfly, then warps in order.
    if (a.ent_partial) {
        __syncthreads();
        float h = (vt && ve) ? -prob * ((logit - m) - logf(s)) : 0.f;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) h += __shfl_xor_sync(0xffffffffu, h, off);
        if (lane == 0) red[warp] = h;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.f;
            for (int w = 0; w < 8; ++w) tot += red[w];
            a.ent_partial[blockIdx.x] = tot;
        }
    }
}

// --------------------------------------------------------------------------
// Any E: a CTA computes the [32 tokens x E] logit tile as a SIMT fp32 GEMM
// (4 tokens x 4 experts per thread, d in steps of 32 through shared memory),
// keeps it in shared memory, then each warp runs softmax and top-k for 4
// tokens with lanes striding over the experts.
// --------------------------------------------------------------------------
constexpr int kTB = 32, kEC = 128, kDK = 32;

// Row stride (floats) of a logit tile in shared memory: E made odd, so that
// reading one expert's column of the tile touches distinct banks.
__host__ __device__ inline int router_lde(int E) { return E | 1; }

__host__ __device__ inline size_t router_tiled_smem(int E) {
    return sizeof(float) *
           ((size_t)kTB * router_lde(E) + kDK * kTB + kDK * (kEC + 4) + 3 * kTB);
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

// Top-k selection over a warp: lane L holds the scores of experts L + 32 i in
// sc[i] (-inf where absent).  next() returns the experts in order of score,
// exactly equal scores going to the lower expert index.  Each lane keeps its
// best two (score, expert) keys, found by one scan in expert order with
// strict comparisons (a later expert displaces an earlier one only with a
// larger score, which is the order's tie rule); a pick is the argmax of the
// lanes' first keys over the warp (5 shuffle steps), and the lane whose key
// was taken moves its second key up.  A lane that has given up both rescans
// its scores for the best two keys after the last one taken (one lane
// providing three or more of a token's picks: a few per cent of tokens).
// Rescanning all scores for each of the 8 picks of the 896-expert layer kept
// the ALU pipe 88 % busy.
constexpr int kTopkPerLane = 32;   // E <= 1024
// Score slots per lane for E experts: 8, 16 or 32.
inline int topk_per_lane(int E) { return E <= 256 ? 8 : E <= 512 ? 16 : 32; }
__device__ __forceinline__ bool key_before(float va, int ea, float vb, int eb) {
    return va > vb || (va == vb && ea < eb);
}
template <int PER>
struct WarpTopK {
    float v0, v1;
    int e0, e1;
    int left;   // keys of the pair not taken yet
    // the lane's best two keys (after (lv, le) unless FIRST)
    template <bool FIRST>
    __device__ __forceinline__ void scan(const float (&sc)[PER], int lane, float lv,
                                         int le) {
        v0 = v1 = -CUDART_INF_F;
        e0 = e1 = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const float x = sc[i];
            const int ex = lane + 32 * i;
            if (!FIRST && !key_before(lv, le, x, ex)) continue;
            if (x > v0) {
                v1 = v0; e1 = e0;
                v0 = x; e0 = ex;
            } else if (x > v1) {
                v1 = x; e1 = ex;
            }
        }
        left = 2;
    }
    __device__ __forceinline__ void init(const float (&sc)[PER], int lane) {
        scan<true>(sc, lane, 0.f, 0);
    }
    __device__ __forceinline__ int next(const float (&sc)[PER], int lane) {
        float bv = v0;
        int be = e0;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (key_before(ov, oe, bv, be)) {
                bv = ov;
                be = oe;
            }
        }
        if (be == e0) {   // this lane's first key was taken
            if (--left == 0) {
                scan<false>(sc, lane, bv, be);
            } else {
                v0 = v1; e0 = e1;
                v1 = -CUDART_INF_F; e1 = 0x7fffffff;
            }
        }
        return be;
    }
};

// Softmax, load-statistics partial sums, optional probs/probsT, optional
// gate-entropy partial sum and top-k with renormalisation for a tile of TB
// tokens whose logits (logit offset included) are in shared memory
// lg[TB][router_lde(E)].  256 threads; warp w owns tokens (TB/8) w ..
// (TB/8)(w+1) - 1.  st_m, st_s, st_h hold TB floats each.  Without top-k
// (do_select = 0) the tile is turned into probabilities in place and the
// expert-major copy probsT is written from it in segments of TB tokens.
template <int TB, int SEL = 2, int PER = kTopkPerLane>
__device__ void router_rows_epilogue(const RouterArgs &a, float *lg, float *st_m, float *st_s,
                                     float *st_h, int t0) {
    // SEL: 0 no top-k (probabilities only), 1 top-k, 2 as a.do_select says
    const bool do_select = SEL == 2 ? (a.do_select != 0) : SEL == 1;
    constexpr int TPWR = TB / 8;
    const int E = a.E, lde = router_lde(E);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Softmax statistics per token (warp per 4 tokens), optional probs rows.
    for (int r = 0; r < TPWR; ++r) {
        const int tt = TPWR * warp + r, t = t0 + tt;
        float *row = lg + tt * lde;
        float m = -CUDART_INF_F;
        for (int e = lane; e < E; e += 32) m = fmaxf(m, row[e]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        float s = 0.f;
        for (int e = lane; e < E; e += 32) s += expf(row[e] - m);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        float hz = 0.f;      // sum_e exp(z) z, z = logit - max: entropy = ln s - hz / s
        if (a.ent_partial) {
            for (int e = lane; e < E; e += 32) {
                const float z = row[e] - m;
                hz += expf(z) * z;
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) hz += __shfl_xor_sync(0xffffffffu, hz, off);
        }
        if (lane == 0) {
            st_m[tt] = m;
            st_s[tt] = s;
            st_h[tt] = t < a.T ? logf(s) - hz / s : 0.f;
        }
        if (!do_select) {
            for (int e = lane; e < E; e += 32) {
                const float p = expf(row[e] - m) / s;
                row[e] = p;
                if (t < a.T && a.probs) a.probs[(size_t)t * E + e] = p;
            }
        } else if (t < a.T && a.probs) {
            for (int e = lane; e < E; e += 32) a.probs[(size_t)t * E + e] = expf(row[e] - m) / s;
        }
    }
    __syncthreads();

    // Column pass: per-block partial sums of probs (fixed token order) and
    // the expert-major copy used by quantile balancing and expert choice.
    const int nt = min(TB, a.T - t0);
    if (!do_select) {
        for (int e = tid; e < E; e += 256) {
            float sum = 0.f;
            for (int tt = 0; tt < nt; ++tt) sum += lg[tt * lde + e];
            if (a.p_partial) a.p_partial[(size_t)blockIdx.x * E + e] = sum;
        }
        if (a.probsT)
            for (int i = tid; i < TB * E; i += 256) {
                const int e = i / TB, tt = i - e * TB;
                if (tt < nt) a.probsT[(size_t)e * a.T + t0 + tt] = lg[tt * lde + e];
            }
    } else {
        for (int e = tid; e < E; e += 256) {
            float sum = 0.f;
            for (int tt = 0; tt < nt; ++tt) {
                const float p = expf(lg[tt * lde + e] - st_m[tt]) / st_s[tt];
                sum += p;
                if (a.probsT) a.probsT[(size_t)e * a.T + t0 + tt] = p;
            }
            if (a.p_partial) a.p_partial[(size_t)blockIdx.x * E + e] = sum;
        }
    }
    if (a.ent_partial && tid == 0) {
        float tot = 0.f;
        for (int tt = 0; tt < TB; ++tt) tot += st_h[tt];
        a.ent_partial[blockIdx.x] = tot;
    }
    if (!do_select) return;
    __syncthreads();

    // Top-k per token from the selection scores held in registers.
    for (int r = 0; r < TPWR; ++r) {
        const int tt = TPWR * warp + r, t = t0 + tt;
        if (t >= a.T) break;
        const float *row = lg + tt * lde;
        const float m = st_m[tt], s = st_s[tt];
        float sc[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e = lane + 32 * i;
            sc[i] = -CUDART_INF_F;
            if (e < E)
                sc[i] = (a.select_space == MOE_SELECT_PROBS ? expf(row[e] - m) / s : row[e]) +
                        (a.select_bias ? a.select_bias[e] : 0.f);
        }
        float psum = 0.f, my_p = 0.f;
        int my_e = 0;
        WarpTopK<PER> topk;
        topk.init(sc, lane);
        for (int j = 0; j < a.k + a.n_cand; ++j) {
            const int bi = topk.next(sc, lane);
            const float pw = expf(row[bi] - m) / s;
            if (j < a.k) psum += pw;
            if (lane == j) { my_e = bi; my_p = pw; }
        }
        if (lane < a.k) {
            a.idx[(size_t)t * a.k + lane] = my_e;
            a.w[(size_t)t * a.k + lane] = my_p / psum;
        } else if (lane < a.k + a.n_cand) {
            a.cand_idx[(size_t)t * a.n_cand + lane - a.k] = my_e;
            a.cand_w[(size_t)t * a.n_cand + lane - a.k] = my_p / psum;
        }
    }
}

template <typename TX>
__global__ void __launch_bounds__(256) router_tiled_kernel(RouterArgs a) {
    extern __shared__ __align__(16) float smem[];
    const int E = a.E, d = a.d, lde = router_lde(E);
    float *lg = smem;                         // [kTB][lde]
    float *xs = lg + kTB * lde;               // [kDK][kTB]
    float *wsh = xs + kDK * kTB;              // [kDK][kEC + 4]
    float *st_m = wsh + kDK * (kEC + 4);      // [kTB]
    float *st_s = st_m + kTB;                 // [kTB]
    float *st_h = st_s + kTB;                 // [kTB]

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
                for (int r = 0; r < 4; ++r) lg[(4 * warp + r) * lde + e] = acc[r][i] + lb;
            }
        }
    }
    __syncthreads();
    router_rows_epilogue<kTB>(a, lg, st_m, st_s, st_h, t0);
}

// --------------------------------------------------------------------------
// Tensor-core router support.  W_r (fp32) is split into `parts` bf16 parts,
// each the nearest bf16 of what the earlier parts leave (two parts: w = hi +
// lo + r with |r| <= 2^-18 |w|; three: |r| <= 2^-24 |w|), laid out as one
// [E, parts*dp] bf16 matrix (dp = d rounded up to 64, zero padded), so that
// x W_r^T = x [hi|lo|..]^T over a parts*dp reduction with x's column taken
// mod dp.  bf16 x bf16 products are exact in fp32.
// --------------------------------------------------------------------------
// A thread takes 8 consecutive columns (dp is a multiple of 64) and stores
// each part as one 16-byte vector.  Block 0 also writes the logit GEMM's tile
// table for its single group of T rows in 128-row tiles (offsets {0, T},
// tile_e = 0, tile_start {0, tiles}, n_tiles), the table the grouped GEMM
// reads.
constexpr int kRouterMaxParts = 3;
__global__ void split_router_weight_kernel(const float *w_r, int E, int d, int dp, int parts,
                                           __nv_bfloat16 *out, int T, int32_t *offsets,
                                           int32_t *tile_e, int32_t *tile_start,
                                           int32_t *n_tiles) {
    const long long n8 = (long long)E * (dp / 8);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8;
         i += (long long)gridDim.x * blockDim.x) {
        const int e = (int)(i / (dp / 8)), c0 = 8 * (int)(i % (dp / 8));
        const float *src = w_r + (size_t)e * d;
        float r[8];
        if (c0 + 8 <= d && (d & 3) == 0) {
            const float4 a = *reinterpret_cast<const float4 *>(src + c0);
            const float4 b = *reinterpret_cast<const float4 *>(src + c0 + 4);
            r[0] = a.x; r[1] = a.y; r[2] = a.z; r[3] = a.w;
            r[4] = b.x; r[5] = b.y; r[6] = b.z; r[7] = b.w;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) r[j] = c0 + j < d ? src[c0 + j] : 0.f;
        }
        __nv_bfloat16 *row = out + (size_t)e * parts * dp + c0;
        // each part is the round-to-nearest bf16 of what the earlier parts left
#pragma unroll
        for (int q = 0; q < kRouterMaxParts; ++q) {
            if (q >= parts) break;
            uint32_t packed[4];
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                const __nv_bfloat162 b = __floats2bfloat162_rn(r[j], r[j + 1]);
                r[j] -= __low2float(b);
                r[j + 1] -= __high2float(b);
                packed[j / 2] = *reinterpret_cast<const uint32_t *>(&b);
            }
            *reinterpret_cast<uint4 *>(row + (size_t)q * dp) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
    }
    if (blockIdx.x == 0) {
        const int tiles = (T + 127) / 128;
        for (int i = threadIdx.x; i < tiles; i += blockDim.x) tile_e[i] = 0;
        if (threadIdx.x == 0) {
            offsets[0] = 0;
            offsets[1] = T;
            tile_start[0] = 0;
            tile_start[1] = tiles;
            *n_tiles = tiles;
        }
    }
}

// Logits = sum of S partial products (fixed order) + logit offset, then the
// same per-token epilogue as the SIMT router.
template <int TB, int SEL, int PER>
__global__ void __launch_bounds__(256) router_from_logits_kernel(RouterArgs a,
                                                                 const float *part, int S) {
    extern __shared__ __align__(16) float smem[];
    const int E = a.E, lde = router_lde(E);
    float *lg = smem;
    float *st_m = lg + TB * lde;
    float *st_s = st_m + TB;
    float *st_h = st_s + TB;
    const int t0 = blockIdx.x * TB;
    const size_t plane = (size_t)a.T * E;
    // The tile's logits are TB * E consecutive floats of each plane: read
    // them as float4 (E % 4 == 0), four per thread in flight.
    const int n = min(TB, a.T - t0) * E;
    const float *src = part + (size_t)t0 * E;
    if ((E & 3) == 0) {
        constexpr int kV = 4;
        for (int j0 = threadIdx.x; j0 < TB * E / 4; j0 += kV * blockDim.x) {
            float4 v[kV];
#pragma unroll
            for (int q = 0; q < kV; ++q) {
                const int j = j0 + q * blockDim.x;
                v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (4 * j < n)
                    for (int sp = 0; sp < S; ++sp) {
                        const float4 u =
                            reinterpret_cast<const float4 *>(src + sp * plane)[j];
                        v[q].x += u.x; v[q].y += u.y; v[q].z += u.z; v[q].w += u.w;
                    }
            }
#pragma unroll
            for (int q = 0; q < kV; ++q) {
                const int j = j0 + q * blockDim.x;
                if (j >= TB * E / 4) break;
                const int i = 4 * j, tt = i / E, e = i - tt * E;
                const float w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    lg[tt * lde + e + c] =
                        w[c] + (a.logit_bias && i < n ? a.logit_bias[e + c] : 0.f);
            }
        }
    } else {
        for (int i = threadIdx.x; i < TB * E; i += blockDim.x) {
            const int tt = i / E, e = i - tt * E;
            float v = 0.f;
            if (i < n) {
                for (int sp = 0; sp < S; ++sp) v += src[sp * plane + i];
                if (a.logit_bias) v += a.logit_bias[e];
            }
            lg[tt * lde + e] = v;
        }
    }
    __syncthreads();
    router_rows_epilogue<TB, SEL, PER>(a, lg, st_m, st_s, st_h, t0);
}

// --------------------------------------------------------------------------
// Quantile bias: b_e = -(v_lo + frac (v_hi - v_lo)) with v_lo, v_hi the
// order statistics of rank lo and lo+1 of column e (linear interpolation,
// h = (T-1) q, lo = floor h, frac = h - lo).  One CTA of 512 threads per
// expert.  v_lo by a 4-pass radix select on the fp32 bit patterns (8 bits a
// pass; probabilities are >= 0, so bit order equals value order);
// v_hi from one more pass: v_lo again if at least lo + 2 values are <= v_lo,
// else the smallest value above it.
// --------------------------------------------------------------------------

// Exclusive scan of one value per thread of a 512-thread block; *total gets
// the block sum.  warp_tot holds 16 ints.
__device__ int block_exclusive_scan_512(int v, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int wt = lane < 16 ? warp_tot[lane] : 0;
        int wi = wt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        if (lane < 16) warp_tot[lane] = wi - wt;
        if (lane == 15) *total = wi;
    }
    __syncthreads();
    const int r = warp_tot[warp] + incl - v;
    __syncthreads();
    return r;
}

constexpr int kRadixDigit = 8;                   // bits resolved per pass (4 passes)
constexpr int kRadixBins = 1 << kRadixDigit;
constexpr int kRadixWarps = 16;                  // 512 threads
constexpr int kRadixBatch = 8;       // column values loaded per thread before binning

// Shared scratch of the 512-thread radix select: one histogram per warp, so
// that warps never contend for a counter (probabilities of similar size share
// their top bits, and one block-wide histogram serialised on a few bins).
struct RadixScratch {
    unsigned hist[kRadixWarps][kRadixBins];
    int warp_tot[16];
    int total;
    unsigned sel[2];
};

// A column of at most kStageMaxT values is copied to shared memory `buf`
// first (one coalesced pass, all threads of the block); the selection passes
// then read it there.  Longer columns are read in place.
constexpr int kStageMaxT = 16384;
__device__ const float *stage_col(const float *col, int T, float *buf) {
    if (T > kStageMaxT) return col;
    if ((reinterpret_cast<uintptr_t>(col) & 15) == 0) {
        const int n4 = T / 4;
#pragma unroll 4
        for (int i = threadIdx.x; i < n4; i += blockDim.x)
            reinterpret_cast<float4 *>(buf)[i] = reinterpret_cast<const float4 *>(col)[i];
        for (int i = 4 * n4 + threadIdx.x; i < T; i += blockDim.x) buf[i] = col[i];
    } else {
        for (int i = threadIdx.x; i < T; i += blockDim.x) buf[i] = col[i];
    }
    __syncthreads();
    return buf;
}
inline size_t stage_col_bytes(int T) { return T <= kStageMaxT ? sizeof(float) * T : 0; }

// Value of rank r (0-based, ascending) of col[0..T); 512 threads.  Four
// passes of 8 bits over the fp32 bit patterns (values >= 0, so bit order is
// value order), per-warp histograms.  After the first pass only the values
// that share the selected prefix are counted, and a warp none of whose values
// does skips the histogram update.
__device__ float radix_select_col(const float *col, int T, long long r, RadixScratch &sc) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned prefix = 0, mask = 0;
    unsigned *my_hist = sc.hist[warp];
    for (int shift = 32 - kRadixDigit; shift >= 0; shift -= kRadixDigit) {
        for (int i = tid; i < kRadixWarps * kRadixBins; i += blockDim.x)
            (&sc.hist[0][0])[i] = 0;
        __syncthreads();
        // kRadixBatch loads in flight per thread; every lane of a warp runs
        // the same number of iterations (n is a multiple of the block size)
        const int n = (T + blockDim.x - 1) / blockDim.x * blockDim.x;
        for (int i0 = tid; i0 < n; i0 += kRadixBatch * blockDim.x) {
            unsigned v[kRadixBatch];
#pragma unroll
            for (int q = 0; q < kRadixBatch; ++q) {
                const int i = i0 + q * blockDim.x;
                v[q] = i < T ? __float_as_uint(col[i]) : 0u;
            }
#pragma unroll
            for (int q = 0; q < kRadixBatch; ++q) {
                const int i = i0 + q * blockDim.x;
                if (i0 - tid + q * (int)blockDim.x >= n) break;     // uniform over the block
                const bool match = i < T && (v[q] & mask) == prefix;
                if (!__any_sync(0xffffffffu, match)) continue;          // uniform over the warp
                const unsigned bin = match ? (v[q] >> shift) & (kRadixBins - 1) : 0xffffffffu;
                const unsigned peers = __match_any_sync(0xffffffffu, bin);
                if (bin != 0xffffffffu && lane == __ffs(peers) - 1)
                    atomicAdd(&my_hist[bin], __popc(peers));
            }
        }
        __syncthreads();
        // thread tid < 256 owns bin tid: its count over all warps, then the
        // bin holding rank r
        int local = 0;
        if (tid < kRadixBins)
            for (int w = 0; w < kRadixWarps; ++w) local += (int)sc.hist[w][tid];
        const int ex = block_exclusive_scan_512(local, sc.warp_tot, &sc.total);
        if (local > 0 && (long long)ex <= r && r < (long long)ex + local) {
            sc.sel[0] = (unsigned)tid;
            sc.sel[1] = (unsigned)(r - ex);
        }
        __syncthreads();
        prefix |= sc.sel[0] << shift;
        mask |= (unsigned)(kRadixBins - 1) << shift;
        r = sc.sel[1];
        __syncthreads();
    }
    return __uint_as_float(prefix);
}

// (v_lo, v_hi): the values of rank lo and lo + 1 (v_lo when lo + 1 == n) of
// col[0..n); 512 threads, all of which must call it.
__device__ float2 rank_pair(const float *col, int n, long long lo, RadixScratch &sc,
                            unsigned *min_gt) {
    const float v_lo = radix_select_col(col, n, lo, sc);
    float v_hi = v_lo;
    if (lo + 1 < n) {
        if (threadIdx.x == 0) *min_gt = 0xffffffffu;
        __syncthreads();
        const unsigned vb = __float_as_uint(v_lo);
        int le = 0;
        unsigned mn = 0xffffffffu;
        for (int i0 = threadIdx.x; i0 < n; i0 += kRadixBatch * blockDim.x) {
            unsigned v[kRadixBatch];
#pragma unroll
            for (int q = 0; q < kRadixBatch; ++q) {
                const int i = i0 + q * blockDim.x;
                v[q] = i < n ? __float_as_uint(col[i]) : 0xffffffffu;
            }
#pragma unroll
            for (int q = 0; q < kRadixBatch; ++q) {
                if (i0 + q * (int)blockDim.x >= n) break;
                if (v[q] <= vb) ++le;
                else mn = min(mn, v[q]);
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        if ((threadIdx.x & 31) == 0) atomicMin(min_gt, mn);
        block_exclusive_scan_512(le, sc.warp_tot, &sc.total);
        const long long n_le = sc.total;
        v_hi = n_le >= lo + 2 ? v_lo : __uint_as_float(*min_gt);
    }
    __syncthreads();
    return make_float2(v_lo, v_hi);
}

__global__ void __launch_bounds__(512) quantile_bias_kernel(const float *probsT, int T,
                                                            long long lo, float frac,
                                                            float *bias_out) {
    __shared__ RadixScratch sc;
    __shared__ unsigned min_gt;
    extern __shared__ float colbuf[];
    const float *col = stage_col(probsT + (size_t)blockIdx.x * T, T, colbuf);
    const float2 r = rank_pair(col, T, lo, sc, &min_gt);
    if (threadIdx.x == 0) bias_out[blockIdx.x] = -(r.x + frac * (r.y - r.x));
}

// The same order statistics when they lie in the column's top tail (n_top =
// T - lo values at ranks >= lo, a few hundred of T, as with many experts and
// q = 1 - k/E).  The ranks are found by narrowing the column with thresholds
// and counting, with few block barriers (a radix pass over a small array
// costs about five):
//  1. a threshold L from a fixed sample of kQSample values (every
//     (T / kQSample)-th): kQPivots of the sample values are pivots, each
//     counted against the whole sample; L is the largest pivot with at least
//     m sample values >= it, m chosen so that about 3 n_top column values
//     are >= L;
//  2. one pass copies the column's values >= L (its c largest) to shared
//     memory; ranks lo and lo + 1 of the column are then descending ranks
//     n_top and n_top - 1 of the copies, provided c >= n_top;
//  3. pivots taken from the copies, counted against them, give the largest
//     threshold A with at least n_top copies >= A, and the copies >= A (c2 of
//     them, a few more than n_top) are copied once more;
//  4. each thread takes one of those and counts the ones above it and not
//     below it: the value whose descending rank range holds n_top is v_lo,
//     the one holding n_top - 1 is v_hi.
// Whenever a count falls outside what the buffers hold (c outside [n_top,
// kQCand], c2 > blockDim.x, no pivot qualifies) the kernel runs the radix
// select of quantile_bias_kernel on the copies or on the whole column, so the
// result is exact either way.
constexpr int kQSample = 512, kQCand = 2048, kQPivots = 64;
__device__ __forceinline__ void count_pivots(const float *vals, int n, const float *piv,
                                             int *cnt) {
    // kQPivots pivots x (blockDim.x / kQPivots) threads, each counting a
    // slice of vals against its pivot; blockDim.x = 512
    const int p = threadIdx.x >> 3, q = threadIdx.x & 7;
    const float x = piv[p];
    int c = 0;
#pragma unroll 8
    for (int i = q; i < n; i += 8) c += vals[i] >= x;
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 4);
    if (q == 0) cnt[p] = c;
}
// The largest pivot with at least `need` values >= it (warp 0 of the block
// writes it to *out, or -1 as a bit pattern when no pivot qualifies).
__device__ __forceinline__ void pick_pivot(const float *piv, const int *cnt, long long need,
                                           unsigned *out) {
    if (threadIdx.x >= 32) return;
    unsigned best = 0u;
    bool any = false;
    for (int p = threadIdx.x; p < kQPivots; p += 32)
        if (cnt[p] >= need) {
            best = max(best, __float_as_uint(piv[p]));
            any = true;
        }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, off));
    any = __any_sync(0xffffffffu, any);
    if (threadIdx.x == 0) *out = any ? best : 0xffffffffu;
}
// Copies the values of src[0..n) >= thr (a bit pattern; values >= 0) to
// dst[0..cap) in any order; returns their count (all threads).
__device__ __forceinline__ int compact_ge(const float *src, int n, unsigned thr, float *dst,
                                          int cap, int *counter) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) *counter = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kRadixBatch * blockDim.x) {
        unsigned xs[kRadixBatch];
#pragma unroll
        for (int q = 0; q < kRadixBatch; ++q) {
            const int i = i0 + q * blockDim.x + tid;
            xs[q] = i < n ? __float_as_uint(src[i]) : 0u;
        }
#pragma unroll
        for (int q = 0; q < kRadixBatch; ++q) {
            const int i = i0 + q * blockDim.x + tid;
            const bool take = i < n && xs[q] >= thr;
            const unsigned bal = __ballot_sync(0xffffffffu, take);
            if (!bal) continue;                          // uniform over the warp
            int base = 0;
            if (lane == 0) base = atomicAdd(counter, __popc(bal));
            base = __shfl_sync(0xffffffffu, base, 0);
            const int pos = base + __popc(bal & ((1u << lane) - 1u));
            if (take && pos < cap) dst[pos] = __uint_as_float(xs[q]);
        }
    }
    __syncthreads();
    return *counter;
}
__global__ void __launch_bounds__(512) quantile_tail_kernel(const float *probsT, int T,
                                                            long long lo, float frac,
                                                            float *bias_out) {
    __shared__ RadixScratch sc;
    __shared__ unsigned min_gt, thr;
    __shared__ int counter, cnt[kQPivots];
    __shared__ float samp[kQSample], piv[kQPivots];
    __shared__ __align__(16) float cand[kQCand];
    __shared__ __align__(16) float cand2[512];
    __shared__ float res[2];
    const int tid = threadIdx.x;
    const float *col = probsT + (size_t)blockIdx.x * T;
    const long long n_top = (long long)T - lo;
    float2 r = make_float2(0.f, 0.f);
    int path = 0;                    // 0: whole column, 1: the copies, 2: counted
    int c = -1;                      // column values >= L
    const long long m = (3 * n_top * kQSample + T - 1) / T + 2;   // sample count wanted
    if (m <= kQSample) {
        for (int j = tid; j < kQSample; j += blockDim.x) samp[j] = col[(long long)j * T / kQSample];
        __syncthreads();
        if (tid < kQPivots) piv[tid] = samp[tid * (kQSample / kQPivots) + kQSample / kQPivots / 2];
        __syncthreads();
        count_pivots(samp, kQSample, piv, cnt);
        __syncthreads();
        pick_pivot(piv, cnt, m, &thr);
        __syncthreads();
        const unsigned L = thr;
        c = L == 0xffffffffu ? -1 : compact_ge(col, T, L, cand, kQCand, &counter);
        if (c >= n_top && c <= kQCand) {
            path = 1;
            if (tid < kQPivots) piv[tid] = cand[(long long)tid * c / kQPivots];
            __syncthreads();
            count_pivots(cand, c, piv, cnt);
            __syncthreads();
            pick_pivot(piv, cnt, n_top, &thr);
            __syncthreads();
            const unsigned A = thr;
            const int c2 = A == 0xffffffffu ? -1 : compact_ge(cand, c, A, cand2, 512, &counter);
            if (c2 >= n_top && c2 <= (int)blockDim.x) {
                path = 2;
                // descending ranks (gt, ge]: v_lo holds n_top, v_hi holds n_top - 1
                if (tid < c2) {
                    const float v = cand2[tid];
                    int gt = 0, ge = 0;
                    const int c4 = c2 & ~3;
                    for (int i = 0; i < c4; i += 4) {   // 16-byte reads (cand2 is 16-byte aligned)
                        const float4 u = *reinterpret_cast<const float4 *>(cand2 + i);
                        gt += (u.x > v) + (u.y > v) + (u.z > v) + (u.w > v);
                        ge += (u.x >= v) + (u.y >= v) + (u.z >= v) + (u.w >= v);
                    }
                    for (int i = c4; i < c2; ++i) {
                        gt += cand2[i] > v;
                        ge += cand2[i] >= v;
                    }
                    if (gt < n_top && n_top <= ge) res[0] = v;
                    if (n_top >= 2 && gt < n_top - 1 && n_top - 1 <= ge) res[1] = v;
                }
                __syncthreads();
                r = make_float2(res[0], n_top >= 2 ? res[1] : res[0]);
            }
        }
    }
    if (path == 1) r = rank_pair(cand, c, c - n_top, sc, &min_gt);
    if (path == 0) r = rank_pair(col, T, lo, sc, &min_gt);
    if (tid == 0) bias_out[blockIdx.x] = -(r.x + frac * (r.y - r.x));
}

// --------------------------------------------------------------------------
// Top-k from stored probabilities [T, E] plus a bias (second pass of
// quantile balancing, and the plain top-k of the unbiased counts): one warp
// per token, the row read coalesced, top-k from registers.
// --------------------------------------------------------------------------
template <int PER>
__global__ void __launch_bounds__(256, 3) select_rows_kernel(const float *probs, const float *bias,
                                                          int T, int E, int k, int32_t *idx,
                                                          float *w, int n_cand,
                                                          int32_t *cand_idx, float *cand_w) {
    extern __shared__ float srows[];      // [8][E]: the probabilities of the block's tokens
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int t = blockIdx.x * 8 + wib;
    if (t >= T) return;
    const float *row = probs + (size_t)t * E;
    float *srow = srows + wib * E;
    float sc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        sc[i] = -CUDART_INF_F;
        if (e < E) {
            const float p = row[e];
            srow[e] = p;
            sc[i] = p + (bias ? bias[e] : 0.f);
        }
    }
    __syncwarp();
    float psum = 0.f, my_p = 0.f;
    int my_e = 0;
    WarpTopK<PER> topk;
    topk.init(sc, lane);
    for (int j = 0; j < k + n_cand; ++j) {
        const int bi = topk.next(sc, lane);
        const float pw = srow[bi];
        if (j < k) psum += pw;
        if (lane == j) { my_e = bi; my_p = pw; }
    }
    if (lane < k) {
        if (idx) idx[(size_t)t * k + lane] = my_e;
        if (w) w[(size_t)t * k + lane] = my_p / psum;
    } else if (lane < k + n_cand) {
        cand_idx[(size_t)t * n_cand + lane - k] = my_e;
        cand_w[(size_t)t * n_cand + lane - k] = my_p / psum;
    }
}

// --------------------------------------------------------------------------
// Host launchers
// --------------------------------------------------------------------------
// Grid of the partial-logit kernels: about `per_sm` resident CTAs per SM
// over all slices, each striding over the token groups of its slice.
static dim3 partial_grid(const void *kern, size_t smem, int S, int tok_per_cta, int T) {
    int dev = 0, sms = 148, per_sm = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int groups = (T + tok_per_cta - 1) / tok_per_cta;
    return dim3(std::max(1, std::min(groups, (sms * per_sm + S - 1) / S)), S);
}

template <typename TX>
static cudaError_t launch_partial_w8(const RouterArgs &a, float *part, cudaStream_t st) {
    auto kern = router_partial_w8_kernel<TX>;
    const int dtype = sizeof(TX) == 2 ? MOE_DTYPE_BF16 : MOE_DTYPE_FP32;
    const dim3 grid = partial_grid(reinterpret_cast<const void *>(kern), 0,
                                   router_slices(a.d, a.E, dtype), 8 * 4, a.T);
    kern<<<grid, 256, 0, st>>>(a, part);
    note_launch();
    return cudaGetLastError();
}

template <typename TX, int EP>
static cudaError_t launch_partial(const RouterArgs &a, float *part, cudaStream_t st) {
    constexpr int TPW = 32 / EP;
    const size_t smem = sizeof(float) * EP * kRouterSlice;
    auto kern = router_partial_kernel<TX, EP>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int dtype = sizeof(TX) == 2 ? MOE_DTYPE_BF16 : MOE_DTYPE_FP32;
    const dim3 grid = partial_grid(reinterpret_cast<const void *>(kern), smem,
                                   router_slices(a.d, a.E, dtype), 8 * TPW, a.T);
    kern<<<grid, 256, smem, st>>>(a, part);
    note_launch();
    return cudaGetLastError();
}

// Tokens per CTA of the router's softmax kernels: 8 warps x 32/EP tokens for
// E <= 32; for E > 32, kTB (the CUDA-core tiled router: fp32 layers, and bf16
// ones whose E is not a multiple of 4) or, for the softmax over the
// tensor-core logits, kTBLogits with top-k selection and
// kTBLogitsProbs without it (quantile balance, expert choice): a tile of 8
// tokens (29 KB of shared memory at E = 896) and no top-k state in registers
// let more CTAs share an SM, which the latency-bound kernel needs.
constexpr int kTBLogits = 16, kTBLogitsProbs = 8;
static int router_tokens_per_block(int E, int dtype, bool select) {
    if (E <= 8) return 32;
    if (E <= 16) return 16;
    if (E <= 32) return 8;
    if (!router_on_tensor_cores(E, dtype)) return kTB;   // router_tiled_kernel
    return select ? kTBLogits : kTBLogitsProbs;
}

// Blocks of the router's softmax kernels: the row count of the per-block
// partial sums (p_partial, ent_partial).
int router_blocks(int T, int E, int dtype, bool select) {
    const int tb = router_tokens_per_block(E, dtype, select);
    return (T + tb - 1) / tb;
}

template <int EP>
static cudaError_t launch_small_epilogue(const RouterArgs &a, const float *part, int S,
                                         cudaStream_t st) {
    router_small_epilogue_kernel<EP><<<router_blocks(a.T, a.E, MOE_DTYPE_FP32, true), 256, 0, st>>>(
        a, part, S);
    note_launch();
    return cudaGetLastError();
}

size_t router_smem_bytes(int E, int dtype) {
    if (E <= 32) return 0;
    (void)dtype;
    return router_tiled_smem(E);
}

template <typename TX>
static cudaError_t launch_router_t(const RouterArgs &a, float *part, cudaStream_t st) {
    if (a.E <= 32) {
        cudaError_t err = a.E <= 8    ? launch_partial_w8<TX>(a, part, st)
                          : a.E <= 16 ? launch_partial<TX, 16>(a, part, st)
                                      : launch_partial<TX, 32>(a, part, st);
        if (err != cudaSuccess) return err;
        const int S = router_slices(a.d, a.E, sizeof(TX) == 2 ? MOE_DTYPE_BF16 : MOE_DTYPE_FP32);
        return a.E <= 8    ? launch_small_epilogue<8>(a, part, S, st)
               : a.E <= 16 ? launch_small_epilogue<16>(a, part, S, st)
                           : launch_small_epilogue<32>(a, part, S, st);
    }
    const size_t smem = router_tiled_smem(a.E);
    auto kern = router_tiled_kernel<TX>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<(a.T + kTB - 1) / kTB, 256, smem, st>>>(a);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_router(const RouterArgs &a, int dtype, float *part, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    return dtype == MOE_DTYPE_FP32 ? launch_router_t<float>(a, part, st)
                                   : launch_router_t<__nv_bfloat16>(a, part, st);
}

cudaError_t launch_split_router_weight(const float *w_r, int E, int d, int dp, int parts,
                                       __nv_bfloat16 *out, int T, int32_t *offsets,
                                       int32_t *tile_e, int32_t *tile_start, int32_t *n_tiles,
                                       cudaStream_t st) {
    if (parts < 1 || parts > kRouterMaxParts || dp % 64 != 0) return cudaErrorInvalidValue;
    const long long n8 = (long long)E * (dp / 8);
    const int grid = (int)std::max<long long>(1, std::min<long long>((n8 + 255) / 256, 148 * 4));
    split_router_weight_kernel<<<grid, 256, 0, st>>>(w_r, E, d, dp, parts, out, T, offsets,
                                                     tile_e, tile_start, n_tiles);
    note_launch();
    return cudaGetLastError();
}

template <int TB, int SEL, int PER>
static cudaError_t launch_from_logits_tb(const RouterArgs &a, const float *part, int S,
                                         cudaStream_t st) {
    const size_t smem = sizeof(float) * ((size_t)TB * router_lde(a.E) + 3 * TB);
    auto kern = router_from_logits_kernel<TB, SEL, PER>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<(a.T + TB - 1) / TB, 256, smem, st>>>(a, part, S);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_router_from_logits(const RouterArgs &a, const float *part, int S,
                                      cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    if (!a.do_select) return launch_from_logits_tb<kTBLogitsProbs, 0, 8>(a, part, S, st);
    switch (topk_per_lane(a.E)) {
        case 8: return launch_from_logits_tb<kTBLogits, 1, 8>(a, part, S, st);
        case 16: return launch_from_logits_tb<kTBLogits, 1, 16>(a, part, S, st);
        default: return launch_from_logits_tb<kTBLogits, 1, 32>(a, part, S, st);
    }
}

cudaError_t launch_select_rows(const float *probs, const float *bias, int T, int E, int k,
                               int32_t *idx, float *w, cudaStream_t st, int n_cand,
                               int32_t *cand_idx, float *cand_w) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((T + 7) / 8);
    const size_t smem = sizeof(float) * 8 * E;
    const int per = topk_per_lane(E);
    if (per == 8)
        select_rows_kernel<8><<<grid, 256, smem, st>>>(probs, bias, T, E, k, idx, w, n_cand,
                                                       cand_idx, cand_w);
    else if (per == 16)
        select_rows_kernel<16><<<grid, 256, smem, st>>>(probs, bias, T, E, k, idx, w, n_cand,
                                                        cand_idx, cand_w);
    else
        select_rows_kernel<32><<<grid, 256, smem, st>>>(probs, bias, T, E, k, idx, w, n_cand,
                                                        cand_idx, cand_w);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_quantile_bias(const float *probsT, int T, int E, long long lo, float frac,
                                 float *bias_out, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    // a top tail of at most a sixth of the candidate buffer: the sampled kernel
    const long long n_top = (long long)T - lo;
    if (T >= 4 * kQSample && n_top * 6 <= kQCand) {
        quantile_tail_kernel<<<E, 512, 0, st>>>(probsT, T, lo, frac, bias_out);
        note_launch();
        return cudaGetLastError();
    }
    const size_t smem = stage_col_bytes(T);
    cudaError_t err = cudaFuncSetAttribute(quantile_bias_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    quantile_bias_kernel<<<E, 512, smem, st>>>(probsT, T, lo, frac, bias_out);
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
