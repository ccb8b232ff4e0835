// Expert-choice routing: every expert takes the tokens it scores highest.
//
// Sources: "混合エキスパートモデル（MoE）実践" (deepseekmodel.com), TopKRouter
// discussion: instead of tokens choosing experts, each expert picks the top-C
// tokens for its capacity, so every expert is exactly full; "Mixture of
// Experts (MoE) memo" (iwashi.co), routing table: expert choice, each expert
// chooses its top tokens.  Expert e takes the Cn = min(C, T) tokens with the
// largest router probability probs[t, e] (exactly equal values: lower token
// index first) with gate weight probs[t, e]; a token may be taken by any
// number of experts, including none.
//
// Per expert one CTA finds the Cn-th largest value v of its column by radix
// select on the fp32 bit patterns (probabilities are >= 0, so bit order is
// value order), then keeps, in token order, every token above v and the
// first (Cn - #above) tokens equal to v.  The combine needs each token's
// rows: a per-token walk over the experts in order builds them as a
// compressed list (counts, scan, fill), so the sum over a token's experts has
// a fixed order.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__global__ void __launch_bounds__(512) ec_select_kernel(const float *probsT, int T, int E, int Cn,
                                                        int32_t *perm, float *row_w,
                                                        int32_t *rowidx, int32_t *counts,
                                                        int32_t *offsets) {
    __shared__ RadixScratch sc;
    int *warp_tot = sc.warp_tot;
    __shared__ int total;
    extern __shared__ float colbuf[];
    const int e = blockIdx.x;
    const float *col = probsT + (size_t)e * T;
    if (threadIdx.x == 0) {
        counts[e] = Cn;
        offsets[e] = e * Cn;
        if (e == E - 1) offsets[E] = E * Cn;
    }
    if (Cn == 0) {
        for (int t = threadIdx.x; t < T; t += blockDim.x) rowidx[(size_t)e * T + t] = -1;
        return;
    }
    col = stage_col(col, T, colbuf);
    const float v = radix_select_col(col, T, (long long)(T - Cn), sc);
    // tokens strictly above v
    int above = 0;
    for (int t = threadIdx.x; t < T; t += blockDim.x) above += col[t] > v ? 1 : 0;
    block_exclusive_scan_512(above, warp_tot, &total);
    const int need_eq = Cn - total;
    __syncthreads();
    int eq_seen = 0, pos = 0;     // carries across chunks (uniform)
    for (int t0 = 0; t0 < T; t0 += blockDim.x) {
        const int t = t0 + threadIdx.x;
        const float p = t < T ? col[t] : -1.f;
        const int is_eq = (t < T && p == v) ? 1 : 0;
        const int eq_rank = eq_seen + block_exclusive_scan_512(is_eq, warp_tot, &total);
        const int eq_tot = total;
        const int take = (t < T && (p > v || (is_eq && eq_rank < need_eq))) ? 1 : 0;
        const int at = pos + block_exclusive_scan_512(take, warp_tot, &total);
        const int take_tot = total;
        if (t < T) {
            if (take) {
                const int row = e * Cn + at;
                perm[row] = t;
                row_w[row] = p;
                rowidx[(size_t)e * T + t] = row;
            } else {
                rowidx[(size_t)e * T + t] = -1;
            }
        }
        eq_seen += eq_tot;
        pos += take_tot;
    }
}

// Per token: the number of experts that took it.
__global__ void ec_token_count_kernel(const int32_t *rowidx, int T, int E, int32_t *tok_cnt) {
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
        int n = 0;
        for (int e = 0; e < E; ++e) n += rowidx[(size_t)e * T + t] >= 0 ? 1 : 0;
        tok_cnt[t] = n;
    }
}

// One CTA: tok_start = exclusive scan of tok_cnt (T + 1 entries); tokens no
// expert took.
__global__ void __launch_bounds__(1024) ec_token_scan_kernel(const int32_t *tok_cnt, int T,
                                                             int32_t *tok_start,
                                                             int32_t *n_unchosen) {
    __shared__ int warp_tot[32];
    __shared__ int total;
    int carry = 0, zeros = 0;
    for (int t0 = 0; t0 < T; t0 += 1024) {
        const int t = t0 + threadIdx.x;
        const int v = t < T ? tok_cnt[t] : 0;
        if (t < T && v == 0) ++zeros;
        const int ex = block_exclusive_scan_1024(v, warp_tot, &total);
        if (t < T) tok_start[t] = carry + ex;
        carry += total;
        __syncthreads();
    }
    const int z = block_exclusive_scan_1024(zeros, warp_tot, &total);
    (void)z;
    if (threadIdx.x == 0) {
        tok_start[T] = carry;
        *n_unchosen = total;
    }
}

// Per token: its rows, experts in ascending order.
__global__ void ec_token_fill_kernel(const int32_t *rowidx, int T, int E,
                                     const int32_t *tok_start, int32_t *tok_rows) {
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
        int o = tok_start[t];
        for (int e = 0; e < E; ++e) {
            const int r = rowidx[(size_t)e * T + t];
            if (r >= 0) tok_rows[o++] = r;
        }
    }
}

cudaError_t launch_expert_choice(const float *probsT, int T, int E, int Cn, int32_t *perm,
                                 float *row_w, int32_t *rowidx, int32_t *counts,
                                 int32_t *offsets, int32_t *tok_cnt, int32_t *tok_start,
                                 int32_t *tok_rows, int32_t *n_unchosen, cudaStream_t st) {
    const size_t smem = stage_col_bytes(T);
    cudaError_t err = cudaFuncSetAttribute(ec_select_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    ec_select_kernel<<<E, 512, smem, st>>>(probsT, T, E, Cn, perm, row_w, rowidx, counts,
                                           offsets);
    note_launch();
    const int grid = std::max(1, std::min((T + 255) / 256, 148 * 8));
    if (T > 0) {
        ec_token_count_kernel<<<grid, 256, 0, st>>>(rowidx, T, E, tok_cnt);
        note_launch();
    }
    ec_token_scan_kernel<<<1, 1024, 0, st>>>(tok_cnt, T, tok_start, n_unchosen);
    note_launch();
    if (T > 0) {
        ec_token_fill_kernel<<<grid, 256, 0, st>>>(rowidx, T, E, tok_start, tok_rows);
        note_launch();
    }
    return cudaGetLastError();
}

}  // namespace moe
