// Internal launchers of the MoE layer kernels (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <cuda_bf16.h>

namespace moe {

constexpr int kErrBadIndex = 2;   // device error bit: an expert index out of [0, E)

struct RouterArgs {
    const void *x;
    const float *w_r, *logit_bias, *select_bias;
    int T, d, E, k, select_space, do_select;
    int32_t *idx;
    float *w, *probs, *probsT, *p_partial;
    float *ent_partial;   // per-block sums of the tokens' gate entropies, or NULL
    int n_cand;           // experts ranked after the top k to report (0: none)
    int32_t *cand_idx;    // [T, n_cand] next-best experts, descending score
    float *cand_w;        // [T, n_cand] their probability over the top-k sum
    float *p_direct;      // E <= 32 with one softmax block: p [E] written by that block
};

// router.cu
// E <= 32: the logits are computed in slices of d, written as partial planes
// [slices][T][E] (caller's buffer) and added in slice order by the softmax
// kernel.  E <= 8: a slice is 32 lanes x one 16-byte vector of x (256 bf16
// or 128 fp32 columns), its W_r columns held in registers; 8 < E <= 32:
// kRouterSlice columns, its W_r columns staged in shared memory.
constexpr int kRouterSlice = 512;
inline int router_slice_cols(int E, int dtype) {
    return E <= 8 ? 32 * (dtype == MOE_DTYPE_BF16 ? 8 : 4) : kRouterSlice;
}
inline int router_slices(int d, int E, int dtype) {
    const int c = router_slice_cols(E, dtype);
    return (d + c - 1) / c;
}
// The router's logits come from the tensor-core GEMM (bf16 x, E > 32,
// E % 4 == 0: its fp32 planes are stored as float4 rows); otherwise from the
// CUDA-core kernels of router.cu.
inline bool router_on_tensor_cores(int E, int dtype) {
    return dtype == MOE_DTYPE_BF16 && E > 32 && E % 4 == 0;
}
// select: the softmax kernel also takes the top-k (false: quantile balance
// and expert choice, which select later)
int router_blocks(int T, int E, int dtype, bool select);
size_t router_smem_bytes(int E, int dtype);
cudaError_t launch_router(const RouterArgs &a, int dtype, float *part, cudaStream_t st);
// W_r split into bf16 parts, and the tile table of the logit GEMM's single
// group of T rows (128-row tiles).
cudaError_t launch_split_router_weight(const float *w_r, int E, int d, int dp, int parts,
                                       __nv_bfloat16 *out, int T, int32_t *offsets,
                                       int32_t *tile_e, int32_t *tile_start, int32_t *n_tiles,
                                       cudaStream_t st);
cudaError_t launch_router_from_logits(const RouterArgs &a, const float *part, int S,
                                      cudaStream_t st);
cudaError_t launch_select_rows(const float *probs, const float *bias, int T, int E, int k,
                               int32_t *idx, float *w, cudaStream_t st, int n_cand = 0,
                               int32_t *cand_idx = nullptr, float *cand_w = nullptr);
cudaError_t launch_quantile_bias(const float *probsT, int T, int E, long long lo, float frac,
                                 float *bias_out, cudaStream_t st);

// Optional observability outputs of the load statistics (any pointer may be
// NULL).
struct ObsArgs {
    const int32_t *n_dropped;   // in: dropped assignments
    const float *bias;          // in: selection bias in effect [E]
    float *drop_ratio, *bias_mean_abs, *bias_max_abs;
};

// dispatch.cu
constexpr int kDispatchChunk = 1024;
inline int dispatch_blocks(long long n) { return (int)((n + kDispatchChunk - 1) / kDispatchChunk); }
// Work that the dispatch kernel computing the counts and offsets does after
// them, in place of separate launches: the router's mean probabilities p_out
// from its per-block partials (p_finalize, up to 32 experts), the load
// statistics (stats_finalize's outputs, from counts, n_dropped and p) and the
// tile table of the up projection (build_tiles with tile_rows-row tiles).
struct DispatchTail {
    const float *p_partial;      // p_nblk > 0: p_out = block sums of p_partial / T
    int p_nblk;
    float *p_out;
    bool stats;
    const float *p;
    int T, k;
    float *f, *aux, *load;
    ObsArgs o;                   // o.n_dropped: the dispatch's own n_dropped
    int tile_rows;               // 0: no tile table
    int32_t *tile_e, *tile_start, *n_tiles;
};
cudaError_t launch_dispatch(const int32_t *idx, long long n, int E, int k, long long C,
                            int32_t *hist, int32_t *block_base, int32_t *counts,
                            int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *n_dropped,
                            cudaStream_t st, const DispatchTail *tail = nullptr);
cudaError_t launch_histogram(const int32_t *idx, long long n, int E, int32_t *hist,
                             int32_t *counts, cudaStream_t st);

// reroute.cu: capacity overflow redirected to the next-best experts.
struct RerouteWork {             // device scratch
    int32_t *slot_e;             // [T*k] current target expert of each slot (-1: none)
    float *slot_w;               // [T*k] its gate weight
    int32_t *served;             // [T*k] rank in the serving expert's rows, -1 if unserved
    int32_t *nxt;                // [T] next unused candidate of each token
    int32_t *filled, *filled_before;   // [E]
    int32_t *hist, *block_base;  // [chunks][E]
};
cudaError_t launch_dispatch_reroute(const int32_t *topk_idx, const float *topk_w,
                                    const int32_t *cand_idx, const float *cand_w, int n_cand,
                                    long long T, int k, int E, long long C, int rounds,
                                    const RerouteWork &w, int32_t *counts, int32_t *offsets,
                                    int32_t *perm, int32_t *inv, int32_t *slot_expert,
                                    float *slot_w_out, int32_t *n_dropped, cudaStream_t st);

// misc.cu
cudaError_t launch_p_finalize(const float *p_partial, int nblk, int E, int T, float *p,
                              cudaStream_t st);
cudaError_t launch_prob_partials(const float *probs, int T, int E, float *p_partial,
                                 cudaStream_t st);
cudaError_t launch_stats_finalize(const int32_t *counts, const float *p, int T, int E, int k,
                                  float *f, float *p_out, float *aux, float *load,
                                  cudaStream_t st, const ObsArgs &o = ObsArgs{});
cudaError_t launch_entropy_partials(const float *probs, int T, int E, float *ent_partial,
                                    cudaStream_t st);
// Expert outputs o in row order: `planes` fp32 planes `plane` elements apart
// (partial sums of a split reduction, added in plane order; one plane when
// the reduction is not split).
struct ExpertOut {
    const float *p;
    int planes;
    long long plane;
};
inline ExpertOut expert_out_f32(const float *p, int planes = 1, long long plane = 0) {
    return ExpertOut{p, planes, plane};
}
// Expert output scale over the dispatched rows: row statistics into
// rs [max_rows][3] (fp64), then per expert mean, std and max |o| (each
// output pointer may be NULL).
cudaError_t launch_expert_scale(const ExpertOut &o, int d, const int32_t *offsets, int E,
                                long long max_rows, double *rs, float *mean, float *std_,
                                float *maxabs, cudaStream_t st);
cudaError_t launch_gather_rows(const void *x, int elem_bytes, int d, const int32_t *perm,
                               const int32_t *offsets_end, int k, long long max_rows, void *xs,
                               cudaStream_t st);
// The same rows, token-major: x[t] to row inv[t*k+j] of xs for every kept slot.
cudaError_t launch_scatter_rows(const void *x, int elem_bytes, int d, const int32_t *inv, int k,
                                long long T, void *xs, cudaStream_t st);
// y[t] = sum_j w o[row] + s[t]; `sh` (the shared expert's output, p NULL
// when there is none) is read like `o`.
cudaError_t launch_combine(const ExpertOut &o, const int32_t *inv, const float *w,
                           const ExpertOut &sh, int T, int k, int d, int out_dtype, void *y,
                           cudaStream_t st);
cudaError_t launch_combine_rows(const ExpertOut &o, const int32_t *tok_start,
                                const int32_t *tok_rows, const float *row_w, const ExpertOut &sh,
                                int T, int d, int out_dtype, void *y, cudaStream_t st);
// expert_choice.cu: each expert takes its top-Cn tokens by probability from
// probsT [E, T]; rows of expert e are [e*Cn, (e+1)*Cn) in token order.
// rowidx [E][T] (row or -1), per-token row lists tok_start [T+1], tok_rows.
cudaError_t launch_expert_choice(const float *probsT, int T, int E, int Cn, int32_t *perm,
                                 float *row_w, int32_t *rowidx, int32_t *counts,
                                 int32_t *offsets, int32_t *tok_cnt, int32_t *tok_start,
                                 int32_t *tok_rows, int32_t *n_unchosen, cudaStream_t st);
cudaError_t launch_slot_outputs(const int32_t *idx, const float *w, const int32_t *inv,
                                long long n, int32_t *slot_expert, float *slot_w,
                                cudaStream_t st);
// h[r] = act(sum_s P_s[r]) in bf16 for rows r < *rows_end of the split
// partial sums of an up projection (SwiGLU: W1 part at f, W3 part at N + f).
cudaError_t launch_split_activation(const float *P, int splits, long long plane, int N,
                                    int swiglu, const int32_t *rows_end, long long max_rows,
                                    __nv_bfloat16 *h, cudaStream_t st);
// out[r] = sum_s P_s[r] (fp32, in split order) for rows r < *rows_end.
cudaError_t launch_sum_planes(const float *P, int splits, long long plane, int d,
                              const int32_t *rows_end, long long max_rows, float *out,
                              cudaStream_t st);
cudaError_t launch_build_tiles(const int32_t *offsets, int E, int BM, int32_t *tile_e,
                               int32_t *tile_m0, int32_t *tile_start, int32_t *n_tiles,
                               cudaStream_t st);
inline long long max_tiles(long long rows, int E, int BM) { return (rows + BM - 1) / BM + E; }

// ffn_simt.cu: SIMT grouped GEMM (fp32 accumulate) for the fp32 workloads.
constexpr int kSimtBM = 64, kSimtBN = 64;
// GEMM_LOGITS: fp32 C = A B^T over K in chains of chain_kb K blocks, each
// split of whole chains summed on chip in chain order into its own plane (the
// tensor-core router).
enum { GEMM_UP_SWIGLU = 0, GEMM_UP_RELU = 1, GEMM_DOWN = 2, GEMM_LOGITS = 3 };
struct GroupedGemmArgs {
    const void *A;               // rows of A: [rows, K] (K contiguous)
    const int32_t *a_gather;     // NULL, or A row of sorted row s = a_gather[s] / gather_k
    int gather_k;
    const void *B1, *B3;         // [E][N][K] (K contiguous); B3 only for SwiGLU
    long long b_expert_stride;   // elements between experts (N*K), 0 for a single matrix
    int N, K;
    void *C;                     // [rows, ldc]
    int ldc;
    const int32_t *tile_e, *tile_m0, *n_tiles, *offsets;
    long long max_tiles;
};
cudaError_t launch_simt_gemm(const GroupedGemmArgs &g, int mode, int dtype, cudaStream_t st);

// gemm_tcgen05.cu: tcgen05/TMEM grouped GEMM for the bf16 workloads.
constexpr int kTcBM = 128;
// Token-row tiling of the nt = 0 geometries (launch_tc_gemm's mh): 128-row
// tiles; 256-row tiles on one SM (two M = 128 MMAs per weight stage, one
// accumulator); 256-row tiles on a pair of SMs (a cluster of two CTAs,
// tcgen05.mma.cta_group::2 with M = 256, two accumulators).
enum { TILE_ROWS_128 = 1, TILE_ROWS_256 = 2, TILE_ROWS_256_PAIR = 3 };
inline int tile_rows(int mh) { return mh == TILE_ROWS_128 ? kTcBM : 2 * kTcBM; }
cudaError_t launch_tc_gemm(int mode, int nt, int bn, int mh, const void *A, long long a_rows,
                           int a_cols,
                           const void *B0, const void *B1, int E, int b_rows, int N, int K,
                           int a_k_period, int k_splits, long long split_stride,
                           const int32_t *tile_e, const int32_t *tile_start,
                           const int32_t *n_mtiles, const int32_t *offsets, void *C, int ldc,
                           cudaStream_t st, int chain_kb = 0);
namespace tc {
// Test hooks of the grouped GEMM's bounded waits on the current device: the
// main-loop wait limit in ns and a stall of the MMA issuer (see
// moe_debug_set_wait_hooks).
cudaError_t set_wait_hooks(unsigned long long main_limit_ns, int stall_mma);
}  // namespace tc

}  // namespace moe
