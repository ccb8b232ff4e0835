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
};

// router.cu
int router_blocks(int T, int E);
size_t router_smem_bytes(int E, int dtype);
cudaError_t launch_router(const RouterArgs &a, int dtype, cudaStream_t st);
cudaError_t launch_split_router_weight(const float *w_r, int E, int d, int dp,
                                       __nv_bfloat16 *out, cudaStream_t st);
cudaError_t launch_router_from_logits(const RouterArgs &a, const float *part, int S,
                                      cudaStream_t st);
cudaError_t launch_select_from_probsT(const float *probsT, const float *bias, int T, int E,
                                      int k, int32_t *idx, float *w, cudaStream_t st);
cudaError_t launch_quantile_bias(const float *probsT, int T, int E, long long lo, float frac,
                                 float *bias_out, cudaStream_t st);

// dispatch.cu
constexpr int kDispatchChunk = 1024;
inline int dispatch_blocks(long long n) { return (int)((n + kDispatchChunk - 1) / kDispatchChunk); }
cudaError_t launch_dispatch(const int32_t *idx, long long n, int E, int k, long long C,
                            int32_t *hist, int32_t *block_base, int32_t *counts,
                            int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *n_dropped,
                            cudaStream_t st);
cudaError_t launch_histogram(const int32_t *idx, long long n, int E, int32_t *hist,
                             int32_t *counts, cudaStream_t st);

// misc.cu
cudaError_t launch_p_finalize(const float *p_partial, int nblk, int E, int T, float *p,
                              cudaStream_t st);
cudaError_t launch_prob_partials(const float *probs, int T, int E, float *p_partial,
                                 cudaStream_t st);
cudaError_t launch_stats_finalize(const int32_t *counts, const float *p, int T, int E, int k,
                                  float *f, float *p_out, float *aux, float *load,
                                  cudaStream_t st);
cudaError_t launch_gather_rows(const void *x, int elem_bytes, int d, const int32_t *perm,
                               const int32_t *offsets_end, int k, long long max_rows, void *xs,
                               cudaStream_t st);
cudaError_t launch_combine(const float *out_sorted, const int32_t *inv, const float *w,
                           const float *shared_out, int T, int k, int d, int out_dtype, void *y,
                           cudaStream_t st);
cudaError_t launch_build_tiles(const int32_t *offsets, int E, int BM, int32_t *tile_e,
                               int32_t *tile_m0, int32_t *tile_start, int32_t *n_tiles,
                               cudaStream_t st);
inline long long max_tiles(long long rows, int E, int BM) { return (rows + BM - 1) / BM + E; }

// ffn_simt.cu: SIMT grouped GEMM (fp32 accumulate) for the fp32 workloads.
constexpr int kSimtBM = 64, kSimtBN = 64;
enum { GEMM_UP_SWIGLU = 0, GEMM_UP_RELU = 1, GEMM_DOWN = 2 };
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
cudaError_t launch_tc_gemm(int mode, const void *A, long long a_rows, int a_cols, const void *B0,
                           const void *B1, int E, int b_rows, int N, int K, int a_k_period,
                           int k_splits, long long split_stride, const int32_t *tile_e,
                           const int32_t *tile_start, const int32_t *n_mtiles,
                           const int32_t *offsets, void *C, int ldc, cudaStream_t st);

}  // namespace moe
