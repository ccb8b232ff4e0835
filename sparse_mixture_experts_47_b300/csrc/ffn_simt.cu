// SIMT grouped GEMM with fp32 accumulation, used for the fp32 layer (tf32
// tensor cores carry a 10-bit mantissa, too coarse for a 1e-4 x RMS bound).
//
// Expert FFN ("Mixture of Experts", waylandz.com ch. 30, §30.2.4 / §30.6.1):
//   up   (SwiGLU) H = silu(A W1_e^T) * (A W3_e^T)   (ReLU) H = relu(A W1_e^T)
//   down O = H W2_e^T
// over each expert's contiguous rows [offsets[e], offsets[e+1]) of the
// grouped layout.  Tiles of 64 rows x 64 columns come from a device-side tile
// table (expert, first row), so the host never reads the expert counts.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kBK = 16;

__device__ __forceinline__ void load4_any(const float *p, float *v) {
    float4 a = *reinterpret_cast<const float4 *>(p);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void load4_any(const __nv_bfloat16 *p, float *v) {
    uint2 a = *reinterpret_cast<const uint2 *>(p);
    v[0] = __uint_as_float(a.x << 16); v[1] = __uint_as_float(a.x & 0xffff0000u);
    v[2] = __uint_as_float(a.y << 16); v[3] = __uint_as_float(a.y & 0xffff0000u);
}

template <typename TI, int MODE>
__global__ void __launch_bounds__(256) simt_gemm_kernel(GroupedGemmArgs g) {
    constexpr int BM = kSimtBM, BN = kSimtBN;
    constexpr bool DUAL = MODE == GEMM_UP_SWIGLU;
    __shared__ __align__(16) float As[kBK][BM + 4];
    __shared__ __align__(16) float Bs[kBK][BN + 4];
    __shared__ __align__(16) float B3s[DUAL ? kBK : 1][BN + 4];
    __shared__ int a_row[BM];

    const int tile = blockIdx.y;
    if (tile >= *g.n_tiles) return;
    const int e = g.tile_e[tile];
    const int m0 = g.tile_m0[tile];
    const int mend = g.offsets[e + 1];
    const int n0 = blockIdx.x * BN;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;

    const TI *A = static_cast<const TI *>(g.A);
    const TI *B1 = static_cast<const TI *>(g.B1) + (size_t)e * g.b_expert_stride;
    const TI *B3 = DUAL ? static_cast<const TI *>(g.B3) + (size_t)e * g.b_expert_stride : nullptr;

    if (tid < BM) {
        const int s = m0 + tid;
        int r = -1;
        if (s < mend) r = g.a_gather ? g.a_gather[s] / g.gather_k : s;
        a_row[tid] = r;
    }
    __syncthreads();

    float acc[4][4], acc3[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) { acc[i][j] = 0.f; acc3[i][j] = 0.f; }

    const int lr = tid >> 2, lk = (tid & 3) * 4;   // loader: row 0..63, k 0,4,8,12
    for (int k0 = 0; k0 < g.K; k0 += kBK) {
        float va[4] = {0.f, 0.f, 0.f, 0.f}, vb[4] = {0.f, 0.f, 0.f, 0.f}, v3[4] = {0.f, 0.f, 0.f, 0.f};
        const bool kin = k0 + lk < g.K;
        const int ar = a_row[lr];
        if (kin && ar >= 0) load4_any(A + (size_t)ar * g.K + k0 + lk, va);
        if (kin && n0 + lr < g.N) {
            load4_any(B1 + (size_t)(n0 + lr) * g.K + k0 + lk, vb);
            if (DUAL) load4_any(B3 + (size_t)(n0 + lr) * g.K + k0 + lk, v3);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            As[lk + i][lr] = va[i];
            Bs[lk + i][lr] = vb[i];
            if (DUAL) B3s[lk + i][lr] = v3[i];
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kBK; ++kk) {
            const float4 a4 = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
            const float4 b4 = *reinterpret_cast<const float4 *>(&Bs[kk][tx * 4]);
            const float a[4] = {a4.x, a4.y, a4.z, a4.w}, b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            if (DUAL) {
                const float4 c4 = *reinterpret_cast<const float4 *>(&B3s[kk][tx * 4]);
                const float c[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc3[i][j] = fmaf(a[i], c[j], acc3[i][j]);
            }
        }
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int s = m0 + ty * 4 + i;
        if (s >= mend) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= g.N) continue;
            float v = acc[i][j];
            if (MODE == GEMM_UP_SWIGLU) v = silu(v) * acc3[i][j];
            if (MODE == GEMM_UP_RELU) v = fmaxf(v, 0.f);
            if (MODE == GEMM_DOWN)
                static_cast<float *>(g.C)[(size_t)s * g.ldc + n] = v;
            else
                static_cast<TI *>(g.C)[(size_t)s * g.ldc + n] = from_f32<TI>(v);
        }
    }
}

template <typename TI>
static cudaError_t launch_t(const GroupedGemmArgs &g, int mode, cudaStream_t st) {
    if (g.max_tiles == 0) return cudaSuccess;
    dim3 grid((g.N + kSimtBN - 1) / kSimtBN, (unsigned)g.max_tiles);
    if (mode == GEMM_UP_SWIGLU) simt_gemm_kernel<TI, GEMM_UP_SWIGLU><<<grid, 256, 0, st>>>(g);
    else if (mode == GEMM_UP_RELU) simt_gemm_kernel<TI, GEMM_UP_RELU><<<grid, 256, 0, st>>>(g);
    else simt_gemm_kernel<TI, GEMM_DOWN><<<grid, 256, 0, st>>>(g);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_simt_gemm(const GroupedGemmArgs &g, int mode, int dtype, cudaStream_t st) {
    return dtype == MOE_DTYPE_FP32 ? launch_t<float>(g, mode, st)
                                   : launch_t<__nv_bfloat16>(g, mode, st);
}

}  // namespace moe
