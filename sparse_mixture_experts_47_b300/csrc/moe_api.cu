// C ABI of the MoE layer forward (declared in include/moe.h).
//
// This file is the library's single translation unit: it includes every
// kernel file, validates arguments on the host, carves the caller's
// workspace and enqueues the kernels on the caller's stream.  It allocates
// nothing and never synchronises, except moe_device_status().
#include "common.cuh"
#include "kernels.h"

#include "router.cu"
#include "dispatch.cu"
#include "misc.cu"
#include "ffn_simt.cu"
#include "gemm_tcgen05.cu"

#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

inline int elem_bytes(int dtype) { return dtype == MOE_DTYPE_FP32 ? 4 : 2; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace regions (byte offsets from the workspace base).
struct Layout {
    size_t p_partial, probsT, hist, block_base, idx, w, counts, offsets, perm, inv, ndrop,
        pvec, sbias, idx_unb, tile_e, tile_m0, tile_start, ntiles, sh_offsets, sh_tile_e,
        sh_tile_m0, sh_tile_start, sh_ntiles, xs, h, out_sorted, sh_h, sh_out, rt_wsplit,
        rt_logits, rt_offsets, rt_tile_e, rt_tile_start, rt_ntiles, total;
};

struct Sizes {
    long long T, d, E, k, F, Fs, Tk;
};

Sizes sizes(const moe_config *c) {
    Sizes s;
    s.T = c->T; s.d = c->d_model; s.E = c->n_experts; s.k = c->top_k; s.F = c->d_ff;
    s.Fs = c->d_ff_shared; s.Tk = s.T * s.k;
    return s;
}

// Router logits on the tensor cores (bf16 x, E > 32, E % 4 == 0): W_r split
// into three bf16 parts over a 3*dp reduction.  The tensor core's fp32
// accumulation loses a little with every step of a long chain (measured on
// B300: logit error up to 1.3e-4 over one 192-block chain, 1e-5 over chains of
// about 20 blocks, where the fp32 CUDA-core router reaches 1.4e-5), so the
// reduction is cut into S chains of at most 16 K blocks, each written as an
// fp32 partial plane and summed in fixed order by the softmax kernel.  Small T
// uses more, shorter chains to fill the SMs.
bool tc_router(const moe_config *c) {
    return c->dtype == MOE_DTYPE_BF16 && c->n_experts > 32 && c->n_experts % 4 == 0;
}
long long router_dp(const moe_config *c) { return (c->d_model + 63) / 64 * 64; }
constexpr int kRouterChainBlocks = 16;
int router_splits(const moe_config *c) {
    const long long tiles = ((long long)c->T + 127) / 128 * ((c->n_experts + 255) / 256);
    const long long nk = 3 * router_dp(c) / 64;
    long long S = (nk + kRouterChainBlocks - 1) / kRouterChainBlocks;
    if (tiles > 0) S = std::max<long long>(S, std::min<long long>((296 + tiles - 1) / tiles,
                                                                    std::max<long long>(1, nk / 4)));
    const long long kbps = (nk + S - 1) / S;
    return (int)((nk + kbps - 1) / kbps);
}

Layout layout(const moe_config *c) {
    const Sizes s = sizes(c);
    const size_t eb = elem_bytes(c->dtype);
    const long long rb = router_blocks((int)s.T, (int)s.E);
    const long long nb = dispatch_blocks(s.Tk);
    const long long mt = max_tiles(s.Tk, (int)s.E, kSimtBM);
    const long long mts = max_tiles(s.T, 1, kSimtBM);
    Layout L;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o += align_up(bytes); return r; };
    L.p_partial = take(sizeof(float) * rb * s.E);
    L.probsT = take(sizeof(float) * s.E * s.T);
    L.hist = take(sizeof(int32_t) * nb * s.E);
    L.block_base = take(sizeof(int32_t) * nb * s.E);
    L.idx = take(sizeof(int32_t) * s.Tk);
    L.w = take(sizeof(float) * s.Tk);
    L.counts = take(sizeof(int32_t) * s.E);
    L.offsets = take(sizeof(int32_t) * (s.E + 1));
    L.perm = take(sizeof(int32_t) * s.Tk);
    L.inv = take(sizeof(int32_t) * s.Tk);
    L.ndrop = take(sizeof(int32_t));
    L.pvec = take(sizeof(float) * s.E);
    L.sbias = take(sizeof(float) * s.E);
    L.idx_unb = take(sizeof(int32_t) * s.Tk);
    L.tile_e = take(sizeof(int32_t) * mt);
    L.tile_m0 = take(sizeof(int32_t) * mt);
    L.tile_start = take(sizeof(int32_t) * (s.E + 1));
    L.ntiles = take(sizeof(int32_t));
    L.sh_offsets = take(sizeof(int32_t) * 2);
    L.sh_tile_e = take(sizeof(int32_t) * mts);
    L.sh_tile_m0 = take(sizeof(int32_t) * mts);
    L.sh_tile_start = take(sizeof(int32_t) * 2);
    L.sh_ntiles = take(sizeof(int32_t));
    L.xs = take(eb * s.Tk * s.d);
    L.h = take(eb * s.Tk * s.F);
    L.out_sorted = take(sizeof(float) * s.Tk * s.d);
    L.sh_h = take(eb * s.T * s.Fs);
    L.sh_out = take(sizeof(float) * s.T * s.d);
    const bool rt = tc_router(c);
    L.rt_wsplit = take(rt ? 2 * s.E * 3 * router_dp(c) : 0);
    L.rt_logits = take(rt ? sizeof(float) * router_splits(c) * s.T * s.E : 0);
    L.rt_offsets = take(sizeof(int32_t) * 2);
    L.rt_tile_e = take(sizeof(int32_t) * max_tiles(s.T, 1, kTcBM));
    L.rt_tile_start = take(sizeof(int32_t) * 2);
    L.rt_ntiles = take(sizeof(int32_t));
    L.total = o;
    return L;
}

int check_cfg(const moe_config *c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->T < 0 || c->d_model <= 0 || c->n_experts < 1 || c->n_experts > 1024) return MOE_ERR_INVALID_ARG;
    if (c->top_k < 1 || c->top_k > c->n_experts || c->top_k > 16) return MOE_ERR_INVALID_ARG;
    if (c->d_ff <= 0 || c->d_ff_shared < 0) return MOE_ERR_INVALID_ARG;
    if (c->act != MOE_ACT_RELU && c->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_DTYPE_FP32 && c->dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->out_dtype != MOE_DTYPE_FP32 && c->out_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->select_space != MOE_SELECT_PROBS && c->select_space != MOE_SELECT_LOGITS) return MOE_ERR_INVALID_ARG;
    if (c->quantile_balance != 0 && c->quantile_balance != 1) return MOE_ERR_INVALID_ARG;
    if (!(c->capacity_factor == c->capacity_factor)) return MOE_ERR_INVALID_ARG;   // NaN
    const int vec = 16 / elem_bytes(c->dtype);
    if (c->d_model % vec || c->d_ff % vec || c->d_ff_shared % vec) return MOE_ERR_INVALID_ARG;
    if ((long long)c->T * c->top_k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
    if (c->quantile_balance && c->select_space != MOE_SELECT_PROBS) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

#define MOE_REQUIRE(cond) do { if (!(cond)) return MOE_ERR_INVALID_ARG; } while (0)
#define MOE_PTR(p) MOE_REQUIRE((p) != nullptr && aligned16(p))
#define MOE_OPT_PTR(p) MOE_REQUIRE((p) == nullptr || aligned16(p))
#define MOE_CUDA(call) do { cudaError_t e_ = (call); if (e_ != cudaSuccess) return MOE_ERR_CUDA; } while (0)

template <typename P> P *at(void *ws, size_t off) {
    return reinterpret_cast<P *>(static_cast<char *>(ws) + off);
}

long long capacity_of(const moe_config *c) {
    const long long Tk = (long long)c->T * c->top_k;
    if (!(c->capacity_factor > 0.f)) return Tk;
    return (long long)ceil((double)c->capacity_factor * (double)c->T * (double)c->top_k /
                           (double)c->n_experts);
}

__global__ void set_pair_kernel(int32_t *p, int a, int b) { p[0] = a; p[1] = b; }

// Optional per-stage event timing of moe_layer_forward (host state, not
// thread-safe; meant for benchmarking).
struct StageTimer {
    bool on = false;
    struct Rec { int stage; cudaEvent_t a, b; };
    std::vector<Rec> recs;
    std::vector<cudaEvent_t> pool;
    long long calls = 0;
    cudaEvent_t get() {
        if (!pool.empty()) { cudaEvent_t e = pool.back(); pool.pop_back(); return e; }
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        return e;
    }
    void recycle() {
        for (auto &r : recs) { pool.push_back(r.a); pool.push_back(r.b); }
        recs.clear();
        calls = 0;
    }
} g_timer;

cudaEvent_t stage_begin(cudaStream_t st) {
    if (!g_timer.on) return nullptr;
    cudaEvent_t e = g_timer.get();
    if (e) cudaEventRecord(e, st);
    return e;
}
void stage_end(int stage, cudaEvent_t a, cudaStream_t st) {
    if (!a) return;
    cudaEvent_t b = g_timer.get();
    if (!b) return;
    cudaEventRecord(b, st);
    g_timer.recs.push_back({stage, a, b});
}

// Router incl. quantile balancing; p (mean probs) when p_out != NULL.
int run_router(const moe_config *c, const void *x, const float *w_r, const float *logit_bias,
               const float *select_bias, int32_t *idx, float *w, float *probs, float *p_out,
               float *sbias_out, bool want_probsT, void *ws, const Layout &L, cudaStream_t st) {
    const Sizes s = sizes(c);
    RouterArgs a;
    a.x = x; a.w_r = w_r; a.logit_bias = logit_bias;
    a.select_bias = c->quantile_balance ? nullptr : select_bias;
    a.T = (int)s.T; a.d = (int)s.d; a.E = (int)s.E; a.k = (int)s.k;
    a.select_space = c->select_space;
    a.do_select = c->quantile_balance ? 0 : 1;
    a.idx = idx; a.w = w; a.probs = probs;
    a.probsT = (c->quantile_balance || want_probsT) ? at<float>(ws, L.probsT) : nullptr;
    a.p_partial = at<float>(ws, L.p_partial);
    if (tc_router(c)) {
        const int dp = (int)router_dp(c);
        const int S = router_splits(c);
        __nv_bfloat16 *wsplit = at<__nv_bfloat16>(ws, L.rt_wsplit);
        float *part = at<float>(ws, L.rt_logits);
        int32_t *off = at<int32_t>(ws, L.rt_offsets);
        int32_t *te = at<int32_t>(ws, L.rt_tile_e), *ts = at<int32_t>(ws, L.rt_tile_start);
        int32_t *nt = at<int32_t>(ws, L.rt_ntiles);
        MOE_CUDA(launch_split_router_weight(w_r, a.E, a.d, dp, wsplit, st));
        set_pair_kernel<<<1, 1, 0, st>>>(off, 0, a.T);
        note_launch();
        MOE_CUDA(cudaGetLastError());
        MOE_CUDA(launch_build_tiles(off, 1, kTcBM, te, nullptr, ts, nt, st));
        MOE_CUDA(launch_tc_gemm(GEMM_DOWN, x, s.T, a.d, wsplit, nullptr, 1, a.E, a.E, 3 * dp, dp,
                                S, s.T * s.E, te, ts, nt, off, part, a.E, st));
        MOE_CUDA(launch_router_from_logits(a, part, S, st));
    } else {
        MOE_CUDA(launch_router(a, c->dtype, st));
    }
    if (p_out && s.T > 0)
        MOE_CUDA(launch_p_finalize(a.p_partial, router_blocks(a.T, a.E), a.E, a.T, p_out, st));
    if (c->quantile_balance && s.T > 0) {
        // Linear interpolation between order statistics: h = (T-1) q,
        // q = 1 - k/E, lo = floor(h), frac = h - lo.
        const double q = 1.0 - (double)s.k / (double)s.E;
        const double h = (double)(s.T - 1) * q;
        const double lo = floor(h);
        MOE_CUDA(launch_quantile_bias(a.probsT, a.T, a.E, (long long)lo, (float)(h - lo),
                                      sbias_out, st));
        MOE_CUDA(launch_select_from_probsT(a.probsT, sbias_out, a.T, a.E, a.k, idx, w, st));
    }
    return MOE_OK;
}

// Grouped expert FFN over the dispatched rows; out_sorted fp32.
// bf16: gather the rows into x_sorted, tcgen05 up (+activation) into h, tcgen05
// down into out_sorted.  fp32: SIMT GEMMs reading x through perm directly.
int run_experts(const moe_config *c, const void *x, const int32_t *perm, const int32_t *offsets,
                const void *w1, const void *w3, const void *w2, float *out_sorted, void *ws,
                const Layout &L, cudaStream_t st) {
    const Sizes s = sizes(c);
    if (s.Tk == 0) return MOE_OK;
    int32_t *tile_e = at<int32_t>(ws, L.tile_e), *tile_m0 = at<int32_t>(ws, L.tile_m0);
    int32_t *tile_start = at<int32_t>(ws, L.tile_start), *ntiles = at<int32_t>(ws, L.ntiles);
    const int up_mode = c->act == MOE_ACT_SWIGLU ? GEMM_UP_SWIGLU : GEMM_UP_RELU;
    if (c->dtype == MOE_DTYPE_BF16) {
        void *xs = at<void>(ws, L.xs), *h = at<void>(ws, L.h);
        cudaEvent_t ev = stage_begin(st);
        MOE_CUDA(launch_gather_rows(x, 2, (int)s.d, perm, offsets + s.E, (int)s.k, s.Tk, xs, st));
        MOE_CUDA(launch_build_tiles(offsets, (int)s.E, kTcBM, tile_e, nullptr, tile_start, ntiles,
                                    st));
        stage_end(MOE_STAGE_GATHER, ev, st);
        ev = stage_begin(st);
        MOE_CUDA(launch_tc_gemm(up_mode, xs, s.Tk, (int)s.d, w1, w3, (int)s.E, (int)s.F,
                                (int)s.F, (int)s.d, (int)s.d, 1, 0, tile_e, tile_start, ntiles,
                                offsets, h, (int)s.F, st));
        stage_end(MOE_STAGE_UP, ev, st);
        ev = stage_begin(st);
        MOE_CUDA(launch_tc_gemm(GEMM_DOWN, h, s.Tk, (int)s.F, w2, nullptr, (int)s.E, (int)s.d,
                                (int)s.d, (int)s.F, (int)s.F, 1, 0, tile_e, tile_start, ntiles,
                                offsets, out_sorted, (int)s.d, st));
        stage_end(MOE_STAGE_DOWN, ev, st);
        return MOE_OK;
    }
    cudaEvent_t ev = stage_begin(st);
    MOE_CUDA(launch_build_tiles(offsets, (int)s.E, kSimtBM, tile_e, tile_m0, nullptr, ntiles, st));
    stage_end(MOE_STAGE_GATHER, ev, st);
    ev = stage_begin(st);
    GroupedGemmArgs up;
    up.A = x; up.a_gather = perm; up.gather_k = (int)s.k;
    up.B1 = w1; up.B3 = w3; up.b_expert_stride = s.F * s.d; up.N = (int)s.F; up.K = (int)s.d;
    up.C = at<void>(ws, L.h); up.ldc = (int)s.F;
    up.tile_e = tile_e; up.tile_m0 = tile_m0; up.n_tiles = ntiles; up.offsets = offsets;
    up.max_tiles = max_tiles(s.Tk, (int)s.E, kSimtBM);
    MOE_CUDA(launch_simt_gemm(up, up_mode, c->dtype, st));
    stage_end(MOE_STAGE_UP, ev, st);
    ev = stage_begin(st);
    GroupedGemmArgs dn = up;
    dn.A = at<void>(ws, L.h); dn.a_gather = nullptr; dn.gather_k = 1;
    dn.B1 = w2; dn.B3 = nullptr; dn.b_expert_stride = s.d * s.F; dn.N = (int)s.d; dn.K = (int)s.F;
    dn.C = out_sorted; dn.ldc = (int)s.d;
    MOE_CUDA(launch_simt_gemm(dn, GEMM_DOWN, c->dtype, st));
    stage_end(MOE_STAGE_DOWN, ev, st);
    return MOE_OK;
}

// Shared expert (SwiGLU) on all T rows -> sh_out fp32 [T, d]: the same
// grouped kernels with one group {0, T} and x read in place.
int run_shared(const moe_config *c, const void *x, const void *ws1, const void *ws3,
               const void *ws2, void *ws, const Layout &L, cudaStream_t st) {
    const Sizes s = sizes(c);
    if (s.T == 0) return MOE_OK;
    int32_t *off = at<int32_t>(ws, L.sh_offsets);
    set_pair_kernel<<<1, 1, 0, st>>>(off, 0, (int)s.T);
    note_launch();
    MOE_CUDA(cudaGetLastError());
    int32_t *te = at<int32_t>(ws, L.sh_tile_e), *tm = at<int32_t>(ws, L.sh_tile_m0);
    int32_t *ts = at<int32_t>(ws, L.sh_tile_start), *nt = at<int32_t>(ws, L.sh_ntiles);
    void *h = at<void>(ws, L.sh_h);
    float *o = at<float>(ws, L.sh_out);
    if (c->dtype == MOE_DTYPE_BF16) {
        MOE_CUDA(launch_build_tiles(off, 1, kTcBM, te, nullptr, ts, nt, st));
        MOE_CUDA(launch_tc_gemm(GEMM_UP_SWIGLU, x, s.T, (int)s.d, ws1, ws3, 1, (int)s.Fs,
                                (int)s.Fs, (int)s.d, (int)s.d, 1, 0, te, ts, nt, off, h,
                                (int)s.Fs, st));
        MOE_CUDA(launch_tc_gemm(GEMM_DOWN, h, s.T, (int)s.Fs, ws2, nullptr, 1, (int)s.d,
                                (int)s.d, (int)s.Fs, (int)s.Fs, 1, 0, te, ts, nt, off, o,
                                (int)s.d, st));
        return MOE_OK;
    }
    MOE_CUDA(launch_build_tiles(off, 1, kSimtBM, te, tm, nullptr, nt, st));
    GroupedGemmArgs up;
    up.A = x; up.a_gather = nullptr; up.gather_k = 1;
    up.B1 = ws1; up.B3 = ws3; up.b_expert_stride = 0; up.N = (int)s.Fs; up.K = (int)s.d;
    up.C = h; up.ldc = (int)s.Fs;
    up.tile_e = te; up.tile_m0 = tm; up.n_tiles = nt; up.offsets = off;
    up.max_tiles = max_tiles(s.T, 1, kSimtBM);
    MOE_CUDA(launch_simt_gemm(up, GEMM_UP_SWIGLU, c->dtype, st));
    GroupedGemmArgs dn = up;
    dn.A = h; dn.B1 = ws2; dn.B3 = nullptr; dn.N = (int)s.d; dn.K = (int)s.Fs;
    dn.C = o; dn.ldc = (int)s.d;
    MOE_CUDA(launch_simt_gemm(dn, GEMM_DOWN, c->dtype, st));
    return MOE_OK;
}

// Fixed scratch of moe_dispatch_static (no workspace, no allocation).  In host
// code g_dispatch_scratch only names the symbol; its device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
__device__ __align__(256) unsigned char g_dispatch_scratch[MOE_DISPATCH_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

int dispatch_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p)
            return MOE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" {

int64_t moe_capacity(const moe_config *cfg) {
    if (check_cfg(cfg) != MOE_OK) return -1;
    return capacity_of(cfg);
}

size_t moe_workspace_size(const moe_config *cfg) {
    if (check_cfg(cfg) != MOE_OK) return 0;
    return layout(cfg).total;
}

int moe_router_topk(const moe_config *cfg, const void *x, const float *w_r,
                    const float *logit_bias, const float *select_bias, int32_t *topk_idx,
                    float *topk_w, float *probs, float *p_mean, float *select_bias_out, void *ws,
                    size_t ws_bytes, moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    if (cfg->T == 0) return MOE_OK;
    MOE_PTR(x); MOE_PTR(w_r); MOE_PTR(topk_idx); MOE_PTR(topk_w); MOE_PTR(ws);
    MOE_OPT_PTR(logit_bias); MOE_OPT_PTR(select_bias); MOE_OPT_PTR(probs); MOE_OPT_PTR(p_mean);
    if (cfg->quantile_balance) MOE_PTR(select_bias_out);
    const Layout L = layout(cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    return run_router(cfg, x, w_r, logit_bias, select_bias, topk_idx, topk_w, probs, p_mean,
                      select_bias_out, false, ws, L, (cudaStream_t)stream);
}

int moe_dispatch(const moe_config *cfg, const int32_t *topk_idx, int32_t *counts,
                 int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *n_dropped, void *ws,
                 size_t ws_bytes, moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    MOE_PTR(counts); MOE_PTR(offsets); MOE_PTR(n_dropped); MOE_PTR(ws);
    if (cfg->T > 0) { MOE_PTR(topk_idx); MOE_PTR(perm); MOE_PTR(inv); }
    const Layout L = layout(cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    const Sizes s = sizes(cfg);
    MOE_CUDA(launch_dispatch(topk_idx, s.Tk, (int)s.E, (int)s.k, capacity_of(cfg),
                             at<int32_t>(ws, L.hist), at<int32_t>(ws, L.block_base), counts,
                             offsets, perm, inv, n_dropped, (cudaStream_t)stream));
    return MOE_OK;
}

int moe_dispatch_static(const moe_config *cfg, const int32_t *topk_idx, int32_t *counts,
                        int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *n_dropped,
                        moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    MOE_PTR(counts); MOE_PTR(offsets); MOE_PTR(n_dropped);
    if (cfg->T > 0) { MOE_PTR(topk_idx); MOE_PTR(perm); MOE_PTR(inv); }
    const Sizes s = sizes(cfg);
    const size_t half = sizeof(int32_t) * (size_t)dispatch_blocks(s.Tk) * (size_t)s.E;
    if (2 * half > MOE_DISPATCH_STATIC_SCRATCH_BYTES) return MOE_ERR_TOO_LARGE;
    void *scratch = nullptr;
    rc = dispatch_scratch(&scratch);
    if (rc != MOE_OK) return rc;
    int32_t *hist = static_cast<int32_t *>(scratch);
    int32_t *base = reinterpret_cast<int32_t *>(static_cast<char *>(scratch) + half);
    MOE_CUDA(launch_dispatch(topk_idx, s.Tk, (int)s.E, (int)s.k, capacity_of(cfg), hist, base,
                             counts, offsets, perm, inv, n_dropped, (cudaStream_t)stream));
    return MOE_OK;
}

int moe_expert_ffn(const moe_config *cfg, const void *x, const int32_t *perm,
                   const int32_t *offsets, const void *w1, const void *w3, const void *w2,
                   float *out_sorted, void *ws, size_t ws_bytes, moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    if (cfg->T == 0) return MOE_OK;
    MOE_PTR(x); MOE_PTR(perm); MOE_PTR(offsets); MOE_PTR(w1); MOE_PTR(w2); MOE_PTR(out_sorted);
    MOE_PTR(ws);
    if (cfg->act == MOE_ACT_SWIGLU) MOE_PTR(w3);
    const Layout L = layout(cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    return run_experts(cfg, x, perm, offsets, w1, w3, w2, out_sorted, ws, L,
                       (cudaStream_t)stream);
}

int moe_combine(const moe_config *cfg, const float *out_sorted, const int32_t *inv,
                const float *topk_w, const float *shared_out, void *y, moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    if (cfg->T == 0) return MOE_OK;
    MOE_PTR(out_sorted); MOE_PTR(inv); MOE_PTR(topk_w); MOE_PTR(y); MOE_OPT_PTR(shared_out);
    MOE_CUDA(launch_combine(out_sorted, inv, topk_w, shared_out, cfg->T, cfg->top_k,
                            cfg->d_model, cfg->out_dtype, y, (cudaStream_t)stream));
    return MOE_OK;
}

int moe_load_stats(const moe_config *cfg, const int32_t *topk_idx, const float *probs,
                   int32_t *counts, float *f, float *p, float *aux, float *load_max_over_mean,
                   void *ws, size_t ws_bytes, moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    MOE_PTR(f); MOE_PTR(p); MOE_PTR(aux); MOE_PTR(ws);
    MOE_OPT_PTR(counts); MOE_OPT_PTR(load_max_over_mean);
    if (cfg->T > 0) { MOE_PTR(topk_idx); MOE_PTR(probs); }
    const Layout L = layout(cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    const Sizes s = sizes(cfg);
    cudaStream_t st = (cudaStream_t)stream;
    int32_t *cnt = counts ? counts : at<int32_t>(ws, L.counts);
    MOE_CUDA(launch_histogram(topk_idx, s.Tk, (int)s.E, at<int32_t>(ws, L.hist), cnt, st));
    float *part = at<float>(ws, L.p_partial);
    MOE_CUDA(launch_prob_partials(probs, (int)s.T, (int)s.E, part, st));
    MOE_CUDA(launch_p_finalize(part, (int)((s.T + 31) / 32), (int)s.E, (int)s.T, p, st));
    MOE_CUDA(launch_stats_finalize(cnt, p, (int)s.T, (int)s.E, (int)s.k, f, nullptr, aux,
                                   load_max_over_mean, st));
    return MOE_OK;
}

int moe_layer_forward(const moe_config *cfg, const void *x, const moe_layer_weights *wts,
                      const moe_layer_outputs *out, void *ws, size_t ws_bytes,
                      moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    MOE_REQUIRE(wts != nullptr && out != nullptr);
    MOE_PTR(ws);
    if (cfg->T > 0) { MOE_PTR(x); MOE_PTR(out->y); }
    MOE_PTR(wts->w_r); MOE_PTR(wts->w1); MOE_PTR(wts->w2);
    if (cfg->act == MOE_ACT_SWIGLU) MOE_PTR(wts->w3);
    MOE_OPT_PTR(wts->logit_bias); MOE_OPT_PTR(wts->select_bias);
    if (cfg->d_ff_shared > 0) { MOE_PTR(wts->ws1); MOE_PTR(wts->ws3); MOE_PTR(wts->ws2); }
    MOE_OPT_PTR(out->topk_idx); MOE_OPT_PTR(out->topk_w); MOE_OPT_PTR(out->counts);
    MOE_OPT_PTR(out->n_dropped); MOE_OPT_PTR(out->f); MOE_OPT_PTR(out->p); MOE_OPT_PTR(out->aux);
    MOE_OPT_PTR(out->load_max_over_mean); MOE_OPT_PTR(out->select_bias_out);
    MOE_OPT_PTR(out->counts_unbiased);
    const Layout L = layout(cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const Sizes s = sizes(cfg);

    int32_t *idx = out->topk_idx ? out->topk_idx : at<int32_t>(ws, L.idx);
    float *w = out->topk_w ? out->topk_w : at<float>(ws, L.w);
    float *p = out->p ? out->p : at<float>(ws, L.pvec);
    int32_t *counts = out->counts ? out->counts : at<int32_t>(ws, L.counts);
    int32_t *ndrop = out->n_dropped ? out->n_dropped : at<int32_t>(ws, L.ndrop);
    float *sbias = out->select_bias_out ? out->select_bias_out : at<float>(ws, L.sbias);
    int32_t *offsets = at<int32_t>(ws, L.offsets);
    int32_t *perm = at<int32_t>(ws, L.perm), *inv = at<int32_t>(ws, L.inv);
    float *out_sorted = at<float>(ws, L.out_sorted);

    const bool biased = cfg->quantile_balance || wts->select_bias != nullptr;
    const bool want_unb = out->counts_unbiased != nullptr;

    if (g_timer.on) ++g_timer.calls;
    cudaEvent_t ev = stage_begin(st);
    if (s.T > 0) {
        rc = run_router(cfg, x, wts->w_r, wts->logit_bias, wts->select_bias, idx, w, nullptr, p,
                        sbias, want_unb && biased, ws, L, st);
        if (rc != MOE_OK) return rc;
    }
    stage_end(MOE_STAGE_ROUTER, ev, st);
    ev = stage_begin(st);
    MOE_CUDA(launch_dispatch(idx, s.Tk, (int)s.E, (int)s.k, capacity_of(cfg),
                             at<int32_t>(ws, L.hist), at<int32_t>(ws, L.block_base), counts,
                             offsets, perm, inv, ndrop, st));
    stage_end(MOE_STAGE_DISPATCH, ev, st);
    ev = stage_begin(st);
    if (want_unb) {
        if (biased && s.T > 0) {
            int32_t *iu = at<int32_t>(ws, L.idx_unb);
            MOE_CUDA(launch_select_from_probsT(at<float>(ws, L.probsT), nullptr, (int)s.T,
                                               (int)s.E, (int)s.k, iu, nullptr, st));
            MOE_CUDA(launch_histogram(iu, s.Tk, (int)s.E, at<int32_t>(ws, L.hist),
                                      out->counts_unbiased, st));
        } else {
            MOE_CUDA(cudaMemcpyAsync(out->counts_unbiased, counts, sizeof(int32_t) * s.E,
                                     cudaMemcpyDeviceToDevice, st));
        }
    }
    if (s.T == 0) {
        MOE_CUDA(cudaMemsetAsync(p, 0, sizeof(float) * s.E, st));
    }
    MOE_CUDA(launch_stats_finalize(counts, p, (int)s.T, (int)s.E, (int)s.k, out->f, nullptr,
                                   out->aux, out->load_max_over_mean, st));
    stage_end(MOE_STAGE_STATS, ev, st);
    if (s.T == 0) return MOE_OK;
    rc = run_experts(cfg, x, perm, offsets, wts->w1, wts->w3, wts->w2, out_sorted, ws, L, st);
    if (rc != MOE_OK) return rc;
    const float *shared = nullptr;
    if (s.Fs > 0) {
        ev = stage_begin(st);
        rc = run_shared(cfg, x, wts->ws1, wts->ws3, wts->ws2, ws, L, st);
        if (rc != MOE_OK) return rc;
        stage_end(MOE_STAGE_SHARED, ev, st);
        shared = at<float>(ws, L.sh_out);
    }
    ev = stage_begin(st);
    MOE_CUDA(launch_combine(out_sorted, inv, w, shared, (int)s.T, (int)s.k, (int)s.d,
                            cfg->out_dtype, out->y, st));
    stage_end(MOE_STAGE_COMBINE, ev, st);
    return MOE_OK;
}

int moe_device_status(moe_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    if (v & kErrTimeout) return MOE_ERR_DEVICE_TIMEOUT;
    if (v & kErrBadIndex) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

int64_t moe_kernel_launches(void) {
    return __atomic_load_n(&g_kernel_launches, __ATOMIC_RELAXED);
}

int moe_stage_timing_enable(int on) {
    for (auto &r : g_timer.recs) cudaEventSynchronize(r.b);
    g_timer.recycle();
    g_timer.on = on != 0;
    return MOE_OK;
}

int moe_stage_timing_read(double *stage_ms, int64_t *calls) {
    if (!stage_ms || !calls) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < MOE_NUM_STAGES; ++i) stage_ms[i] = 0.0;
    int rc = MOE_OK;
    for (auto &r : g_timer.recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess ||
            cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
            rc = MOE_ERR_CUDA;
            continue;
        }
        stage_ms[r.stage] += ms;
    }
    *calls = g_timer.calls;
    g_timer.recycle();
    return rc;
}

const char *moe_strerror(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or option";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_TIMEOUT: return "a device-side bounded wait timed out";
        case MOE_ERR_TOO_LARGE:
            return "problem exceeds the fixed scratch of moe_dispatch_static";
        default: return "unknown status";
    }
}

}  // extern "C"
