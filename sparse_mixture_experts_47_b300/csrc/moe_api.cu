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
#include "reroute.cu"
#include "expert_choice.cu"
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
        rt_logits, rt_offsets, rt_tile_e, rt_tile_start, rt_ntiles, up_part, sh_up_part,
        ent_partial, row_stats, cand_idx, cand_w, rr_slot_e, rr_slot_w, rr_served, rr_nxt,
        rr_filled, rr_filled_before, slot_w, ec_row_w, ec_rowidx, ec_tok_cnt, ec_tok_start,
        ec_tok_rows, probs_rows, total;
};

long long capacity_of(const moe_config *c) {
    const long long Tk = (long long)c->T * c->top_k;
    if (!(c->capacity_factor > 0.f)) return Tk;
    return (long long)ceil((double)c->capacity_factor * (double)c->T * (double)c->top_k /
                           (double)c->n_experts);
}

bool expert_choice(const moe_config *c) { return c->routing == MOE_ROUTING_EXPERT_CHOICE; }

// Rows each expert takes under expert choice: min(C, T).
long long ec_rows_per_expert(const moe_config *c) {
    return std::min<long long>(capacity_of(c), c->T);
}

// Tk: token-choice slots (T*k).  R: rows of the grouped layout, at most Tk
// for token choice, E * min(C, T) for expert choice.
struct Sizes {
    long long T, d, E, k, F, Fs, Tk, R;
};

Sizes sizes(const moe_config *c) {
    Sizes s;
    s.T = c->T; s.d = c->d_model; s.E = c->n_experts; s.k = c->top_k; s.F = c->d_ff;
    s.Fs = c->d_ff_shared; s.Tk = s.T * s.k;
    s.R = expert_choice(c) ? s.E * ec_rows_per_expert(c) : s.Tk;
    return s;
}

// Router logits on the tensor cores (bf16 x, E > 32, E % 4 == 0): W_r split
// into kRouterParts bf16 parts over a kRouterParts*dp reduction.  Two parts
// (hi + lo) leave a residual of at most 2^-18 |w| per weight, a logit error
// of about 2e-6 rms at d = 4096, the size of the fp32 CUDA-core router's
// rounding.  The tensor
// core's fp32 accumulation loses a little with every step of a long chain
// (measured on B300: logit error up to 1.3e-4 over one 192-block chain, 1e-5
// over chains of about 20 blocks, where the fp32 CUDA-core router reaches
// 1.4e-5), so the reduction is cut into S chains of at most 16 K blocks.
// Groups of 4 chains are summed on chip in chain order (GEMM_LOGITS), each
// group into its own fp32 plane, and the softmax adds the planes in group
// order.  Chains and groups depend on d only, so a token's logits do not
// depend on the batch it comes in (batch invariance).
// The router's softmax kernel also takes the top-k, unless the selection
// comes later (quantile balance, expert choice).
bool router_selects(const moe_config *c) {
    return !(c->quantile_balance || c->routing == MOE_ROUTING_EXPERT_CHOICE);
}
bool tc_router(const moe_config *c) { return router_on_tensor_cores(c->n_experts, c->dtype); }
long long router_dp(const moe_config *c) { return (c->d_model + 63) / 64 * 64; }
constexpr int kRouterChainBlocks = 16;
constexpr int kRouterParts = 2;
constexpr int kRouterGroupChains = 4;
// Chains: S equal K ranges of at most kRouterChainBlocks K blocks.
int router_chain_kb(const moe_config *c) {
    const long long nk = kRouterParts * router_dp(c) / 64;
    const long long S = (nk + kRouterChainBlocks - 1) / kRouterChainBlocks;
    return (int)((nk + S - 1) / S);
}
// Groups of up to kRouterGroupChains consecutive chains: one work item per
// group and tile, one fp32 plane per group (summed in group order by the
// softmax).  Both depend on d only.
int router_groups(const moe_config *c) {
    const long long nk = kRouterParts * router_dp(c) / 64;
    const long long kb = router_chain_kb(c);
    const long long chains = (nk + kb - 1) / kb;
    return (int)((chains + kRouterGroupChains - 1) / kRouterGroupChains);
}
// How the grouped GEMMs of one expert FFN run.  nt = 0: 128 token rows per
// tile on the MMA's M side.  nt = 16/32/64: weights on the M side and nt
// token rows per tile, for a few rows per expert, where the layer streams
// weights from HBM and a 128-row token tile would be mostly padding.  With
// few tiles the reduction is split (s_up, s_down) so that every SM streams
// weights; the splits' fp32 partial sums are added in split order later.
// nt_down = 256 (with nt = 0): the down projection runs on tiles of up to 256
// rows whose MMA N is each tile's row count rounded to 16.
struct FfnPlan {
    int nt, s_up, s_down;
    int bn_up, bn_down;     // nt = 0: MMA N (256, or 128 when tiles are few)
    int nt_down;            // geometry of the down projection
    int mh_down;            // nt_down = 0: token-row tiling (TILE_ROWS_*)
    int mh_up;              // nt = 0: token-row tiling of the up projection
};
constexpr int kPlanSMs = 148;   // SM count the split choice assumes (B300)
constexpr int kVarTileRows = 256;
// Measured on B300: with the same work per tile, the per-tile-width geometry
// runs the down projection 1.26x slower than 128-row tiles (DeepSeek shape,
// at most 256 rows per expert), and 1.49x faster where the last 128-row tile
// of every expert is mostly padding (896 experts of about 146 rows).  It is
// chosen when the padding of 128-row tiles exceeds its own by more than this.
constexpr double kVarPadGain = 1.3;
// 256-row tiles for the down projection (two M = 128 MMAs per weight stage;
// one TMEM accumulator, so the epilogue is not overlapped) when the experts
// hold at least kWideMinRows rows on average and the reduction is at least
// kWideMinK long.  Measured at the Mixtral shape (K = 14336): down 2.70 ->
// 2.41 ms at T = 16384; the SwiGLU up projection (K = 4096) went 5.0 ->
// 6.1 ms, its unoverlapped epilogue being a fifth of a tile.
constexpr long long kWideMinRows = 512;
constexpr long long kWideMinK = 8192;
// 256-row tiles on SM pairs (cta_group::2: 32 KB stages per SM, two
// accumulators) for an nt = 0, N = 256 projection whose experts hold at least
// kPairMinRows rows on average, or whose loads are balanced by construction
// (quantile balancing, expert choice).  Measured on B300 against the one-SM
// tiles: Switch T = 8192 (1024 rows per expert) 0.184 -> 0.170 ms and Mixtral
// T = 4096 2.06 -> 2.00 ms at the same clock; Mixtral T = 16384 5 % fewer
// cycles, about even in time under the power cap; the 896-expert layer
// (quantile-balanced, about 146 rows per expert, bound by HBM) 3.57 -> 3.49 ms,
// one 256-row tile per expert reading each weight tile once instead of two
// 128-row tiles reading it twice.  DeepSeek T = 8192 (256 rows on average,
// most experts far fewer under its selection bias) and its capacity-limited
// variant ran 10-15 % slower on pairs, at lower clocks: the padding rows of
// light experts' 256-row tiles cost MMA work and power.
constexpr long long kPairMinRows = 512;
static int g_pair_policy = 0;
static bool use_pair(long long per, int bn, int splits, bool balanced) {
    if (g_pair_policy < 0 || bn != 256 || splits != 1) return false;
    return g_pair_policy > 0 || per >= kPairMinRows || balanced;
}
// The up projection on the per-tile-width geometry (weights on the MMA's M
// side, up to 256 of one expert's rows on its N side, rounded up to 16) only
// on request (g_var_up_policy 1: wherever the experts average more than 64
// rows; 0 and -1: never).  Measured on the 896-expert layer (about 146 rows
// per expert), whose SwiGLU up projection streams 7.5 GB of W1 and W3 and is
// bound by HBM: 1.56 ms against 1.46 ms on 256-row SM-pair tiles.  One
// SwiGLU tile fills the 512 TMEM columns (no second accumulator), and its
// 64 KB stages leave room for 3 (the pairs keep 7 of 32 KB in flight).
static int g_var_up_policy = 0;

// Split the reduction only when the tiles do not fill the SMs once, and then
// only up to one round of work items: measured at the Mixtral shape, a split
// that spreads the items over more rounds, or any split of the up projection
// at T = 1 and 16, costs more in partial sums than it gains in balance (a
// split chosen to fill the rounds to 95 %, 7-way for the up projection at
// T = 1: 0.152 -> 0.163 ms per layer), while splitting the down projection at
// T = 1 (64 tiles) in two cuts it from 68 to 45 us.
int split_count(long long tiles, long long nk) {
    if (tiles <= 0 || nk <= 0 || tiles >= kPlanSMs) return 1;
    long long S = kPlanSMs / tiles;
    S = std::min<long long>(S, std::min<long long>(16, std::max<long long>(1, nk / 8)));
    const long long kbps = (nk + S - 1) / S;
    return (int)((nk + kbps - 1) / kbps);
}

// rows: dispatched rows (T*k routed, T shared); groups: experts; K = d.
FfnPlan ffn_plan(const moe_config *c, long long rows, long long groups, long long F,
                 bool swiglu) {
    FfnPlan p{0, 1, 1, 256, 256, 0, TILE_ROWS_128, TILE_ROWS_128};
    if (c->dtype != MOE_DTYPE_BF16 || rows <= 0 || F <= 0) return p;
    const long long d = c->d_model;
    const long long active = std::min(groups, rows);
    const long long per = (rows + active - 1) / active;
    const long long up_cols = swiglu ? 128 : 256;
    const long long normal_items = active * ((per + 127) / 128) * ((F + up_cols - 1) / up_cols);
    if (per <= 16) p.nt = 16;
    else if (per <= 32) p.nt = 32;
    else if (per <= 64 || (per <= 256 && normal_items < kPlanSMs)) p.nt = 64;
    else {
        // 128-row tiles; halve the MMA N when there are too few output tiles
        // (down projection: fewer than one round of SMs; at the Switch shape
        // 288 tiles of N = 256 ran in 65 us against 69 us for 576 of N = 128,
        // and 66 against 89 us with redirected overflow)
        const long long mt = (rows + 127) / 128 + active;
        if (mt * ((F + up_cols - 1) / up_cols) < 2 * kPlanSMs) p.bn_up = 128;
        if (mt * ((d + 255) / 256) < kPlanSMs) p.bn_down = 128;
        if (g_pair_policy > 0) p.bn_up = p.bn_down = 256;
        if (per >= kWideMinRows && F >= kWideMinK && p.bn_down == 256) p.mh_down = TILE_ROWS_256;
        // expert loads equal by construction: quantile balancing, expert choice
        const bool balanced = groups > 1 && (c->quantile_balance ||
                                             c->routing == MOE_ROUTING_EXPERT_CHOICE);
        if (use_pair(per, p.bn_up, p.s_up, balanced)) p.mh_up = TILE_ROWS_256_PAIR;
        // the long-reduction down projection keeps its one-SM 256-row tiles
        // (measured at Mixtral T = 16384: 2.48 ms against 2.54-2.58 on pairs)
        if (use_pair(per, p.bn_down, p.s_down, balanced) &&
            (p.mh_down != TILE_ROWS_256 || g_pair_policy > 0))
            p.mh_down = TILE_ROWS_256_PAIR;
        const double pad128 = (double)((per + 127) / 128 * 128) / per;
        const double pad16 = (double)((per + 15) / 16 * 16) / per;
        const long long var_tiles = active * ((per + kVarTileRows - 1) / kVarTileRows);
        if (pad128 > kVarPadGain * pad16) {
            p.nt_down = kVarTileRows;
            p.s_down = split_count(var_tiles * ((d + 127) / 128), (F + 63) / 64);
        }
        if (g_var_up_policy > 0) {
            p.nt = kVarTileRows;
            p.mh_up = TILE_ROWS_128;
            p.s_up = split_count(var_tiles * ((F + 127) / 128), (d + 63) / 64);
        }
        return p;
    }
    p.nt_down = p.nt;
    const long long ttiles = active * ((per + p.nt - 1) / p.nt);
    p.s_up = split_count(ttiles * ((F + 127) / 128), (d + 63) / 64);
    p.s_down = split_count(ttiles * ((d + 127) / 128), (F + 63) / 64);
    return p;
}
FfnPlan routed_plan(const moe_config *c) {
    return ffn_plan(c, sizes(c).R, c->n_experts, c->d_ff, c->act == MOE_ACT_SWIGLU);
}
FfnPlan shared_plan(const moe_config *c) {
    return ffn_plan(c, c->T, 1, c->d_ff_shared, true);
}

// Experts ranked after the top k that the router reports for redirected
// overflow: each round gives every unserved slot one more candidate.
long long n_candidates(const moe_config *c) {
    if (c->reroute_rounds <= 0) return 0;
    return std::min<long long>((long long)c->n_experts - c->top_k,
                               (long long)c->top_k * c->reroute_rounds);
}

Layout layout(const moe_config *c) {
    const Sizes s = sizes(c);
    const size_t eb = elem_bytes(c->dtype);
    const long long rb = router_blocks((int)s.T, (int)s.E, c->dtype, router_selects(c));
    const long long nb = dispatch_blocks(s.Tk);
    const FfnPlan rp = routed_plan(c), sp = shared_plan(c);
    const long long mt = max_tiles(s.R, (int)s.E, std::min(kSimtBM, rp.nt ? rp.nt : kSimtBM));
    const long long mts = max_tiles(s.T, 1, std::min(kSimtBM, sp.nt ? sp.nt : kSimtBM));
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
    L.perm = take(sizeof(int32_t) * s.R);
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
    L.xs = take(eb * s.R * s.d);
    L.h = take(eb * s.R * s.F);
    L.out_sorted = take(sizeof(float) * rp.s_down * s.R * s.d);
    L.sh_h = take(eb * s.T * s.Fs);
    L.sh_out = take(sizeof(float) * sp.s_down * s.T * s.d);
    const bool rt = tc_router(c);
    L.rt_wsplit = take(rt ? 2 * s.E * kRouterParts * router_dp(c) : 0);
    const long long planes =
        rt ? router_groups(c) : (s.E <= 32 ? router_slices((int)s.d, (int)s.E, c->dtype) : 0);
    L.rt_logits = take(sizeof(float) * planes * s.T * s.E);
    L.rt_offsets = take(sizeof(int32_t) * 2);
    L.rt_tile_e = take(sizeof(int32_t) * max_tiles(s.T, 1, kTcBM));
    L.rt_tile_start = take(sizeof(int32_t) * 2);
    L.rt_ntiles = take(sizeof(int32_t));
    const long long upw = c->act == MOE_ACT_SWIGLU ? 2 : 1;
    L.up_part = take(rp.s_up > 1 ? sizeof(float) * rp.s_up * s.R * upw * s.F : 0);
    L.sh_up_part = take(sp.s_up > 1 ? sizeof(float) * sp.s_up * s.T * 2 * s.Fs : 0);
    L.ent_partial = take(sizeof(float) * std::max<long long>(rb, (s.T + 31) / 32));
    L.row_stats = take(sizeof(double) * 3 * s.R);
    const long long nc = n_candidates(c);
    L.cand_idx = take(sizeof(int32_t) * s.T * nc);
    L.cand_w = take(sizeof(float) * s.T * nc);
    const bool rr = c->reroute_rounds > 0;
    L.rr_slot_e = take(rr ? sizeof(int32_t) * s.Tk : 0);
    L.rr_slot_w = take(rr ? sizeof(float) * s.Tk : 0);
    L.rr_served = take(rr ? sizeof(int32_t) * s.Tk : 0);
    L.rr_nxt = take(rr ? sizeof(int32_t) * s.T : 0);
    L.rr_filled = take(rr ? sizeof(int32_t) * s.E : 0);
    L.rr_filled_before = take(rr ? sizeof(int32_t) * s.E : 0);
    L.slot_w = take(rr ? sizeof(float) * s.Tk : 0);
    const bool ec = expert_choice(c);
    L.ec_row_w = take(ec ? sizeof(float) * s.R : 0);
    L.ec_rowidx = take(ec ? sizeof(int32_t) * s.E * s.T : 0);
    L.ec_tok_cnt = take(ec ? sizeof(int32_t) * s.T : 0);
    L.ec_tok_start = take(ec ? sizeof(int32_t) * (s.T + 1) : 0);
    L.ec_tok_rows = take(ec ? sizeof(int32_t) * s.R : 0);
    L.probs_rows = take(sizeof(float) * s.T * s.E);
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
    if (c->reroute_rounds < 0 || (c->routing != MOE_ROUTING_TOKEN_CHOICE &&
                                  c->routing != MOE_ROUTING_EXPERT_CHOICE))
        return MOE_ERR_INVALID_ARG;
    if (c->routing == MOE_ROUTING_EXPERT_CHOICE && c->quantile_balance)
        return MOE_ERR_UNSUPPORTED;
    if (c->reroute_rounds > 0) {
        if (!(c->capacity_factor > 0.f) || c->routing != MOE_ROUTING_TOKEN_CHOICE)
            return MOE_ERR_INVALID_ARG;
        if ((long long)c->top_k * (1 + c->reroute_rounds) > 32) return MOE_ERR_UNSUPPORTED;
    }
    return MOE_OK;
}

#define MOE_REQUIRE(cond) do { if (!(cond)) return MOE_ERR_INVALID_ARG; } while (0)
#define MOE_PTR(p) MOE_REQUIRE((p) != nullptr && aligned16(p))
#define MOE_OPT_PTR(p) MOE_REQUIRE((p) == nullptr || aligned16(p))
#define MOE_CUDA(call) do { cudaError_t e_ = (call); if (e_ != cudaSuccess) return MOE_ERR_CUDA; } while (0)

template <typename P> P *at(void *ws, size_t off) {
    return reinterpret_cast<P *>(static_cast<char *>(ws) + off);
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

// Inside a stream capture a plain event record only orders the captured
// work; the External flag makes it a real record node of the graph, so the
// event can be timed after a replay.
void timer_record(cudaEvent_t e, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
    else
        cudaEventRecord(e, st);
}
cudaEvent_t stage_begin(cudaStream_t st) {
    if (!g_timer.on) return nullptr;
    cudaEvent_t e = g_timer.get();
    if (e) timer_record(e, st);
    return e;
}
void stage_end(int stage, cudaEvent_t a, cudaStream_t st) {
    if (!a) return;
    cudaEvent_t b = g_timer.get();
    if (!b) return;
    timer_record(b, st);
    g_timer.recs.push_back({stage, a, b});
}

// Router incl. quantile balancing; p (mean probs) when p_out != NULL.
// The layer's dispatch computes p from the router's per-block partials
// (DispatchTail) instead of a p_finalize launch: token choice without
// redirection, up to 32 experts on the CUDA-core router, more than one
// softmax block (one block writes p itself).
bool p_from_dispatch(const moe_config *c) {
    const Sizes s = sizes(c);
    return s.T > 0 && !expert_choice(c) && c->reroute_rounds == 0 && !tc_router(c) &&
           s.E <= 32 && router_blocks((int)s.T, (int)s.E, c->dtype, router_selects(c)) > 1;
}

// defer_p: leave p to the dispatch (p_from_dispatch(c) must hold).
int run_router(const moe_config *c, const void *x, const float *w_r, const float *logit_bias,
               const float *select_bias, int32_t *idx, float *w, float *probs, float *p_out,
               float *sbias_out, bool want_probsT, void *ws, const Layout &L, cudaStream_t st,
               float *entropy_out = nullptr, int32_t *cand_out = nullptr, bool defer_p = false) {
    const Sizes s = sizes(c);
    RouterArgs a{};
    a.x = x; a.w_r = w_r; a.logit_bias = logit_bias;
    const bool ec = expert_choice(c);
    a.select_bias = (c->quantile_balance || ec) ? nullptr : select_bias;
    a.T = (int)s.T; a.d = (int)s.d; a.E = (int)s.E; a.k = (int)s.k;
    a.select_space = c->select_space;
    a.do_select = (c->quantile_balance || ec) ? 0 : 1;
    a.idx = idx; a.w = w;
    // expert-major probabilities for the per-expert passes (quantile bias,
    // expert choice); row-major ones for a second selection pass
    a.probsT = (c->quantile_balance || ec) ? at<float>(ws, L.probsT) : nullptr;
    a.probs = probs ? probs
                    : ((c->quantile_balance || want_probsT) ? at<float>(ws, L.probs_rows) : nullptr);
    a.p_partial = at<float>(ws, L.p_partial);
    a.ent_partial = entropy_out ? at<float>(ws, L.ent_partial) : nullptr;
    a.n_cand = (int)n_candidates(c);
    a.cand_idx = cand_out ? cand_out : at<int32_t>(ws, L.cand_idx);
    a.cand_w = at<float>(ws, L.cand_w);
    // E <= 32 with a single softmax block (at most 32, 16 or 8 tokens for
    // E <= 8, 16, 32): that block writes p itself, one launch fewer
    a.p_direct = (!tc_router(c) && s.E <= 32 && p_out &&
                  router_blocks(a.T, a.E, c->dtype, a.do_select != 0) == 1) ? p_out : nullptr;
    if (tc_router(c)) {
        const int dp = (int)router_dp(c);
        const int G = router_groups(c);
        __nv_bfloat16 *wsplit = at<__nv_bfloat16>(ws, L.rt_wsplit);
        float *part = at<float>(ws, L.rt_logits);
        int32_t *off = at<int32_t>(ws, L.rt_offsets);
        int32_t *te = at<int32_t>(ws, L.rt_tile_e), *ts = at<int32_t>(ws, L.rt_tile_start);
        int32_t *nt = at<int32_t>(ws, L.rt_ntiles);
        MOE_CUDA(launch_split_router_weight(w_r, a.E, a.d, dp, kRouterParts, wsplit, a.T, off,
                                            te, ts, nt, st));
        // chains of router_chain_kb K blocks summed on chip in chain order,
        // one plane per group of chains; the softmax adds the G planes in order
        // column tiles of 224 where they pad the experts less than 256 (896:
        // four tiles of 224 instead of 1024 columns)
        const int rbn = (a.E + 223) / 224 * 224 < (a.E + 255) / 256 * 256 ? 224 : 256;
        MOE_CUDA(launch_tc_gemm(GEMM_LOGITS, 0, rbn, 1, x, s.T, a.d, wsplit, nullptr, 1, a.E,
                                a.E, kRouterParts * dp, dp, G, s.T * s.E, te, ts, nt, off, part,
                                a.E, st, router_chain_kb(c)));
        MOE_CUDA(launch_router_from_logits(a, part, G, st));
    } else {
        MOE_CUDA(launch_router(a, c->dtype, at<float>(ws, L.rt_logits), st));
    }
    if (p_out && s.T > 0 && !a.p_direct && !defer_p)
        MOE_CUDA(launch_p_finalize(a.p_partial,
                                   router_blocks(a.T, a.E, c->dtype, a.do_select != 0), a.E, a.T,
                                   p_out, st));
    if (entropy_out && s.T > 0)
        MOE_CUDA(launch_p_finalize(a.ent_partial,
                                   router_blocks(a.T, a.E, c->dtype, a.do_select != 0), 1, a.T,
                                   entropy_out,
                                   st));
    if (c->quantile_balance && s.T > 0) {
        // Linear interpolation between order statistics: h = (T-1) q,
        // q = 1 - k/E, lo = floor(h), frac = h - lo.
        const double q = 1.0 - (double)s.k / (double)s.E;
        const double h = (double)(s.T - 1) * q;
        const double lo = floor(h);
        MOE_CUDA(launch_quantile_bias(a.probsT, a.T, a.E, (long long)lo, (float)(h - lo),
                                      sbias_out, st));
        MOE_CUDA(launch_select_rows(a.probs, sbias_out, a.T, a.E, a.k, idx, w, st, a.n_cand,
                                    a.cand_idx, a.cand_w));
    }
    return MOE_OK;
}

// Rows per tile of the up projection's tile table.
int up_tile_rows(const FfnPlan &plan) { return plan.nt ? plan.nt : tile_rows(plan.mh_up); }

// Up and down projections of one grouped FFN on the tensor cores: rows of A
// (x_sorted, or x itself for the shared expert) grouped by `offsets` into
// `groups` experts; h gets the activation in bf16; the down projection's
// output goes to `out`: plan.s_down fp32 planes of rows*d elements.
// tiles_built: the up projection's tile table is already in tile_e /
// tile_start / ntiles (up_tile_rows rows per tile).
int run_tc_ffn(const moe_config *c, const FfnPlan &plan, int up_mode, const void *A,
               long long rows, int groups, int F, const int32_t *offsets, const void *w1,
               const void *w3, const void *w2, void *h, float *up_part, float *out,
               int32_t *tile_e, int32_t *tile_start, int32_t *ntiles, int up_stage,
               int down_stage, cudaStream_t st, bool tiles_built = false) {
    const int d = c->d_model;
    const int nt = plan.nt;
    cudaEvent_t ev = up_stage >= 0 ? stage_begin(st) : nullptr;
    const int up_rows = up_tile_rows(plan);
    if (!tiles_built)
        MOE_CUDA(launch_build_tiles(offsets, groups, up_rows, tile_e, nullptr, tile_start, ntiles,
                                    st));
    if (plan.s_up > 1) {
        const int upw = up_mode == GEMM_UP_SWIGLU ? 2 : 1;
        MOE_CUDA(launch_tc_gemm(up_mode, nt, plan.bn_up, 1, A, rows, d, w1, w3, groups, F, F, d,
                                d, plan.s_up,
                                rows * upw * F, tile_e, tile_start, ntiles, offsets, up_part,
                                upw * F, st));
        MOE_CUDA(launch_split_activation(up_part, plan.s_up, rows * upw * F, F,
                                         up_mode == GEMM_UP_SWIGLU, offsets + groups, rows,
                                         static_cast<__nv_bfloat16 *>(h), st));
    } else {
        MOE_CUDA(launch_tc_gemm(up_mode, nt, plan.bn_up, nt ? TILE_ROWS_128 : plan.mh_up, A, rows,
                                d, w1, w3, groups, F, F, d, d, 1, 0, tile_e, tile_start, ntiles,
                                offsets, h, F, st));
    }
    if (up_stage >= 0) {
        stage_end(up_stage, ev, st);
        ev = stage_begin(st);
    }
    const int mh_down = plan.nt_down ? TILE_ROWS_128 : plan.mh_down;
    const int down_rows = plan.nt_down ? plan.nt_down : tile_rows(mh_down);
    if (down_rows != up_rows)
        MOE_CUDA(launch_build_tiles(offsets, groups, down_rows, tile_e, nullptr, tile_start,
                                    ntiles, st));
    MOE_CUDA(launch_tc_gemm(GEMM_DOWN, plan.nt_down, plan.bn_down, mh_down, h, rows, F, w2, nullptr,
                            groups, d, d, F, F, plan.s_down, rows * d, tile_e, tile_start, ntiles,
                            offsets, out, d, st));
    if (down_stage >= 0) stage_end(down_stage, ev, st);
    return MOE_OK;
}

// Grouped expert FFN over the dispatched rows; out_sorted fp32 (plan.s_down
// planes of R*d elements).  bf16: gather the rows into x_sorted, tcgen05 up
// (+activation, h in bf16) into h, tcgen05 down into out_sorted.  fp32: SIMT
// GEMMs reading x through perm directly.
// inv (token choice, may be NULL): the slots' rows, for the token-major copy.
// tiles_built: the dispatch already wrote the up projection's tile table
// (bf16 layers; DispatchTail).
int run_experts(const moe_config *c, const void *x, const int32_t *perm, const int32_t *offsets,
                const void *w1, const void *w3, const void *w2, float *out_sorted, void *ws,
                const Layout &L, cudaStream_t st, const int32_t *inv = nullptr,
                bool tiles_built = false) {
    const Sizes s = sizes(c);
    if (s.R == 0) return MOE_OK;
    const int gk = expert_choice(c) ? 1 : (int)s.k;   // perm holds t*k+j, or t itself
    int32_t *tile_e = at<int32_t>(ws, L.tile_e), *tile_m0 = at<int32_t>(ws, L.tile_m0);
    int32_t *tile_start = at<int32_t>(ws, L.tile_start), *ntiles = at<int32_t>(ws, L.ntiles);
    const int up_mode = c->act == MOE_ACT_SWIGLU ? GEMM_UP_SWIGLU : GEMM_UP_RELU;
    if (c->dtype == MOE_DTYPE_BF16) {
        void *xs = at<void>(ws, L.xs), *h = at<void>(ws, L.h);
        cudaEvent_t ev = stage_begin(st);
        if (inv && !expert_choice(c))
            MOE_CUDA(launch_scatter_rows(x, 2, (int)s.d, inv, (int)s.k, s.T, xs, st));
        else
            MOE_CUDA(launch_gather_rows(x, 2, (int)s.d, perm, offsets + s.E, gk, s.R, xs, st));
        stage_end(MOE_STAGE_GATHER, ev, st);
        return run_tc_ffn(c, routed_plan(c), up_mode, xs, s.R, (int)s.E, (int)s.F, offsets, w1,
                          w3, w2, h, at<float>(ws, L.up_part), out_sorted, tile_e,
                          tile_start, ntiles, MOE_STAGE_UP, MOE_STAGE_DOWN, st, tiles_built);
    }
    cudaEvent_t ev = stage_begin(st);
    MOE_CUDA(launch_build_tiles(offsets, (int)s.E, kSimtBM, tile_e, tile_m0, nullptr, ntiles, st));
    stage_end(MOE_STAGE_GATHER, ev, st);
    ev = stage_begin(st);
    GroupedGemmArgs up;
    up.A = x; up.a_gather = perm; up.gather_k = gk;
    up.B1 = w1; up.B3 = w3; up.b_expert_stride = s.F * s.d; up.N = (int)s.F; up.K = (int)s.d;
    up.C = at<void>(ws, L.h); up.ldc = (int)s.F;
    up.tile_e = tile_e; up.tile_m0 = tile_m0; up.n_tiles = ntiles; up.offsets = offsets;
    up.max_tiles = max_tiles(s.R, (int)s.E, kSimtBM);
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

// Shared expert (SwiGLU) on all T rows -> sh_out: shared_plan.s_down fp32
// planes of T*d elements: the same grouped kernels with one group {0, T} and
// x read in place.
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
    if (c->dtype == MOE_DTYPE_BF16)
        return run_tc_ffn(c, shared_plan(c), GEMM_UP_SWIGLU, x, s.T, 1, (int)s.Fs, off, ws1, ws3,
                          ws2, h, at<float>(ws, L.sh_up_part), o, te, ts, nt, -1,
                          -1, st);
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

RerouteWork reroute_work(void *ws, const Layout &L) {
    RerouteWork w;
    w.slot_e = at<int32_t>(ws, L.rr_slot_e);
    w.slot_w = at<float>(ws, L.rr_slot_w);
    w.served = at<int32_t>(ws, L.rr_served);
    w.nxt = at<int32_t>(ws, L.rr_nxt);
    w.filled = at<int32_t>(ws, L.rr_filled);
    w.filled_before = at<int32_t>(ws, L.rr_filled_before);
    w.hist = at<int32_t>(ws, L.hist);
    w.block_base = at<int32_t>(ws, L.block_base);
    return w;
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

int moe_dispatch_reroute(const moe_config *cfg, const int32_t *topk_idx, const float *topk_w,
                         const int32_t *cand_idx, const float *cand_w, int32_t *counts,
                         int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *slot_expert,
                         float *slot_w, int32_t *n_dropped, void *ws, size_t ws_bytes,
                         moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    if (cfg->reroute_rounds <= 0) return MOE_ERR_INVALID_ARG;
    MOE_PTR(counts); MOE_PTR(offsets); MOE_PTR(n_dropped); MOE_PTR(ws);
    const long long nc = n_candidates(cfg);
    if (cfg->T > 0) {
        MOE_PTR(topk_idx); MOE_PTR(topk_w); MOE_PTR(perm); MOE_PTR(inv);
        if (nc > 0) { MOE_PTR(cand_idx); MOE_PTR(cand_w); }
    }
    MOE_OPT_PTR(slot_expert); MOE_OPT_PTR(slot_w);
    const Layout L = layout(cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    MOE_CUDA(launch_dispatch_reroute(topk_idx, topk_w, cand_idx, cand_w, (int)nc, cfg->T,
                                     cfg->top_k, cfg->n_experts, capacity_of(cfg),
                                     cfg->reroute_rounds, reroute_work(ws, L), counts, offsets,
                                     perm, inv, slot_expert, slot_w, n_dropped,
                                     (cudaStream_t)stream));
    return MOE_OK;
}

int64_t moe_reroute_candidates(const moe_config *cfg) {
    if (check_cfg(cfg) != MOE_OK) return -1;
    return n_candidates(cfg);
}

int moe_ffn_plan(const moe_config *cfg, int32_t shared, moe_ffn_plan_info *out) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    MOE_REQUIRE(out != nullptr);
    if (cfg->dtype != MOE_DTYPE_BF16 || (shared && cfg->d_ff_shared <= 0))
        return MOE_ERR_UNSUPPORTED;
    const FfnPlan p = shared ? shared_plan(cfg) : routed_plan(cfg);
    out->rows_per_tile = p.nt;
    out->up_splits = p.s_up;
    out->down_splits = p.s_down;
    out->up_n = p.bn_up;
    out->down_n = p.bn_down;
    out->down_rows_per_tile = p.nt_down;
    out->down_halves = p.nt_down || p.mh_down == TILE_ROWS_128 ? 1 : 2;
    out->up_pair = !p.nt && p.s_up == 1 && p.mh_up == TILE_ROWS_256_PAIR;
    out->down_pair = !p.nt_down && p.mh_down == TILE_ROWS_256_PAIR;
    return MOE_OK;
}

int moe_debug_set_pair_tiles(int32_t policy) {
    if (policy < -1 || policy > 1) return MOE_ERR_INVALID_ARG;
    g_pair_policy = policy;
    return MOE_OK;
}

int moe_debug_set_var_up_tiles(int32_t policy) {
    if (policy < -1 || policy > 1) return MOE_ERR_INVALID_ARG;
    g_var_up_policy = policy;
    return MOE_OK;
}

int64_t moe_expert_choice_rows(const moe_config *cfg) {
    if (check_cfg(cfg) != MOE_OK) return -1;
    return ec_rows_per_expert(cfg);
}

int moe_expert_choice(const moe_config *cfg, const float *probs_t, int32_t *perm, float *row_w,
                      int32_t *counts, int32_t *offsets, int32_t *tok_start, int32_t *tok_rows,
                      int32_t *n_unchosen, void *ws, size_t ws_bytes, moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    if (!expert_choice(cfg)) return MOE_ERR_INVALID_ARG;
    MOE_PTR(counts); MOE_PTR(offsets); MOE_PTR(tok_start); MOE_PTR(n_unchosen); MOE_PTR(ws);
    if (cfg->T > 0) { MOE_PTR(probs_t); MOE_PTR(perm); MOE_PTR(row_w); MOE_PTR(tok_rows); }
    const Layout L = layout(cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    const Sizes s = sizes(cfg);
    MOE_CUDA(launch_expert_choice(probs_t, (int)s.T, (int)s.E, (int)ec_rows_per_expert(cfg), perm,
                                  row_w, at<int32_t>(ws, L.ec_rowidx), counts, offsets,
                                  at<int32_t>(ws, L.ec_tok_cnt), tok_start, tok_rows, n_unchosen,
                                  (cudaStream_t)stream));
    return MOE_OK;
}

int moe_combine_rows(const moe_config *cfg, const float *out_sorted, const float *row_w,
                     const int32_t *tok_start, const int32_t *tok_rows, const float *shared_out,
                     void *y, moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    if (cfg->T == 0) return MOE_OK;
    MOE_PTR(out_sorted); MOE_PTR(row_w); MOE_PTR(tok_start); MOE_PTR(tok_rows); MOE_PTR(y);
    MOE_OPT_PTR(shared_out);
    MOE_CUDA(launch_combine_rows(expert_out_f32(out_sorted), tok_start, tok_rows,
                                 row_w, expert_out_f32(shared_out),
                                 cfg->T, cfg->d_model, cfg->out_dtype, y, (cudaStream_t)stream));
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
    const FfnPlan plan = routed_plan(cfg);
    if (plan.s_down == 1)
        return run_experts(cfg, x, perm, offsets, w1, w3, w2, out_sorted, ws, L,
                           (cudaStream_t)stream);
    // split reduction: partial planes in the workspace, summed into out_sorted
    float *planes = at<float>(ws, L.out_sorted);
    rc = run_experts(cfg, x, perm, offsets, w1, w3, w2, planes, ws, L, (cudaStream_t)stream);
    if (rc != MOE_OK) return rc;
    const long long R = sizes(cfg).R;
    MOE_CUDA(launch_sum_planes(planes, plan.s_down, R * cfg->d_model, cfg->d_model,
                               offsets + cfg->n_experts, R, out_sorted, (cudaStream_t)stream));
    return MOE_OK;
}

int moe_combine(const moe_config *cfg, const float *out_sorted, const int32_t *inv,
                const float *topk_w, const float *shared_out, void *y, moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    if (cfg->T == 0) return MOE_OK;
    MOE_PTR(out_sorted); MOE_PTR(inv); MOE_PTR(topk_w); MOE_PTR(y); MOE_OPT_PTR(shared_out);
    MOE_CUDA(launch_combine(expert_out_f32(out_sorted), inv, topk_w,
                            expert_out_f32(shared_out), cfg->T, cfg->top_k,
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

int moe_observe(const moe_config *cfg, const float *probs, const float *out_sorted,
                const int32_t *offsets, const float *select_bias, const int32_t *n_dropped,
                const moe_observability *obs, void *ws, size_t ws_bytes, moe_stream_t stream) {
    int rc = check_cfg(cfg);
    if (rc != MOE_OK) return rc;
    MOE_REQUIRE(obs != nullptr);
    MOE_PTR(ws);
    MOE_OPT_PTR(probs); MOE_OPT_PTR(out_sorted); MOE_OPT_PTR(offsets);
    MOE_OPT_PTR(select_bias); MOE_OPT_PTR(n_dropped);
    MOE_REQUIRE((out_sorted == nullptr) == (offsets == nullptr));
    MOE_OPT_PTR(obs->drop_ratio); MOE_OPT_PTR(obs->gate_entropy);
    MOE_OPT_PTR(obs->bias_mean_abs); MOE_OPT_PTR(obs->bias_max_abs);
    MOE_OPT_PTR(obs->expert_out_mean); MOE_OPT_PTR(obs->expert_out_std);
    MOE_OPT_PTR(obs->expert_out_max_abs);
    const Layout L = layout(cfg);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    const Sizes s = sizes(cfg);
    cudaStream_t st = (cudaStream_t)stream;
    if (obs->gate_entropy) {
        if (probs && s.T > 0) {
            float *part = at<float>(ws, L.ent_partial);
            MOE_CUDA(launch_entropy_partials(probs, (int)s.T, (int)s.E, part, st));
            MOE_CUDA(launch_p_finalize(part, (int)((s.T + 31) / 32), 1, (int)s.T,
                                       obs->gate_entropy, st));
        } else {
            MOE_CUDA(cudaMemsetAsync(obs->gate_entropy, 0, sizeof(float), st));
        }
    }
    ObsArgs oa{};
    oa.n_dropped = n_dropped;
    oa.bias = select_bias;
    oa.drop_ratio = obs->drop_ratio;
    oa.bias_mean_abs = obs->bias_mean_abs;
    oa.bias_max_abs = obs->bias_max_abs;
    if (oa.drop_ratio || oa.bias_mean_abs || oa.bias_max_abs)
        MOE_CUDA(launch_stats_finalize(nullptr, nullptr, (int)s.T, (int)s.E, (int)s.k, nullptr,
                                       nullptr, nullptr, nullptr, st, oa));
    float *outs[3] = {obs->expert_out_mean, obs->expert_out_std, obs->expert_out_max_abs};
    for (float *o : outs) {
        if (o && !out_sorted) MOE_CUDA(cudaMemsetAsync(o, 0, sizeof(float) * s.E, st));
    }
    if (out_sorted && (outs[0] || outs[1] || outs[2]))
        MOE_CUDA(launch_expert_scale(expert_out_f32(out_sorted), (int)s.d, offsets, (int)s.E,
                                     s.Tk, at<double>(ws, L.row_stats), outs[0], outs[1],
                                     outs[2], st));
    return MOE_OK;
}

int moe_layer_forward(const moe_config *cfg, const void *x, const moe_layer_weights *wts,
                      const moe_layer_outputs *out, void *ws, size_t ws_bytes,
                      moe_stream_t stream) {
    return moe_layer_forward_observed(cfg, x, wts, out, nullptr, ws, ws_bytes, stream);
}

int moe_layer_forward_observed(const moe_config *cfg, const void *x,
                               const moe_layer_weights *wts, const moe_layer_outputs *out,
                               const moe_observability *obs, void *ws, size_t ws_bytes,
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
    MOE_OPT_PTR(out->counts_unbiased); MOE_OPT_PTR(out->slot_expert); MOE_OPT_PTR(out->slot_w);
    MOE_OPT_PTR(out->offsets); MOE_OPT_PTR(out->perm); MOE_OPT_PTR(out->cand_idx);
    if (obs) {
        MOE_OPT_PTR(obs->drop_ratio); MOE_OPT_PTR(obs->gate_entropy);
        MOE_OPT_PTR(obs->bias_mean_abs); MOE_OPT_PTR(obs->bias_max_abs);
        MOE_OPT_PTR(obs->expert_out_mean); MOE_OPT_PTR(obs->expert_out_std);
        MOE_OPT_PTR(obs->expert_out_max_abs);
    }
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
    int32_t *offsets = out->offsets ? out->offsets : at<int32_t>(ws, L.offsets);
    int32_t *perm = out->perm ? out->perm : at<int32_t>(ws, L.perm);
    int32_t *inv = at<int32_t>(ws, L.inv);
    int32_t *cand = out->cand_idx && cfg->reroute_rounds > 0 ? out->cand_idx
                                                             : at<int32_t>(ws, L.cand_idx);
    // Expert outputs: fp32 planes (one per split of the down projection's
    // reduction, added in split order by their readers), routed and shared.
    float *out_sorted = at<float>(ws, L.out_sorted);
    const FfnPlan rplan = routed_plan(cfg), splan = shared_plan(cfg);
    const ExpertOut eo = expert_out_f32(out_sorted, rplan.s_down, s.R * s.d);
    ExpertOut sh = expert_out_f32(nullptr, splan.s_down, s.T * s.d);

    const bool biased = cfg->quantile_balance || wts->select_bias != nullptr;
    const bool want_unb = out->counts_unbiased != nullptr;

    if (g_timer.on) ++g_timer.calls;
    cudaEvent_t ev = stage_begin(st);
    if (s.T > 0) {
        rc = run_router(cfg, x, wts->w_r, wts->logit_bias, wts->select_bias, idx, w, nullptr, p,
                        sbias, want_unb && biased, ws, L, st, obs ? obs->gate_entropy : nullptr,
                        cand, p_from_dispatch(cfg));
        if (rc != MOE_OK) return rc;
    } else if (obs && obs->gate_entropy) {
        MOE_CUDA(cudaMemsetAsync(obs->gate_entropy, 0, sizeof(float), st));
    }
    stage_end(MOE_STAGE_ROUTER, ev, st);
    ev = stage_begin(st);
    const float *comb_w = w;           // gate weight of each slot in the combine
    const bool ec = expert_choice(cfg);
    ObsArgs oa{};
    if (obs) {
        oa.n_dropped = ndrop;
        oa.bias = cfg->quantile_balance ? sbias : wts->select_bias;
        oa.drop_ratio = obs->drop_ratio;
        oa.bias_mean_abs = obs->bias_mean_abs;
        oa.bias_max_abs = obs->bias_max_abs;
    }
    DispatchTail tail{};
    if (ec) {
        MOE_CUDA(launch_expert_choice(at<float>(ws, L.probsT), (int)s.T, (int)s.E,
                                      (int)ec_rows_per_expert(cfg), perm,
                                      at<float>(ws, L.ec_row_w), at<int32_t>(ws, L.ec_rowidx),
                                      counts, offsets, at<int32_t>(ws, L.ec_tok_cnt),
                                      at<int32_t>(ws, L.ec_tok_start),
                                      at<int32_t>(ws, L.ec_tok_rows), ndrop, st));
    } else if (cfg->reroute_rounds > 0) {
        float *sw = out->slot_w ? out->slot_w : at<float>(ws, L.slot_w);
        MOE_CUDA(launch_dispatch_reroute(idx, w, cand,
                                         at<float>(ws, L.cand_w), (int)n_candidates(cfg), s.T,
                                         (int)s.k, (int)s.E, capacity_of(cfg),
                                         cfg->reroute_rounds, reroute_work(ws, L), counts,
                                         offsets, perm, inv, out->slot_expert, sw, ndrop, st));
        comb_w = sw;
    } else {
        // the dispatch's offsets CTA also computes p (when the router left
        // it), the load statistics and, for the tensor-core FFN, the up
        // projection's tile table
        if (p_from_dispatch(cfg)) {
            tail.p_partial = at<float>(ws, L.p_partial);
            tail.p_nblk = router_blocks((int)s.T, (int)s.E, cfg->dtype, router_selects(cfg));
            tail.p_out = p;
        }
        tail.stats = s.T > 0;
        tail.p = p;
        tail.T = (int)s.T;
        tail.k = (int)s.k;
        tail.f = out->f;
        tail.aux = out->aux;
        tail.load = out->load_max_over_mean;
        tail.o = oa;
        if (cfg->dtype == MOE_DTYPE_BF16 && s.T > 0) {
            tail.tile_rows = up_tile_rows(rplan);
            tail.tile_e = at<int32_t>(ws, L.tile_e);
            tail.tile_start = at<int32_t>(ws, L.tile_start);
            tail.n_tiles = at<int32_t>(ws, L.ntiles);
        }
        MOE_CUDA(launch_dispatch(idx, s.Tk, (int)s.E, (int)s.k, capacity_of(cfg),
                                 at<int32_t>(ws, L.hist), at<int32_t>(ws, L.block_base), counts,
                                 offsets, perm, inv, ndrop, st, &tail));
        if (out->slot_expert || out->slot_w)
            MOE_CUDA(launch_slot_outputs(idx, w, inv, s.Tk, out->slot_expert, out->slot_w, st));
    }
    stage_end(MOE_STAGE_DISPATCH, ev, st);
    ev = stage_begin(st);
    if (want_unb) {
        if (biased && s.T > 0 && !ec) {
            int32_t *iu = at<int32_t>(ws, L.idx_unb);
            MOE_CUDA(launch_select_rows(at<float>(ws, L.probs_rows), nullptr, (int)s.T,
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
    if (!tail.stats)
        MOE_CUDA(launch_stats_finalize(counts, p, (int)s.T, (int)s.E, (int)s.k, out->f, nullptr,
                                       out->aux, out->load_max_over_mean, st, oa));
    stage_end(MOE_STAGE_STATS, ev, st);
    const bool want_scale =
        obs && (obs->expert_out_mean || obs->expert_out_std || obs->expert_out_max_abs);
    if (s.T == 0) {
        if (want_scale)
            MOE_CUDA(launch_expert_scale(eo, (int)s.d, offsets, (int)s.E, 0,
                                         at<double>(ws, L.row_stats), obs->expert_out_mean,
                                         obs->expert_out_std, obs->expert_out_max_abs, st));
        return MOE_OK;
    }
    rc = run_experts(cfg, x, perm, offsets, wts->w1, wts->w3, wts->w2, out_sorted, ws, L, st,
                     expert_choice(cfg) ? nullptr : inv, tail.tile_rows > 0);
    if (rc != MOE_OK) return rc;
    if (want_scale)
        MOE_CUDA(launch_expert_scale(eo, (int)s.d, offsets, (int)s.E, s.R,
                                     at<double>(ws, L.row_stats),
                                     obs->expert_out_mean, obs->expert_out_std,
                                     obs->expert_out_max_abs, st));
    if (s.Fs > 0) {
        ev = stage_begin(st);
        rc = run_shared(cfg, x, wts->ws1, wts->ws3, wts->ws2, ws, L, st);
        if (rc != MOE_OK) return rc;
        stage_end(MOE_STAGE_SHARED, ev, st);
        sh.p = at<float>(ws, L.sh_out);
    }
    ev = stage_begin(st);
    if (ec)
        MOE_CUDA(launch_combine_rows(eo, at<int32_t>(ws, L.ec_tok_start),
                                     at<int32_t>(ws, L.ec_tok_rows), at<float>(ws, L.ec_row_w),
                                     sh, (int)s.T, (int)s.d, cfg->out_dtype, out->y, st));
    else
        MOE_CUDA(launch_combine(eo, inv, comb_w, sh, (int)s.T, (int)s.k, (int)s.d,
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

int moe_debug_set_wait_hooks(uint64_t main_loop_limit_ns, int32_t stall_mma) {
    if (main_loop_limit_ns == 0 || stall_mma < 0 || stall_mma > 1) return MOE_ERR_INVALID_ARG;
    if (tc::set_wait_hooks(main_loop_limit_ns, stall_mma) != cudaSuccess) {
        (void)cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

int moe_kernel_binary_version(int32_t *version) {
    if (!version) return MOE_ERR_INVALID_ARG;
    cudaFuncAttributes a{};
    if (cudaFuncGetAttributes(&a, set_pair_kernel) != cudaSuccess) {
        (void)cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    *version = a.binaryVersion;
    return MOE_OK;
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
            (void)cudaGetLastError();   // keep the failure out of later launch checks
            rc = MOE_ERR_CUDA;
            continue;
        }
        stage_ms[r.stage] += ms;
    }
    *calls = g_timer.calls;
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
