// Grouped expert GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// operands staged by TMA, for the bf16 layer.
//
// Expert FFN ("Mixture of Experts", waylandz.com ch. 30, §30.2.4 / §30.6.1),
// on the rows grouped by expert ("混合エキスパートモデル（MoE）実践",
// deepseekmodel.com: contiguous per-expert rows make one grouped GEMM over
// all experts possible):
//   up   SwiGLU: H = silu(A W1_e^T) * (A W3_e^T)    ReLU: H = relu(A W1_e^T)
//   down O = H W2_e^T  (fp32 expert outputs)
// A [rows, K] and all weights [E*N, K] are K-major bf16, exactly the
// nn.Linear layout, so both operands are "K-major" for tcgen05.mma.
//
// One CTA per SM, persistent over output tiles of 128 rows.  Tile order:
// experts in order; inside an expert, N-tiles outer and M-tiles inner, so the
// CTAs running at the same time share one expert's weight tiles through L2
// and each expert's weights stream from HBM about once.
//   warp 0     TMA producer: A tile [128 x 64] + B tile [256 x 64] per stage
//              (SwiGLU: 128 rows of W1 and the same 128 rows of W3),
//              128-byte swizzle, 4 stages in shared memory
//   warp 1     MMA issuer: tcgen05.mma.cta_group::1.kind::f16, M=128, N=256,
//              K=16 per instruction, fp32 accumulator in TMEM
//   warp 2     TMEM allocator (512 columns: two 256-column accumulators)
//   warps 4-7  epilogue: tcgen05.ld of 32 TMEM lanes each, activation,
//              bf16 (up) stores; down: fp32 stores (partial sums for a
//              split)
// Small batches (a few rows per expert) run the same pipeline with the
// operands swapped (NT > 0): 128 weight rows are the MMA's M side and NT = 16,
// 32 or 64 token rows its N side, so a tile streams 128 rows of W1 (and W3)
// against a narrow token tile instead of padding 128 token rows.  The
// reduction can then be split over CTAs (k_splits): each split writes fp32
// partial sums that a later kernel adds in split order.
// NT = 256 is the same swapped pipeline with the MMA's N chosen per tile: a
// tile holds up to 256 of one expert's rows and its MMA N is that count
// rounded up to 16, so an expert with 146 rows costs a 160-wide tile instead
// of two 128-row tiles.  For SwiGLU the W1 and W3 parts of a tile fill the 512
// TMEM columns, so there is one accumulator.
// GEMM_LOGITS (NT = 0, N = 256, or 224 where that pads the experts less):
// the router's logits x W_r^T over a long reduction cut into chains of equal
// K ranges (the tensor core's fp32
// accumulation loses precision along one long chain).  Chain 0 of a tile
// accumulates into TMEM columns 0-255 (S), every later chain into columns
// 256-511 (A); after each later chain the epilogue adds A into S in TMEM
// (tcgen05.ld / st), so S = ((c0 + c1) + c2) + ..., and stores S once.
// MH = 2 (NT = 0, N = 256): tiles of 256 token rows, two M = 128 MMAs per
// K step sharing the weight tile, so a 64 KB stage feeds twice the MMA work
// of a 48 KB one; the 256 x 256 fp32 accumulator fills TMEM, so there is one
// accumulator and the epilogue does not overlap the next tile's MMAs.
// SM pairs (grouped_gemm_pair_kernel, below): tiles of 256 token rows on a
// cluster of two CTAs running one tcgen05.mma.cta_group::2 of M = 256, each
// CTA staging half of the rows and half of the weight tile (32 KB stages,
// two accumulators).
// Every mbarrier wait is bounded (about 2 s of no progress); on expiry the
// kernel sets the device error word, stops issuing, lets its own copies and
// MMAs land, frees TMEM and returns.
#include "common.cuh"
#include "kernels.h"

#include <cuda.h>

#include <algorithm>

namespace moe {
namespace tc {

constexpr int BM = 128;              // rows per tile (UMMA M)
constexpr int BNM = 256;             // UMMA N (B rows per stage)
constexpr int BK = 64;               // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int WROWS = 128;           // weight rows of one TMA box
constexpr int TMEM_COLS = 512;
constexpr int ACC_COLS = 256;        // columns of one of the two accumulators
constexpr int kSmemLimit = 232448;   // dynamic shared memory per CTA (227 KB)
constexpr int kSmemBase = 1024 /* alignment slack */ + 256 /* barriers */;
// Epilogue staging per CTA (4 epilogue warps).  Swapped geometries: a
// [16 tokens][32 features] bf16 block per warp.  NT = 0 fp32 outputs: a
// [32 rows][32 or 16 columns] fp32 block per warp (Geo::EPI_COLS).
constexpr int kEpiSwapBytes = 4 * 16 * 32 * 2;
constexpr int kVarRows = 256;        // NT of the per-tile-width geometry
constexpr int kLogitsN224 = 224;     // GEMM_LOGITS column tile that divides 896 experts
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s without progress

// Failure-detection test hooks (moe_debug_set_wait_hooks).  The limit of the
// main-loop waits (producer, MMA issuer, epilogue); the drain waits after an
// abort keep kWaitLimitNs.  g_stall_mma != 0 makes the MMA issuer first wait
// on a barrier phase that nothing completes, so that its bounded wait runs
// out and the abort path runs.
__device__ unsigned long long g_main_wait_limit_ns = kWaitLimitNs;
__device__ int g_stall_mma = 0;

// Tile geometry of one kernel instantiation.  NT = 0: token rows on the M
// side (A = 128 activation rows, B = 256 weight rows).  NT > 0: weight rows on
// the M side (A = 128 rows of W1, plus 128 rows of W3 for SwiGLU), token rows
// on the N side (NT rows).  A stage holds the activation tile first, then the
// weight tile(s); every tile is a multiple of 1024 bytes.
template <int MODE, int NT, int BN, int MH> struct Geo {
    static_assert(MH == 1 || (MH == 2 && NT == 0 && BN == BNM), "256-row tiles: NT 0, N 256");
    static constexpr bool SWAP = NT > 0;
    static constexpr bool VARN = NT == kVarRows;                 // MMA N chosen per tile
    static_assert(!VARN || MODE != GEMM_LOGITS, "per-tile width: expert projections only");
    static constexpr int ROWS = SWAP ? NT : BM * MH;             // activation rows per tile
    static constexpr int WT = (SWAP && MODE == GEMM_UP_SWIGLU) ? 2 : 1;
    // rows of one weight TMA box: 128 (NT > 0), BN / 2 (NT = 0: two boxes)
    static constexpr int BOX = SWAP ? WROWS : BN / 2;
    static constexpr int ACT_BYTES = ROWS * BK * 2;
    static constexpr int W_BYTES = SWAP ? WT * WROWS * BK * 2 : BN * BK * 2;
    static constexpr int STAGE_BYTES = ACT_BYTES + W_BYTES;
    // fp32 epilogue staging: [32 rows][EPI_COLS] per warp, rows EPI_STRIDE
    // floats apart (16-byte aligned; a quarter-warp's float4 writes hit
    // distinct banks)
    static constexpr int EPI_COLS = 32;
    static constexpr int EPI_STRIDE = EPI_COLS + 4;
    static constexpr int EPI =
        SWAP ? kEpiSwapBytes
             : ((MODE == GEMM_DOWN || MODE == GEMM_LOGITS) ? 4 * 32 * EPI_STRIDE * 4 : 0);
    static constexpr int EXTRA = kSmemBase + EPI;
    static constexpr int FIT = (kSmemLimit - EXTRA) / STAGE_BYTES;
    static constexpr int STAGES =
        SWAP ? (FIT < 8 ? FIT : 8)
             : MH == 2 ? 3
                       : (MODE == GEMM_LOGITS && BN != BNM) ? (FIT < 8 ? FIT : 8)
                                                            : (BN == BNM ? 4 : 6);
    // accumulator buffers: one where a tile fills all 512 TMEM columns (two
    // 256-column MMA halves, or SwiGLU's W1 and W3 parts of up to 256 tokens)
    static constexpr int NACC = (MH == 2 || (VARN && MODE == GEMM_UP_SWIGLU)) ? 1 : 2;
    // output columns (features) of one tile
    static constexpr int OUTC = SWAP ? WROWS : (MODE == GEMM_UP_SWIGLU ? BN / 2 : BN);
    static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + EXTRA;
};

struct Args {
    int mode;          // GEMM_UP_SWIGLU, GEMM_UP_RELU, GEMM_DOWN
    int N;             // output columns
    int K;             // reduction length (B's columns)
    int a_k_period;    // A's column of reduction index k is k mod a_k_period
    int n_ntiles;      // output-column tiles (OUTC columns each)
    int b_rows;        // weight rows per expert (F for up, d for down)
    int k_splits;      // work items per output tile along K
    int kb_per_split;  // K blocks of one split
    long long split_stride;   // output elements between the partial results of splits
    const int32_t *tile_e, *tile_start, *n_mtiles, *offsets;
    void *C;
    int ldc;
    int chain_kb;      // GEMM_LOGITS: K blocks per chain (a split holds whole chains)
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait; false when the limit expired or another role aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    const uint64_t limit = g_main_wait_limit_ns;
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit) {
            flag_error(kErrTimeout);
            *abort_flag = 1;
            return false;
        }
    }
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// 32 TMEM lanes x 16 consecutive 32-bit columns; thread i reads lane base+i.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 TMEM lanes x 16 consecutive 32-bit columns; thread i writes lane base+i.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32"
        " [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
        ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
          "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
          "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
          "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
          "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
          "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes in 8-row (1024-byte) atoms.  Fields: start address >> 4 (bits
// 0-13), leading byte offset >> 4 (16-29; unused for this layout), stride
// byte offset >> 4 = 1024 >> 4 (32-45), descriptor version 1 (bits 46-47),
// swizzle mode 2 = 128-byte (bits 61-63).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

struct TileCoord {
    int e, m0, mend, n0, split, kb0, kb1;
};

// Serpentine reduction order: a CTA walks the K blocks of every second work
// item backwards, so that each wave of tiles starts on the K blocks the
// previous wave loaded last, which are still in L2 (token-row tiles only: the
// router's chains keep their order, and swapped tiles stream weights that no
// other item reads).  Only the fp32 order of the K blocks within a tile
// changes, fixed by the item's position.
template <int MODE, int NT>
__device__ __forceinline__ bool serpentine(int it) {
    return MODE != GEMM_LOGITS && NT == 0 && (it & 1);
}

// Work item L -> (split, expert, row tile, output-column tile, K-block
// range).  Splits are outermost so that the CTAs in flight work on the same K
// slice.  Inside an expert, output-column tiles are outer and row tiles inner
// (the CTAs in flight share a weight tile); with ROWS_OUTER the other way
// round (they share the activation rows: the router's logits, whose split
// spans all of x's columns and whose weights stay in L2).  ROWS = activation
// rows per tile, OUTC = output columns per tile.
template <int ROWS, int OUTC, bool ROWS_OUTER = false>
__device__ __forceinline__ TileCoord decode_tile(const Args &g, int L, int tiles, int nk) {
    const int split = L / tiles;
    L -= split * tiles;
    const int gm = L / g.n_ntiles;
    const int e = g.tile_e[gm];
    const int st = g.tile_start[e];
    const int mt_e = g.tile_start[e + 1] - st;
    const int local = L - st * g.n_ntiles;
    const int nt = ROWS_OUTER ? local % g.n_ntiles : local / mt_e;
    const int mt = ROWS_OUTER ? local / g.n_ntiles : local - nt * mt_e;
    TileCoord c;
    c.e = e;
    c.m0 = g.offsets[e] + mt * ROWS;
    c.mend = g.offsets[e + 1];
    c.n0 = nt * OUTC;
    c.split = split;
    c.kb0 = split * g.kb_per_split;
    c.kb1 = min(nk, c.kb0 + g.kb_per_split);
    return c;
}

// Token rows a tile covers, rounded up to the MMA's N granularity of 16
// (NT = 256 geometry; rows past the expert's end are computed, never stored).
template <int ROWS>
__device__ __forceinline__ int tile_n16(const TileCoord &c) {
    const int r = min(ROWS, c.mend - c.m0);
    return (r + 15) & ~15;
}

__device__ __forceinline__ uint4 pack_bf16x8(const float *v) {
    uint4 u;
    uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&b);
    }
    return u;
}

// fp32 results of this warp's 32 TMEM lanes (rows row0 .. row0 + 31) and BNT
// columns from taddr, stored to O [rows, ldc] through the warp's staging
// block stg [32][EC + 4]: lane = row in, EC/4 lanes per row out, so that a
// warp store writes whole EC*4-byte row segments of 32/(EC/4) rows.
template <int EC, int BNT>
__device__ __forceinline__ void store_f32_rows(uint32_t taddr, float *stg, int lane, float *O,
                                               int ldc, int row0, int mend, int n0, int N) {
    constexpr int ES = EC + 4, LPR = EC / 4, RPI = 32 / LPR;
#pragma unroll 1
    for (int cc = 0; cc < BNT; cc += EC) {
        float v[EC];
#pragma unroll
        for (int h = 0; h < EC; h += 16) tmem_ld16(taddr + cc + h, v + h);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < EC / 4; ++q)
            *reinterpret_cast<float4 *>(stg + lane * ES + 4 * q) =
                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        __syncwarp();
        const int col = n0 + cc + 4 * (lane % LPR);
#pragma unroll
        for (int it = 0; it < 32 / RPI; ++it) {
            const int r = RPI * it + lane / LPR;
            const float4 q = *reinterpret_cast<const float4 *>(stg + r * ES + 4 * (lane % LPR));
            if (row0 + r < mend && col < N)
                *reinterpret_cast<float4 *>(O + (size_t)(row0 + r) * ldc + col) = q;
        }
        __syncwarp();
    }
}

template <int MODE, int NT, int BN, int MH>
__global__ void __launch_bounds__(256, 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmA64,
                       const __grid_constant__ CUtensorMap tmA32,
                       const __grid_constant__ CUtensorMap tmA16,
                       const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1, Args g) {
    using G = Geo<MODE, NT, BN, MH>;
    constexpr int STAGES = G::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * G::STAGE_BYTES);
    // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], done[1]
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t tfull0 = smem_u32(bars + 2 * STAGES), tempty0 = smem_u32(bars + 2 * STAGES + 2);
    const uint32_t done_bar = smem_u32(bars + 2 * STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // swapped epilogue: per epilogue warp a [16 tokens][32 features] bf16 block
    __nv_bfloat16 *epi_stage =
        reinterpret_cast<__nv_bfloat16 *>(smem + STAGES * G::STAGE_BYTES + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, 4);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int tiles = (*g.n_mtiles) * g.n_ntiles;
    const int total = tiles * g.k_splits;
    const int nk = (g.K + BK - 1) / BK;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0;       // stages that received a load
        uint32_t issued_par = 0;   // bit s: phase parity of stage s's last load
        bool ok = true;
        for (int L = blockIdx.x, it = 0; L < total && ok; L += gridDim.x, ++it) {
            const TileCoord c = decode_tile<G::ROWS, G::OUTC, MODE == GEMM_LOGITS>(g, L, tiles, nk);
            const bool rev = serpentine<MODE, NT>(it);
            int b0, b1;
            if (G::SWAP) { b0 = c.e * g.b_rows + c.n0; b1 = b0; }
            else if (MODE == GEMM_UP_SWIGLU) { b0 = c.e * g.b_rows + c.n0; b1 = b0; }
            else { b0 = c.e * g.b_rows + c.n0; b1 = b0 + BN / 2; }
            const int n16 = G::VARN ? tile_n16<G::ROWS>(c) : G::ROWS;
            const uint32_t stage_tx = G::W_BYTES + n16 * BK * 2;
            for (int i = 0; i < c.kb1 - c.kb0; ++i) {
                const int kb = rev ? c.kb1 - 1 - i : c.kb0 + i;
                if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) { ok = false; break; }
                const uint32_t fb = full0 + 8 * stage;
                mbar_expect_tx(fb, stage_tx);
                const uint32_t sa = smem_u32(smem + stage * G::STAGE_BYTES);
                const uint32_t sb = sa + G::ACT_BYTES;
                const int ka = (kb * BK) % g.a_k_period;
                if (G::VARN) {
                    // n16 token rows as boxes of 128, 64, 32 and 16 rows
                    int r = 0;
                    for (; r + 128 <= n16; r += 128)
                        tma_load_2d(sa + r * BK * 2, &tmA, ka, c.m0 + r, fb);
                    if (n16 - r >= 64) {
                        tma_load_2d(sa + r * BK * 2, &tmA64, ka, c.m0 + r, fb);
                        r += 64;
                    }
                    if (n16 - r >= 32) {
                        tma_load_2d(sa + r * BK * 2, &tmA32, ka, c.m0 + r, fb);
                        r += 32;
                    }
                    if (n16 - r >= 16) tma_load_2d(sa + r * BK * 2, &tmA16, ka, c.m0 + r, fb);
                } else {
                    tma_load_2d(sa, &tmA, ka, c.m0, fb);
                }
                tma_load_2d(sb, &tmB0, kb * BK, b0, fb);
                if (!G::SWAP || MODE == GEMM_UP_SWIGLU)
                    tma_load_2d(sb + G::BOX * BK * 2, &tmB1, kb * BK, b1, fb);
                issued |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
        }
        if (!ok) {
            // Let the copies already issued land before the CTA can exit: the
            // last load into stage s completes the full barrier's phase of
            // parity issued_par[s] (only this thread arrives on it, so that
            // phase stays the last completed one).
            for (int s = 0; s < STAGES; ++s) {
                if (!(issued >> s & 1u)) continue;
                const uint32_t par = issued_par >> s & 1u;
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(full0 + 8 * s, par) && globaltimer() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        constexpr uint32_t idesc_fixed = G::SWAP ? idesc_bf16(WROWS, NT) : idesc_bf16(BM, BN);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        // test hook: done_bar's first phase completes only at the commit
        // below, so this wait can only run out
        if (g_stall_mma && !mbar_wait(done_bar, 0, abort_flag)) ok = false;
        if constexpr (MODE == GEMM_LOGITS) {
            // a work item is a tile and a split of whole chains; chain 0 of
            // an item into S (columns 0-255), later chains into A (256-511);
            // sp, ap: uses of S and A so far (wait parities)
            uint32_t sp = 0, ap = 0;
            for (int L = blockIdx.x; L < total && ok; L += gridDim.x) {
                const int kbs = (L / tiles) * g.kb_per_split;
                const int kbe = min(nk, kbs + g.kb_per_split);
                const int nch = (kbe - kbs + g.chain_kb - 1) / g.chain_kb;
                for (int ch = 0; ch < nch; ++ch) {
                    const int slot = ch == 0 ? 0 : 1;
                    if (!mbar_wait(tempty0 + 8 * slot, (slot ? ap : sp) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (slot) ap ^= 1; else sp ^= 1;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + slot * ACC_COLS;
                    const int kb0 = kbs + ch * g.chain_kb, kb1 = min(kbe, kb0 + g.chain_kb);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t sa = smem_u32(smem + stage * G::STAGE_BYTES);
                        const uint32_t sb = sa + G::ACT_BYTES;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            tc_mma(d_tmem, desc_sw128(sa + kk * 32), desc_sw128(sb + kk * 32),
                                   idesc_fixed, (kb > kb0 || kk > 0) ? 1u : 0u);
                        tc_commit(empty0 + 8 * stage);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    // A's commit also covers chain 0's MMAs into S
                    if (slot || nch == 1) tc_commit(tfull0 + 8 * slot);
                }
            }
        } else {
            for (int L = blockIdx.x, it = 0; L < total && ok; L += gridDim.x, ++it) {
                // The K range depends on the split alone; only the per-tile
                // width (NT = 256) needs the tile table here.
                const int kb0 = (L / tiles) * g.kb_per_split;
                const int kb1 = min(nk, kb0 + g.kb_per_split);
                uint32_t idesc = idesc_fixed;
                if (G::VARN)
                    idesc = idesc_bf16(
                        WROWS, tile_n16<G::ROWS>(decode_tile<G::ROWS, G::OUTC, MODE == GEMM_LOGITS>(g, L, tiles, nk)));
                if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
                // (the K blocks arrive in the producer's order; the first of
                // them starts the accumulator)
                for (int i = 0; i < kb1 - kb0; ++i) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * G::STAGE_BYTES);
                    const uint32_t sb = sa + G::ACT_BYTES;
    #pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint32_t accum = (i > 0 || kk > 0) ? 1u : 0u;
                        if (G::SWAP) {
                            // weights (M side) x tokens (N side)
                            tc_mma(d_tmem, desc_sw128(sb + kk * 32), desc_sw128(sa + kk * 32), idesc,
                                   accum);
                            if (MODE == GEMM_UP_SWIGLU)
                                tc_mma(d_tmem + NT, desc_sw128(sb + WROWS * BK * 2 + kk * 32),
                                       desc_sw128(sa + kk * 32), idesc, accum);
                        } else {
                            tc_mma(d_tmem, desc_sw128(sa + kk * 32), desc_sw128(sb + kk * 32), idesc,
                                   accum);
                            if (MH == 2)    // rows 128..255 of the tile into columns 256..511
                                tc_mma(d_tmem + BN, desc_sw128(sa + BM * BK * 2 + kk * 32),
                                       desc_sw128(sb + kk * 32), idesc, accum);
                        }
                    }
                    tc_commit(empty0 + 8 * stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit(tfull0 + 8 * acc);
                if (++acc == G::NACC) { acc = 0; acc_phase ^= 1; }
            }
        }
        // All MMAs of this thread complete before TMEM can be freed.
        tc_commit(done_bar);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(done_bar, 0) && globaltimer() - t0 < kWaitLimitNs) {
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue
        const int quarter = warp - 4;                     // TMEM lanes 32*quarter..
        if constexpr (MODE == GEMM_LOGITS) {
            uint32_t sf = 0, af = 0;   // fills of S and A seen so far (wait parities)
            float *stg = reinterpret_cast<float *>(epi_stage) + quarter * (32 * G::EPI_STRIDE);
            bool ok = true;
            for (int L = blockIdx.x; L < total && ok; L += gridDim.x) {
                const TileCoord c = decode_tile<G::ROWS, G::OUTC, MODE == GEMM_LOGITS>(g, L, tiles, nk);
                const int nch = (c.kb1 - c.kb0 + g.chain_kb - 1) / g.chain_kb;
                float *O = static_cast<float *>(g.C) + (size_t)c.split * g.split_stride;
                const uint32_t tS = tmem_base + ((uint32_t)(quarter * 32) << 16);
                const uint32_t tA = tS + ACC_COLS;
                if (nch == 1) {
                    if (!mbar_wait(tfull0, sf, abort_flag)) break;
                    sf ^= 1;
                    tc_fence_after();
                }
                // S += A after every later chain, in chain order
                for (int ch = 1; ch < nch; ++ch) {
                    if (!mbar_wait(tfull0 + 8, af, abort_flag)) { ok = false; break; }
                    af ^= 1;
                    tc_fence_after();
#pragma unroll 1
                    for (int cc = 0; cc < BN; cc += 16) {
                        float a[16], b[16];
                        tmem_ld16(tS + cc, a);
                        tmem_ld16(tA + cc, b);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) a[i] += b[i];
                        tmem_st16(tS + cc, a);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty0 + 8);
                }
                if (!ok) break;
                // S out as fp32 row segments through the staging block
                store_f32_rows<G::EPI_COLS, BN>(tS, stg, lane, O, g.ldc, c.m0 + quarter * 32,
                                                c.mend, c.n0, g.N);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty0);
            }
        } else {
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int L = blockIdx.x; L < total; L += gridDim.x) {
                const TileCoord c = decode_tile<G::ROWS, G::OUTC, MODE == GEMM_LOGITS>(g, L, tiles, nk);
                if (!mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag)) break;
                tc_fence_after();
                const uint32_t tbase0 =
                    tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * ACC_COLS;
                if (G::SWAP) {
                    const uint32_t tbase = tbase0;
                    // TMEM lane = output feature f, column = token row m0 + j.
                    const int f = c.n0 + quarter * 32 + lane;
                    const bool vf = f < g.N;
                    const bool raw = MODE == GEMM_DOWN || g.k_splits > 1;
                    // bf16 results (the activation h) leave through shared
                    // memory: lane = feature in, 16-byte vectors of 8 features of
                    // one token out
                    const bool bf16_out = !raw;
                    const int ncols = G::VARN ? tile_n16<G::ROWS>(c) : NT;
                    float *P = static_cast<float *>(g.C) + (size_t)c.split * g.split_stride;
                    __nv_bfloat16 *H = static_cast<__nv_bfloat16 *>(g.C);
                    __nv_bfloat16 *stg = epi_stage + quarter * (16 * 32);
    #pragma unroll 1
                    for (int j0 = 0; j0 < ncols; j0 += 16) {
                        float a[16], b[16];
                        tmem_ld16(tbase + j0, a);
                        if (MODE == GEMM_UP_SWIGLU) tmem_ld16(tbase + NT + j0, b);
                        tmem_ld_wait();
                        if (bf16_out) {
    #pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                float v;
                                if (MODE == GEMM_UP_SWIGLU) v = silu(a[i]) * b[i];
                                else v = fmaxf(a[i], 0.f);
                                stg[i * 32 + lane] = __float2bfloat16_rn(v);
                            }
                            __syncwarp();
    #pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                const int vi = lane + 32 * q, i = vi >> 2, part = vi & 3;
                                const int row = c.m0 + j0 + i;
                                const int fc = c.n0 + quarter * 32 + 8 * part;
                                if (row < c.mend && fc < g.N)
                                    *reinterpret_cast<uint4 *>(H + (size_t)row * g.ldc + fc) =
                                        *reinterpret_cast<const uint4 *>(stg + i * 32 + 8 * part);
                            }
                            __syncwarp();
                            continue;
                        }
    #pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int row = c.m0 + j0 + i;
                            if (!vf || row >= c.mend) continue;
                            if (raw) {
                                float *dst = P + (size_t)row * g.ldc + f;
                                dst[0] = a[i];
                                if (MODE == GEMM_UP_SWIGLU) dst[g.N] = b[i];
                            } else if (MODE == GEMM_UP_SWIGLU) {
                                H[(size_t)row * g.ldc + f] = __float2bfloat16_rn(silu(a[i]) * b[i]);
                            } else {
                                H[(size_t)row * g.ldc + f] = __float2bfloat16_rn(fmaxf(a[i], 0.f));
                            }
                        }
                    }
                } else {
    #pragma unroll 1
                  for (int hh = 0; hh < MH; ++hh) {    // 128-row halves (MH = 2)
                    const int row = c.m0 + hh * BM + quarter * 32 + lane;
                    const bool vrow = row < c.mend;
                    const uint32_t tbase = tbase0 + hh * BN;
                    if (MODE == GEMM_UP_SWIGLU) {
                        __nv_bfloat16 *H = static_cast<__nv_bfloat16 *>(g.C);
    #pragma unroll 1
                        for (int cc = 0; cc < BN / 2; cc += 16) {
                            float gt[16], up[16];
                            tmem_ld16(tbase + cc, gt);
                            tmem_ld16(tbase + BN / 2 + cc, up);
                            tmem_ld_wait();
                            float h[16];
    #pragma unroll
                            for (int i = 0; i < 16; ++i) h[i] = silu(gt[i]) * up[i];
                            const int col = c.n0 + cc;
                            if (vrow) {
                                __nv_bfloat16 *dst = H + (size_t)row * g.ldc + col;
                                if (col < g.N) *reinterpret_cast<uint4 *>(dst) = pack_bf16x8(h);
                                if (col + 8 < g.N)
                                    *reinterpret_cast<uint4 *>(dst + 8) = pack_bf16x8(h + 8);
                            }
                        }
                    } else if (MODE == GEMM_UP_RELU) {
                        __nv_bfloat16 *H = static_cast<__nv_bfloat16 *>(g.C);
    #pragma unroll 1
                        for (int cc = 0; cc < BN; cc += 16) {
                            float v[16];
                            tmem_ld16(tbase + cc, v);
                            tmem_ld_wait();
    #pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = fmaxf(v[i], 0.f);
                            const int col = c.n0 + cc;
                            if (vrow) {
                                __nv_bfloat16 *dst = H + (size_t)row * g.ldc + col;
                                if (col < g.N) *reinterpret_cast<uint4 *>(dst) = pack_bf16x8(v);
                                if (col + 8 < g.N)
                                    *reinterpret_cast<uint4 *>(dst + 8) = pack_bf16x8(v + 8);
                            }
                        }
                    } else {
                        // fp32 outputs: each warp stores its 32 rows as whole row
                        // segments through its staging block
                        float *O = static_cast<float *>(g.C) + (size_t)c.split * g.split_stride;
                        float *stg = reinterpret_cast<float *>(epi_stage) +
                                     quarter * (32 * G::EPI_STRIDE);
                        store_f32_rows<G::EPI_COLS, BN>(tbase, stg, lane, O, g.ldc,
                                                        c.m0 + hh * BM + quarter * 32, c.mend,
                                                        c.n0, g.N);
                    }
                  }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
                if (++acc == G::NACC) { acc = 0; acc_phase ^= 1; }
            }
    
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------- SM-pair tiles
// Tiles of 256 token rows x 256 MMA columns on a cluster of two CTAs (two
// SMs) with tcgen05.mma.cta_group::2 (M = 256).  CTA r of the pair stages
// rows m0 + 128 r .. + 127 of A and the r-th 128-row box of the weight tile
// (SwiGLU: r = 0 the W1 rows, r = 1 the same W3 rows; otherwise weight rows
// n0 + 128 r ..), so a stage is 32 KB per SM where the one-SM 128 x 256 tile
// needs 48 KB, and 6 (down) or 7 (up) stages fit.  The MMA reads each CTA's
// A rows from that CTA's shared memory and the two B boxes from both, and
// leaves each CTA's 128 rows x 256 columns in that CTA's TMEM, where the
// CTA's own epilogue reads them.  Two accumulators of 256 columns: a tile's
// epilogue overlaps the next tile's MMAs.
//   rank 0 (even CTA): the MMA issuer for both; its full barriers collect
//     both CTAs' TMA bytes; its commits arrive on both CTAs' barriers
//     (multicast); its accumulator-empty barriers count both epilogues.
//   rank 1: producer and epilogue only.
template <int MODE> struct PairGeo {
    static constexpr int A_BYTES = BM * BK * 2;              // 16 KB
    static constexpr int STAGE_BYTES = A_BYTES + WROWS * BK * 2;   // + 16 KB of weights
    static constexpr int EPI_COLS = 32;
    static constexpr int EPI_STRIDE = EPI_COLS + 4;
    static constexpr int EPI = MODE == GEMM_DOWN ? 4 * 32 * EPI_STRIDE * 4 : 0;
    static constexpr int EXTRA = kSmemBase + EPI;
    static constexpr int FIT = (kSmemLimit - EXTRA) / STAGE_BYTES;
    static constexpr int STAGES = FIT < 8 ? FIT : 8;
    static constexpr int OUTC = MODE == GEMM_UP_SWIGLU ? BNM / 2 : BNM;
    static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + EXTRA;
};
constexpr int kPairRows = 2 * BM;
// After an abort, how long a CTA waits for its own copies in flight: they
// land within microseconds, and rank 1 cannot observe their completion (it is
// counted on rank 0's barrier), so it waits this long.
constexpr uint64_t kPairDrainNs = 20000000ull;   // 20 ms

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of `addr` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// mbar_wait for a barrier that the other CTA of the pair arrives on.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int *abort_flag) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    const uint64_t limit = g_main_wait_limit_ns;
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit) {
            flag_error(kErrTimeout);
            *abort_flag = 1;
            return false;
        }
    }
}
// TMA load into this CTA's shared memory, completing on a barrier of either
// CTA of the pair (a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *tm, int c0,
                                                 int c1, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile"
        ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}
// Arrive on the barrier at offset `bar` in both CTAs of the pair once this
// thread's MMAs have completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar), "h"((uint16_t)3) : "memory");
}
__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB0,
                         const __grid_constant__ CUtensorMap tmB1, Args g) {
    using P = PairGeo<MODE>;
    constexpr int STAGES = P::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * P::STAGE_BYTES);
    // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], done[1]
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t tfull0 = smem_u32(bars + 2 * STAGES), tempty0 = smem_u32(bars + 2 * STAGES + 2);
    const uint32_t done_bar = smem_u32(bars + 2 * STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *epi_stage = reinterpret_cast<float *>(smem + STAGES * P::STAGE_BYTES + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);       // rank 0's arrive.expect_tx of both CTAs' bytes
            mbar_init(empty0 + 8 * s, 1);      // rank 0's commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);      // rank 0's commit
            mbar_init(tempty0 + 8 * a, 8);     // 4 epilogue warps of each CTA
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 2) {
        // one warp of each CTA allocates, collectively, the same columns in both
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync_all();      // both CTAs' barriers are initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int tiles = (*g.n_mtiles) * g.n_ntiles;
    const int nk = (g.K + BK - 1) / BK;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        const uint32_t full_r0 = map_to_rank(full0, 0);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0, issued_par = 0;
        bool ok = true;
        for (int L = pair, it = 0; L < tiles && ok; L += npairs, ++it) {
            const TileCoord c = decode_tile<kPairRows, P::OUTC>(g, L, tiles, nk);
            const CUtensorMap *tb = (MODE == GEMM_UP_SWIGLU && rank) ? &tmB1 : &tmB0;
            const int brow = c.e * g.b_rows + c.n0 + (MODE == GEMM_UP_SWIGLU ? 0 : WROWS * (int)rank);
            const bool rev = serpentine<MODE, 0>(it);
            for (int i = 0; i < c.kb1 - c.kb0; ++i) {
                const int kb = rev ? c.kb1 - 1 - i : c.kb0 + i;
                if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) { ok = false; break; }
                if (rank == 0) mbar_expect_tx(full0 + 8 * stage, 2 * P::STAGE_BYTES);
                const uint32_t sa = smem_u32(smem + stage * P::STAGE_BYTES);
                const uint32_t fb = full_r0 + 8 * stage;
                tma_load_2d_pair(sa, &tmA, (kb * BK) % g.a_k_period, c.m0 + BM * (int)rank, fb);
                tma_load_2d_pair(sa + P::A_BYTES, tb, kb * BK, brow, fb);
                issued |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
        }
        if (!ok) {
            // Let the copies already issued land before the CTA can exit.
            // Rank 0: the last load into stage s completes the phase of parity
            // issued_par[s] (once rank 1's bytes for it have landed too).
            // Rank 1 cannot see its copies complete; it waits the drain time.
            const uint64_t t0 = globaltimer();
            if (rank == 0) {
                for (int s = 0; s < STAGES; ++s) {
                    if (!(issued >> s & 1u)) continue;
                    const uint32_t par = issued_par >> s & 1u;
                    while (!mbar_try_wait(full0 + 8 * s, par) && globaltimer() - t0 < kPairDrainNs) {
                    }
                }
            } else {
                while (globaltimer() - t0 < kPairDrainNs) {
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        if (rank == 0) {
            // -------------------------------------------- MMA issuer (rank 0)
            constexpr uint32_t idesc = idesc_bf16(kPairRows, BNM);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            if (g_stall_mma && !mbar_wait(done_bar, 0, abort_flag)) ok = false;
            for (int L = pair; L < tiles && ok; L += npairs) {
                if (!mbar_wait_cluster(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
                for (int i = 0; i < nk; ++i) {   // in the producers' order (serpentine)
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * P::STAGE_BYTES);
                    const uint32_t sb = sa + P::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma_pair(d_tmem, desc_sw128(sa + kk * 32), desc_sw128(sb + kk * 32),
                                    idesc, (i > 0 || kk > 0) ? 1u : 0u);
                    tc_commit_pair(empty0 + 8 * stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit_pair(tfull0 + 8 * acc);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            // Every MMA of the pair completes (both CTAs' done barriers) before
            // either CTA frees its tensor memory.
            tc_commit_pair(done_bar);
        }
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(done_bar, 0) && globaltimer() - t0 < kWaitLimitNs) {
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue (both CTAs)
        const int quarter = warp - 4;
        const uint32_t tempty_r0 = map_to_rank(tempty0, 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int L = pair; L < tiles; L += npairs) {
            const TileCoord c = decode_tile<kPairRows, P::OUTC>(g, L, tiles, nk);
            if (!mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * ACC_COLS;
            const int row0 = c.m0 + BM * (int)rank + quarter * 32;
            const int row = row0 + lane;
            const bool vrow = row < c.mend;
            if (MODE == GEMM_UP_SWIGLU) {
                __nv_bfloat16 *H = static_cast<__nv_bfloat16 *>(g.C);
#pragma unroll 1
                for (int cc = 0; cc < BNM / 2; cc += 16) {
                    float gt[16], up[16];
                    tmem_ld16(tbase + cc, gt);
                    tmem_ld16(tbase + BNM / 2 + cc, up);
                    tmem_ld_wait();
                    float h[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) h[i] = silu(gt[i]) * up[i];
                    const int col = c.n0 + cc;
                    if (vrow) {
                        __nv_bfloat16 *dst = H + (size_t)row * g.ldc + col;
                        if (col < g.N) *reinterpret_cast<uint4 *>(dst) = pack_bf16x8(h);
                        if (col + 8 < g.N) *reinterpret_cast<uint4 *>(dst + 8) = pack_bf16x8(h + 8);
                    }
                }
            } else if (MODE == GEMM_UP_RELU) {
                __nv_bfloat16 *H = static_cast<__nv_bfloat16 *>(g.C);
#pragma unroll 1
                for (int cc = 0; cc < BNM; cc += 16) {
                    float v[16];
                    tmem_ld16(tbase + cc, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = fmaxf(v[i], 0.f);
                    const int col = c.n0 + cc;
                    if (vrow) {
                        __nv_bfloat16 *dst = H + (size_t)row * g.ldc + col;
                        if (col < g.N) *reinterpret_cast<uint4 *>(dst) = pack_bf16x8(v);
                        if (col + 8 < g.N) *reinterpret_cast<uint4 *>(dst + 8) = pack_bf16x8(v + 8);
                    }
                }
            } else {
                float *O = static_cast<float *>(g.C);
                float *stg = epi_stage + quarter * (32 * P::EPI_STRIDE);
                store_f32_rows<P::EPI_COLS, BNM>(tbase, stg, lane, O, g.ldc, row0, c.mend, c.n0,
                                                 g.N);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(tempty_r0 + 8 * acc);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    tc_fence_before();
    __syncthreads();
    // Neither CTA leaves while the other may still reach its shared memory
    // (rank 0's MMAs read rank 1's, the barriers are signalled across).
    cluster_sync_all();
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
    }
    cluster_sync_all();
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D bf16 tensor [rows, K] (K contiguous), box [box_rows, 64], 128-B swizzle.
static bool make_map(CUtensorMap *m, const void *base, long long rows, long long K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// moe_debug_set_wait_hooks: the current device's copies of the test hooks.
cudaError_t set_wait_hooks(unsigned long long main_limit_ns, int stall_mma) {
    cudaError_t e = cudaMemcpyToSymbol(tc::g_main_wait_limit_ns, &main_limit_ns,
                                       sizeof(main_limit_ns));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(tc::g_stall_mma, &stall_mma, sizeof(stall_mma));
}

static int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

struct Maps {
    CUtensorMap a, a64, a32, a16, b0, b1;
};

template <int MODE, int NT, int BN, int MH = 1>
static cudaError_t launch_geo(const Maps &m, const Args &g, cudaStream_t st) {
    using G = Geo<MODE, NT, BN, MH>;
    static_assert(G::SMEM <= (size_t)kSmemLimit, "shared memory");
    auto kern = grouped_gemm_tc_kernel<MODE, NT, BN, MH>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G::SMEM);
    if (err != cudaSuccess) return err;
    kern<<<num_sms(), 256, G::SMEM, st>>>(m.a, m.a64, m.a32, m.a16, m.b0, m.b1, g);
    note_launch();
    return cudaGetLastError();
}

// SM-pair geometry: as many pairs as can be resident at once (clusters of two
// CTAs of about 200 KB of shared memory each), every pair persistent.
template <int MODE>
static cudaError_t launch_pair(const Maps &m, const Args &g, cudaStream_t st) {
    using P = PairGeo<MODE>;
    static_assert(P::SMEM <= (size_t)kSmemLimit, "shared memory");
    auto kern = grouped_gemm_pair_kernel<MODE>;
    static int grid = 0;
    if (!grid) {
        cudaError_t err =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P::SMEM);
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(num_sms());
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = P::SMEM;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            clusters = num_sms() / 2;
        }
        grid = 2 * std::min(clusters, num_sms() / 2);
    }
    kern<<<grid, 256, P::SMEM, st>>>(m.a, m.b0, m.b1, g);
    note_launch();
    return cudaGetLastError();
}

template <int MODE>
static cudaError_t launch_mode(int nt, int bn, int mh, const Maps &m, const Args &g,
                               cudaStream_t st) {
    switch (nt) {
        case 0:
            if (mh == TILE_ROWS_256_PAIR) {
                if constexpr (MODE == GEMM_LOGITS) return cudaErrorInvalidValue;
                else return launch_pair<MODE>(m, g, st);
            }
            if (mh == 2) return launch_geo<MODE, 0, BNM, 2>(m, g, st);
            return bn == BNM ? launch_geo<MODE, 0, BNM>(m, g, st)
                             : launch_geo<MODE, 0, BNM / 2>(m, g, st);
        case 16: return launch_geo<MODE, 16, BNM>(m, g, st);
        case 32: return launch_geo<MODE, 32, BNM>(m, g, st);
        case 64: return launch_geo<MODE, 64, BNM>(m, g, st);
        case kVarRows:
            if constexpr (MODE != GEMM_LOGITS) return launch_geo<MODE, kVarRows, BNM>(m, g, st);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tc

// A [a_rows, a_cols], weights B0/B1 [E*b_rows, K]; tile table from
// launch_build_tiles with row tiles of 128 (nt = 0) or nt rows (nt = 16, 32,
// 64, 256: weights on the MMA's M side; 256 sets the MMA N per tile).  bn (nt = 0 only): MMA N of 256 or 128; 128 doubles the
// output tiles when there are too few to fill the SMs.  mh (nt = 0, bn = 256
// only; tile table built with 256-row tiles): TILE_ROWS_256, 256-row tiles on
// one SM; TILE_ROWS_256_PAIR, 256-row tiles on an SM pair (the up and down
// modes, k_splits = 1).  A's column for
// reduction index k is k mod a_k_period (a_k_period = K: no wrap).  With k_splits > 1 split s of
// every tile writes fp32 partial sums to C + s * split_stride: GEMM_DOWN
// always (row-major [rows, ldc]); the up modes only with nt > 0, writing the
// pre-activation sums (SwiGLU: W1 part at column f, W3 part at N + f).
// k_splits = 1 up modes write the activation in bf16; GEMM_DOWN writes fp32.
// GEMM_LOGITS (nt = 0, bn = 256 or 224, mh = 1): the reduction is cut into chains of
// chain_kb K blocks, and k_splits splits of whole chains; each split sums its
// chains on chip in chain order and writes one fp32 plane.
cudaError_t launch_tc_gemm(int mode, int nt, int bn, int mh, const void *A, long long a_rows,
                           int a_cols,
                           const void *B0, const void *B1, int E, int b_rows, int N, int K,
                           int a_k_period, int k_splits, long long split_stride,
                           const int32_t *tile_e, const int32_t *tile_start,
                           const int32_t *n_mtiles, const int32_t *offsets, void *C, int ldc,
                           cudaStream_t st, int chain_kb) {
    using namespace tc;
    if (a_rows == 0) return cudaSuccess;
    const int nk = (K + BK - 1) / BK;
    if (nt != 0 && nt != 16 && nt != 32 && nt != 64 && nt != kVarRows) return cudaErrorInvalidValue;
    if (bn != BNM && bn != BNM / 2 && !(mode == GEMM_LOGITS && bn == kLogitsN224))
        return cudaErrorInvalidValue;
    if (mh != 1 && ((mh != 2 && mh != TILE_ROWS_256_PAIR) || nt != 0 || bn != BNM))
        return cudaErrorInvalidValue;
    if (mh == TILE_ROWS_256_PAIR && (k_splits != 1 || mode == GEMM_LOGITS || a_k_period != K))
        return cudaErrorInvalidValue;
    if (mode == GEMM_LOGITS &&
        (nt != 0 || (bn != BNM && bn != kLogitsN224) || mh != 1 || chain_kb < 1))
        return cudaErrorInvalidValue;
    if (k_splits < 1 || (k_splits > 1 && mode != GEMM_DOWN && mode != GEMM_LOGITS && nt == 0) ||
        (a_k_period % BK != 0 && a_k_period != K))
        return cudaErrorInvalidValue;
    // GEMM_LOGITS: a split holds whole chains of chain_kb K blocks
    const int chains = mode == GEMM_LOGITS ? (nk + chain_kb - 1) / chain_kb : nk;
    const int unit = mode == GEMM_LOGITS ? chain_kb : 1;
    const int kbps = (chains + k_splits - 1) / k_splits * unit;
    k_splits = (nk + kbps - 1) / kbps;          // every split gets at least one K block
    const bool var = nt == kVarRows;
    if (var && mode == GEMM_LOGITS) return cudaErrorInvalidValue;
    // rows of one A box: one CTA's share of a tile
    const int rows = var ? 128 : nt ? nt : mh == TILE_ROWS_256_PAIR ? BM : BM * mh;
    Maps m;
    if (!make_map(&m.a, A, a_rows, a_cols, rows)) return cudaErrorInvalidValue;
    m.a64 = m.a32 = m.a16 = m.a;
    if (var && (!make_map(&m.a64, A, a_rows, a_cols, 64) ||
                !make_map(&m.a32, A, a_rows, a_cols, 32) ||
                !make_map(&m.a16, A, a_rows, a_cols, 16)))
        return cudaErrorInvalidValue;
    const int box = nt ? WROWS : bn / 2;
    if (!make_map(&m.b0, B0, (long long)E * b_rows, K, box)) return cudaErrorInvalidValue;
    if (!make_map(&m.b1, B1 ? B1 : B0, (long long)E * b_rows, K, box))
        return cudaErrorInvalidValue;
    const int outc = nt ? WROWS : (mode == GEMM_UP_SWIGLU ? bn / 2 : bn);
    Args g;
    g.mode = mode;
    g.N = N;
    g.K = K;
    g.a_k_period = a_k_period;
    g.n_ntiles = (N + outc - 1) / outc;
    g.b_rows = b_rows;
    g.k_splits = k_splits;
    g.kb_per_split = kbps;
    g.split_stride = split_stride;
    g.tile_e = tile_e;
    g.tile_start = tile_start;
    g.n_mtiles = n_mtiles;
    g.offsets = offsets;
    g.C = C;
    g.ldc = ldc;
    g.chain_kb = chain_kb;
    if (mode == GEMM_UP_SWIGLU) return launch_mode<GEMM_UP_SWIGLU>(nt, bn, mh, m, g, st);
    if (mode == GEMM_UP_RELU) return launch_mode<GEMM_UP_RELU>(nt, bn, mh, m, g, st);
    if (mode == GEMM_LOGITS)
        return bn == kLogitsN224 ? launch_geo<GEMM_LOGITS, 0, kLogitsN224>(m, g, st)
                                 : launch_geo<GEMM_LOGITS, 0, BNM>(m, g, st);
    return launch_mode<GEMM_DOWN>(nt, bn, mh, m, g, st);
}

}  // namespace moe
