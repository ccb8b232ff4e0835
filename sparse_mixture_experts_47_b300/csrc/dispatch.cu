// Dispatch: group the T*k (token, slot) assignments by expert, keeping the
// flattened (t*k + j) order inside each expert, and apply the capacity cap.
//
// Sources: "混合エキスパートモデル（MoE）実践" (deepseekmodel.com), expert
// parallelism section (stable argsort by destination, bincount; the grouped
// layout is what makes one grouped GEMM over all experts possible) and the
// capacity section (hard cap C per expert, overflow dropped).
//
// Three launches, all integer work and exactly reproducible:
//   1. per-chunk histograms hist[b][e] (chunks of 1024 slots),
//   2. one CTA: counts[e] = sum_b hist[b][e], per-chunk bases
//      base[b][e] = sum_{b'<b} hist[b'][e], offsets = exclusive scan of
//      min(counts, C), n_dropped,
//   3. per chunk, 8 warps each walk 128 of its slots in order; the rank of
//      a slot in its expert is base[b][e] + (earlier slots of e in the
//      chunk: in earlier warps' ranges, counted first, then in its own warp,
//      found with __match_any_sync); rank < C keeps the slot at row
//      offsets[e] + rank.
// A batch of at most one chunk (T*k <= 1024) runs the three steps in one
// CTA instead, with the same results.  In the layer, the CTA that computes
// the offsets (step 2, or the one-CTA form) also computes the load
// statistics and the up projection's tile table from them (DispatchTail).
#include "block_ops.cuh"
#include "common.cuh"
#include "kernels.h"

namespace moe {

__global__ void dispatch_hist_kernel(const int32_t *idx, long long n, int E, int32_t *hist) {
    extern __shared__ int h[];
    for (int i = threadIdx.x; i < E; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const long long base = (long long)blockIdx.x * kDispatchChunk;
    for (int i = threadIdx.x; i < kDispatchChunk && base + i < n; i += blockDim.x) {
        const int e = idx[base + i];
        if (e >= 0 && e < E) atomicAdd(&h[e], 1);
        else flag_error(kErrBadIndex);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) hist[(size_t)blockIdx.x * E + i] = h[i];
}

// Exclusive scan of one value per thread over a 1024-thread block.
__device__ int block_exclusive_scan_1024(int v, int *warp_tot, int *total) {
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
        int wt = warp_tot[lane], wi = wt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        warp_tot[lane] = wi - wt;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    return warp_tot[warp] + incl - v;
}

__global__ void __launch_bounds__(1024) dispatch_scan_kernel(
        const int32_t *hist, int nblk, int E, long long C, int32_t *block_base,
        int32_t *counts, int32_t *offsets, int32_t *n_dropped, DispatchTail tail) {
    __shared__ int warp_tot[32];
    __shared__ int total;
    const int e = threadIdx.x;
    int kept = 0, run = 0;
    if (e < E) {
        // 8 histogram loads in flight per step; the running sum stays in order
        for (int b0 = 0; b0 < nblk; b0 += 8) {
            int hv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                hv[u] = b0 + u < nblk ? hist[(size_t)(b0 + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (b0 + u < nblk && block_base) block_base[(size_t)(b0 + u) * E + e] = run;
                run += hv[u];
            }
        }
        if (counts) counts[e] = run;
        kept = (long long)run < C ? run : (int)C;
    }
    block_exclusive_scan_1024(run, warp_tot, &total);
    const int all_total = total;
    __syncthreads();
    const int ex = block_exclusive_scan_1024(kept, warp_tot, &total);
    if (offsets && e < E) offsets[e] = ex;
    if (e == 0) {
        if (offsets) offsets[E] = total;
        if (n_dropped) *n_dropped = all_total - total;
    }
    if (tail.stats || tail.tile_rows > 0 || tail.p_nblk > 0) {
        __syncthreads();
        dispatch_tail(tail, run, E, offsets);
    }
}

// One CTA of kScatterWarps warps per chunk; warp w walks its kScatterSlots
// consecutive slots of the chunk in order.  Its starting rank in expert e is
// the chunk's base[b][e] plus the slots of e in the chunk's earlier warps,
// so the ranks are those of one in-order walk over the chunk.  The expert
// indices are loaded up front and the ranks and offsets kept in shared
// memory, so each walk touches only registers and shared memory.
constexpr int kScatterWarps = 8;
constexpr int kScatterSlots = kDispatchChunk / kScatterWarps;
__global__ void __launch_bounds__(32 * kScatterWarps) dispatch_scatter_kernel(
        const int32_t *idx, long long n, int E, long long C, const int32_t *block_base,
        const int32_t *offsets, int32_t *perm, int32_t *inv) {
    extern __shared__ int sh[];          // [kScatterWarps][E] counts, then ranks; [E] offsets
    int *off = sh + kScatterWarps * E;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kScatterWarps * E; i += blockDim.x) sh[i] = 0;
    for (int i = threadIdx.x; i < E; i += blockDim.x) off[i] = offsets[i];
    __syncthreads();
    const long long base = (long long)blockIdx.x * kDispatchChunk + warp * kScatterSlots;
    constexpr int kIter = kScatterSlots / 32;
    int *run = sh + warp * E;
    int ev[kIter];
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        const long long f = base + it * 32 + lane;
        int e = -1;
        if (f < n) {
            e = idx[f];
            if (e < 0 || e >= E) e = -1;
        }
        ev[it] = e;
        if (e >= 0) atomicAdd(&run[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int r = block_base[(size_t)blockIdx.x * E + e];
        for (int w = 0; w < kScatterWarps; ++w) {
            const int c = sh[w * E + e];
            sh[w * E + e] = r;
            r += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        const long long f = base + it * 32 + lane;
        if (base + it * 32 >= n) break;
        const int e = ev[it];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int rank = 0;
        if (e >= 0) rank = run[e] + __popc(peers & lanemask_lt());
        __syncwarp();
        if (e >= 0 && lane == 31 - __clz(peers)) run[e] += __popc(peers);
        __syncwarp();
        if (f < n) {
            if (e >= 0 && rank < C) {
                const int s = off[e] + rank;
                perm[s] = (int32_t)f;
                inv[f] = s;
            } else {
                inv[f] = -1;
            }
        }
    }
}

// n <= kDispatchChunk slots: histogram, counts and offsets, then warp 0's
// in-order walk, in one CTA of 1024 threads (E <= 1024).
__global__ void __launch_bounds__(1024) dispatch_small_kernel(const int32_t *idx, int n, int E,
                                                              long long C, int32_t *counts,
                                                              int32_t *offsets, int32_t *perm,
                                                              int32_t *inv, int32_t *n_dropped,
                                                              DispatchTail tail) {
    extern __shared__ int sh[];          // [E] counts, then running ranks; [E] offsets
    int *h = sh, *off = sh + E;
    __shared__ int warp_tot[32];
    __shared__ int total;
    const int tid = threadIdx.x;
    for (int i = tid; i < E; i += blockDim.x) h[i] = 0;
    __syncthreads();
    if (tid < n) {
        const int e = idx[tid];
        if (e >= 0 && e < E) atomicAdd(&h[e], 1);
        else flag_error(kErrBadIndex);
    }
    __syncthreads();
    int run = 0, kept = 0;
    if (tid < E) {
        run = h[tid];
        kept = (long long)run < C ? run : (int)C;
        if (counts) counts[tid] = run;
    }
    block_exclusive_scan_1024(run, warp_tot, &total);
    const int all_total = total;
    __syncthreads();
    const int ex = block_exclusive_scan_1024(kept, warp_tot, &total);
    if (tid < E) {
        off[tid] = ex;
        h[tid] = 0;
        if (offsets) offsets[tid] = ex;
    }
    if (tid == 0) {
        if (offsets) offsets[E] = total;
        if (n_dropped) *n_dropped = all_total - total;
    }
    __syncthreads();
    if (tail.stats || tail.tile_rows > 0 || tail.p_nblk > 0) dispatch_tail(tail, run, E, offsets);
    if (tid >= 32) return;
    const int lane = tid;
    for (int b = 0; b < n; b += 32) {
        const int f = b + lane;
        int e = -1;
        if (f < n) {
            e = idx[f];
            if (e < 0 || e >= E) e = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int rank = 0;
        if (e >= 0) rank = h[e] + __popc(peers & lanemask_lt());
        __syncwarp();
        if (e >= 0 && lane == 31 - __clz(peers)) h[e] += __popc(peers);
        __syncwarp();
        if (f < n) {
            if (e >= 0 && rank < C) {
                const int s = off[e] + rank;
                perm[s] = f;
                inv[f] = s;
            } else {
                inv[f] = -1;
            }
        }
    }
}

cudaError_t launch_dispatch(const int32_t *idx, long long n, int E, int k, long long C,
                            int32_t *hist, int32_t *block_base, int32_t *counts,
                            int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *n_dropped,
                            cudaStream_t st, const DispatchTail *tail) {
    (void)k;
    DispatchTail t{};
    if (tail) {
        t = *tail;
        // the tail reads offsets and n_dropped as this launch writes them
        if ((t.tile_rows > 0 && !offsets) || (t.o.drop_ratio && t.o.n_dropped != n_dropped) ||
            (t.p_nblk > 0 && (E > 32 || !t.p_partial || !t.p_out)))
            return cudaErrorInvalidValue;
    }
    const int nblk = dispatch_blocks(n);
    if (nblk == 1) {
        dispatch_small_kernel<<<1, 1024, 2 * sizeof(int) * E, st>>>(
            idx, (int)n, E, C, counts, offsets, perm, inv, n_dropped, t);
        note_launch();
        return cudaGetLastError();
    }
    if (nblk > 0) {
        dispatch_hist_kernel<<<nblk, 256, sizeof(int) * E, st>>>(idx, n, E, hist);
        note_launch();
    }
    dispatch_scan_kernel<<<1, 1024, 0, st>>>(hist, nblk, E, C, block_base, counts, offsets,
                                             n_dropped, t);
    note_launch();
    if (nblk > 0) {
        dispatch_scatter_kernel<<<nblk, 32 * kScatterWarps,
                                  (kScatterWarps + 1) * sizeof(int) * E, st>>>(
            idx, n, E, C, block_base, offsets, perm, inv);
        note_launch();
    }
    return cudaGetLastError();
}

cudaError_t launch_histogram(const int32_t *idx, long long n, int E, int32_t *hist,
                             int32_t *counts, cudaStream_t st) {
    const int nblk = dispatch_blocks(n);
    if (nblk > 0) {
        dispatch_hist_kernel<<<nblk, 256, sizeof(int) * E, st>>>(idx, n, E, hist);
        note_launch();
    }
    dispatch_scan_kernel<<<1, 1024, 0, st>>>(hist, nblk, E, (long long)1 << 40, nullptr, counts,
                                             nullptr, nullptr, DispatchTail{});
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
