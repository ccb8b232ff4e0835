// Capacity overflow sent to the next-best experts instead of being dropped.
//
// Source: "Mixture of Experts" (waylandz.com LLM book, ch. 30) §30.5.2:
// tokens beyond an expert's capacity are dropped or redirected to the next
// best expert.  The rule computed here, in rounds:
//   round 0   the plain capacity rule: slots in flattened (t*k + j) order, a
//             slot is served by its expert while the expert has room (C rows);
//   round r   every slot still unserved takes its token's next unused expert
//             down the token's score ranking (the token's unserved slots in
//             j order take consecutive candidates), and the slots are served
//             in (t*k + j) order by experts that still have room;
//   at the end, slots still unserved are dropped.  An expert's rows are
//   grouped in the order they were served (round 0 first).
// Every round is a histogram / scan / in-order scatter over chunks of 1024
// slots, like the plain dispatch; all integer work, exactly reproducible.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Round-0 state: each slot targets its top-k expert with its gate weight.
__global__ void rr_init_kernel(const int32_t *topk_idx, const float *topk_w, long long n, int k,
                               int E, int32_t *slot_e, float *slot_w, int32_t *served,
                               int32_t *nxt) {
    for (long long f = blockIdx.x * (long long)blockDim.x + threadIdx.x; f < n;
         f += (long long)gridDim.x * blockDim.x) {
        int e = topk_idx[f];
        if (e < 0 || e >= E) {
            flag_error(kErrBadIndex);
            e = -1;
        }
        slot_e[f] = e;
        slot_w[f] = topk_w[f];
        served[f] = -1;
        if (f % k == 0) nxt[f / k] = 0;
    }
}

// Unserved live slots of token t take its next candidates, in slot order.
__global__ void rr_next_kernel(long long T, int k, int n_cand, int E, const int32_t *cand_idx,
                               const float *cand_w, int32_t *slot_e, float *slot_w,
                               const int32_t *served, int32_t *nxt) {
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < T;
         t += (long long)gridDim.x * blockDim.x) {
        int q = nxt[t];
        for (int j = 0; j < k; ++j) {
            const long long f = t * k + j;
            if (served[f] >= 0 || slot_e[f] < 0) continue;
            if (q < n_cand) {
                int e = cand_idx[t * n_cand + q];
                if (e < 0 || e >= E) {
                    flag_error(kErrBadIndex);
                    e = -1;
                }
                slot_e[f] = e;
                slot_w[f] = cand_w[t * n_cand + q];
                ++q;
            } else {
                slot_e[f] = -1;        // no candidate left: dropped
            }
        }
        nxt[t] = q;
    }
}

// Per-chunk histogram of the targets of the slots still looking for an expert.
__global__ void rr_hist_kernel(const int32_t *slot_e, const int32_t *served, long long n, int E,
                               int32_t *hist) {
    extern __shared__ int h[];
    for (int i = threadIdx.x; i < E; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const long long base = (long long)blockIdx.x * kDispatchChunk;
    for (int i = threadIdx.x; i < kDispatchChunk && base + i < n; i += blockDim.x) {
        const long long f = base + i;
        const int e = slot_e[f];
        if (served[f] < 0 && e >= 0) atomicAdd(&h[e], 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) hist[(size_t)blockIdx.x * E + i] = h[i];
}

// One CTA, thread e: per-chunk bases of this round's slots of expert e, the
// rows the expert held before the round and after it (at most C).
__global__ void __launch_bounds__(1024) rr_scan_kernel(const int32_t *hist, int nblk, int E,
                                                       long long C, int round,
                                                       int32_t *block_base, int32_t *filled,
                                                       int32_t *filled_before,
                                                       int32_t *counts) {
    const int e = threadIdx.x;
    if (e >= E) return;
    int run = 0;
    for (int b0 = 0; b0 < nblk; b0 += 8) {
        int hv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) hv[u] = b0 + u < nblk ? hist[(size_t)(b0 + u) * E + e] : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (b0 + u < nblk) block_base[(size_t)(b0 + u) * E + e] = run;
            run += hv[u];
        }
    }
    const int fb = round == 0 ? 0 : filled[e];
    const long long room = C - fb > 0 ? C - fb : 0;
    filled_before[e] = fb;
    filled[e] = fb + (int)((long long)run < room ? run : room);
    if (counts) counts[e] = run;
}

// Per chunk, 8 warps each walk 128 of its slots in order: the rank of a live
// slot among this round's slots of its expert is block_base + earlier slots
// of the same expert in the chunk (in earlier warps' ranges, counted first,
// then in its own warp); it is served when the rank fits in the room left.
constexpr int kRrWarps = 8;
constexpr int kRrSlots = kDispatchChunk / kRrWarps;
__global__ void __launch_bounds__(32 * kRrWarps) rr_scatter_kernel(
        const int32_t *slot_e, int32_t *served, long long n, int E, long long C,
        const int32_t *block_base, const int32_t *filled_before) {
    extern __shared__ int sh[];    // [kRrWarps][E] counts, then ranks; [E] rows before the round
    int *fb = sh + kRrWarps * E;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kRrWarps * E; i += blockDim.x) sh[i] = 0;
    for (int i = threadIdx.x; i < E; i += blockDim.x) fb[i] = filled_before[i];
    __syncthreads();
    const long long base = (long long)blockIdx.x * kDispatchChunk + warp * kRrSlots;
    constexpr int kIter = kRrSlots / 32;
    int *run = sh + warp * E;
    int ev[kIter];
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        const long long f = base + it * 32 + lane;
        const int e = (f < n && served[f] < 0) ? slot_e[f] : -1;
        ev[it] = e;
        if (e >= 0) atomicAdd(&run[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int r = block_base[(size_t)blockIdx.x * E + e];
        for (int w = 0; w < kRrWarps; ++w) {
            const int c = sh[w * E + e];
            sh[w * E + e] = r;
            r += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        if (base + it * 32 >= n) break;
        const long long f = base + it * 32 + lane;
        const int e = ev[it];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int rank = 0;
        if (e >= 0) rank = run[e] + __popc(peers & lanemask_lt());
        __syncwarp();
        if (e >= 0 && lane == 31 - __clz(peers)) run[e] += __popc(peers);
        __syncwarp();
        if (e >= 0 && (long long)rank < C - fb[e]) served[f] = fb[e] + rank;
    }
}

// offsets = exclusive scan of the rows each expert serves; n_dropped.
__global__ void __launch_bounds__(1024) rr_offsets_kernel(const int32_t *filled, int E,
                                                          long long n, int32_t *offsets,
                                                          int32_t *n_dropped) {
    __shared__ int warp_tot[32];
    __shared__ int total;
    const int e = threadIdx.x;
    const int v = e < E ? filled[e] : 0;
    const int ex = block_exclusive_scan_1024(v, warp_tot, &total);
    if (e < E) offsets[e] = ex;
    if (e == 0) {
        offsets[E] = total;
        *n_dropped = (int)(n - total);
    }
}

// Grouped layout and the per-slot result.
__global__ void rr_final_kernel(const int32_t *slot_e, const float *slot_w, const int32_t *served,
                                const int32_t *offsets, long long n, int32_t *perm, int32_t *inv,
                                int32_t *slot_expert, float *slot_w_out) {
    for (long long f = blockIdx.x * (long long)blockDim.x + threadIdx.x; f < n;
         f += (long long)gridDim.x * blockDim.x) {
        const int r = served[f];
        if (r >= 0) {
            const int e = slot_e[f];
            const int row = offsets[e] + r;
            perm[row] = (int32_t)f;
            inv[f] = row;
            if (slot_expert) slot_expert[f] = e;
            if (slot_w_out) slot_w_out[f] = slot_w[f];
        } else {
            inv[f] = -1;
            if (slot_expert) slot_expert[f] = -1;
            if (slot_w_out) slot_w_out[f] = 0.f;
        }
    }
}

static inline int grid_for(long long n) {
    return (int)std::min<long long>((n + 255) / 256, 148 * 8);
}

cudaError_t launch_dispatch_reroute(const int32_t *topk_idx, const float *topk_w,
                                    const int32_t *cand_idx, const float *cand_w, int n_cand,
                                    long long T, int k, int E, long long C, int rounds,
                                    const RerouteWork &w, int32_t *counts, int32_t *offsets,
                                    int32_t *perm, int32_t *inv, int32_t *slot_expert,
                                    float *slot_w_out, int32_t *n_dropped, cudaStream_t st) {
    const long long n = T * k;
    const int nblk = dispatch_blocks(n);
    if (n > 0) {
        rr_init_kernel<<<grid_for(n), 256, 0, st>>>(topk_idx, topk_w, n, k, E, w.slot_e,
                                                    w.slot_w, w.served, w.nxt);
        note_launch();
    }
    for (int r = 0; r <= rounds; ++r) {
        if (r > 0 && n > 0) {
            rr_next_kernel<<<grid_for(T), 256, 0, st>>>(T, k, n_cand, E, cand_idx, cand_w,
                                                        w.slot_e, w.slot_w, w.served, w.nxt);
            note_launch();
        }
        if (nblk > 0) {
            rr_hist_kernel<<<nblk, 256, sizeof(int) * E, st>>>(w.slot_e, w.served, n, E, w.hist);
            note_launch();
        }
        rr_scan_kernel<<<1, 1024, 0, st>>>(w.hist, nblk, E, C, r, w.block_base, w.filled,
                                           w.filled_before, r == 0 ? counts : nullptr);
        note_launch();
        if (nblk > 0) {
            rr_scatter_kernel<<<nblk, 32 * kRrWarps, (kRrWarps + 1) * sizeof(int) * E, st>>>(
                w.slot_e, w.served, n, E, C, w.block_base, w.filled_before);
            note_launch();
        }
    }
    rr_offsets_kernel<<<1, 1024, 0, st>>>(w.filled, E, n, offsets, n_dropped);
    note_launch();
    if (n > 0) {
        rr_final_kernel<<<grid_for(n), 256, 0, st>>>(w.slot_e, w.slot_w, w.served, offsets, n,
                                                     perm, inv, slot_expert, slot_w_out);
        note_launch();
    }
    return cudaGetLastError();
}

}  // namespace moe
