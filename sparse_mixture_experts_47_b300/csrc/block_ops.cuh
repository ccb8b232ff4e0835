// Block-wide steps shared by a standalone kernel and the dispatch kernels
// that run them after their offsets (one CTA; see DispatchTail).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

// Load statistics over the first n threads of a CTA (n a power of two,
// E <= n <= 1024, n <= the CTA's size; every thread of the CTA calls it),
// thread e < E holding count_e:
//   f_e = count_e / (T k); aux = E * sum_e f_e p_e (fp64, fixed tree order);
//   load = max_e count_e / (T k / E).
// The tree over n leaves adds the same nonzero terms in the same order as
// over 1024 (the other leaves are exact zeros), so the result does not
// depend on n.  Optional observability outputs (ObsArgs): drop_ratio =
// n_dropped / (T k); bias_mean_abs, bias_max_abs = mean and max |b_e| of the
// selection bias in effect.  p_out, if not p, receives a copy of p.
struct StatsSmem {
    double red[1024], redb[1024];
    float redbm[1024];
    int redmax[1024];
};
__device__ inline void block_load_stats(StatsSmem &sm, int n, int c, const float *p, int T,
                                        int E, int k, float *f, float *p_out, float *aux,
                                        float *load, const ObsArgs &o) {
    const int e = threadIdx.x;
    const double tk = (double)T * (double)k;
    double fp = 0.0;
    float b = 0.f;
    if (e < E) {
        const double fe = tk > 0 ? (double)c / tk : 0.0;
        if (f) f[e] = (float)fe;
        if (p && p_out && p_out != p) p_out[e] = p[e];
        fp = p ? fe * (double)p[e] : 0.0;
        if (o.bias) b = fabsf(o.bias[e]);
    } else {
        c = 0;
    }
    if (e < n) {
        sm.red[e] = fp;
        sm.redmax[e] = c;
        sm.redb[e] = b;
        sm.redbm[e] = b;
    }
    __syncthreads();
    for (int off = n / 2; off >= 1; off >>= 1) {
        if (e < off) {
            sm.red[e] += sm.red[e + off];
            sm.redmax[e] = max(sm.redmax[e], sm.redmax[e + off]);
            sm.redb[e] += sm.redb[e + off];
            sm.redbm[e] = fmaxf(sm.redbm[e], sm.redbm[e + off]);
        }
        __syncthreads();
    }
    if (e == 0) {
        if (aux) *aux = (float)((double)E * sm.red[0]);
        if (load) *load = tk > 0 ? (float)((double)sm.redmax[0] / (tk / (double)E)) : 0.f;
        if (o.drop_ratio)
            *o.drop_ratio = (o.n_dropped && tk > 0) ? (float)((double)*o.n_dropped / tk) : 0.f;
        if (o.bias_mean_abs) *o.bias_mean_abs = (float)(sm.redb[0] / (double)E);
        if (o.bias_max_abs) *o.bias_max_abs = sm.redbm[0];
    }
}

// p_e = (sum over blocks b of p_partial[b][e]) / T for the 32 experts e0 ..
// e0 + 31, over a CTA of 1024 threads: lane = expert (128-byte rows of the
// partials), warp w of 32 sums blocks w, w + 32, ... in order in fp32 with 8
// loads in flight, and the 32 warp sums are added in warp order in fp64
// (fixed order, no atomics).  fp64 arithmetic runs at a few operations per
// clock per SM on this part, so it is kept to the final 32 terms: an fp64
// sum of every partial on 28 SMs took 25 us for the 896-expert layer.
__device__ inline void block_p_finalize(const float *p_partial, int nblk, int E, int T,
                                        float *p, int e0) {
    __shared__ double red[32][33];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = e0 + lane;
    float s = 0.f;
    if (e < E) {
        int b = warp;
        for (; b + 7 * 32 < nblk; b += 8 * 32) {
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = p_partial[(size_t)(b + 32 * q) * E + e];
#pragma unroll
            for (int q = 0; q < 8; ++q) s += v[q];
        }
        for (; b < nblk; b += 32) s += p_partial[(size_t)b * E + e];
    }
    red[warp][lane] = (double)s;
    __syncthreads();
    if (warp == 0 && e < E) {
        double t = 0.0;
        for (int w = 0; w < 32; ++w) t += red[w][lane];
        p[e] = T > 0 ? (float)(t / (double)T) : 0.f;
    }
}

// Tile table of a grouped GEMM with BM-row tiles, over a CTA of 1024
// threads: expert e owns ceil((offsets[e+1]-offsets[e]) / BM) tiles starting
// at row offsets[e]; tile_start[e] is the index of its first tile
// (tile_start[E] = total).  offsets may have been written by this CTA before
// a __syncthreads().
__device__ inline void block_build_tiles(const int32_t *offsets, int E, int BM, int32_t *tile_e,
                                         int32_t *tile_m0, int32_t *tile_start,
                                         int32_t *n_tiles) {
    __shared__ int warp_tot[32];
    __shared__ int carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int e0 = 0; e0 < E; e0 += 1024) {
        const int e = e0 + threadIdx.x;
        int mt = 0;
        if (e < E) mt = (offsets[e + 1] - offsets[e] + BM - 1) / BM;
        int incl = mt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int wt = warp_tot[lane];
            int wi = wt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, wi, off);
                if (lane >= off) wi += o;
            }
            warp_tot[lane] = wi - wt;
        }
        __syncthreads();
        const int start = carry + warp_tot[warp] + incl - mt;
        if (e < E && tile_start) tile_start[e] = start;
        for (int i = 0; i < mt; ++i) {
            tile_e[start + i] = e;
            if (tile_m0) tile_m0[start + i] = offsets[e] + i * BM;
        }
        __syncthreads();
        if (threadIdx.x == 1023) carry = start + mt;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        *n_tiles = carry;
        if (tile_start) tile_start[E] = carry;
    }
}

// The dispatch tail in a CTA of 1024 threads, thread e < E holding count_e,
// after the CTA wrote offsets and n_dropped and passed a __syncthreads().
__device__ inline void dispatch_tail(const DispatchTail &t, int c, int E, const int32_t *offsets) {
    __shared__ StatsSmem sm;
    if (t.p_nblk > 0) {                      // p of up to 32 experts from the router's partials
        block_p_finalize(t.p_partial, t.p_nblk, E, t.T, t.p_out, 0);
        __syncthreads();
    }
    int n = 32;                              // the statistics' tree: the power of two >= E
    while (n < E) n *= 2;
    if (t.stats) block_load_stats(sm, n, c, t.p, t.T, E, t.k, t.f, nullptr, t.aux, t.load, t.o);
    if (t.tile_rows > 0)
        block_build_tiles(offsets, E, t.tile_rows, t.tile_e, nullptr, t.tile_start, t.n_tiles);
}

}  // namespace moe
