// Device helpers shared by the routing kernels: the logit order key, the warp
// top-k with softmax over the k, and the deterministic block-wide dispatch.
#pragma once

#include "common.cuh"

namespace colibri {

// Total order on float logits as an unsigned key: larger value -> larger key,
// -0 == +0, NaN below -inf.
__device__ __forceinline__ uint32_t logit_order_key(float v) {
    if (v != v) return 0u;
    if (v == 0.0f) v = 0.0f;
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Top-k of one token's E logits (shared memory) by one warp: k rounds of a
// warp arg-max over a 64-bit key (ordered value, then ~expert so that the
// lower index wins a tie), then the softmax over the k selected logits with
// the largest subtracted first.  Lane 0 writes idx[0..k) and w[0..k).
__device__ __forceinline__ void warp_topk_softmax(const float* logit, int E, int k, int lane,
                                                  int32_t* idx, float* w) {
    uint32_t taken = 0;
    int sel_e[8];
    float sel_l[8];
    for (int j = 0; j < k; ++j) {
        unsigned long long best = 0ull;
        for (int s = 0, e = lane; e < E; ++s, e += 32) {
            if (taken & (1u << s)) continue;
            const unsigned long long key =
                ((unsigned long long)logit_order_key(logit[e]) << 32) | (uint32_t)(~(uint32_t)e);
            best = key > best ? key : best;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
            best = other > best ? other : best;
        }
        const int e = (int)(~(uint32_t)(best & 0xffffffffull));
        if ((e & 31) == lane) taken |= 1u << (e >> 5);
        sel_e[j] = e;
        sel_l[j] = logit[e];
    }
    if (lane == 0) {
        const float m = sel_l[0];
        float sum = 0.f;
        for (int j = 0; j < k; ++j) sum += expf(sel_l[j] - m);
        for (int j = 0; j < k; ++j) {
            idx[j] = sel_e[j];
            w[j] = expf(sel_l[j] - m) / sum;
        }
    }
}

constexpr int kDispatchWarps = 32;
constexpr int kDispatchChunk = 2048;   // pairs per CTA of the multi-CTA dispatch
constexpr int kMaxBand = 16;   // tiles of up to 256 rows per raster band

__host__ __device__ constexpr size_t dispatch_smem_bytes(int E) {
    return (size_t)(kDispatchWarps * E + 3 * E + 2) * sizeof(int32_t);
}

// Building blocks of the deterministic dispatch (a stable counting sort of
// the pairs r = t*k + j by expert; zskr.cn "Colibri：面向MoE架构的C语言高效推理
// 引擎解析" section 3.3 stage 3: the input slices of one expert packed into one
// mini-batch).  A warp walks a contiguous range [lo, hi) of r, 32 at a time.

// Both passes read the warp's expert ids kWalkBatch * 32 at a time, the
// loads of a batch issued before any is used, so that a pass waits for one
// memory latency per batch instead of one per 32 pairs.
constexpr int kWalkBatch = 8;

// Pass 1: add the warp's per-expert counts into my[E]: lanes holding the
// same expert are found with __match_any_sync and the group leader adds the
// group size (no atomics, so the counts never depend on timing).
__device__ __forceinline__ void warp_count_pass(const int32_t* __restrict__ topk_idx, int lo,
                                                int hi, int E, int32_t* my, int* status) {
    const int lane = threadIdx.x & 31;
    for (int b0 = lo; b0 < hi; b0 += kWalkBatch * 32) {
        int ev[kWalkBatch];
#pragma unroll
        for (int i = 0; i < kWalkBatch; ++i) {
            const int r = b0 + i * 32 + lane;
            ev[i] = r < hi ? topk_idx[r] : -1;
        }
#pragma unroll
        for (int i = 0; i < kWalkBatch; ++i) {
            const int r = b0 + i * 32 + lane;
            int e = ev[i];
            if (e >= E || (e < 0 && r < hi)) {
                atomicExch(status, DEV_BAD_INDEX);
                e = -1;
            }
            const unsigned m = __match_any_sync(0xffffffffu, e);
            if (e >= 0 && lane == __ffs(m) - 1) my[e] += __popc(m);
            __syncwarp();
        }
    }
}

// Pass 2: the same walk; my[e] holds the warp's next position inside expert
// e's segment (which starts at seg_start[e]).  perm[p] = r, and inv[r] = p —
// or -1 when p is the segment's cap-th pair or later (dropped by the expert's
// capacity; cf-1.com sections 2.3 and 4.2: a hard per-expert token limit).
__device__ __forceinline__ void warp_scatter_pass(const int32_t* __restrict__ topk_idx, int lo,
                                                  int hi, int E, int32_t* my,
                                                  const int32_t* seg_start, int cap,
                                                  int32_t* __restrict__ perm,
                                                  int32_t* __restrict__ inv) {
    const int lane = threadIdx.x & 31;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int b0 = lo; b0 < hi; b0 += kWalkBatch * 32) {
        int ev[kWalkBatch];
#pragma unroll
        for (int i = 0; i < kWalkBatch; ++i) {
            const int r = b0 + i * 32 + lane;
            ev[i] = r < hi ? topk_idx[r] : -1;
        }
#pragma unroll
        for (int i = 0; i < kWalkBatch; ++i) {
            const int r = b0 + i * 32 + lane;
            int e = ev[i];
            if (e >= E) e = -1;
            const unsigned m = __match_any_sync(0xffffffffu, e);
            int32_t start = 0;
            if (e >= 0) start = my[e];
            __syncwarp();
            if (e >= 0) {
                const int p = start + __popc(m & lt_mask);
                perm[p] = r;
                inv[r] = p - seg_start[e] < cap ? p : -1;
                if (lane == __ffs(m) - 1) my[e] = start + __popc(m);
            } else if (r < hi) {
                inv[r] = -1;     // an expert id out of range (reported by pass 1): adds nothing
            }
            __syncwarp();
        }
    }
}

// The grouped GEMM's tile list for expert e (kept pairs c, first pair eoff,
// first tile tb): one entry per block of `bm` consecutive pairs, grouped into raster
// bands that never cross an expert boundary (at most kMaxBand tiles of one
// expert per band), so the GEMM walks all of a band's m-tiles against one
// weight block at a time and every weight block is streamed from HBM once.
// tile_info[t] packs: bits 0-9 valid rows (1..bm, bm <= 512), bits 10-17 the
// tile's position inside its band, bits 18-25 the band's length in tiles.
__device__ __forceinline__ void write_tiles(int e, int c, int eoff, int tb, int bm,
                                            int32_t* __restrict__ tile_expert,
                                            int32_t* __restrict__ tile_row,
                                            int32_t* __restrict__ tile_info) {
    const int nt = (c + bm - 1) / bm;
    for (int i = 0; i < nt; ++i, ++tb) {
        const int band_len = min(kMaxBand, nt - (i / kMaxBand) * kMaxBand);
        tile_expert[tb] = e;
        tile_row[tb] = eoff + i * bm;
        tile_info[tb] = min(bm, c - i * bm) | ((i % kMaxBand) << 10) | (band_len << 18);
    }
}

// Dispatch of n = T*k pairs by one block of kDispatchWarps warps: counts[E],
// offsets[E+1] (exclusive scan), perm[p] = r, inv[r] = p (-1 when dropped),
// kept[E] = min(counts, cap) and the tile list over the kept pairs.
// Warp w owns a contiguous range of r; after pass 1 the per-warp counts are
// turned into each warp's base inside every expert segment (warps in order),
// and pass 2 writes the positions.
// Every thread of the block must call it; `sh` is dispatch_smem_bytes(E).
__device__ __forceinline__ void dispatch_block(
    const int32_t* __restrict__ topk_idx, int n, int E, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv, int bm,
    int32_t* __restrict__ tile_expert, int32_t* __restrict__ tile_row,
    int32_t* __restrict__ tile_info, int32_t* __restrict__ num_tiles, int* __restrict__ status,
    int cap, int32_t* __restrict__ kept, int32_t* sh) {
    int32_t* wcnt = sh;                           // [kDispatchWarps][E]
    int32_t* ecount = wcnt + kDispatchWarps * E;  // [E]
    int32_t* eoff = ecount + E;                   // [E + 1]
    int32_t* tbase = eoff + E + 1;                // [E + 1]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Warp w walks pairs [w*chunk, (w+1)*chunk); only the first `nw` warps
    // hold any (a small batch fills one warp), so only their counts are kept.
    const int chunk = ((n + kDispatchWarps - 1) / kDispatchWarps + 31) & ~31;
    const int nw = chunk > 0 ? min(kDispatchWarps, (n + chunk - 1) / chunk) : 0;
    for (int i = threadIdx.x; i < nw * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();

    const int lo = warp * chunk;
    const int hi = min(n, lo + chunk);
    int32_t* my = wcnt + warp * E;
    warp_count_pass(topk_idx, lo, hi, E, my, status);
    __syncthreads();

    if (threadIdx.x < E) {
        const int e = threadIdx.x;
        int32_t c = 0;
        for (int w = 0; w < nw; ++w) c += wcnt[w * E + e];
        ecount[e] = c;
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scans of the counts and of the tile counts: lane l sums
        // experts [l*per, (l+1)*per), a warp scan gives each lane its base
        const int per = (E + 31) / 32;
        const int e0 = lane * per;
        int32_t c_sum = 0, t_sum = 0;
        for (int i = 0; i < per; ++i) {
            const int e = e0 + i;
            if (e < E) {
                c_sum += ecount[e];
                t_sum += (min(ecount[e], cap) + bm - 1) / bm;
            }
        }
        int32_t c_inc = c_sum, t_inc = t_sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t a = __shfl_up_sync(0xffffffffu, c_inc, o);
            const int32_t b = __shfl_up_sync(0xffffffffu, t_inc, o);
            if (lane >= o) c_inc += a, t_inc += b;
        }
        int32_t acc = c_inc - c_sum, tacc = t_inc - t_sum;
        for (int i = 0; i < per; ++i) {
            const int e = e0 + i;
            if (e < E) {
                eoff[e] = acc;
                tbase[e] = tacc;
                acc += ecount[e];
                tacc += (min(ecount[e], cap) + bm - 1) / bm;
            }
        }
        if (lane == 31) {
            eoff[E] = c_inc;
            tbase[E] = t_inc;
            *num_tiles = t_inc;
        }
    }
    __syncthreads();
    if (threadIdx.x < E) {
        const int e = threadIdx.x;
        int32_t run = eoff[e];
        for (int w = 0; w < nw; ++w) {
            const int32_t c = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += c;
        }
        counts[e] = ecount[e];
        kept[e] = min(ecount[e], cap);
        offsets[e] = eoff[e];
        write_tiles(e, min(ecount[e], cap), eoff[e], tbase[e], bm, tile_expert, tile_row,
                    tile_info);
    }
    if (threadIdx.x == 0) offsets[E] = eoff[E];
    __syncthreads();

    warp_scatter_pass(topk_idx, lo, hi, E, my, eoff, cap, perm, inv);
}

}  // namespace colibri
