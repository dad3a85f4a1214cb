// Dispatch: group the (token, slot) pairs by expert, deterministically.
//
// zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析" section 3.3 stage 3
// (dispatch_kernel: every input slice that belongs to one expert is packed
// into one mini-batch for that expert's GEMM).
//
// Pairs are numbered r = t*k + j.  The result is a stable counting sort of r
// by expert: counts[E], offsets[E+1] (exclusive scan), perm[p] = r and
// inv[r] = p.  One CTA of 32 warps; warp w owns a contiguous range of r.
//   pass 1  per-warp histograms in shared memory: lanes holding the same
//           expert are found with __match_any_sync and the group leader adds
//           the group size (no atomics, so the counts never depend on timing)
//   scan    counts -> offsets, and each warp's base inside every expert
//           segment (warps in order)
//   pass 2  the same walk again: position = warp base + running count + rank
//           of the lane inside its match group.
// The same kernel also writes the grouped GEMM's tile list: one entry per
// block of `bm` consecutive pairs of one expert.  Tiles are grouped into
// raster bands that never cross an expert boundary (at most kMaxBand tiles of
// one expert per band), so that the GEMM walks all of a band's m-tiles against
// one weight block at a time and every weight block is streamed from HBM once.
// tile_info[t] packs: bits 0-9 valid rows (1..bm, bm <= 512), bits 10-17 the
// tile's position inside its band, bits 18-25 the band's length in tiles.
#include "common.cuh"
#include "kernels.h"

namespace colibri {

namespace {

constexpr int kDispatchWarps = 32;
constexpr int kMaxBand = 16;   // tiles of up to 256 rows

__global__ void __launch_bounds__(kDispatchWarps * 32)
dispatch_kernel(const int32_t* __restrict__ topk_idx, int n, int E, int32_t* __restrict__ counts,
                int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                int32_t* __restrict__ inv, int bm, int32_t* __restrict__ tile_expert,
                int32_t* __restrict__ tile_row, int32_t* __restrict__ tile_info,
                int32_t* __restrict__ num_tiles, int* __restrict__ status) {
    extern __shared__ int32_t sh[];
    int32_t* wcnt = sh;                           // [kDispatchWarps][E]
    int32_t* ecount = wcnt + kDispatchWarps * E;  // [E]
    int32_t* eoff = ecount + E;                   // [E + 1]
    int32_t* tbase = eoff + E + 1;                // [E + 1]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i < kDispatchWarps * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();

    const int chunk = ((n + kDispatchWarps - 1) / kDispatchWarps + 31) & ~31;
    const int lo = warp * chunk;
    const int hi = min(n, lo + chunk);
    int32_t* my = wcnt + warp * E;
    const unsigned lt_mask = (1u << lane) - 1u;

    for (int base = lo; base < hi; base += 32) {
        const int r = base + lane;
        int e = r < hi ? topk_idx[r] : -1;
        if (e >= E || (e < 0 && r < hi)) {
            atomicExch(status, DEV_BAD_INDEX);
            e = -1;
        }
        const unsigned m = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(m) - 1) my[e] += __popc(m);
        __syncwarp();
    }
    __syncthreads();

    if (threadIdx.x < E) {
        const int e = threadIdx.x;
        int32_t c = 0;
        for (int w = 0; w < kDispatchWarps; ++w) c += wcnt[w * E + e];
        ecount[e] = c;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t acc = 0, tacc = 0;
        for (int e = 0; e < E; ++e) {
            eoff[e] = acc;
            tbase[e] = tacc;
            acc += ecount[e];
            tacc += (ecount[e] + bm - 1) / bm;
        }
        eoff[E] = acc;
        tbase[E] = tacc;
        *num_tiles = tacc;
    }
    __syncthreads();
    if (threadIdx.x < E) {
        const int e = threadIdx.x;
        int32_t run = eoff[e];
        for (int w = 0; w < kDispatchWarps; ++w) {
            const int32_t c = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += c;
        }
        counts[e] = ecount[e];
        offsets[e] = eoff[e];
        const int32_t c = ecount[e];
        const int nt = (c + bm - 1) / bm;
        for (int i = 0, tb = tbase[e]; i < nt; ++i, ++tb) {
            const int band_len = min(kMaxBand, nt - (i / kMaxBand) * kMaxBand);
            tile_expert[tb] = e;
            tile_row[tb] = eoff[e] + i * bm;
            tile_info[tb] = min(bm, c - i * bm) | ((i % kMaxBand) << 10) | (band_len << 18);
        }
    }
    if (threadIdx.x == 0) offsets[E] = eoff[E];
    __syncthreads();

    for (int base = lo; base < hi; base += 32) {
        const int r = base + lane;
        int e = r < hi ? topk_idx[r] : -1;
        if (e >= E) e = -1;
        const unsigned m = __match_any_sync(0xffffffffu, e);
        int32_t start = 0;
        if (e >= 0) start = my[e];
        __syncwarp();
        if (e >= 0) {
            const int p = start + __popc(m & lt_mask);
            perm[p] = r;
            inv[r] = p;
            if (lane == __ffs(m) - 1) my[e] = start + __popc(m);
        }
        __syncwarp();
    }
}

}  // namespace

size_t dispatch_smem(int E) { return (size_t)(kDispatchWarps * E + 3 * E + 2) * sizeof(int32_t); }

cudaError_t launch_dispatch(const int32_t* topk_idx, int n, int E, int32_t* counts,
                            int32_t* offsets, int32_t* perm, int32_t* inv, int bm,
                            int32_t* tile_expert, int32_t* tile_row, int32_t* tile_info,
                            int32_t* num_tiles, int* status, cudaStream_t s) {
    const size_t smem = dispatch_smem(E);
    cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dispatch_kernel<<<1, kDispatchWarps * 32, smem, s>>>(topk_idx, n, E, counts, offsets, perm,
                                                         inv, bm, tile_expert, tile_row,
                                                         tile_info, num_tiles, status);
    return cudaGetLastError();
}

}  // namespace colibri
