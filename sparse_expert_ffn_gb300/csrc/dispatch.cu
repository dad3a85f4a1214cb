// Dispatch: group the (token, slot) pairs by expert, deterministically: one
// CTA of 32 warps running dispatch_block (see routing.cuh), or for large
// batches the same counting sort spread over many CTAs in three launches.
//
// zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析" section 3.3 stage 3
// (dispatch_kernel: every input slice that belongs to one expert is packed
// into one mini-batch for that expert's GEMM).
#include "common.cuh"
#include "kernels.h"
#include "routing.cuh"

namespace colibri {

namespace {

__global__ void __launch_bounds__(kDispatchWarps * 32)
dispatch_kernel(const int32_t* __restrict__ topk_idx, int n, int E, int32_t* __restrict__ counts,
                int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                int32_t* __restrict__ inv, int bm, int32_t* __restrict__ tile_expert,
                int32_t* __restrict__ tile_row, int32_t* __restrict__ tile_info,
                int32_t* __restrict__ num_tiles, int* __restrict__ status, int cap,
                int32_t* __restrict__ kept) {
    pdl_enter();
    extern __shared__ int32_t sh[];
    dispatch_block(topk_idx, n, E, counts, offsets, perm, inv, bm, tile_expert, tile_row,
                   tile_info, num_tiles, status, cap, kept, sh);
}

// ---- Multi-CTA dispatch for large batches: CTA b owns the pairs
// [b * kChunk, (b + 1) * kChunk), warp w of it a contiguous 1/32 of those, so
// the order (CTA, warp, lane rank) is still increasing r.

// 1. per-CTA, per-expert counts
__global__ void __launch_bounds__(kDispatchWarps * 32)
dispatch_count_kernel(const int32_t* __restrict__ topk_idx, int n, int E,
                      int32_t* __restrict__ block_counts, int* __restrict__ status) {
    pdl_enter();
    extern __shared__ int32_t wcnt[];  // [kDispatchWarps][E]
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kDispatchWarps * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const int lo = blockIdx.x * kDispatchChunk + warp * (kDispatchChunk / kDispatchWarps);
    const int hi = min(n, lo + kDispatchChunk / kDispatchWarps);
    warp_count_pass(topk_idx, lo, hi, E, wcnt + warp * E, status);
    __syncthreads();
    if (threadIdx.x < E) {
        int32_t c = 0;
        for (int w = 0; w < kDispatchWarps; ++w) c += wcnt[w * E + threadIdx.x];
        block_counts[blockIdx.x * E + threadIdx.x] = c;
    }
}

constexpr size_t kScanSmemMax = 160 * 1024;   // block counts staged in shared memory up to this

// 2. one CTA: expert counts, offsets, every CTA's base in every expert
//    segment (CTAs in order), and the tile list
__global__ void __launch_bounds__(kDispatchWarps * 32)
dispatch_scan_kernel(int32_t* block_counts, int nb, int E, int staged,
                     int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int bm,
                     int32_t* __restrict__ tile_expert, int32_t* __restrict__ tile_row,
                     int32_t* __restrict__ tile_info, int32_t* __restrict__ num_tiles, int cap,
                     int32_t* __restrict__ kept) {
    pdl_enter();
    __shared__ int32_t ecount[256], eoff[257], tbase[257];
    const int e = threadIdx.x;
    // every (block, expert) count is read once into shared memory, eight
    // loads in flight per thread, then walked from there (batches whose
    // counts do not fit walk them in global memory)
    extern __shared__ int32_t bc_sh[];   // [nb][E] when staged
    const int32_t* bc = staged ? bc_sh : block_counts;
    if (staged) {
        for (int i = threadIdx.x; i < nb * E; i += blockDim.x * 8) {
            int32_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = i + u * blockDim.x;
                v[u] = j < nb * E ? block_counts[j] : 0;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = i + u * blockDim.x;
                if (j < nb * E) bc_sh[j] = v[u];
            }
        }
    }
    __syncthreads();
    if (e < E) {
        int32_t c = 0;
        for (int b = 0; b < nb; ++b) c += bc[b * E + e];
        ecount[e] = c;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t acc = 0, tacc = 0;
        for (int i = 0; i < E; ++i) {
            eoff[i] = acc;
            tbase[i] = tacc;
            acc += ecount[i];
            tacc += (min(ecount[i], cap) + bm - 1) / bm;
        }
        eoff[E] = acc;
        *num_tiles = tacc;
        offsets[E] = acc;
    }
    __syncthreads();
    if (e < E) {
        int32_t run = eoff[e];
        for (int b = 0; b < nb; ++b) {     // counts -> bases
            const int32_t c = bc[b * E + e];
            block_counts[b * E + e] = run;
            run += c;
        }
        counts[e] = ecount[e];
        kept[e] = min(ecount[e], cap);
        offsets[e] = eoff[e];
        write_tiles(e, min(ecount[e], cap), eoff[e], tbase[e], bm, tile_expert, tile_row,
                    tile_info);
    }
}

// 3. per CTA: the warps' bases from the CTA's bases, then the positions
__global__ void __launch_bounds__(kDispatchWarps * 32)
dispatch_scatter_kernel(const int32_t* __restrict__ topk_idx, int n, int E,
                        const int32_t* __restrict__ block_base,
                        const int32_t* __restrict__ offsets, int cap,
                        int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                        int* __restrict__ status) {
    pdl_enter();
    extern __shared__ int32_t wcnt[];  // [kDispatchWarps][E]
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kDispatchWarps * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const int lo = blockIdx.x * kDispatchChunk + warp * (kDispatchChunk / kDispatchWarps);
    const int hi = min(n, lo + kDispatchChunk / kDispatchWarps);
    int32_t* my = wcnt + warp * E;
    warp_count_pass(topk_idx, lo, hi, E, my, status);
    __syncthreads();
    if (threadIdx.x < E) {
        int32_t run = block_base[blockIdx.x * E + threadIdx.x];
        for (int w = 0; w < kDispatchWarps; ++w) {
            const int32_t c = wcnt[w * E + threadIdx.x];
            wcnt[w * E + threadIdx.x] = run;
            run += c;
        }
    }
    __syncthreads();
    warp_scatter_pass(topk_idx, lo, hi, E, my, offsets, cap, perm, inv);
}

}  // namespace

size_t dispatch_smem(int E) { return dispatch_smem_bytes(E); }

int dispatch_blocks(int n) { return (n + kDispatchChunk - 1) / kDispatchChunk; }

cudaError_t launch_dispatch_multi(const int32_t* topk_idx, int n, int E, int32_t* block_counts,
                                  int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                  int bm, int32_t* tile_expert, int32_t* tile_row,
                                  int32_t* tile_info, int32_t* num_tiles, int* status,
                                  int cap, int32_t* kept, cudaStream_t s) {
    const int nb = dispatch_blocks(n);
    const size_t smem = (size_t)kDispatchWarps * E * sizeof(int32_t);
    const dim3 block(kDispatchWarps * 32);
    cudaError_t e = launch_pdl(dispatch_count_kernel, nb, block, smem, s, topk_idx, n, E,
                               block_counts, status);
    if (e == cudaSuccess) {
        const size_t need = (size_t)nb * E * sizeof(int32_t);
        const int staged = need <= kScanSmemMax ? 1 : 0;
        const size_t scan_smem = staged ? need : 0;
        if (staged) smem_attr((const void*)dispatch_scan_kernel, (int)scan_smem);
        e = launch_pdl(dispatch_scan_kernel, 1, block, scan_smem, s, block_counts, nb, E, staged,
                       counts, offsets, bm, tile_expert, tile_row, tile_info, num_tiles, cap, kept);
    }
    if (e == cudaSuccess)
        e = launch_pdl(dispatch_scatter_kernel, nb, block, smem, s, topk_idx, n, E, block_counts,
                       offsets, cap, perm, inv, status);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_dispatch(const int32_t* topk_idx, int n, int E, int32_t* counts,
                            int32_t* offsets, int32_t* perm, int32_t* inv, int bm,
                            int32_t* tile_expert, int32_t* tile_row, int32_t* tile_info,
                            int32_t* num_tiles, int* status, int cap, int32_t* kept,
                            cudaStream_t s) {
    const size_t smem = dispatch_smem(E);
    smem_attr((const void*)dispatch_kernel, (int)smem);
    const cudaError_t e = launch_pdl(dispatch_kernel, 1, kDispatchWarps * 32, smem, s, topk_idx, n,
                                     E, counts, offsets, perm, inv, bm, tile_expert, tile_row,
                                     tile_info, num_tiles, status, cap, kept);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace colibri
