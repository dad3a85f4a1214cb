// Launchers of the MoE layer kernels (host-side declarations, internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace colibri {

enum class DType : int;

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per kernel and size:
// a host-side cache keeps it off the per-launch path.
cudaError_t smem_attr(const void* kernel, int bytes);

// The CUDA-core router keeps one token row of d floats (+256 logits) in
// shared memory: d_model beyond that limit (about 57 000) is not supported.
bool router_simt_fits(int d);
cudaError_t launch_router_simt(DType dt, const void* x, const void* wr, const float* bias,
                               int ntok, int d, int E, int k, int32_t* idx, float* w,
                               cudaStream_t s, bool soft = false);

size_t dispatch_smem(int E);
cudaError_t launch_dispatch(const int32_t* topk_idx, int n, int E, int32_t* counts,
                            int32_t* offsets, int32_t* perm, int32_t* inv, int bm,
                            int32_t* tile_expert, int32_t* tile_row, int32_t* tile_info,
                            int32_t* num_tiles, int* status, int cap, int32_t* kept,
                            cudaStream_t s);

// The same dispatch over ceil(n / 2048) CTAs (three launches); block_counts
// holds dispatch_blocks(n) * E int32.
int dispatch_blocks(int n);
cudaError_t launch_dispatch_multi(const int32_t* topk_idx, int n, int E, int32_t* block_counts,
                                  int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                  int bm, int32_t* tile_expert, int32_t* tile_row,
                                  int32_t* tile_info, int32_t* num_tiles, int* status,
                                  int cap, int32_t* kept, cudaStream_t s);

// Router + top-k + softmax + dispatch (+ gather when xp != null) in one
// launch for decode-sized batches (route_decode_fits()): every warp one
// partial logit (in `part`, route_decode_part_floats() floats), the CTA that
// draws the last `ticket` (zero at rest) does the rest.  With gamma the
// routed rows are u = RMSNorm(x) * gamma, written to u.
bool route_decode_fits(int ntok, int d, int E, int k);
size_t route_decode_part_floats(int max_tok, int E);
cudaError_t launch_route_decode(DType dt, const void* x, const void* wr, const float* bias,
                                int ntok, int d, int E, int k, float* part, unsigned int* ticket,
                                int32_t* topk_idx, float* topk_w, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* inv, int bm,
                                int32_t* tile_expert, int32_t* tile_row, int32_t* tile_info,
                                int32_t* num_tiles, int* status, int cap, int32_t* kept, void* xp,
                                const void* gamma, float eps, void* u, cudaStream_t s,
                                bool xp_f16 = false);

// `kept` = pairs each expert accepted (its first kept[e] segment rows).
cudaError_t launch_ffn_up_stream(DType dt, const void* x, const void* wgu, const int32_t* kept,
                                 const int32_t* offsets, const int32_t* perm, int k, int d, int f,
                                 int E, void* H, cudaStream_t s);
cudaError_t launch_ffn_down_stream(DType dt, const void* H, const void* wdT, const int32_t* kept,
                                   const int32_t* offsets, int d, int f, int E, float* Y,
                                   cudaStream_t s);
// Int8-weight variants (64x64 blocks, w = (q - zp) * scale); scales and zero
// points per 64-row block of the packed weight rows, [packed row / 64][K / 64].
cudaError_t launch_ffn_up_stream_i8(DType dt, const void* x, const int8_t* wq, const float* sc,
                                    const int32_t* zp, const int32_t* kept,
                                    const int32_t* offsets, const int32_t* perm, int k, int d,
                                    int f, int E, void* H, cudaStream_t s);
cudaError_t launch_ffn_down_stream_i8(DType dt, const void* H, const int8_t* wq, const float* sc,
                                      const int32_t* zp, const int32_t* kept,
                                      const int32_t* offsets, int d, int f, int E, float* Y,
                                      cudaStream_t s);

// Int8-weight expert FFN for a few tokens per expert on CUDA cores, bf16
// layers (gemv_i8.cu): items of 64 weight rows x one K slice per CTA over the
// dispatch's tile list, codes streamed by bulk copies into a shared-memory
// ring, activations as 16-bit integers per 64-wide k-tile, integer dot
// products; S token rows per pass (1, 2 or 4; more rows take several passes).
// gemv_i8_fits: the ring and the staging area of S rows of one item fit.
struct GemvTiles {
    const int32_t* tile_expert;
    const int32_t* tile_row;
    const int32_t* tile_info;
    const int32_t* num_tiles;
    int E;                    // experts: tile_expert values are checked against it
    int* status;              // DEV_TIMEOUT when a wait gave up, DEV_BAD_INDEX on a bad expert
    uint64_t wait_limit_ns;   // bound of every wait
    int stall_producer;       // failure-detection tests only: issue no copy, so the
                              // consumers' first wait runs out its bound
};
int gemv_i8_slots(int max_rows_per_expert);
bool gemv_i8_fits(int S, int d, int f, int ks);
int gemv_i8_items(bool up, int tiles, int d, int f, int ks);
// H[p, n] = silu(g) * u as bf16, x the bf16 token rows (pair p: row perm[p] / k).
cudaError_t launch_ffn_up_gemv_i8(int S, const void* x, const int32_t* perm, int k,
                                  const int8_t* wq, const float* sc, const int32_t* zp,
                                  const GemvTiles& t, int d, int f, int grid, void* H,
                                  cudaStream_t s);
// Y + s * y_split_stride: the float32 partial of K slice s, [pairs][d].
cudaError_t launch_ffn_down_gemv_i8(int S, const void* H, const int8_t* wq, const float* sc,
                                    const int32_t* zp, const GemvTiles& t, int d, int f, int ks,
                                    int grid, float* Y, size_t y_split_stride, cudaStream_t s);

// xp[p] = x[perm[p] / k] for p < npairs; a perm value outside [0, src_pairs)
// gathers a zero row.
cudaError_t launch_gather(int elem_bytes, const void* x, const int32_t* perm, int k, int d,
                          int npairs, int src_pairs, void* xp, cudaStream_t s, bool to_f16 = false);
// y_bf16: Y holds the down projection's rows as bf16 (no K slices).
cudaError_t launch_combine(DType dt, const float* Y, bool y_bf16, const float* topk_w,
                           const int32_t* inv, int T, int k, int d, int nsplit, size_t split_stride,
                           const void* resid, void* y, cudaStream_t s);
// inv[perm[p]] = p for p < n.
cudaError_t launch_invert_perm(const int32_t* perm, int n, int32_t* inv, cudaStream_t s);
cudaError_t launch_rmsnorm(DType dt, const void* h, const void* gamma, int T, int d, float eps,
                           void* u, cudaStream_t s);
cudaError_t launch_transpose_remap(int elem_bytes, const void* in, void* out, int batch, int R,
                                   int C, size_t in_batch, size_t out_batch, int blk, int period,
                                   int which, cudaStream_t s, bool tiled = false);

}  // namespace colibri
