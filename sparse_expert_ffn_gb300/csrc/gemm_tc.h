// Host interface of the tcgen05 grouped GEMM (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace colibri {

enum : int { kGateUp = 0, kDown = 1, kRouter = 2 };

struct TcGemmArgs {
    const int32_t* tile_expert;  // [max_tiles] expert of each m-tile
    const int32_t* tile_row;     // [max_tiles] first pair row of each m-tile
    const int32_t* tile_info;    // [max_tiles] rows | band position << 10 | band length << 18
    const int32_t* num_tiles;    // device scalar: number of m-tiles
    int n_blocks;                // n-blocks per expert
    int k_blocks;                // K / 64
    int k_splits;                // K split into this many slices (1 = none); every slice
                                 // non-empty; kDown: slice s writes out + s * out_split_stride
    int b_rows_per_expert;       // rows of the packed B operand per expert
    void* out;                   // H (bf16, kGateUp) or Y (float32, kDown)
    int y_bf16;                  // kDown without K slices: Y stored as bf16 (one rounding)
    int out_ld;                  // row stride of `out` in elements
    size_t out_split_stride;     // elements between the outputs of two K slices
    // kGateUp with k_splits > 1 (single CTAs only): float32 G|U partials
    // [k_splits][pairs][2 f] and one arrival counter per (m-tile, n-block),
    // zero between launches
    float* partial;
    size_t partial_split_stride; // elements between two slices' partials
    int32_t* tile_counter;
    int* status;                 // device status word (DEV_TIMEOUT on a wait that gave up)
    uint64_t wait_limit_ns;      // bound of every mbarrier wait
    // router mode (kRouter): dense tiles over dense_rows tokens, MMA N = bn_rows
    int dense_rows;
    int bn_rows;
    int n_experts, top_k;
    const float* bias;           // [E] or null
    int32_t* topk_idx;           // [T, k]
    float* topk_w;               // [T, k]
    // int8 B (launch_tc_gemm with int8_b): block scales and zero points per
    // 64 packed B rows, [B rows / 64][k_blocks]
    const float* q_scale;
    const int32_t* q_zp;
    const int8_t* q_codes;       // tile-major codes (code_index), read by bulk copies
    int stall_producer;          // failure-detection tests only: issue no TMA copy, so
                                 // the first wait on a full stage runs out its bound
};

size_t tc_gemm_smem_bytes();
int tc_gemm_block_m();
int tc_gemm_pair_rows();     // rows of one expert tile of a CTA pair (256)
int tc_gemm_max_pairs();     // CTA pairs resident at once (0 if unknown)
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows, bool f16 = false);
// The packed bf16 gate/up weights (rows = E * 2 * d_ff, d columns) as the
// 5-D view the weights-as-M gate/up GEMM loads one CTA's A stage through.
bool make_tmap_gate_up_wm(CUtensorMap* map, const void* wgu, uint64_t rows, uint64_t d);
// Token-row tensor maps of Xp or H for the weights-as-M GEMMs: box heights of
// 16, 32, ..., 128 rows (map i: 16 * (i + 1) rows), 64 columns, the layout of
// make_tmap_bf16.  A tile whose token columns per CTA are h loads its B stage
// through map h / 16 - 1, so a narrow tile moves only the rows its MMA reads.
struct TokenRowMaps {
    CUtensorMap m[8];
};
bool make_tmap_token_rows(TokenRowMaps* maps, const void* base, uint64_t rows, uint64_t cols);
// pair: run the expert GEMMs on CTA pairs (256-row tiles, B tensor map with
// 128-row boxes) instead of single CTAs (128-row tiles, 256-row B boxes).
// int8_b: B is int8 codes (args.q_codes, tile-major, two 128-row tiles per
// stage by bulk copies; tmB unused) dequantised to f16 in shared memory by
// converter warps; A (Xp, H) is f16 and H is written as f16; single CTAs,
// kGateUp / kDown only.
// weights_m (CTA pairs, bf16, no gate/up K slices): the weights are the MMA's A (M)
// operand and the tile's tokens its B (N) operand, N = the tile's rows
// rounded up to 32, so an expert's last tile computes at most 31 padding
// columns instead of up to 255 padding rows.  tmA: the packed weights (gate/up
// through make_tmap_gate_up_wm: each CTA's 128 A rows are 4 x (16 gate, 16 up)
// rows of its 64 hidden units; down with 128-row boxes), wm_b: the token
// rows (Xp or H) in boxes of the tile's width (make_tmap_token_rows); tmB is
// not read.
cudaError_t launch_tc_gemm(int mode, bool pair, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           const TcGemmArgs& args, int grid, cudaStream_t s, bool int8_b = false,
                           bool weights_m = false, const TokenRowMaps* wm_b = nullptr);

// Decode-sized expert GEMMs with the weights as the MMA's M operand
// (gemm_dec.cu): tiles of 128 weight rows x 32 tokens of one expert (the tile
// list cut with tc_gemm_dec_tile_rows() rows).  tmTok: Xp or H with 32-row
// boxes; tmW: the packed bf16 weights with 128-row boxes, or with int8_w
// unused: the int8 code tiles come from args.q_codes, the block scales from
// args.q_scale / q_zp, and the tokens are f16.  kGateUp: n_blocks = f / 128,
// b_rows_per_expert = 2 f; kDown:
// n_blocks = d / 128, b_rows_per_expert = d.
size_t tc_gemm_dec_smem_bytes();
int tc_gemm_dec_tile_rows();
int tc_gemm_dec_w_rows();
cudaError_t launch_tc_gemm_dec(int mode, const CUtensorMap& tmTok, const CUtensorMap& tmW,
                               const TcGemmArgs& args, int grid, cudaStream_t s, bool int8_w);

}  // namespace colibri
