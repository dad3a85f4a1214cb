// Decode-sized expert GEMMs with the weights as the MMA's M operand.
//
// zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析" section 3.3 stage 4 (per
// expert: gate_proj, up_proj, SiLU, down_proj) for batches with few tokens per
// expert.  grouped_gemm_tc puts the tokens on M (128-row tiles) and, at decode
// sizes, computes mostly padding rows while its shared memory carries 128
// token rows per stage.  Here a tile is 128 weight rows (M) x up to 32 tokens
// of one expert (N = 32); the dispatch kernel cuts each expert's tokens into
// 32-row tiles.
//
//   kGateUp  per n-block of 128 hidden units, two MMAs per K step, the 128
//            gate rows and the 128 up rows, into two accumulators: TMEM lane
//            n holds g and u of hidden unit n for every token of the tile,
//            and the epilogue writes H = silu(g) * u (or, split over K, the
//            float32 G|U partials of the gate/up fixup).
//   kDown    per block of 128 output features, one MMA; lane c holds y_c.
//
// Operands.  B (tokens): the tile's 32 rows of Xp (gate/up) or H (down), 64 K
// columns per stage, TMA with 128-byte swizzle.  A (weights):
//   bf16     TMA boxes of 128 rows x 64 K into shared memory;
//   int8     one bulk copy per 8 KB tile of 128 rows x 64 codes (the codes are
//            stored tile-major and pre-swizzled); converter warps (one weight row
//            per thread) dequantise (q - zp) * scale to f16 and store the row
//            into tensor memory with tcgen05.st, where the MMA reads A.  Shared
//            memory then carries only the codes and the token rows, so a
//            stage is 20 KB (gate/up) and the ring holds 9 of them in flight.
//
// Roles: warp 0 TMA producer (bf16: tokens and weights; int8: code tiles),
// warp 1 TMEM owner + MMA issuer, warps 2-5 epilogue, warps 6-13 converters
// and warp 14 token producer (int8).  Every mbarrier wait is bounded as in
// grouped_gemm_tc; on expiry the kernel records DEV_TIMEOUT, every role stops,
// copies and MMAs in flight are drained and TMEM is freed.
#include <cuda.h>

#include "common.cuh"
#include "gemm_tc.h"
#include "kernels.h"
#include "tc_common.cuh"

namespace colibri {

namespace {

using namespace tc;

constexpr int kDecN = 32;                  // tokens per tile (MMA N)
constexpr int kDecM = 128;                 // weight rows per MMA (MMA M)
constexpr int kDecMaxStages = 16;
constexpr uint32_t kDecRingBytes = 192 * 1024;
constexpr uint32_t kTokStage = kDecN * kBK * 2;   // 4 KB of token rows per stage
constexpr int kDecConvWarps = 8;            // two per SM sub-partition
constexpr int kDecTokWarp = 6 + kDecConvWarps;   // 14, int8: token producer
constexpr int kDecThreads = 192;
constexpr int kDecThreadsI8 = (kDecTokWarp + 1) * 32;
constexpr int kDecTokStages = 4;           // int8: token ring, released by the MMA
constexpr int kDecTmemCols = 512;
constexpr int kDecAccCols = 64;            // per accumulator: gate [0, 32), up [32, 64)
constexpr int kDecAStages = 6;             // int8: A stages in tensor memory (6 x 64 columns)
constexpr int kDecACol0 = 2 * kDecAccCols; // first TMEM column of the A stages

// Weight matrices per tile: gate and up, or down.
template <int kMode> constexpr int n_mats() { return kMode == kGateUp ? 2 : 1; }

// Dequantise kChunks 16-code chunks of row r of a code tile (as stored:
// chunk c at chunk c ^ ((r >> 1) & 3), so that the 8 rows of a quarter warp
// hit 8 different bank groups), starting at chunk c0, to 8 * kChunks words of
// f16 pairs, in K order.
template <int kChunks>
__device__ __forceinline__ void dequant_row(const uint8_t* __restrict__ tile, int r, int c0,
                                            __half2 off2, __half2 s2, uint32_t (&o)[8 * kChunks]) {
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(tile + code_chunk_offset(r, c0 + c));
        uint4 lo, hi;
        dequant16_h2(v, off2, s2, lo, hi);
        o[8 * c + 0] = lo.x, o[8 * c + 1] = lo.y, o[8 * c + 2] = lo.z, o[8 * c + 3] = lo.w;
        o[8 * c + 4] = hi.x, o[8 * c + 5] = hi.y, o[8 * c + 6] = hi.z, o[8 * c + 7] = hi.w;
    }
}

template <int kMode, bool kI8>
__global__ void __launch_bounds__(kI8 ? kDecThreadsI8 : kDecThreads, 1)
grouped_gemm_dec(const __grid_constant__ CUtensorMap tmTok, const __grid_constant__ CUtensorMap tmW,
                 TcGemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    constexpr int kMats = n_mats<kMode>();
    // A bytes per matrix and stage: bf16 rows (SW128) or int8 codes (64-byte rows)
    constexpr uint32_t kMatBytes = kDecM * kBK * (kI8 ? 1 : 2);
    // bf16: one ring of [token rows 4 KB][matrix 0][matrix 1] stages, released
    // by the MMA.  int8: a ring of code stages [matrix 0][matrix 1], released
    // by the converters once read, and a separate 4-stage ring of token rows
    // after it, released by the MMA: the codes, the HBM stream, turn over
    // without waiting for the tensor core.
    constexpr uint32_t kStageBytes = kI8 ? kMats * kMatBytes : kTokStage + kMats * kMatBytes;
    constexpr uint32_t kRing = kDecRingBytes - (kI8 ? kDecTokStages * kTokStage : 0);
    constexpr int kStages =
        (int)(kRing / kStageBytes) < kDecMaxStages ? (int)(kRing / kStageBytes) : kDecMaxStages;
    uint8_t* tok_ring = smem + kRing;               // int8: [kDecTokStages][4 KB]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDecRingBytes);
    uint64_t* full = bars;                          // [kStages]
    uint64_t* empty = bars + kDecMaxStages;         // [kStages]
    uint64_t* acc_full = bars + 2 * kDecMaxStages;  // [2]
    uint64_t* acc_empty = acc_full + 2;             // [2]
    uint64_t* a_full = acc_full + 4;                // [kDecAStages] int8: A rows in TMEM
    uint64_t* a_empty = a_full + kDecAStages;       // [kDecAStages]
    uint64_t* mma_done = a_empty + kDecAStages;     // [1]
    uint64_t* t_full = mma_done + 1;                // [kDecTokStages] int8: token rows landed
    uint64_t* t_empty = t_full + kDecTokStages;     // [kDecTokStages]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(t_empty + kDecTokStages);
    static_assert((2 * kDecMaxStages + 4 + 2 * kDecAStages + 1 + 2 * kDecTokStages) * 8 + 8 <= 512,
                  "barriers, TMEM slot and abort flag fit the 512 bytes after the ring");
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x, n_units = gridDim.x;
    const int kb_per_split = (args.k_blocks + args.k_splits - 1) / args.k_splits;
    const uint64_t limit = args.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            // int8: a code stage is released by every converter warp
            mbar_init(smem_u32(&empty[s]), kI8 ? kDecConvWarps : 1);
        }
        for (int t = 0; t < kDecTokStages; ++t) {
            mbar_init(smem_u32(&t_full[t]), 1);
            mbar_init(smem_u32(&t_empty[t]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&acc_full[a]), 1);
            mbar_init(smem_u32(&acc_empty[a]), 4);
        }
        for (int a = 0; a < kDecAStages; ++a) {
            mbar_init(smem_u32(&a_full[a]), kDecConvWarps);
            mbar_init(smem_u32(&a_empty[a]), 1);
        }
        mbar_init(smem_u32(&mma_done[0]), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<false>(smem_u32(tmem_slot), kDecTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_enter();
    const int num_tiles = *args.num_tiles;
    const int total = num_tiles * args.n_blocks * args.k_splits;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool issued[kDecMaxStages];
            uint32_t issued_phase[kDecMaxStages];
            for (int s = 0; s < kStages; ++s) issued[s] = false, issued_phase[s] = 0;
            for (int w = unit; w < total && !*abort_flag && !args.stall_producer; w += n_units) {
                const Work wk = decode_work(w, args.n_blocks, args.k_splits, args.tile_expert,
                                            args.tile_row, args.tile_info);
                // first weight row of the tile: gate/up n-blocks are 256 packed
                // rows (128 gate, 128 up), down blocks 128 rows
                const int w_row = wk.expert * args.b_rows_per_expert + wk.nblk * kMats * kDecM;
                const int kb0 = wk.split * kb_per_split;
                const int kb1 = min(args.k_blocks, kb0 + kb_per_split);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1, abort_flag, args.status,
                                   limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[stage]);
                    mbar_expect_tx(fb, kStageBytes);
                    uint8_t* st = smem + stage * kStageBytes;
                    if constexpr (!kI8) tma_load_2d(smem_u32(st), &tmTok, kb * kBK, wk.row0, fb);
                    uint8_t* mats = st + (kI8 ? 0 : kTokStage);
#pragma unroll
                    for (int m = 0; m < kMats; ++m) {
                        const uint32_t dst = smem_u32(mats + m * kMatBytes);
                        if constexpr (kI8)   // tile-major codes: tile (row block, kb), 8 KB
                            bulk_load(dst,
                                      args.q_codes +
                                          (((size_t)(w_row + m * kDecM) >> 7) * args.k_blocks + kb) * 8192,
                                      kMatBytes, fb);
                        else
                            tma_load_2d(dst, &tmW, kb * kBK, w_row + m * kDecM, fb);
                    }
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == kStages) stage = 0, phase ^= 1;
                }
                if (!ok) break;
            }
            for (int s = 0; s < kStages; ++s)
                if (issued[s]) mbar_wait_drain(smem_u32(&full[s]), issued_phase[s], kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            // N = 16 for tiles of at most 16 tokens: every MMA reads and
            // rewrites its accumulator in tensor memory, and half the
            // columns halve that traffic (the epilogue uses only the live
            // token columns)
            const uint32_t idesc32 = kI8 ? idesc_f16(kDecM, kDecN) : idesc_bf16(kDecM, kDecN);
            const uint32_t idesc16 = kI8 ? idesc_f16(kDecM, 16) : idesc_bf16(kDecM, 16);
            int stage = 0, as = 0, acc = 0;     // int8: `stage` counts token stages
            uint32_t phase = 0, aphase = 0, acc_phase = 0;
            for (int w = unit; w < total && !*abort_flag; w += n_units) {
                const Work wk = decode_work(w, args.n_blocks, args.k_splits, args.tile_expert,
                                            args.tile_row, args.tile_info);
                const int kb0 = wk.split * kb_per_split;
                const int kb1 = min(args.k_blocks, kb0 + kb_per_split);
                if (!mbar_wait(smem_u32(&acc_empty[acc]), acc_phase ^ 1, abort_flag, args.status,
                               limit))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kDecAccCols;
                const uint32_t idesc = wk.rows <= 16 ? idesc16 : idesc32;
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    const bool got =
                        kI8 ? mbar_wait(smem_u32(&a_full[as]), aphase, abort_flag, args.status,
                                        limit) &&
                                  mbar_wait(smem_u32(&t_full[stage]), phase, abort_flag,
                                            args.status, limit)
                            : mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.status,
                                        limit);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint8_t* st = kI8 ? tok_ring + stage * kTokStage : smem + stage * kStageBytes;
                    const uint64_t db = smem_desc_sw128(smem_u32(st));
#pragma unroll
                    for (int m = 0; m < kMats; ++m) {
#pragma unroll
                        for (int ks = 0; ks < kBK / 16; ++ks) {
                            const uint32_t accf = (kb > kb0) || ks != 0;
                            const uint32_t dm = d_tmem + m * kDecN;
                            if constexpr (kI8) {
                                // A: 16 K values = 8 columns per step
                                const uint32_t at = tmem_base + kDecACol0 +
                                                    (as * kMats + m) * (kBK / 2) + ks * 8;
                                mma_f16_ta(dm, at, db + 2 * ks, idesc, accf);
                            } else {
                                const uint64_t da =
                                    smem_desc_sw128(smem_u32(st + kTokStage + m * kMatBytes));
                                mma_bf16<false>(dm, da + 2 * ks, db + 2 * ks, idesc, accf);
                            }
                        }
                    }
                    if constexpr (kI8) {
                        mma_commit<false>(smem_u32(&t_empty[stage]));
                        mma_commit<false>(smem_u32(&a_empty[as]));
                        if (++stage == kDecTokStages) stage = 0, phase ^= 1;
                        if (++as == kDecAStages) as = 0, aphase ^= 1;
                    } else {
                        mma_commit<false>(smem_u32(&empty[stage]));
                        if (++stage == kStages) stage = 0, phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit<false>(smem_u32(&acc_full[acc]));
                if (++acc == 2) acc = 0, acc_phase ^= 1;
            }
            mma_commit_local<false>(smem_u32(&mma_done[0]));
            mbar_wait_drain(smem_u32(&mma_done[0]), 0, kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;                    // TMEM lane quarter: weight rows 32q..32q+31
        const int wrow = q * 32 + lane;            // weight row of this thread inside the block
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int w = unit; w < total; w += n_units) {
            const Work wk = decode_work(w, args.n_blocks, args.k_splits, args.tile_expert,
                                        args.tile_row, args.tile_info);
            const bool got =
                mbar_wait(smem_u32(&acc_full[acc]), acc_phase, abort_flag, args.status, limit);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + acc * kDecAccCols;
            if constexpr (kMode == kGateUp) {
                uint32_t g[32], u[32];
                tmem_ld32(tb, g);
                tmem_ld32(tb + kDecN, u);
                tmem_ld_wait();
                const int n = wk.nblk * kDecM + wrow;    // hidden unit
                if (args.k_splits > 1) {
                    float* P = args.partial + wk.split * args.partial_split_stride;
                    const size_t pld = (size_t)args.n_blocks * 256;
#pragma unroll
                    for (int t = 0; t < kDecN; ++t) {
                        if (t >= wk.rows) break;
                        float* pr = P + (size_t)(wk.row0 + t) * pld + wk.nblk * 256;
                        pr[wrow] = __uint_as_float(g[t]);
                        pr[128 + wrow] = __uint_as_float(u[t]);
                    }
                } else {
                    uint16_t* H = reinterpret_cast<uint16_t*>(args.out);
#pragma unroll
                    for (int t = 0; t < kDecN; ++t) {
                        if (t >= wk.rows) break;
                        const float h = silu(__uint_as_float(g[t])) * __uint_as_float(u[t]);
                        uint16_t hv;
                        if constexpr (kI8) {
                            const __half hh = __float2half_rn(h);
                            hv = *reinterpret_cast<const uint16_t*>(&hh);
                        } else {
                            const __nv_bfloat16 hb = __float2bfloat16_rn(h);
                            hv = *reinterpret_cast<const uint16_t*>(&hb);
                        }
                        H[(size_t)(wk.row0 + t) * args.out_ld + n] = hv;
                    }
                }
            } else {
                uint32_t v[32];
                tmem_ld32(tb, v);
                tmem_ld_wait();
                float* Y = reinterpret_cast<float*>(args.out) + wk.split * args.out_split_stride;
                const int c = wk.nblk * kDecM + wrow;    // output feature
#pragma unroll
                for (int t = 0; t < kDecN; ++t) {
                    if (t >= wk.rows) break;
                    Y[(size_t)(wk.row0 + t) * args.out_ld + c] = __uint_as_float(v[t]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc_empty[acc]));
            if constexpr (kMode == kGateUp) {
                if (args.k_splits > 1) gate_up_split_fixup<kI8>(args, wk, lane);
            }
            if (++acc == 2) acc = 0, acc_phase ^= 1;
        }
    } else if (kI8 && warp == kDecTokWarp) {
        // ------------------------------------------------ token producer (int8)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool issued[kDecTokStages];
            uint32_t issued_phase[kDecTokStages];
            for (int s = 0; s < kDecTokStages; ++s) issued[s] = false, issued_phase[s] = 0;
            for (int w = unit; w < total && !*abort_flag && !args.stall_producer; w += n_units) {
                const Work wk = decode_work(w, args.n_blocks, args.k_splits, args.tile_expert,
                                            args.tile_row, args.tile_info);
                const int kb0 = wk.split * kb_per_split;
                const int kb1 = min(args.k_blocks, kb0 + kb_per_split);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&t_empty[stage]), phase ^ 1, abort_flag, args.status,
                                   limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t tb = smem_u32(&t_full[stage]);
                    mbar_expect_tx(tb, kTokStage);
                    tma_load_2d(smem_u32(tok_ring + stage * kTokStage), &tmTok, kb * kBK, wk.row0, tb);
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == kDecTokStages) stage = 0, phase ^= 1;
                }
                if (!ok) break;
            }
            for (int s = 0; s < kDecTokStages; ++s)
                if (issued[s]) mbar_wait_drain(smem_u32(&t_full[s]), issued_phase[s], kDrainLimitNs);
        }
        __syncwarp();
    } else if constexpr (kI8) {
        // ------------------------------------------------ converters (warps 6..13)
        // Thread = one weight row (lane quarter = warp % 4, the only TMEM
        // lanes this warp may write); warp group g = 0, 1 takes the gate or
        // the up matrix (gate/up), or the first or second 32 codes of the
        // row (down).  Each dequantises its codes of the stage and stores
        // them as columns of f16 pairs.
        const int q = warp & 3;
        const int grp = (warp - 6) >> 2;
        const int wrow = q * 32 + lane;
        constexpr int kChunks = kMats == 2 ? 4 : 2;     // 16-code chunks per thread
        const int mat = kMats == 2 ? grp : 0;
        const int c0 = kMats == 2 ? 0 : 2 * grp;
        int stage = 0, as = 0;
        uint32_t phase = 0, aphase = 0;
        for (int w = unit; w < total && !*abort_flag; w += n_units) {
            const Work wk = decode_work(w, args.n_blocks, args.k_splits, args.tile_expert,
                                        args.tile_row, args.tile_info);
            const int kb0 = wk.split * kb_per_split;
            const int kb1 = min(args.k_blocks, kb0 + kb_per_split);
            // this thread's 64-row block of scales (of its matrix)
            const int rb = (wk.expert * args.b_rows_per_expert + wk.nblk * kMats * kDecM +
                            mat * kDecM + wrow) >> 6;
            const float* sc_row = args.q_scale + (size_t)rb * args.k_blocks;
            const int32_t* zp_row = args.q_zp + (size_t)rb * args.k_blocks;
            // Scales and zero points are loaded kPf k-blocks ahead (a rotating
            // window of registers), so that their L2 latency hides behind the
            // conversions of the stages in between.
            constexpr int kPf = 3;
            float pscl[kPf], pzp[kPf];
#pragma unroll
            for (int i = 0; i < kPf; ++i) {
                const int kc = min(kb0 + i, kb1 - 1);
                pscl[i] = __ldg(sc_row + kc);
                pzp[i] = (float)__ldg(zp_row + kc);
            }
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                const __half2 off2 = __float2half2_rn(1152.0f + pzp[0]);
                const __half2 s2 = __float2half2_rn(pscl[0]);
#pragma unroll
                for (int i = 0; i + 1 < kPf; ++i) pscl[i] = pscl[i + 1], pzp[i] = pzp[i + 1];
                {
                    const int kc = min(kb + kPf, kb1 - 1);
                    pscl[kPf - 1] = __ldg(sc_row + kc);
                    pzp[kPf - 1] = (float)__ldg(zp_row + kc);
                }
                const bool got =
                    mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.status, limit) &&
                    mbar_wait(smem_u32(&a_empty[as]), aphase ^ 1, abort_flag, args.status, limit);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* st = smem + stage * kStageBytes + mat * kMatBytes;
                uint32_t o[8 * kChunks];
                dequant_row<kChunks>(st, wrow, c0, off2, s2, o);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));   // codes read
                const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + kDecACol0 +
                                    (as * kMats + mat) * (kBK / 2) + c0 * 8;
                if constexpr (kChunks == 4) tmem_st32(ta, o);
                else tmem_st16(ta, o);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&a_full[as]));
                if (++stage == kStages) stage = 0, phase ^= 1;
                if (++as == kDecAStages) as = 0, aphase ^= 1;
            }
            if (!ok) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<false>(tmem_base, kDecTmemCols);
}

template <int kMode, bool kI8>
cudaError_t launch_dec(const CUtensorMap& tmTok, const CUtensorMap& tmW, const TcGemmArgs& args,
                       int grid, cudaStream_t s) {
    const size_t smem = tc_gemm_dec_smem_bytes();
    auto k = grouped_gemm_dec<kMode, kI8>;
    smem_attr((const void*)k, (int)smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kI8 ? kDecThreadsI8 : kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, tmTok, tmW, args);
}

}  // namespace

size_t tc_gemm_dec_smem_bytes() { return (size_t)kDecRingBytes + 512 + 1024; }
int tc_gemm_dec_tile_rows() { return kDecN; }
int tc_gemm_dec_w_rows() { return kDecM; }

cudaError_t launch_tc_gemm_dec(int mode, const CUtensorMap& tmTok, const CUtensorMap& tmW,
                               const TcGemmArgs& args, int grid, cudaStream_t s, bool int8_w) {
    if (grid <= 0) return cudaSuccess;
    if (mode != kGateUp && mode != kDown) return cudaErrorInvalidValue;
    if (mode == kGateUp && args.k_splits > 1 && (!args.partial || !args.tile_counter))
        return cudaErrorInvalidValue;
    if (int8_w && (!args.q_scale || !args.q_zp || !args.q_codes || args.b_rows_per_expert % 128))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (mode == kGateUp)
        e = int8_w ? launch_dec<kGateUp, true>(tmTok, tmW, args, grid, s)
                   : launch_dec<kGateUp, false>(tmTok, tmW, args, grid, s);
    else
        e = int8_w ? launch_dec<kDown, true>(tmTok, tmW, args, grid, s)
                   : launch_dec<kDown, false>(tmTok, tmW, args, grid, s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace colibri
