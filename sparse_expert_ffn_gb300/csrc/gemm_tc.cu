// Grouped GEMM for the expert FFN on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bf16 operands, float32 accumulation.
//
// zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析" section 3.3 stages 3-4
// (the tokens of one expert batched into one GEMM; gate_proj, up_proj, SiLU and
// down_proj per expert).  Three instantiations:
//
//   kGateUp  A = Xp (tokens of each expert, consecutive rows) [pairs, d]
//            B = packed [W_gate^T | W_up^T] blocks of 128 rows each, K = d
//            one tile = 128 rows x (128 gate + 128 up) columns; the epilogue
//            reads both halves from TMEM and writes H = silu(G) * U (bf16).
//   kDown    A = H [pairs, f], B = W_down^T [d, f] per expert, K = f
//            one tile = 128 rows x 256 output features.  Without K slices
//            the rows Y are stored as bf16 (one rounding of each element, as
//            for H; the combine then adds the k rows in float32 and rounds y
//            once more); with K slices (small batches) each slice is stored
//            as float32 and the combine adds the slices first.
//   kRouter  A = x [T, d] (the caller's tokens), B = packed router [E_pad, d]:
//            the router logits of 128 tokens per tile (N = E rounded up to 16),
//            top-k and softmax in the epilogue (p1 section 3.3 stage 2).
//
// Work items are (m-tile, n-block) pairs.  An m-tile is up to 128 consecutive
// pair rows of one expert (the dispatch kernel's tile list), so experts with
// no token have no tile at all.  The kernel is persistent: CTA b takes work
// b, b + grid, ...; work is walked band by band (a band = up to 32 m-tiles of
// one expert), n-block-major inside a band, so one weight block is read from
// HBM once and reused from L2 by all of the band's m-tiles, while the band's A
// rows stay resident in L2 across the n-blocks.
//
// Roles (192 threads):
//   warp 0      TMA producer: A and B tiles of 64 K-columns into a ring of
//               128B-swizzled shared-memory stages (4 deep for a single CTA,
//               6 deep for a CTA of a pair).
//   warp 1      TMEM owner; lane 0 issues tcgen05.mma (M=128, N=256, K=16)
//               into one of two 256-column accumulators, commits each stage
//               back to the producer and each finished tile to the epilogue.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4)..+31, i.e. tile rows), activation, stores.
// Every mbarrier wait is bounded by a time limit: on expiry the CTA records
// DEV_TIMEOUT in the status word, every role stops, outstanding TMA copies
// and MMAs are waited for (again bounded) and TMEM is freed before exit.
#include <cuda.h>

#include "common.cuh"
#include "gemm_tc.h"
#include "kernels.h"
#include "routing.cuh"
#include "tc_common.cuh"

namespace colibri {

namespace {

using namespace tc;

// Shared-memory ring: a single CTA holds 4 stages of A (16 KB) + B (up to
// 256 rows, 32 KB); a CTA of a pair loads only half of B (16 KB), so it
// holds 6 stages.  Both keep ~192 KB of copies in flight per SM.
template <bool kPair> struct Ring {
    static constexpr int kStages = kPair ? 6 : 4;
    static constexpr uint32_t kStageB = (kPair ? 128 : 256) * 64 * 2;
};
constexpr int kThreads = 192;
// Int8 B operand (single CTAs).  Three rings: 5 stages of int8 B codes
// (256 x 64 bytes, 16 KB) fed by TMA from warp 0 and released by the
// converters as soon as they are read; 3 stages of A (16 KB) fed by TMA from
// warp 14 and released by the MMA; 2 stages of dequantised f16 B (32 KB,
// 128-byte swizzle) written by 8 converter warps (warps 6-13) and released by
// the MMA.  The codes, the only HBM stream at decode sizes, thus turn over
// without waiting for the tensor core.
constexpr int kConvWarps = 8;
constexpr int kAWarp = 6 + kConvWarps;                  // 14: A producer
constexpr int kThreadsI8 = (kAWarp + 1) * 32;           // 480
constexpr int kQStages = 5;
constexpr int kAStagesI8 = 3;
constexpr int kBStages = 2;
constexpr uint32_t kStageQ = 256 * 64;        // int8 codes of one B stage
constexpr uint32_t kStageBf = 256 * 64 * 2;   // the same stage in bf16
constexpr uint32_t kRingBytes = 192 * 1024;   // shared-memory ring of every instantiation
// Per epilogue warp, a 32-row tile of one 32-column accumulator chunk in
// shared memory (rows padded to 36 floats): the warp turns its 32 per-thread
// rows into 128-byte row segments for the global stores, and the router reads
// its logits back with a rolled loop instead of a fully unrolled one.
constexpr uint32_t kStagingOffset = kRingBytes + 512;   // after the ring and the barriers
constexpr int kStgStride = 36;                           // floats per staged row
constexpr uint32_t kStgWarpBytes = 32 * kStgStride * 4;  // 4608
// Router: each epilogue warp's copy of the logit offset (E <= 256 floats),
// so that the top-k insertion loop reads it from shared memory
constexpr uint32_t kBiasOffset = kStagingOffset + 4 * kStgWarpBytes;
constexpr uint32_t kBiasWarpBytes = 256 * 4;
constexpr int kMaxRouterStages = 12;
constexpr int kAccCols = 256;     // TMEM columns per accumulator
constexpr int kTmemCols = 512;    // two accumulators
constexpr uint32_t kStageA = kBM * kBK * 2;   // 16 KB


// ---------------------------------------------------------------- the kernel

// Dequantise one stage of int8 B codes (two 128-row code tiles of 64-byte
// rows, as stored: code_chunk_offset) into the f16 128-byte-swizzled layout
// the MMA reads (16-byte chunk j
// of row r at chunk j ^ (r & 7), as TMA would have written it).  Converter
// thread ct (0..255) takes the 16-byte code chunks ct + 256 j, j = 0..3: row
// ct/4 + 64 j (64-row block j), chunk ct % 4.  off2[j] = 1152 + zp and s2[j] =
// scale of block j, as half2.
__device__ __forceinline__ void convert_stage(const uint8_t* __restrict__ sq, uint8_t* __restrict__ sb,
                                              int ct, const __half2 (&off2)[4], const __half2 (&s2)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int id = ct + 256 * j;
        const int r = id >> 2, c = id & 3;
        // the two 128-row code tiles as stored (chunk c of row r at c ^ ((r >> 1) & 3))
        const uint4 v = *reinterpret_cast<const uint4*>(sq + (r >> 7) * 8192 + code_chunk_offset(r, c));
        uint4 lo, hi;
        dequant16_h2(v, off2[j], s2[j], lo, hi);
        uint8_t* row = sb + r * 128;
        *reinterpret_cast<uint4*>(row + (((2 * c) ^ (r & 7)) << 4)) = lo;
        *reinterpret_cast<uint4*>(row + (((2 * c + 1) ^ (r & 7)) << 4)) = hi;
    }
}

// Router epilogue: top-k by insertion over a key that puts the larger logit
// first and the lower expert id first on ties (as the CUDA-core router), then
// the softmax over the k.  Logits arrive 32 at a time in shared memory (a
// rolled loop over them keeps the instruction footprint small).  K >= k
// slots: every logit runs a chain of K compare-and-swaps, the thread's
// critical path when E is large, so the list is as short as the layer's k
// allows (1, 2, 4 or 8).
template <int K>
struct RouterTopk {
    unsigned long long key[K];
    float val[K];
    __device__ __forceinline__ RouterTopk() {
#pragma unroll
        for (int j = 0; j < K; ++j) key[j] = 0ull, val[j] = 0.f;
    }
    // logits of experts c .. c + n - 1 in l[0 .. n)
    __device__ __forceinline__ void insert(const float* l, int c, int n, const float* bias) {
#pragma unroll 1
        for (int i = 0; i < n; ++i) {
            const int e = c + i;
            float v = l[i];
            if (bias) v += bias[e];
            unsigned long long kk =
                ((unsigned long long)logit_order_key(v) << 32) | (uint32_t)(~(uint32_t)e);
            float vv = v;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (kk > key[j]) {
                    const unsigned long long tk = key[j];
                    const float tv = val[j];
                    key[j] = kk, val[j] = vv;
                    kk = tk, vv = tv;
                }
            }
        }
    }
    __device__ __forceinline__ void write(const TcGemmArgs& args, size_t t) const {
        const int k = args.top_k;
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (j < k) sum += expf(val[j] - val[0]);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (j < k) {
                args.topk_idx[t * k + j] = (int)(~(uint32_t)(key[j] & 0xffffffffull));
                args.topk_w[t * k + j] = expf(val[j] - val[0]) / sum;
            }
        }
    }
};

// The last slice's rows: slices' logits added in slice order, then routed.
template <int K>
__device__ __forceinline__ void router_fixup_rows(const TcGemmArgs& args, const Work& wk, int q,
                                                  int lane, float* mine, const float* bias) {
    const int E = args.n_experts;
    const int ld = args.bn_rows;                  // partial row stride: E padded to 16
    const int row = q * 32 + lane;
    const size_t t = (size_t)wk.row0 + row;
    if (row < wk.rows) {
        RouterTopk<K> top;
        for (int c = 0; c < E; c += 32) {
            const int n = min(32, E - c);
            const int nv = min(32, ld - c) / 4;   // float4 groups present in the row
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.f;
            for (int sl = 0; sl < args.k_splits; ++sl) {
                // the slice's 32 logits of this chunk: eight loads in flight
                const float4* src =
                    reinterpret_cast<const float4*>(args.partial + sl * args.partial_split_stride + t * ld + c);
                float4 v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = i < nv ? __ldcg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    acc[4 * i] += v[i].x;
                    acc[4 * i + 1] += v[i].y;
                    acc[4 * i + 2] += v[i].z;
                    acc[4 * i + 3] += v[i].w;
                }
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) mine[i] = acc[i];
            top.insert(mine, c, n, bias);
        }
        top.write(args, t);
    }
}


// Whole-K router rows: the thread's E logits from its TMEM lane, 32 at a
// time through shared memory, then the top-k and softmax.
template <int K>
__device__ __forceinline__ void router_rows_tmem(uint32_t tbase, int bn, float* mine,
                                                 const TcGemmArgs& args, const float* bias, bool live,
                                                 size_t orow) {
    RouterTopk<K> top;
#pragma unroll 1
    for (int c = 0; c < bn; c += 32) {
        uint32_t v[32];
        tmem_ld32(tbase + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) mine[i] = __uint_as_float(v[i]);
        top.insert(mine, c, min(32, args.n_experts - c), bias);
    }
    if (live) top.write(args, orow);
}

// Router with K split into slices: every slice's epilogue warp counts itself
// in on a counter per (tile, lane quarter) once its partial logits are
// globally visible; the warp that arrives last adds the slices' logits of its
// 32 rows in slice order (so the sum does not depend on arrival order), routes
// them and rearms the counter.  Nothing waits on another CTA.
__device__ __noinline__ void router_split_fixup(const TcGemmArgs& args, const Work& wk, int q,
                                                int lane, float* mine, const float* bias) {
    __threadfence();
    __syncwarp();
    int* ctr = args.tile_counter + (size_t)wk.tile * 4 + q;
    int old = 0;
    if (lane == 0) old = atomicAdd(ctr, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old != args.k_splits - 1) return;
    __threadfence();
    const int k = args.top_k;
    if (k <= 1) router_fixup_rows<1>(args, wk, q, lane, mine, bias);
    else if (k <= 2) router_fixup_rows<2>(args, wk, q, lane, mine, bias);
    else if (k <= 4) router_fixup_rows<4>(args, wk, q, lane, mine, bias);
    else router_fixup_rows<8>(args, wk, q, lane, mine, bias);
    __syncwarp();
    if (lane == 0) *ctr = 0;
}

// Order in which the CTAs of the expert GEMMs take the work list when the
// expert sizes are skewed: even positions walk it from the front, odd ones
// from the back.  The list is in expert order, so the units of the large
// experts (many m-tiles per weight block: bound by the tensor pipe) then run
// beside those of the small ones (one m-tile per weight block: bound by the
// weight stream from HBM) instead of in separate waves.  A bijection of
// [0, total): front positions j < ceil(total / 2), back ones the rest.
__device__ __forceinline__ int both_ends(int w, int total) {
    const int j = w >> 1;
    return (w & 1) ? total - 1 - j : j;
}

// Skewed: the first expert's raster band is at least four times as long as
// the last one's (a Zipf-like load puts the large experts first).  Under
// even loads a second stream costs L2 locality, so the list is walked in
// order.
__device__ __forceinline__ bool work_skewed(const int32_t* tile_info, int num_tiles) {
    if (num_tiles < 2) return false;
    const int first = (tile_info[0] >> 18) & 0xFF;
    const int last = (tile_info[num_tiles - 1] >> 18) & 0xFF;
    return first >= 4 * last;
}

// Weights as M (kWM): token columns of a tile, its valid rows rounded up to
// 32 (each CTA of the pair holds half of them as MMA B rows).
__device__ __forceinline__ int wm_cols(int rows) { return min(2 * kBM, max(32, (rows + 31) & ~31)); }

template <int kMode, bool kPair, bool kI8, bool kWM>
__global__ void __launch_bounds__(kI8 ? kThreadsI8 : kThreads, 1)
grouped_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ TokenRowMaps tmBr, TcGemmArgs args) {
    static_assert(!kI8 || (!kPair && kMode != kRouter), "int8 B: single-CTA expert GEMMs only");
    static_assert(!kWM || (kPair && !kI8 && kMode != kRouter), "weights as M: CTA-pair expert GEMMs");
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms.
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    // The router's B tile is only E_pad rows: its ring is as deep as fits
    // (up to kMaxRouterStages) in the same bytes; the expert GEMMs use Ring.
    constexpr int kMaxSt = kMode == kRouter ? kMaxRouterStages : kI8 ? kQStages : Ring<kPair>::kStages;
    // Bytes per stage of the TMA-fed B tile (int8 codes for kI8).
    const uint32_t kStageB = kMode == kRouter ? (uint32_t)args.bn_rows * kBK * 2
                             : kI8            ? kStageQ
                                              : Ring<kPair>::kStageB;
    const int kStages = kMode == kRouter
                            ? min(kMaxRouterStages, (int)(kRingBytes / (kStageA + kStageB)))
                            : kMaxSt;
    // kI8: [A x 3][codes x 5][f16 B x 2]; otherwise [A x kStages][B x kStages]
    uint8_t* stage_a = smem;
    uint8_t* stage_b = smem + (kI8 ? kAStagesI8 : kStages) * kStageA;
    uint8_t* stage_bf = stage_b + kStages * kStageB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage_bf + (kI8 ? kBStages * kStageBf : 0));
    uint64_t* full = bars;                 // [kStages]
    uint64_t* empty = bars + kStages;      // [kStages]
    uint64_t* acc_full = bars + 2 * kStages;     // [2]
    uint64_t* acc_empty = bars + 2 * kStages + 2;  // [2]
    uint64_t* mma_done = bars + 2 * kStages + 4;   // [1]
    uint64_t* bf_full = bars + 2 * kStages + 5;    // [kBStages] kI8: converted B ready
    uint64_t* bf_empty = bars + 2 * kStages + 7;   // [kBStages] kI8: converted B consumed
    uint64_t* a_full = bars + 2 * kStages + 9;     // [kAStagesI8] kI8: A landed
    uint64_t* a_empty = bars + 2 * kStages + 12;   // [kAStagesI8] kI8: A consumed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 15);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTA pair: rank 0 (leader) owns the full / acc_empty barriers and issues
    // the MMAs; both CTAs load their halves of A and B and run an epilogue on
    // their own 128 rows of the 256-row tile.
    const uint32_t rank = kPair ? cluster_rank() : 0;
    const bool leader = rank == 0;
    const int unit = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int n_units = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    // Rows of B this CTA loads per stage (= MMA N, or half of it for a pair).
    const int bn = kMode == kRouter ? args.bn_rows : kBN;
    const int b_rows_cta = kPair ? bn / 2 : bn;
    const uint32_t cta_tx = kI8 ? kStageQ : kStageA + (uint32_t)b_rows_cta * kBK * 2;
    const uint32_t stage_tx = kPair ? 2 * cta_tx : cta_tx;   // bytes landing on `full`
    const int kb_per_split = (args.k_blocks + args.k_splits - 1) / args.k_splits;
    const uint64_t limit = args.wait_limit_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            // kI8: a code stage is released by every converter warp
            mbar_init(smem_u32(&empty[s]), kI8 ? kConvWarps : 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&acc_full[a]), 1);
            // one elected lane per epilogue warp, in each CTA of the pair
            mbar_init(smem_u32(&acc_empty[a]), kPair ? 8 : 4);
        }
        mbar_init(smem_u32(&mma_done[0]), 1);
        if constexpr (kI8) {
            for (int b = 0; b < kBStages; ++b) {
                mbar_init(smem_u32(&bf_full[b]), kConvWarps);
                mbar_init(smem_u32(&bf_empty[b]), 1);
            }
            for (int a = 0; a < kAStagesI8; ++a) {
                mbar_init(smem_u32(&a_full[a]), 1);
                mbar_init(smem_u32(&a_empty[a]), 1);
            }
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<kPair>(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync();   // the peer's barriers exist before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above touched only this CTA's shared and tensor memory; the
    // tile list and the operands come from the kernels before this one.
    pdl_enter();
    const int num_tiles =
        kMode == kRouter ? (args.dense_rows + kBM - 1) / kBM : *args.num_tiles;
    const int total = num_tiles * args.n_blocks * args.k_splits;
    const bool skewed = kMode != kRouter && work_skewed(args.tile_info, num_tiles);
    // every role (producer, MMA, epilogue, both CTAs of a pair) takes the
    // same order
    auto work_at = [&](int w) { return get_work<kMode>(skewed ? both_ends(w, total) : w, args); };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool issued[kMaxSt];
            uint32_t issued_phase[kMaxSt];
            for (int s = 0; s < kStages; ++s) issued[s] = false, issued_phase[s] = 0;
            for (int w = unit; w < total && !*abort_flag && !args.stall_producer; w += n_units) {
                const Work wk = work_at(w);
                const int a_row = wk.row0 + (int)rank * kBM;
                const int b_row = wk.expert * args.b_rows_per_expert + wk.nblk * kBN +
                                  (int)rank * b_rows_cta;
                const int kb0 = wk.split * kb_per_split;
                const int kb1 = min(args.k_blocks, kb0 + kb_per_split);
                // kWM: each CTA loads the tile's token columns it holds
                // (wm_cols / 2 = 16..128 rows) through the map of that height
                const int wm_h = kWM ? wm_cols(wk.rows) / 2 : 0;
                const CUtensorMap* wm_map = &tmBr.m[kWM ? wm_h / 16 - 1 : 0];
                const uint32_t unit_tx = kWM ? 2 * (kStageA + (uint32_t)wm_h * kBK * 2) : stage_tx;
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1, abort_flag, args.status,
                                   limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_u32(&full[stage]);
                    if (leader) mbar_expect_tx(fb_local, unit_tx);
                    const uint32_t sa = smem_u32(stage_a + stage * kStageA);
                    const uint32_t sb = smem_u32(stage_b + stage * kStageB);
                    if constexpr (kWM) {
                        // A: this CTA's 128 weight rows; B: its half of the
                        // tile's token columns, exactly the rows the MMA reads
                        const uint32_t fb = map_to_rank(fb_local, 0);
                        tma_load_2d_pair(sb, wm_map, kb * kBK, wk.row0 + (int)rank * wm_h, fb);
                        if constexpr (kMode == kGateUp) {
                            // 64 hidden units per CTA in four groups of 16:
                            // group g's 16 gate rows (TMEM lanes 32g..32g+15)
                            // then its 16 up rows (32g+16..32g+31), one copy
                            // through the 5-D view of make_tmap_gate_up_wm
                            const int f = args.b_rows_per_expert / 2;
                            tma_load_5d_pair(sa, &tmA, kb * kBK, 0, 0, 0,
                                             4 * (wk.expert * (f / 128) + wk.nblk) + (int)rank, fb);
                        } else {
                            tma_load_2d_pair(sa, &tmA, kb * kBK,
                                             wk.expert * args.b_rows_per_expert + wk.nblk * kBN +
                                                 (int)rank * kBM,
                                             fb);
                        }
                    } else if constexpr (kPair) {
                        // both halves complete on the leader's barrier
                        const uint32_t fb = map_to_rank(fb_local, 0);
                        tma_load_2d_pair(sa, &tmA, kb * kBK, a_row, fb);
                        tma_load_2d_pair(sb, &tmB, kb * kBK, b_row, fb);
                    } else if constexpr (kI8) {
                        // int8 codes only (warp 14 loads A into its own ring):
                        // the 256 B rows are two tile-major 128-row tiles
                        (void)sa;
                        (void)a_row;
                        const int8_t* t0 =
                            args.q_codes + (((size_t)b_row >> 7) * args.k_blocks + kb) * 8192;
                        bulk_load(sb, t0, 8192, fb_local);
                        bulk_load(sb + 8192, t0 + (size_t)args.k_blocks * 8192, 8192, fb_local);
                    } else {
                        tma_load_2d(sa, &tmA, kb * kBK, a_row, fb_local);
                        tma_load_2d(sb, &tmB, kb * kBK, b_row, fb_local);
                    }
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == kStages) stage = 0, phase ^= 1;
                }
                if (!ok) break;
            }
            // Teardown: every copy issued must have landed.  The leader's
            // `full` barriers count the copies of both CTAs of a pair.
            if (leader)
                for (int s = 0; s < kStages; ++s)
                    if (issued[s]) mbar_wait_drain(smem_u32(&full[s]), issued_phase[s], kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader)
        if (lane == 0 && leader) {
            // int8 B: A (Xp / H) and the dequantised B are f16
            const uint32_t idesc =
                kI8 ? idesc_f16(kBM, bn) : idesc_bf16(kPair ? 2 * kBM : kBM, bn);
            int stage = 0;
            uint32_t phase = 0;
            int bs = 0;              // kI8: converted-B stage
            uint32_t bphase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int w = unit; w < total && !*abort_flag; w += n_units) {
                const Work wk = work_at(w);
                const int kb0 = wk.split * kb_per_split;
                const int kb1 = min(args.k_blocks, kb0 + kb_per_split);
                if (!mbar_wait(smem_u32(&acc_empty[acc]), acc_phase ^ 1, abort_flag, args.status,
                               limit))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kAccCols;
                // weights as M: N is the tile's token count rounded up to 32
                const uint32_t idesc_w = kWM ? idesc_bf16(2 * kBM, wm_cols(wk.rows)) : idesc;
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    // kI8: A from its own ring (`stage` counts A stages), B
                    // from the converters' f16 ring
                    const bool got =
                        kI8 ? mbar_wait(smem_u32(&bf_full[bs]), bphase, abort_flag, args.status,
                                        limit) &&
                                  mbar_wait(smem_u32(&a_full[stage]), phase, abort_flag,
                                            args.status, limit)
                            : mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.status,
                                        limit);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = smem_desc_sw128(smem_u32(stage_a + stage * kStageA));
                    const uint64_t db = smem_desc_sw128(
                        smem_u32(kI8 ? stage_bf + bs * kStageBf : stage_b + stage * kStageB));
#pragma unroll
                    for (int ks = 0; ks < kBK / 16; ++ks)
                        // +32 bytes of K per step inside the swizzle atom (encoded >> 4)
                        mma_bf16<kPair>(d_tmem, da + 2 * ks, db + 2 * ks, idesc_w,
                                        (kb > kb0) || ks != 0);
                    if constexpr (kI8) {
                        mma_commit<kPair>(smem_u32(&a_empty[stage]));
                        mma_commit<kPair>(smem_u32(&bf_empty[bs]));
                        if (++stage == kAStagesI8) stage = 0, phase ^= 1;
                        if (++bs == kBStages) bs = 0, bphase ^= 1;
                    } else {
                        mma_commit<kPair>(smem_u32(&empty[stage]));
                        if (++stage == kStages) stage = 0, phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit<kPair>(smem_u32(&acc_full[acc]));
                if (++acc == 2) acc = 0, acc_phase ^= 1;
            }
            // Teardown: all MMAs issued by this thread complete before TMEM is freed.
            mma_commit_local<kPair>(smem_u32(&mma_done[0]));
            mbar_wait_drain(smem_u32(&mma_done[0]), 0, kDrainLimitNs);
        }
        __syncwarp();
    } else if (!kI8 || warp < 6) {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;       // row of this CTA's 128-row half
        // router: this warp's copy of the logit offset
        const float* bias_sh = nullptr;
        if constexpr (kMode == kRouter) {
            if (args.bias) {
                float* b = reinterpret_cast<float*>(smem + kBiasOffset) + (warp - 2) * (kBiasWarpBytes / 4);
                for (int e = lane; e < args.n_experts; e += 32) b[e] = args.bias[e];
                __syncwarp();
                bias_sh = b;
            }
        }
        const uint32_t acc_empty_leader0 =
            kPair ? map_to_rank(smem_u32(&acc_empty[0]), 0) : smem_u32(&acc_empty[0]);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int w = unit; w < total; w += n_units) {
            const Work wk = work_at(w);
            const bool got =
                mbar_wait(smem_u32(&acc_full[acc]), acc_phase, abort_flag, args.status, limit);
            // tcgen05.ld is warp-collective: the whole warp stops if any lane gave up.
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * kAccCols;
            const int my_row = (int)rank * kBM + row;          // row inside the tile
            const bool live = my_row < wk.rows;
            const size_t orow = (size_t)(wk.row0 + my_row);
            float* stg = reinterpret_cast<float*>(smem + kStagingOffset) + (warp - 2) * 32 * kStgStride;
            if constexpr (kWM) {
                // TMEM lane = weight row of this CTA, column = token of the tile
                const int ncol = wm_cols(wk.rows);
                if constexpr (kMode == kGateUp) {
                    // lanes 0-15 hold the gate and lanes 16-31 the up rows of
                    // 16 hidden units; one shuffle per token pairs them, and
                    // lanes 0-15 form and store the chunk's first 16 tokens,
                    // lanes 16-31 the last 16 (a store: 16 consecutive units)
                    uint16_t* H = reinterpret_cast<uint16_t*>(args.out);
                    const int unit = wk.nblk * kBM + (int)rank * 64 + q * 16 + (lane & 15);
                    const int hi = lane >> 4;
#pragma unroll 1
                    for (int c = 0; c < ncol; c += 32) {
                        uint32_t v[32];
                        tmem_ld32(tbase + c, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            // lane < 16 sends its gate of token 16 + i and gets
                            // the up of token i; lane >= 16 the other way round
                            const float mine = __uint_as_float(hi ? v[16 + i] : v[i]);
                            const float other = __shfl_xor_sync(
                                0xffffffffu, __uint_as_float(hi ? v[i] : v[16 + i]), 16);
                            const float g = hi ? other : mine, u = hi ? mine : other;
                            const int t = c + 16 * hi + i;
                            if (t < wk.rows) {
                                // fast exp and divide (|rel err| ~1e-6, far
                                // below the bf16 rounding of H)
                                const float sg = __fdividef(g, 1.0f + __expf(-g));
                                const __nv_bfloat16 hb = __float2bfloat16_rn(sg * u);
                                H[(size_t)(wk.row0 + t) * args.out_ld + unit] =
                                    *reinterpret_cast<const uint16_t*>(&hb);
                            }
                        }
                    }
                } else {
                    const int feat = wk.nblk * kBN + (int)rank * kBM + q * 32 + lane;
                    float* Y = reinterpret_cast<float*>(args.out) + wk.split * args.out_split_stride;
                    uint16_t* Yb = reinterpret_cast<uint16_t*>(args.out);
#pragma unroll 1
                    for (int c = 0; c < ncol; c += 32) {
                        uint32_t v[32];
                        tmem_ld32(tbase + c, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int t = c + i;
                            if (t < wk.rows) {
                                const size_t o = (size_t)(wk.row0 + t) * args.out_ld + feat;
                                if (args.y_bf16) {
                                    const __nv_bfloat16 yb = __float2bfloat16_rn(__uint_as_float(v[i]));
                                    Yb[o] = *reinterpret_cast<const uint16_t*>(&yb);
                                } else {
                                    Y[o] = __uint_as_float(v[i]);
                                }
                            }
                        }
                    }
                }
            } else if constexpr (kMode == kRouter) {
                float* mine = stg + lane * 33;     // own row, stride 33: conflict-free
                if (args.k_splits > 1) {
                    // One K slice: the thread's float32 partial logits go to
                    // the slice's buffer [T][E padded to 16] (all bn
                    // columns); the last slice to arrive on this quarter of
                    // the tile routes its rows (below).
                    float* P = args.partial + wk.split * args.partial_split_stride;
#pragma unroll 1
                    for (int c = 0; c < bn; c += 32) {
                        uint32_t v[32];
                        tmem_ld32(tbase + c, v);
                        tmem_ld_wait();
                        if (live) {
                            float4* dst = reinterpret_cast<float4*>(P + orow * bn + c);
                            const int nv = min(32, bn - c) / 4;
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                if (i < nv)
                                    dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                         __uint_as_float(v[4 * i + 2]),
                                                         __uint_as_float(v[4 * i + 3]));
                        }
                    }
                } else {
                    const int k = args.top_k;
                    if (k <= 1) router_rows_tmem<1>(tbase, bn, mine, args, bias_sh, live, orow);
                    else if (k <= 2) router_rows_tmem<2>(tbase, bn, mine, args, bias_sh, live, orow);
                    else if (k <= 4) router_rows_tmem<4>(tbase, bn, mine, args, bias_sh, live, orow);
                    else router_rows_tmem<8>(tbase, bn, mine, args, bias_sh, live, orow);
                }
            } else if constexpr (kMode == kGateUp) {
              if (args.k_splits > 1) {
                // One K slice: the float32 partial of this thread's G|U row
                // (256 columns) goes to the slice's partial buffer; H is
                // written after the accumulator is released (below).
                float* P = args.partial + wk.split * args.partial_split_stride;
                const int pld = args.n_blocks * 256;
#pragma unroll 1
                for (int c = 0; c < 256 / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tbase + c * 32, v);
                    tmem_ld_wait();
                    if (live) {
                        float4* dst = reinterpret_cast<float4*>(P + orow * pld + wk.nblk * 256 + c * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                 __uint_as_float(v[4 * i + 2]),
                                                 __uint_as_float(v[4 * i + 3]));
                    }
                }
              } else {
                // H = silu(G) * U for this thread's row, 32 columns per chunk,
                // stored straight from registers: each row's 64 bytes are two
                // whole sectors, so staging them buys nothing here.
                uint16_t* H = reinterpret_cast<uint16_t*>(args.out);
#pragma unroll 1
                for (int c = 0; c < 128 / 32; ++c) {
                    uint32_t g[32], u[32];
                    tmem_ld32(tbase + c * 32, g);
                    tmem_ld32(tbase + 128 + c * 32, u);
                    tmem_ld_wait();
                    if (live) {
                        uint4 pk[4];
                        uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float h0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
                            const float h1 =
                                silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
                            pw[i] = pack_h2<kI8>(h0, h1);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(H + orow * args.out_ld +
                                                              wk.nblk * 128 + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = pk[i];
                    }
                }
              }
            } else {
                // Y for this thread's row, 32 columns per chunk, staged and
                // stored as row segments, 4 rows per warp instruction: float32
                // (128 bytes a row), or bf16 (64 bytes) when the GEMM has no K
                // slices and args.y_bf16 is set.
                float* Y = reinterpret_cast<float*>(args.out) + wk.split * args.out_split_stride;
                __nv_bfloat16* Yb = reinterpret_cast<__nv_bfloat16*>(args.out);
                const int row_base = (int)rank * kBM + q * 32;
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tbase + c * 32, v);
                    tmem_ld_wait();
                    float4* mine = reinterpret_cast<float4*>(stg + lane * kStgStride);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        mine[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                              __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                    __syncwarp();
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int rr = it * 4 + (lane >> 3), c4 = lane & 7;
                        if (row_base + rr < wk.rows) {
                            const float4 val = reinterpret_cast<const float4*>(stg + rr * kStgStride)[c4];
                            const size_t o = (size_t)(wk.row0 + row_base + rr) * args.out_ld + wk.nblk * kBN +
                                             c * 32 + c4 * 4;
                            if (args.y_bf16) {
                                uint2 pk;
                                pk.x = pack_h2<false>(val.x, val.y);
                                pk.y = pack_h2<false>(val.z, val.w);
                                *reinterpret_cast<uint2*>(Yb + o) = pk;
                            } else {
                                *reinterpret_cast<float4*>(Y + o) = val;
                            }
                        }
                    }
                    __syncwarp();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                const uint32_t ae = acc_empty_leader0 + acc * 8;   // &acc_empty[acc] in the leader
                if constexpr (kPair) mbar_arrive_cluster(ae);
                else mbar_arrive(ae);
            }
            if constexpr (kMode == kGateUp) {
                if (args.k_splits > 1) gate_up_split_fixup<kI8>(args, wk, lane);
            }
            if constexpr (kMode == kRouter) {
                if (args.k_splits > 1)
                    router_split_fixup(args, wk, q, lane, stg + lane * 33, bias_sh);
            }
            if (++acc == 2) acc = 0, acc_phase ^= 1;
        }
    } else if (kI8 && warp == kAWarp) {
        // ------------------------------------------------ A producer (kI8)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool issued[kAStagesI8];
            uint32_t issued_phase[kAStagesI8];
            for (int s = 0; s < kAStagesI8; ++s) issued[s] = false, issued_phase[s] = 0;
            for (int w = unit; w < total && !*abort_flag && !args.stall_producer; w += n_units) {
                const Work wk = work_at(w);
                const int kb0 = wk.split * kb_per_split;
                const int kb1 = min(args.k_blocks, kb0 + kb_per_split);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&a_empty[stage]), phase ^ 1, abort_flag, args.status,
                                   limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t ab = smem_u32(&a_full[stage]);
                    mbar_expect_tx(ab, kStageA);
                    tma_load_2d(smem_u32(stage_a + stage * kStageA), &tmA, kb * kBK, wk.row0, ab);
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == kAStagesI8) stage = 0, phase ^= 1;
                }
                if (!ok) break;
            }
            for (int s = 0; s < kAStagesI8; ++s)
                if (issued[s]) mbar_wait_drain(smem_u32(&a_full[s]), issued_phase[s], kDrainLimitNs);
        }
        __syncwarp();
    } else if constexpr (kI8) {
        // ------------------------------------------------ converters (warps 6..13)
        // Walk the same k-blocks as the producers and the MMA issuer: wait for
        // the stage's codes to land and for a free f16 B stage, dequantise
        // with the 64-row blocks' scales and zero points, release the codes,
        // make the stores visible to the tensor core's proxy, and count the
        // warp in.
        const int ct = threadIdx.x - 6 * 32;
        int stage = 0;
        uint32_t phase = 0;
        int bs = 0;
        uint32_t bphase = 0;
        for (int w = unit; w < total && !*abort_flag; w += n_units) {
            const Work wk = work_at(w);
            const int kb0 = wk.split * kb_per_split;
            const int kb1 = min(args.k_blocks, kb0 + kb_per_split);
            // first packed B row of the tile; a multiple of 64 (one block row)
            const int rb0 = (wk.expert * args.b_rows_per_expert + wk.nblk * kBN) >> 6;
            const float* sc_row = args.q_scale + (size_t)rb0 * args.k_blocks;
            const int32_t* zp_row = args.q_zp + (size_t)rb0 * args.k_blocks;
            // The four 64-row blocks' scale and zero point of k-block kb; the
            // next k-block's are loaded one stage ahead, so that their L2
            // latency hides behind a conversion.
            float scl[4], zpf[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                scl[j] = __ldg(sc_row + (size_t)j * args.k_blocks + kb0);
                zpf[j] = (float)__ldg(zp_row + (size_t)j * args.k_blocks + kb0);
            }
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                float nscl[4], nzpf[4];
                const int kn = kb + 1 < kb1 ? kb + 1 : kb;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    nscl[j] = __ldg(sc_row + (size_t)j * args.k_blocks + kn);
                    nzpf[j] = (float)__ldg(zp_row + (size_t)j * args.k_blocks + kn);
                }
                const bool got =
                    mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.status, limit) &&
                    mbar_wait(smem_u32(&bf_empty[bs]), bphase ^ 1, abort_flag, args.status, limit);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                __half2 off2[4], s2[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    off2[j] = __float2half2_rn(1152.0f + zpf[j]);   // exact: an integer < 2048
                    s2[j] = __float2half2_rn(scl[j]);
                }
                convert_stage(stage_b + stage * kStageB, stage_bf + bs * kStageBf, ct, off2, s2);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));   // codes read
#pragma unroll
                for (int j = 0; j < 4; ++j) scl[j] = nscl[j], zpf[j] = nzpf[j];
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bf_full[bs]));
                if (++stage == kStages) stage = 0, phase ^= 1;
                if (++bs == kBStages) bs = 0, bphase ^= 1;
            }
            if (!ok) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    // A pair ends together: the leader's MMAs read the peer's shared memory
    // and the peer's copies complete on the leader's barriers.
    if constexpr (kPair) cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<kPair>(tmem_base, kTmemCols);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

}  // namespace

bool make_tmap_gate_up_wm(CUtensorMap* map, const void* wgu, uint64_t rows, uint64_t d) {
    // The packed gate/up rows [E][f/128][2][128][d] seen as 5-D:
    //   (k, i, which, g, j) -> row j*64 + which*128 + g*16 + i, column k,
    // j = 4 * (128-unit block) + half; a box {64, 16, 2, 4, 1} is, in order,
    // group g's 16 gate rows then its 16 up rows for g = 0..3: the 64 hidden
    // units of one half-block with gate and up interleaved per 16 units.
    EncodeTiledFn fn = encode_fn();
    if (!fn || rows % 256 || d % 64) return false;
    const cuuint64_t D = d * 2;
    const cuuint64_t dims[5] = {d, 16, 2, 4, rows / 64};
    const cuuint64_t strides[4] = {D, 128 * D, 16 * D, 64 * D};
    const cuuint32_t box[5] = {(cuuint32_t)kBK, 16, 2, 4, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(wgu), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_token_rows(TokenRowMaps* maps, const void* base, uint64_t rows, uint64_t cols) {
    for (int i = 0; i < 8; ++i)
        if (!make_tmap_bf16(&maps->m[i], base, rows, cols, (uint32_t)(16 * (i + 1)))) return false;
    return true;
}

size_t tc_gemm_smem_bytes() {
    // ring + barriers (512 B) + 4 epilogue staging tiles + 1024-byte alignment slack
    return (size_t)kBiasOffset + 1024;
}
int tc_gemm_block_m() { return kBM; }
int tc_gemm_pair_rows() { return 2 * kBM; }

// Tensor map of a row-major bf16 (or f16) matrix [rows, cols] with a box of
// 64 columns x box_rows rows, 128-byte swizzle, zero fill out of bounds.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows, bool f16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
              const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The B maps of launches that are not weights-as-M (never read).
const TokenRowMaps kNoTokenRowMaps = {};

template <int kMode, bool kPair, bool kI8 = false, bool kWM = false>
cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmB, const TcGemmArgs& args,
                       int grid, cudaStream_t s, const TokenRowMaps& tmBr = kNoTokenRowMaps) {
    // the router's epilogue warps also keep the logit offset in shared memory
    const size_t smem = tc_gemm_smem_bytes() + (kMode == kRouter ? 4 * kBiasWarpBytes : 0);
    auto k = grouped_gemm_tc<kMode, kPair, kI8, kWM>;
    smem_attr((const void*)k, (int)smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kI8 ? kThreadsI8 : kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k, tmA, tmB, tmBr, args);
}

cudaError_t launch_tc_gemm(int mode, bool pair, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           const TcGemmArgs& args, int grid, cudaStream_t s, bool int8_b,
                           bool weights_m, const TokenRowMaps* wm_b) {
    if (grid <= 0) return cudaSuccess;
    if (weights_m) {
        // CTA pairs, bf16, gate/up over the whole K (the down projection may
        // be split into float32 K slices): tmA the weights (make_tmap_gate_up_wm
        // for gate/up, 128-row boxes for down), wm_b the token rows
        if (!pair || int8_b || !wm_b || mode == kRouter || (mode == kGateUp && args.k_splits != 1) ||
            (args.y_bf16 && args.k_splits != 1))
            return cudaErrorInvalidValue;
        const cudaError_t e =
            mode == kGateUp ? launch_one<kGateUp, true, false, true>(tmA, tmB, args, grid & ~1, s, *wm_b)
                            : launch_one<kDown, true, false, true>(tmA, tmB, args, grid & ~1, s, *wm_b);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    // bf16 Y: the down projection's rows, not K slices
    if (args.y_bf16 && (mode != kDown || args.k_splits > 1)) return cudaErrorInvalidValue;
    // the split gate/up and router fixups count epilogue warps of single CTAs
    if ((mode == kGateUp || mode == kRouter) && args.k_splits > 1 &&
        (pair || !args.partial || !args.tile_counter))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (int8_b) {
        // B: two 128-row code tiles per 256-row tile; single CTAs
        if (pair || mode == kRouter || !args.q_scale || !args.q_zp || !args.q_codes ||
            args.b_rows_per_expert % 128)
            return cudaErrorInvalidValue;
        e = mode == kGateUp ? launch_one<kGateUp, false, true>(tmA, tmB, args, grid, s)
                            : launch_one<kDown, false, true>(tmA, tmB, args, grid, s);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    if (mode == kGateUp)
        e = pair ? launch_one<kGateUp, true>(tmA, tmB, args, grid & ~1, s)
                 : launch_one<kGateUp, false>(tmA, tmB, args, grid, s);
    else if (mode == kDown)
        e = pair ? launch_one<kDown, true>(tmA, tmB, args, grid & ~1, s)
                 : launch_one<kDown, false>(tmA, tmB, args, grid, s);
    else
        e = launch_one<kRouter, false>(tmA, tmB, args, grid, s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int tc_gemm_max_pairs() {
    // CTA pairs of the expert GEMMs that can be resident at once.
    static int pairs = -1;
    if (pairs < 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = tc_gemm_smem_bytes();
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        auto k = grouped_gemm_tc<kGateUp, true, false, false>;
        smem_attr((const void*)k, (int)tc_gemm_smem_bytes());
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess || n <= 0) n = 0;
        pairs = n;
    }
    return pairs;
}

}  // namespace colibri
