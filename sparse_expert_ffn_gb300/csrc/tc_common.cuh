// Shared building blocks of the tcgen05 GEMM kernels (sm_103a): PTX wrappers
// for mbarriers, TMA, tensor memory and tcgen05.mma, shared-memory and
// instruction descriptors, the decode of the expert tile list into work
// items, and the split gate/up fixup.  Included by gemm_tc.cu (tokens as the
// MMA's M operand) and gemm_dec.cu (weights as M, for decode-sized batches).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "gemm_tc.h"

namespace colibri {
namespace tc {

constexpr int kBM = 128;          // tile rows (pairs)
constexpr int kBN = 256;          // tile columns of B rows per MMA
constexpr int kBK = 64;           // K per stage: one 128-byte swizzle atom of bf16

// Teardown waits (copies and MMAs already issued) use their own bound,
// independent of the configurable wait limit, so that a CTA never exits with
// a TMA copy or an MMA of its own still in flight.
constexpr uint64_t kDrainLimitNs = 1000000000ull;

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with parity `parity` of `bar` has completed, or the
// time limit passes, or another role has aborted.  Returns false on
// timeout/abort (and records the timeout).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicExch(status, DEV_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait used during teardown: ignores the abort flag.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > limit_ns) return;
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Contiguous copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global memory into this CTA's shared memory, completing on
// the mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// The same copy for a CTA pair: the mbarrier may be the peer CTA's (a
// shared::cluster address), so both halves of a pair's stage complete on the
// leader's barrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0,
                                                 int c1, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}

// A 5-D tile of the same kind (coordinates innermost first).
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                 int c2, int c3, int c4, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
        "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier of another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
                 : "memory");
}

// Tensor-memory allocation: for a CTA pair one warp of each CTA allocates
// the same columns collectively (cta_group::2).
template <bool kPair>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    if constexpr (kPair) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
}

template <bool kPair>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if constexpr (kPair)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, f32 accumulate).
// For a CTA pair (cta_group::2, issued by the leader) A is the 2 x 128 rows
// held by the two CTAs, B the 2 x N/2 rows, and each CTA's TMEM receives its
// own 128 rows of D over all N columns.
template <bool kPair>
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    if constexpr (kPair)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far has
// completed; for a pair, on the barrier at that offset in both CTAs.
template <bool kPair>
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    if constexpr (kPair) {
        const uint16_t both = 0x3;
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
            " [%0], %1;" ::"r"(bar),
            "h"(both)
            : "memory");
    } else {
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
            : "memory");
    }
}

// Commit onto the issuing CTA's own barrier only.
template <bool kPair>
__device__ __forceinline__ void mma_commit_local(uint32_t bar) {
    if constexpr (kPair)
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
            : "memory");
    else
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
            : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr));
}
// 32 consecutive 32-bit TMEM columns of this thread's lane, written.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
// 16 consecutive 32-bit TMEM columns of this thread's lane, written.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16, single CTA: A (M rows in TMEM
// lanes, 16-bit K pairs per 32-bit column) is read from tensor memory.
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), start
// address >> 4 in bits 0-13, descriptor version 1 in bits 46-47, layout
// "128-byte swizzle" (2) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset
    d |= (uint64_t)1 << 46;             // version
    d |= (uint64_t)2 << 61;             // SWIZZLE_128B
    return d;
}

// Instruction descriptor for kind::f16: f32 accumulator (bits 4-5 = 1),
// A and B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
// The same with A and B f16 (format 0 in bits 7-9 and 10-12).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Two floats as the 16-bit H element pair: bf16, or f16 for the int8-weight
// GEMMs (whose A operands are f16).
template <bool kF16>
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    if constexpr (kF16) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// ---------------------------------------------------------------- work decode

struct Work {
    int expert, row0, rows, nblk, split, tile;
};

// Work w -> (m-tile, n-block).  Bands of m-tiles (one expert each, from the
// dispatch kernel) are laid out back to back; inside a band the m-tile index
// runs fastest, so consecutive work items share one weight block.  The band
// holding work w contains the tile w / n_blocks.
__device__ __forceinline__ Work decode_work(int w, int n_blocks, int k_splits,
                                            const int32_t* __restrict__ tile_expert,
                                            const int32_t* __restrict__ tile_row,
                                            const int32_t* __restrict__ tile_info) {
    // (n-block, K slice) pairs act as one combined n index, slices fastest
    n_blocks *= k_splits;
    const int t = w / n_blocks;
    const int info = tile_info[t];
    const int first = t - ((info >> 10) & 0xFF);
    const int len = (info >> 18) & 0xFF;
    const int rem = w - first * n_blocks;
    const int nblk = rem / len;
    const int m = first + (rem - nblk * len);
    Work r;
    r.expert = tile_expert[m];
    r.row0 = tile_row[m];
    r.rows = tile_info[m] & 0x3FF;
    r.nblk = nblk / k_splits;
    r.split = nblk - r.nblk * k_splits;
    r.tile = m;
    return r;
}

// Router mode: dense m-tiles of 128 consecutive tokens, one n-block, K
// slices fastest.
__device__ __forceinline__ Work dense_work(int w, int rows_total, int k_splits) {
    Work r;
    const int t = w / k_splits;
    r.expert = 0;
    r.row0 = t * kBM;
    r.rows = min(kBM, rows_total - r.row0);
    r.nblk = 0;
    r.split = w - t * k_splits;
    r.tile = t;
    return r;
}

template <int kMode>
__device__ __forceinline__ Work get_work(int w, const TcGemmArgs& a) {
    if constexpr (kMode == kRouter) return dense_work(w, a.dense_rows, a.k_splits);
    else return decode_work(w, a.n_blocks, a.k_splits, a.tile_expert, a.tile_row, a.tile_info);
}

// Gate/up with K split into slices (single CTAs, few rows): every epilogue
// warp of every slice counts itself in on the (m-tile, n-block) counter after
// its partial rows are globally visible; the warp that arrives last adds the
// slices in slice order (so the sum does not depend on arrival order), applies
// SiLU(G)*U and writes the tile's H rows, then rearms the counter.  Nothing
// waits on another CTA.
template <bool kF16>
__device__ __noinline__ void gate_up_split_fixup(const TcGemmArgs& args, const Work& wk, int lane) {
    __threadfence();
    __syncwarp();
    int* ctr = args.tile_counter + (size_t)wk.tile * args.n_blocks + wk.nblk;
    int old = 0;
    if (lane == 0) old = atomicAdd(ctr, 1);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old != 4 * args.k_splits - 1) return;
    __threadfence();
    const int pld = args.n_blocks * 256;
    uint16_t* H = reinterpret_cast<uint16_t*>(args.out);
    for (int r = 0; r < wk.rows; ++r) {
        const size_t prow = (size_t)(wk.row0 + r) * pld + (size_t)wk.nblk * 256;
        float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
        for (int sl = 0; sl < args.k_splits; ++sl) {
            const float* ps = args.partial + sl * args.partial_split_stride + prow;
            const float4 gs = __ldcg(reinterpret_cast<const float4*>(ps) + lane);
            const float4 us = __ldcg(reinterpret_cast<const float4*>(ps + 128) + lane);
            g[0] += gs.x, g[1] += gs.y, g[2] += gs.z, g[3] += gs.w;
            u[0] += us.x, u[1] += us.y, u[2] += us.z, u[3] += us.w;
        }
        uint2 pk;
        pk.x = pack_h2<kF16>(silu(g[0]) * u[0], silu(g[1]) * u[1]);
        pk.y = pack_h2<kF16>(silu(g[2]) * u[2], silu(g[3]) * u[3]);
        *reinterpret_cast<uint2*>(H + (size_t)(wk.row0 + r) * args.out_ld + wk.nblk * 128 + lane * 4) = pk;
    }
    if (lane == 0) *ctr = 0;   // rearmed for the next launch
}

}  // namespace tc
}  // namespace colibri
