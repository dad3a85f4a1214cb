// Int8-weight expert FFN for decode batches of a few tokens per expert, on
// CUDA cores, for bf16 layers.
//
// zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析" section 3.3 stage 4
// (gate_proj, up_proj, SiLU, down_proj per activated expert) with the weights
// as int8 codes in 64x64 blocks, w = (q - zp) * scale (m.nxbn.cn section 3.1;
// pnsm.cn section 5.2).  With one to four tokens per expert the layer is a
// stream of weight codes: every code is read from HBM once and takes part in
// one multiply-add per token.  The tensor cores need one M = 128, K = 16 MMA
// per 2 KB of codes whatever the token count, which caps them near 0.7 of
// HBM; here the products are integer dot products on the CUDA cores.
//
// Arithmetic.  Each token's activations are staged per 64-wide k-tile (one
// scale block of K) as 16-bit integers x16 = round(x * 2^e), e the largest
// exponent with max|x| * 2^e < 2^15 over the k-tile: every bf16 activation
// within a factor 2^7 of the k-tile's largest is represented exactly, the
// others to within 2^-16 of that largest.  One dp2a multiplies two codes by
// two x16 and adds them to an int32, so a lane's 16 codes of a k-tile cost
// eight instructions per token and their sum is exact (|sum| < 2^26).  With
// P the k-tile's code-activation sum and X its activation sum,
//   sum_k (q_k - zp) x_k = 2^-e (P - zp X),
// scaled by the block's scale; the zp X part is the same for the 64 rows of a
// block and is formed once per k-tile while staging.
//
// Measured on the Mixtral-shaped layer (two experts, 235 MB of gate/up codes,
// 117 MB of down codes), the access pattern alone (bulk copies, no arithmetic)
// streams at 0.91 of the copy bandwidth with four 8 KB stages per CTA (six
// or more: slower, fewer CTAs fit) and 0.73 for the down projection's
// 896 short items, whose first bytes arrive microseconds after launch: its
// producer therefore starts streaming codes before the gate/up kernel has
// finished (the tile list comes from the routing, which completed before
// the gate/up kernel let this one launch; the codes do not depend on H).
//
// Work.  A CTA takes one item at a time: 64 weight rows (one scale block)
// over the whole K (gate/up: 64 hidden units, gate and up rows) or over one of
// `ks` K slices (down), for the tokens of one expert tile.  A producer warp
// streams the item's codes k-tile by k-tile into a ring of shared-memory
// stages with bulk copies (each k-tile of 64 rows is 4 KB contiguous in the
// 128x64 code tiles); four consumer warps share the staged activations and
// each takes 16 rows as two 8-row groups.  A consumer lane reads 16 bytes of a
// 512-byte group slice: row l/4, 16-code chunk l%4 as stored, which the
// tiles' chunk swizzle makes logical chunk (l%4) ^ ((l/8)%4) for every row the
// lane touches, so each lane multiplies the same 16 activations of a k-tile
// into all its rows.
#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace colibri {

namespace {

constexpr int kGvWarps = 4;                      // consumer warps
constexpr int kGvThreads = (kGvWarps + 1) * 32;  // + the producer warp
constexpr int kGvRows = 64;              // weight rows per item (one scale block)
constexpr int kGvStagesUp = 4;           // 8 KB stages (gate and up k-tiles)
constexpr int kGvStagesDown = 6;         // 4 KB stages
constexpr int kGvBarBytes = 256;         // barriers and the abort flag after the ring

template <bool kUp> constexpr int gv_stage_bytes() { return kUp ? 8192 : 4096; }
template <bool kUp> constexpr int gv_stages() { return kUp ? kGvStagesUp : kGvStagesDown; }

__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kGvWarps * 32) : "memory");
}

// c + a.lo16 * b.byte0 + a.hi16 * b.byte1 (lo) or bytes 2, 3 (hi), signed.
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// P[s] = sum over the 16 codes of v of q * x16_s, x16_s the lane's 16 staged
// activations of token s as 8 packed pairs (xw[s][0] pairs 0-3, [1] 4-7).
template <int NS>
__device__ __forceinline__ void code_dot(const uint4& v, const uint4 (&xw)[NS][2], int (&P)[NS]) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        int p = 0;
        p = dp2a_lo(xw[s][0].x, v.x, p);
        p = dp2a_hi(xw[s][0].y, v.x, p);
        p = dp2a_lo(xw[s][0].z, v.y, p);
        p = dp2a_hi(xw[s][0].w, v.y, p);
        p = dp2a_lo(xw[s][1].x, v.z, p);
        p = dp2a_hi(xw[s][1].y, v.z, p);
        p = dp2a_lo(xw[s][1].z, v.w, p);
        p = dp2a_hi(xw[s][1].w, v.w, p);
        P[s] = p;
    }
}

// mbar_wait for a whole warp, with one outcome for all its lanes: every lane
// polls the barrier (each acquires the completed phase itself), and the warp
// gives up together once the time limit passes or another warp has aborted.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, uint64_t limit_ns) {
    using namespace tc;
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        const bool late = globaltimer() - t0 > limit_ns;
        if (__any_sync(0xffffffffu, late || *abort_flag != 0)) {
            if (__any_sync(0xffffffffu, late) && (threadIdx.x & 31) == 0) {
                *abort_flag = 1;
                atomicExch(status, DEV_TIMEOUT);
            }
            return false;
        }
    }
}

// Row of the packed gate/up weight: [E][f/128][2][128][d], which = 0 gate, 1 up.
__device__ __forceinline__ int64_t gu_row(int e, int n, int which, int f) {
    return ((int64_t)(e * (f / 128) + n / 128) * 2 + which) * 128 + (n % 128);
}

// Staging area of one pass (S token rows, kt_max k-tiles).
struct Staged {
    uint8_t* x16;      // [S][kt_max][64] int16
    float2* comb;      // [S][kt_max] (scale_a, scale_b) * 2^-e
    float2* corr;      // [S][kt_max] comb * zp * X, rows a and b
};

__device__ __forceinline__ Staged staged_at(uint8_t* base, int S, int kt_max) {
    Staged st;
    st.x16 = base;
    st.comb = reinterpret_cast<float2*>(base + (size_t)S * kt_max * 128);
    st.corr = st.comb + (size_t)S * kt_max;
    return st;
}

// The k-tile loop of one pass with NS token rows (NS <= the staged S):
// codes from the ring, activations from the staging area.  Returns false
// when a wait gave up (the pass's remaining stages are left unread).
template <int NS, int S, bool kUp>
__device__ __forceinline__ bool pass_tiles(const uint8_t* ring, uint64_t* full, uint64_t* empty,
                                           int& stage, uint32_t& phase, int nkt, int kt_max,
                                           const Staged& sg, int warp, int lane,
                                           volatile int* abort_flag, int* status, uint64_t limit,
                                           float (&acc_a)[2][S], float (&acc_b)[2][S]) {
    using namespace tc;
    constexpr int kStages = gv_stages<kUp>();
    const int chunk = (lane & 3) ^ ((lane >> 3) & 3);
    const int off = warp * 16 * 64 + lane * 16;
    for (int kt = 0; kt < nkt; ++kt) {
        if (!warp_wait(smem_u32(&full[stage]), phase, abort_flag, status, limit)) return false;
        const uint8_t* st = ring + stage * gv_stage_bytes<kUp>();
        const uint4 a0 = *reinterpret_cast<const uint4*>(st + off);
        const uint4 a1 = *reinterpret_cast<const uint4*>(st + off + 512);
        uint4 b0, b1;
        if (kUp) {
            b0 = *reinterpret_cast<const uint4*>(st + 4096 + off);
            b1 = *reinterpret_cast<const uint4*>(st + 4096 + off + 512);
        }
        uint4 xw[NS][2];
        float2 cs[NS];
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const uint4* xp =
                reinterpret_cast<const uint4*>(sg.x16 + ((size_t)(s * kt_max + kt) * 128 + chunk * 32));
            xw[s][0] = xp[0];
            xw[s][1] = xp[1];
            cs[s] = sg.comb[s * kt_max + kt];
        }
        int P[NS];
        code_dot<NS>(a0, xw, P);
#pragma unroll
        for (int s = 0; s < NS; ++s) acc_a[0][s] = fmaf(cs[s].x, (float)P[s], acc_a[0][s]);
        code_dot<NS>(a1, xw, P);
#pragma unroll
        for (int s = 0; s < NS; ++s) acc_a[1][s] = fmaf(cs[s].x, (float)P[s], acc_a[1][s]);
        if (kUp) {
            code_dot<NS>(b0, xw, P);
#pragma unroll
            for (int s = 0; s < NS; ++s) acc_b[0][s] = fmaf(cs[s].y, (float)P[s], acc_b[0][s]);
            code_dot<NS>(b1, xw, P);
#pragma unroll
            for (int s = 0; s < NS; ++s) acc_b[1][s] = fmaf(cs[s].y, (float)P[s], acc_b[1][s]);
        }
        // the stage's codes are consumed: the warp releases it
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
        if (++stage == kStages) stage = 0, phase ^= 1;
    }
    return true;
}

// kUp: x = token rows (pair p reads row perm[p] / k), K = d, rows = hidden
// units; H[p, n] = silu(g) * u rounded to bf16.  Otherwise x = H rows in pair
// order, K = f, rows = output features, K split into ks slices; slice s
// writes its float32 partial to Y + s * y_split_stride.  Every wait is
// bounded by limit_ns; one that gives up sets DEV_TIMEOUT in *status and the
// CTA winds down (the producer waits for its copies in flight).
template <int S, bool kUp>
__global__ void __launch_bounds__(kGvThreads)
ffn_gemv_i8(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ perm, int k,
            const int8_t* __restrict__ wq, const float* __restrict__ sc,
            const int32_t* __restrict__ zpt, const int32_t* __restrict__ tile_expert,
            const int32_t* __restrict__ tile_row, const int32_t* __restrict__ tile_info,
            const int32_t* __restrict__ num_tiles, int E, int d, int f, int ks,
            __nv_bfloat16* __restrict__ H, float* __restrict__ Y, size_t y_split_stride,
            int* status, uint64_t limit, int stall) {
    using namespace tc;
    constexpr int kStages = gv_stages<kUp>();
    constexpr int kStageBytes = gv_stage_bytes<kUp>();
    extern __shared__ __align__(128) uint8_t gv_smem[];
    uint8_t* ring = gv_smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(gv_smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);
    static_assert(2 * kStages * 8 + 4 <= kGvBarBytes, "barriers fit their area");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = kUp ? d : f;
    const int nkb = K / 64;
    const int groups = (kUp ? f : d) / kGvRows;
    const int kt_max = (nkb + ks - 1) / ks;
    const Staged sg = staged_at(gv_smem + kStages * kStageBytes + kGvBarBytes, S, kt_max);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), kGvWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == kGvWarps) {
        // ------------------------------------------------ producer
        // gate/up: the tile list is the previous launch's output.  Down: it
        // is older (see above), so the codes stream before that wait; the
        // list is read from L2 and checked, never trusted for an address.
        if (kUp) pdl_wait();
        pdl_launch_dependents();
        if (lane == 0) {
            const int nt = __ldcg(num_tiles);
            const int n_items = nt * groups * ks;
            int stage = 0;
            uint32_t phase = 0;
            bool issued[kStages];
            uint32_t issued_phase[kStages];
            for (int i = 0; i < kStages; ++i) issued[i] = false, issued_phase[i] = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok && !stall; it += gridDim.x) {
                const int sl = it % ks;
                const int g = (it / ks) % groups;
                const int tile = it / (ks * groups);
                const int e = __ldcg(tile_expert + tile);
                const int rows = __ldcg(tile_info + tile) & 1023;
                if (e < 0 || e >= E) {
                    atomicExch(status, DEV_BAD_INDEX);
                    *abort_flag = 1;
                    break;
                }
                const int kt0 = (int)((int64_t)sl * nkb / ks);
                const int nkt = (int)((int64_t)(sl + 1) * nkb / ks) - kt0;
                const int64_t ra = kUp ? gu_row(e, g * kGvRows, 0, f) : (int64_t)e * d + g * kGvRows;
                const int8_t* src0 = wq + ((ra >> 7) * nkb + kt0) * 8192 + (ra & 127) * 64;
                for (int r0 = 0; r0 < rows && ok; r0 += S) {
                    for (int kt = 0; kt < nkt; ++kt) {
                        if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1, abort_flag, status, limit)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = smem_u32(&full[stage]);
                        const uint32_t dst = smem_u32(ring + stage * kStageBytes);
                        mbar_expect_tx(fb, kStageBytes);
                        bulk_load(dst, src0 + (int64_t)kt * 8192, 4096, fb);
                        if (kUp) bulk_load(dst + 4096, src0 + ((int64_t)nkb + kt) * 8192, 4096, fb);
                        issued[stage] = true;
                        issued_phase[stage] = phase;
                        if (++stage == kStages) stage = 0, phase ^= 1;
                    }
                }
            }
            for (int i = 0; i < kStages; ++i)
                if (issued[i]) mbar_wait_drain(smem_u32(&full[i]), issued_phase[i], kDrainLimitNs);
        }
        return;
    }

    // ---------------------------------------------------- consumers
    pdl_enter();
    const int n_items = *num_tiles * groups * ks;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;   // false once a wait gave up: the loops still run, doing nothing
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int sl = it % ks;
        const int g = (it / ks) % groups;
        const int tile = it / (ks * groups);
        const int e = min(max(tile_expert[tile], 0), E - 1);   // the producer reports a bad one
        const int p0 = tile_row[tile];
        const int rows = tile_info[tile] & 1023;
        const int kt0 = (int)((int64_t)sl * nkb / ks);
        const int nkt = (int)((int64_t)(sl + 1) * nkb / ks) - kt0;
        const int64_t ra = kUp ? gu_row(e, g * kGvRows, 0, f) : (int64_t)e * d + g * kGvRows;
        const int64_t blk_a = ra >> 6, blk_b = (ra + 128) >> 6;

        for (int r0 = 0; r0 < rows; r0 += S) {
            const int ns = min(S, rows - r0);
            consumers_sync();   // the previous pass is done with the staging area
            // Activations of the pass's tokens as x16 per k-tile: 16 threads
            // per k-tile, four values each; the first of the 16 also forms the
            // k-tile's scales and zero-point terms.
            {
                const __nv_bfloat16* src[S];
#pragma unroll
                for (int s = 0; s < S; ++s) {
                    const int p = p0 + r0 + min(s, ns - 1);
                    src[s] = kUp ? x + (int64_t)(perm[p] / k) * K : x + (int64_t)p * K;
                }
                const int per_tok = nkt * 16;
                for (int b = 0; b < S * per_tok; b += kGvWarps * 32) {
                    const int i = b + threadIdx.x;
                    const bool on = i < S * per_tok;
                    const int s = on ? i / per_tok : 0;
                    const int j = i - s * per_tok;
                    const int kt = j >> 4;
                    uint2 raw = make_uint2(0u, 0u);
                    if (on && s < ns) {
                        const __nv_bfloat16* row = src[0];   // static indices keep src in registers
#pragma unroll
                        for (int q = 1; q < S; ++q)
                            if (s == q) row = src[q];
                        raw = __ldg(reinterpret_cast<const uint2*>(row + (int64_t)(kt0 + kt) * 64 +
                                                                   4 * (j & 15)));
                    }
                    const float v[4] = {__uint_as_float(raw.x << 16),
                                        __uint_as_float(raw.x & 0xffff0000u),
                                        __uint_as_float(raw.y << 16),
                                        __uint_as_float(raw.y & 0xffff0000u)};
                    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
                    for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    // m * 2^e in [2^14, 2^15): e = 14 - exponent(m), kept where
                    // 2^e and 2^-e are normal floats (m == 0: e = 0, all zero)
                    const int em = (int)((__float_as_uint(m) >> 23) & 255) - 127;
                    const int e2 = m > 0.f ? max(-126, min(126, 14 - em)) : 0;
                    const float up = __uint_as_float((uint32_t)(e2 + 127) << 23);
                    int r[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) r[c] = max(-32767, min(32767, __float2int_rn(v[c] * up)));
                    if (on)
                        *reinterpret_cast<uint2*>(sg.x16 + (size_t)(s * kt_max + kt) * 128 + (j & 15) * 8) =
                            make_uint2(((uint32_t)r[0] & 0xffffu) | ((uint32_t)r[1] << 16),
                                       ((uint32_t)r[2] & 0xffffu) | ((uint32_t)r[3] << 16));
                    int t = (r[0] + r[1]) + (r[2] + r[3]);
#pragma unroll
                    for (int o = 1; o < 16; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                    if (on && (j & 15) == 0) {
                        const float down = __uint_as_float((uint32_t)(127 - e2) << 23);
                        const int64_t ia = blk_a * nkb + kt0 + kt;
                        const float ca = __ldg(sc + ia) * down;
                        float cb = 0.f, zb = 0.f;
                        if (kUp) {
                            const int64_t ib = blk_b * nkb + kt0 + kt;
                            cb = __ldg(sc + ib) * down;
                            zb = cb * ((float)__ldg(zpt + ib) * (float)t);
                        }
                        sg.comb[s * kt_max + kt] = make_float2(ca, cb);
                        sg.corr[s * kt_max + kt] =
                            make_float2(ca * ((float)__ldg(zpt + ia) * (float)t), zb);
                    }
                }
            }
            consumers_sync();
            // zero-point terms of the block rows: sum over k-tiles
            float corr_a[S], corr_b[S];
#pragma unroll
            for (int s = 0; s < S; ++s) {
                float ta = 0.f, tb = 0.f;
                for (int kt = lane; kt < nkt; kt += 32) {
                    const float2 c2 = sg.corr[s * kt_max + kt];
                    ta += c2.x;
                    tb += c2.y;
                }
                corr_a[s] = warp_sum(ta);
                corr_b[s] = kUp ? warp_sum(tb) : 0.f;
            }

            float acc_a[2][S], acc_b[2][S];
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int s = 0; s < S; ++s) acc_a[q][s] = acc_b[q][s] = 0.f;
            if (ok) {
                // as many token rows as the pass holds: one, two or S
                if (ns == 1)
                    ok = pass_tiles<1, S, kUp>(ring, full, empty, stage, phase, nkt, kt_max, sg,
                                               warp, lane, abort_flag, status, limit, acc_a, acc_b);
                else if (S >= 4 && ns <= 2)
                    ok = pass_tiles<(S >= 4 ? 2 : 1), S, kUp>(ring, full, empty, stage, phase, nkt,
                                                              kt_max, sg, warp, lane, abort_flag,
                                                              status, limit, acc_a, acc_b);
                else
                    ok = pass_tiles<S, S, kUp>(ring, full, empty, stage, phase, nkt, kt_max, sg,
                                               warp, lane, abort_flag, status, limit, acc_a, acc_b);
            }
            if (!ok) continue;
            // the four lanes of a row hold its four 16-code chunks of every k-tile
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int s = 0; s < S; ++s) {
                    acc_a[q][s] += __shfl_xor_sync(0xffffffffu, acc_a[q][s], 1);
                    acc_a[q][s] += __shfl_xor_sync(0xffffffffu, acc_a[q][s], 2);
                    if (kUp) {
                        acc_b[q][s] += __shfl_xor_sync(0xffffffffu, acc_b[q][s], 1);
                        acc_b[q][s] += __shfl_xor_sync(0xffffffffu, acc_b[q][s], 2);
                    }
                }
            if ((lane & 3) == 0) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int r = g * kGvRows + warp * 16 + q * 8 + (lane >> 2);
#pragma unroll
                    for (int s = 0; s < S; ++s) {
                        if (s < ns) {
                            const int64_t p = p0 + r0 + s;
                            const float va = acc_a[q][s] - corr_a[s];
                            if (kUp) {
                                const float vb = acc_b[q][s] - corr_b[s];
                                H[p * f + r] = __float2bfloat16_rn(silu(va) * vb);
                            } else {
                                Y[sl * y_split_stride + p * d + r] = va;
                            }
                        }
                    }
                }
            }
        }
    }
}

size_t gemv_stage_area(int S, int kt_max) { return (size_t)S * kt_max * (128 + 16); }
template <bool kUp> size_t gemv_smem(int S, int kt_max) {
    return (size_t)gv_stages<kUp>() * gv_stage_bytes<kUp>() + kGvBarBytes +
           gemv_stage_area(S, kt_max);
}

template <int S, bool kUp>
cudaError_t launch_one(const void* x, const int32_t* perm, int k, const int8_t* wq,
                       const float* sc, const int32_t* zp, const GemvTiles& t, int d, int f,
                       int ks, int grid, void* H, float* Y, size_t y_split_stride,
                       cudaStream_t s) {
    auto kern = ffn_gemv_i8<S, kUp>;
    const int nkb = (kUp ? d : f) / 64;
    const int bytes = (int)gemv_smem<kUp>(S, (nkb + ks - 1) / ks);
    cudaError_t e = smem_attr(reinterpret_cast<const void*>(kern), bytes);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(grid), dim3(kGvThreads), (size_t)bytes, s, (const __nv_bfloat16*)x,
                   perm, k, wq, sc, zp, t.tile_expert, t.tile_row, t.tile_info, t.num_tiles, t.E, d,
                   f, ks, (__nv_bfloat16*)H, Y, y_split_stride, t.status, t.wait_limit_ns,
                   t.stall_producer);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <bool kUp>
cudaError_t launch_s(int S, const void* x, const int32_t* perm, int k, const int8_t* wq,
                     const float* sc, const int32_t* zp, const GemvTiles& t, int d, int f, int ks,
                     int grid, void* H, float* Y, size_t y_split_stride, cudaStream_t s) {
    if (S == 1)
        return launch_one<1, kUp>(x, perm, k, wq, sc, zp, t, d, f, ks, grid, H, Y, y_split_stride, s);
    if (S == 2)
        return launch_one<2, kUp>(x, perm, k, wq, sc, zp, t, d, f, ks, grid, H, Y, y_split_stride, s);
    return launch_one<4, kUp>(x, perm, k, wq, sc, zp, t, d, f, ks, grid, H, Y, y_split_stride, s);
}

}  // namespace

int gemv_i8_slots(int max_rows_per_expert) {
    return max_rows_per_expert <= 1 ? 1 : max_rows_per_expert <= 2 ? 2 : 4;
}

bool gemv_i8_fits(int S, int d, int f, int ks) {
    const size_t limit = 112 * 1024;   // two CTAs per SM at least
    return d % kGvRows == 0 && f % 128 == 0 && gemv_smem<true>(S, d / 64) <= limit &&
           gemv_smem<false>(S, (f / 64 + ks - 1) / ks) <= limit;
}

int gemv_i8_items(bool up, int tiles, int d, int f, int ks) {
    return tiles * ((up ? f : d) / kGvRows) * (up ? 1 : ks);
}

cudaError_t launch_ffn_up_gemv_i8(int S, const void* x, const int32_t* perm, int k,
                                  const int8_t* wq, const float* sc, const int32_t* zp,
                                  const GemvTiles& t, int d, int f, int grid, void* H,
                                  cudaStream_t s) {
    return launch_s<true>(S, x, perm, k, wq, sc, zp, t, d, f, 1, grid, H, nullptr, 0, s);
}

cudaError_t launch_ffn_down_gemv_i8(int S, const void* H, const int8_t* wq, const float* sc,
                                    const int32_t* zp, const GemvTiles& t, int d, int f, int ks,
                                    int grid, float* Y, size_t y_split_stride, cudaStream_t s) {
    return launch_s<false>(S, H, nullptr, 0, wq, sc, zp, t, d, f, ks, grid, nullptr, Y,
                           y_split_stride, s);
}

}  // namespace colibri
