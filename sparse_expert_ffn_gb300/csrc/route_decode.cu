// Routing of a decode-sized batch in one launch over many CTAs: router
// logits, top-k, softmax over the k, dispatch and (for the grouped executor)
// the gather of the token rows into expert order.
//
// zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析" section 3.3 stages 2-3.
// For decode-sized batches each of these steps is a few microseconds of work
// but a launch and a memory round trip apiece.  Here:
//   1. every warp of the grid computes one partial logit: token t, expert e,
//      the q-th of nq slices of d (all of the slice's loads issued before
//      the first multiply), and writes it to `part`;
//   2. each CTA then takes a ticket (one atomic add after a memory fence);
//      the CTA that draws the last ticket has every partial in view and does
//      the serial rest alone: adds each logit's slices in slice order, runs
//      top-k and softmax (a warp per token), the block dispatch, and the
//      gather of small batches.  No CTA waits for another: the last one to
//      finish simply continues.
// For a pre-norm layer each warp first computes its token's RMS over the
// whole row (the same arithmetic in every warp, so every warp holds the same
// float) and forms u = bf16(h / rms * gamma) on its slice; the warps of
// expert 0 also write their u slices for the expert GEMMs.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "routing.cuh"

namespace colibri {

namespace {

constexpr int kRouteThreads = kDispatchWarps * 32;
constexpr int kMaxSlices = 16;
// 8-element vectors of a row loaded before any is used (float rows take
// twice the registers)
template <typename T> constexpr int row_batch() { return sizeof(T) == 2 ? 4 : 2; }

// Eight consecutive elements held as raw registers until they are used, so
// that a lane can keep several rows' vectors in flight at once.
template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
    uint4 a;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) {
        a = __ldg(reinterpret_cast<const uint4*>(p));
    }
    __device__ __forceinline__ void get(float (&v)[8]) const {
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(b[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
};
template <> struct Vec8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float* p) {
        a = __ldg(reinterpret_cast<const float4*>(p));
        b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ __forceinline__ void get(float (&v)[8]) const {
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};

// 1 / sqrt(mean(h^2) + eps) of one row by one warp: lane l adds the squares
// of elements 8l + 256j .. 8l + 256j + 7 in order, then the butterfly sum.
template <typename T>
__device__ __forceinline__ float row_inv_rms(const T* __restrict__ hr, int d, float eps, int lane) {
    constexpr int kRowBatch = 2;    // (a slice's loads are in flight meanwhile)
    float ss = 0.f;
    for (int i0 = lane * 8; i0 < d; i0 += 256 * kRowBatch) {
        Vec8<T> r[kRowBatch];
#pragma unroll
        for (int b = 0; b < kRowBatch; ++b)
            if (i0 + b * 256 < d) r[b].load(hr + i0 + b * 256);
#pragma unroll
        for (int b = 0; b < kRowBatch; ++b)
            if (i0 + b * 256 < d) {
                float v[8];
                r[b].get(v);
#pragma unroll
                for (int c = 0; c < 8; ++c) ss = fmaf(v[c], v[c], ss);
            }
    }
    ss = warp_sum(ss);
    return 1.0f / sqrtf(ss / (float)d + eps);
}

// Dispatch of n <= 32 * kWarpDispatchChunks pairs by one warp, pair r in
// lane r % 32 of chunk r / 32: the same counts, offsets, kept counts, stable
// permutation, inverse and tile list as dispatch_block (whose passes,
// barriers and per-warp tables cost microseconds of latency for a few
// hundred pairs).  Chunks are walked in order twice: once counting, once
// placing each pair after the earlier pairs of its expert (earlier chunks
// through `run`, earlier lanes of its chunk by a warp match).  `ecnt`, `run`
// and `eoff` are [E], [E] and [E + 1] ints of shared memory; perm goes to
// `perm_s` (shared).
constexpr int kWarpDispatchChunks = 8;

__device__ __forceinline__ void dispatch_warp(const int32_t* __restrict__ sidx, int n, int E,
                                              int32_t* __restrict__ counts,
                                              int32_t* __restrict__ offsets,
                                              int32_t* __restrict__ perm_s,
                                              int32_t* __restrict__ inv, int bm,
                                              int32_t* __restrict__ tile_expert,
                                              int32_t* __restrict__ tile_row,
                                              int32_t* __restrict__ tile_info,
                                              int32_t* __restrict__ num_tiles,
                                              int* __restrict__ status, int cap,
                                              int32_t* __restrict__ kept, int32_t* ecnt,
                                              int32_t* run, int32_t* eoff, int lane) {
    for (int e = lane; e < E; e += 32) ecnt[e] = 0, run[e] = 0;
    __syncwarp();
    const unsigned lt = (1u << lane) - 1u;
    // pass 1: counts
    for (int r0 = 0; r0 < n; r0 += 32) {
        const int r = r0 + lane;
        int e = r < n ? sidx[r] : -1;
        if (r < n && (e < 0 || e >= E)) {
            atomicExch(status, DEV_BAD_INDEX);
            e = -1;
        }
        const unsigned m = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && __popc(m & lt) == 0) ecnt[e] += __popc(m);
        __syncwarp();
    }
    // exclusive scans of the counts and of the tile counts over the experts
    // in expert order: lane l sums experts [l*per, (l+1)*per), a warp scan
    // gives each lane its base
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int32_t c_sum = 0, t_sum = 0;
    for (int i = 0; i < per; ++i) {
        const int x = e0 + i;
        if (x < E) {
            c_sum += ecnt[x];
            t_sum += (min(ecnt[x], cap) + bm - 1) / bm;
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
        const int x = e0 + i;
        if (x < E) {
            const int c = ecnt[x];
            eoff[x] = acc;
            counts[x] = c;
            kept[x] = min(c, cap);
            offsets[x] = acc;
            write_tiles(x, min(c, cap), acc, tacc, bm, tile_expert, tile_row, tile_info);
            acc += c;
            tacc += (min(c, cap) + bm - 1) / bm;
        }
    }
    if (lane == 31) {
        offsets[E] = c_inc;
        *num_tiles = t_inc;
    }
    __syncwarp();
    // pass 2: positions, chunk by chunk in pair order
    for (int r0 = 0; r0 < n; r0 += 32) {
        const int r = r0 + lane;
        int e = r < n ? sidx[r] : -1;
        if (e >= E) e = -1;
        const unsigned m = __match_any_sync(0xffffffffu, e);
        const int before = __popc(m & lt);                  // earlier lanes, same expert
        int rank = 0;
        if (e >= 0) rank = run[e] + before;                 // within the expert's segment
        __syncwarp();
        if (e >= 0) {
            const int p = eoff[e] + rank;
            perm_s[p] = r;
            inv[r] = rank < cap ? p : -1;
            if (before == 0) run[e] += __popc(m);
        } else if (r < n) {
            inv[r] = -1;      // an expert id out of range (reported above): adds nothing
        }
        __syncwarp();
    }
}

template <typename T>
__global__ void __launch_bounds__(kRouteThreads)
route_decode_kernel(const T* __restrict__ x, const T* __restrict__ wr,
                    const float* __restrict__ bias, int ntok, int d, int E, int k, int nq,
                    float* __restrict__ part, unsigned int* __restrict__ ticket,
                    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ perm, int32_t* __restrict__ inv, int bm,
                    int32_t* __restrict__ tile_expert, int32_t* __restrict__ tile_row,
                    int32_t* __restrict__ tile_info, int32_t* __restrict__ num_tiles,
                    int* __restrict__ status, int cap, int32_t* __restrict__ kept,
                    uint4* __restrict__ xp, const T* __restrict__ gamma, float eps,
                    T* __restrict__ u, int xp_f16) {
    pdl_enter();
    constexpr int kRowBatch = row_batch<T>();
    extern __shared__ int32_t sh[];
    __shared__ int last_cta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- 1. one partial logit per warp
    const int unit = blockIdx.x * kDispatchWarps + warp;
    const int seg = d / nq;
    if (unit < ntok * E * nq) {
        const int p = unit / nq, q = unit - p * nq;
        const int t = p / E, e = p - t * E;
        const T* xr = x + (size_t)t * d;
        const T* w = wr + (size_t)e * d + q * seg;
        float s = 0.f;
        if (gamma) {
            T* ur = (e == 0) ? u + (size_t)t * d + q * seg : nullptr;
            const T* hr = xr + q * seg;
            const T* gr = gamma + q * seg;
            Vec8<T> hv[kRowBatch], wv[kRowBatch];
            auto load_batch = [&](int i0) {
#pragma unroll
                for (int b = 0; b < kRowBatch; ++b)
                    if (i0 + b * 256 < seg) {
                        hv[b].load(hr + i0 + b * 256);
                        wv[b].load(w + i0 + b * 256);
                    }
            };
            // the slice's first row and weight loads go out before the row's
            // RMS pass (gamma, shared by every token, is read after it)
            load_batch(lane * 8);
            const float inv_rms = row_inv_rms(xr, d, eps, lane);
            for (int i0 = lane * 8; i0 < seg; i0 += 256 * kRowBatch) {
                if (i0 != lane * 8) load_batch(i0);
#pragma unroll
                for (int b = 0; b < kRowBatch; ++b)
                    if (i0 + b * 256 < seg) {
                        float hf[8], wf[8], gf[8];
                        hv[b].get(hf);
                        wv[b].get(wf);
                        load8(gr + i0 + b * 256, gf);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const T uv = from_f32<T>(hf[c] * inv_rms * gf[c]);
                            if (ur) ur[i0 + b * 256 + c] = uv;
                            s = fmaf(to_f32(uv), wf[c], s);
                        }
                    }
            }
        } else {
            xr += q * seg;
            for (int i0 = lane * 8; i0 < seg; i0 += 256 * kRowBatch) {
                Vec8<T> xv[kRowBatch], wv[kRowBatch];
#pragma unroll
                for (int b = 0; b < kRowBatch; ++b)
                    if (i0 + b * 256 < seg) {
                        xv[b].load(xr + i0 + b * 256);
                        wv[b].load(w + i0 + b * 256);
                    }
#pragma unroll
                for (int b = 0; b < kRowBatch; ++b)
                    if (i0 + b * 256 < seg) {
                        float xf[8], wf[8];
                        xv[b].get(xf);
                        wv[b].get(wf);
#pragma unroll
                        for (int c = 0; c < 8; ++c) s = fmaf(xf[c], wf[c], s);
                    }
            }
        }
        s = warp_sum(s);
        if (lane == 0) part[unit] = s;
        // the threads that wrote make their writes visible before the ticket
        if (lane == 0 || (gamma && e == 0)) __threadfence();
    }

    // ---- 2. ticket: the last CTA to arrive does the rest
    __syncthreads();
    if (threadIdx.x == 0) last_cta = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last_cta) return;
    __threadfence();
    if (threadIdx.x == 0) *ticket = 0u;     // rearmed for the next launch

    // Shared memory: the logits, then the routing ids and the permutation
    // (the dispatch and the gather read them here, not back through L2),
    // then the dispatch's own scratch.
    const int npairs = ntok * k;
    float* logit = reinterpret_cast<float*>(sh);                  // [ntok][E]
    int32_t* sidx = sh + ((ntok * E + 63) & ~63);                 // [npairs]
    int32_t* sperm = sidx + ((npairs + 63) & ~63);                // [npairs]
    int32_t* dsh = sperm + ((npairs + 63) & ~63);
    for (int p = threadIdx.x; p < ntok * E; p += blockDim.x) {
        float s = 0.f;
        for (int q = 0; q < nq; ++q) s += __ldcg(part + (size_t)p * nq + q);
        logit[p] = bias ? s + bias[p % E] : s;
    }
    __syncthreads();
    for (int t = warp; t < ntok; t += kDispatchWarps)
        warp_topk_softmax(logit + t * E, E, k, lane, sidx + t * k, topk_w + (size_t)t * k);
    __syncthreads();
    for (int i = threadIdx.x; i < npairs; i += blockDim.x) topk_idx[i] = sidx[i];
    if (npairs <= 32 * kWarpDispatchChunks) {
        if (warp == 0)
            dispatch_warp(sidx, npairs, E, counts, offsets, sperm, inv, bm, tile_expert, tile_row,
                          tile_info, num_tiles, status, cap, kept, dsh, dsh + E, dsh + 2 * E,
                          lane);
    } else {
        dispatch_block(sidx, npairs, E, counts, offsets, sperm, inv, bm, tile_expert, tile_row,
                       tile_info, num_tiles, status, cap, kept, dsh);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < npairs; i += blockDim.x) perm[i] = sperm[i];
    if (xp) {
        const int vecs = d * (int)sizeof(T) / 16;
        const uint4* xs = reinterpret_cast<const uint4*>(gamma ? u : x);
        for (int i = threadIdx.x; i < npairs * vecs; i += blockDim.x) {
            const int p = i / vecs, v = i - p * vecs;
            const uint4 val = __ldcg(xs + (size_t)(sperm[p] / k) * vecs + v);
            xp[(size_t)p * vecs + v] = xp_f16 ? bf16x8_to_f16x8(val) : val;
        }
    }
}

// d slices per logit: slices of at most 1024 elements (one batch of loads
// per lane), then more while the grid has fewer than 512 warps, each slice a
// multiple of 8 elements.
int slices_for(int ntok, int E, int d) {
    int nq = 1;
    auto ok = [&](int n) { return n <= kMaxSlices && d % n == 0 && (d / n) % 8 == 0; };
    while (d / nq > 1024 && ok(2 * nq)) nq *= 2;
    while (ntok * E * nq < 512 && d / (2 * nq) >= 256 && ok(2 * nq)) nq *= 2;
    return nq;
}

}  // namespace

bool route_decode_fits(int ntok, int d, int E, int k) {
    // bounded logit work (the router's d x E weights are read by every token
    // from L2), the logits of the batch in one CTA's shared memory, and the
    // pairs in one CTA's dispatch
    return ntok <= 256 && (int64_t)ntok * E * d <= (int64_t)1 << 24 && ntok * E <= 8192 &&
           ntok * k <= 2048;
}

size_t route_decode_part_floats(int max_tok, int E) {
    return (size_t)std::min(max_tok, 256) * E * kMaxSlices;
}

cudaError_t launch_route_decode(DType dt, const void* x, const void* wr, const float* bias,
                                int ntok, int d, int E, int k, float* part, unsigned int* ticket,
                                int32_t* topk_idx, float* topk_w, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* inv, int bm,
                                int32_t* tile_expert, int32_t* tile_row, int32_t* tile_info,
                                int32_t* num_tiles, int* status, int cap, int32_t* kept, void* xp,
                                const void* gamma, float eps, void* u, cudaStream_t s,
                                bool xp_f16) {
    if (ntok <= 0) return cudaSuccess;
    const int nq = slices_for(ntok, E, d);
    const int units = ntok * E * nq;
    const int grid = (units + kDispatchWarps - 1) / kDispatchWarps;
    const size_t smem = (size_t)((ntok * E + 63) & ~63) * 4 + (size_t)2 * ((ntok * k + 63) & ~63) * 4 +
                        dispatch_smem_bytes(E);
    cudaError_t e;
    if (dt == DType::BF16) {
        auto kern = route_decode_kernel<__nv_bfloat16>;
        smem_attr((const void*)kern, (int)smem);
        e = launch_pdl(kern, grid, kRouteThreads, smem, s, (const __nv_bfloat16*)x,
                       (const __nv_bfloat16*)wr, bias, ntok, d, E, k, nq, part, ticket, topk_idx,
                       topk_w, counts, offsets, perm, inv, bm, tile_expert, tile_row, tile_info,
                       num_tiles, status, cap, kept, (uint4*)xp, (const __nv_bfloat16*)gamma, eps,
                       (__nv_bfloat16*)u, xp_f16 ? 1 : 0);
    } else {
        auto kern = route_decode_kernel<float>;
        smem_attr((const void*)kern, (int)smem);
        e = launch_pdl(kern, grid, kRouteThreads, smem, s, (const float*)x, (const float*)wr, bias,
                       ntok, d, E, k, nq, part, ticket, topk_idx, topk_w, counts, offsets, perm,
                       inv, bm, tile_expert, tile_row, tile_info, num_tiles, status, cap, kept,
                       (uint4*)xp, (const float*)gamma, eps, (float*)u, 0);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace colibri
