// Routing of a small batch in one CTA: router logits, top-k, softmax over
// the k, dispatch and (for the grouped executor) the gather of the token rows
// into expert order, in a single launch.
//
// zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析" section 3.3 stages 2-3.
// For decode-sized batches these steps are a few microseconds of work each
// but a launch and a round trip through global memory apiece; one CTA of 32
// warps does them back to back with block barriers in between:
//   1. logits: the T x E dot products of token rows and packed router rows,
//      each cut into d slices so that all 32 warps work, into shared memory
//   2. top-k + softmax: warp w routes tokens w, w + 32, ...
//   3. dispatch_block: the same deterministic counting sort as the dispatch kernel
//   4. gather: Xp[p] = x[perm[p] / k] with 16-byte vectors (converted to
//      f16 for the int8-weight GEMMs).
// For a pre-norm layer it first normalises the token rows (RMSNorm * gamma)
// into u and routes u.
#include "common.cuh"
#include "kernels.h"
#include "routing.cuh"

namespace colibri {

namespace {

template <typename T>
__global__ void __launch_bounds__(kDispatchWarps * 32)
route_small_kernel(const T* __restrict__ x, const T* __restrict__ wr,
                   const float* __restrict__ bias, int ntok, int d, int E, int k,
                   int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                   int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                   int32_t* __restrict__ perm, int32_t* __restrict__ inv, int bm,
                   int32_t* __restrict__ tile_expert, int32_t* __restrict__ tile_row,
                   int32_t* __restrict__ tile_info, int32_t* __restrict__ num_tiles,
                   int* __restrict__ status, int cap, int32_t* __restrict__ kept,
                   uint4* __restrict__ xp, int nq, const T* __restrict__ gamma, float eps,
                   T* __restrict__ u, int xp_f16) {
    pdl_enter();
    extern __shared__ int32_t sh[];
    float* logit = reinterpret_cast<float*>(sh);                 // [ntok][E]
    float* part = logit + ((ntok * E + 63) & ~63);               // [ntok * E][nq]
    int32_t* dsh = reinterpret_cast<int32_t*>(part + ((ntok * E * nq + 63) & ~63));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // 0. (pre-norm layer) u = RMSNorm(x) * gamma; the rest of the kernel
    // routes and gathers u, read back through L2.  With fewer tokens than
    // warps each row is cut into wpt slices of whole 256-element steps (a
    // warp each): the slices' sums of squares go through shared memory and
    // are added in slice order.  Otherwise one warp per token.
    const T* src = x;
    if (gamma) {
        int wpt = 1;
        while (ntok * wpt * 2 <= kDispatchWarps && d % (256 * wpt * 2) == 0) wpt *= 2;
        if (wpt == 1) {
            for (int t = warp; t < ntok; t += kDispatchWarps)
                rmsnorm_row_warp(x + (size_t)t * d, gamma, d, eps, u + (size_t)t * d, lane);
        } else {
            float* ssp = part;                    // [ntok * wpt] <= kDispatchWarps
            const int seg = d / wpt;
            const int unit = ntok * wpt;
            if (warp < unit) {
                const int t = warp / wpt, sl = warp - t * wpt;
                const T* hr = x + (size_t)t * d + sl * seg;
                float ss = 0.f;
#pragma unroll 4
                for (int i = lane * 8; i < seg; i += 256) {
                    float v[8];
                    load8(hr + i, v);
#pragma unroll
                    for (int c = 0; c < 8; ++c) ss = fmaf(v[c], v[c], ss);
                }
                ss = warp_sum(ss);
                if (lane == 0) ssp[warp] = ss;
            }
            __syncthreads();
            if (warp < unit) {
                const int t = warp / wpt, sl = warp - t * wpt;
                float tot = 0.f;
                for (int i = 0; i < wpt; ++i) tot += ssp[t * wpt + i];
                const float inv_rms = 1.0f / sqrtf(tot / (float)d + eps);
                const T* hr = x + (size_t)t * d + sl * seg;
                T* ur = u + (size_t)t * d + sl * seg;
                const T* gr = gamma + sl * seg;
#pragma unroll 4
                for (int i = lane * 8; i < seg; i += 256) {
                    float v[8], g[8];
                    load8(hr + i, v);
                    load8(gr + i, g);
#pragma unroll
                    for (int c = 0; c < 8; ++c) ur[i + c] = from_f32<T>(v[c] * inv_rms * g[c]);
                }
            }
        }
        __syncthreads();
        src = u;
    }

    // Logit p over d slice q (the d range is cut into nq slices so that the
    // 32 warps stay busy when T x E is small); slices are added in order.
    const int seg = d / nq;
    for (int u = warp; u < ntok * E * nq; u += kDispatchWarps) {
        const int p = u / nq, q = u - p * nq;
        const int t = p / E, e = p - t * E;
        const T* xr = src + (size_t)t * d + q * seg;
        const T* w = wr + (size_t)e * d + q * seg;
        float s = 0.f;
#pragma unroll 4
        for (int i = lane * 8; i < seg; i += 256) {
            float xv[8], wv[8];
            load8_cg(xr + i, xv);
            load8(w + i, wv);
#pragma unroll
            for (int c = 0; c < 8; ++c) s = fmaf(xv[c], wv[c], s);
        }
        s = warp_sum(s);
        if (lane == 0) part[u] = s;
    }
    __syncthreads();
    for (int p = threadIdx.x; p < ntok * E; p += blockDim.x) {
        float s = 0.f;
        for (int q = 0; q < nq; ++q) s += part[p * nq + q];
        logit[p] = bias ? s + bias[p % E] : s;
    }
    __syncthreads();
    for (int t = warp; t < ntok; t += kDispatchWarps)
        warp_topk_softmax(logit + t * E, E, k, lane, topk_idx + (size_t)t * k,
                          topk_w + (size_t)t * k);
    __syncthreads();
    dispatch_block(topk_idx, ntok * k, E, counts, offsets, perm, inv, bm, tile_expert, tile_row,
                   tile_info, num_tiles, status, cap, kept, dsh);
    if (xp) {
        __syncthreads();
        const int vecs = d * (int)sizeof(T) / 16;
        const uint4* xs = reinterpret_cast<const uint4*>(src);
        for (int i = threadIdx.x; i < ntok * k * vecs; i += blockDim.x) {
            const int p = i / vecs, v = i - p * vecs;
            const uint4 val = __ldcg(xs + (size_t)(perm[p] / k) * vecs + v);
            xp[(size_t)p * vecs + v] = xp_f16 ? bf16x8_to_f16x8(val) : val;
        }
    }
}

}  // namespace

bool route_small_fits(int ntok, int d, int E, int k) {
    // a few microseconds of logits for one CTA: beyond that the router and
    // dispatch kernels, spread over the GPU, are faster
    return (int64_t)ntok * E * d <= (int64_t)1 << 18 && ntok * k <= 1024 && ntok * E <= 2048;
}

namespace {
// d slices per logit: enough (warp, logit, slice) units for 32 warps, each
// slice a multiple of 8 elements (d is a multiple of 64).
int slices_for(int ntok, int E, int d) {
    int nq = 1;
    while (nq < 8 && ntok * E * nq < kDispatchWarps && (d / (2 * nq)) % 8 == 0) nq *= 2;
    return nq;
}
}  // namespace

cudaError_t launch_route_small(DType dt, const void* x, const void* wr, const float* bias,
                               int ntok, int d, int E, int k, int32_t* topk_idx, float* topk_w,
                               int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                               int bm, int32_t* tile_expert, int32_t* tile_row,
                               int32_t* tile_info, int32_t* num_tiles, int* status, int cap,
                               int32_t* kept, void* xp, const void* gamma, float eps, void* u,
                               cudaStream_t s, bool xp_f16) {
    const int nq = slices_for(ntok, E, d);
    const size_t smem = (size_t)((ntok * E + 63) & ~63) * 4 +
                        (size_t)((ntok * E * nq + 63) & ~63) * 4 + dispatch_smem_bytes(E);
    const dim3 block(kDispatchWarps * 32);
    cudaError_t e;
    if (dt == DType::BF16) {
        auto kern = route_small_kernel<__nv_bfloat16>;
        smem_attr((const void*)kern, (int)smem);
        e = launch_pdl(kern, 1, block, smem, s, (const __nv_bfloat16*)x, (const __nv_bfloat16*)wr,
                       bias, ntok, d, E, k, topk_idx, topk_w, counts, offsets, perm, inv, bm,
                       tile_expert, tile_row, tile_info, num_tiles, status, cap, kept, (uint4*)xp,
                       nq, (const __nv_bfloat16*)gamma, eps, (__nv_bfloat16*)u, xp_f16 ? 1 : 0);
    } else {
        auto kern = route_small_kernel<float>;
        smem_attr((const void*)kern, (int)smem);
        e = launch_pdl(kern, 1, block, smem, s, (const float*)x, (const float*)wr, bias, ntok, d, E,
                       k, topk_idx, topk_w, counts, offsets, perm, inv, bm, tile_expert, tile_row,
                       tile_info, num_tiles, status, cap, kept, (uint4*)xp, nq, (const float*)gamma,
                       eps, (float*)u, 0);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace colibri
