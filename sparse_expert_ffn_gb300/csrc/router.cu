// Router: logits x . W_r (+ offset), per-token top-k, softmax over the k.
//
// zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析" section 3.3 stage 2 (a
// routing kernel with one warp per sequence, warp-level partial top-k, outputs
// expert_indices [batch, top_k] and expert_scores [batch, top_k]); lmnt.cn
// section 2.2 (route_tokens: logits, top-k, softmax over the top-k logits).
//
// The token's row is widened to float in shared memory; every logit is a warp
// dot product over d against one packed router row (W_r repacked to [E, d],
// K contiguous).  Top-k runs as k rounds of a warp
// arg-max over a 64-bit key (ordered value, then ~expert so that the lower
// index wins a tie); NaN ranks below -inf.  The softmax is over the k
// selected logits, with the largest subtracted first.
#include "common.cuh"
#include "kernels.h"
#include "routing.cuh"

namespace colibri {

namespace {

constexpr int kRouterWarps = 8;
// Opt-in shared memory per CTA on sm_103 (227 KB).
constexpr size_t kRouterSmemMax = 227 * 1024;

// One CTA of kRouterWarps warps routes kRouterWarps / kWarpsPerToken tokens;
// the kWarpsPerToken warps of a token split its experts (e = sub, sub + W, ...).
// Large batches use one warp per token; small ones spread a token over all
// warps of the CTA so that the E dot products run in parallel.
template <typename T, int kWarpsPerToken>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_topk_simt(const T* __restrict__ x, const T* __restrict__ wr, const float* __restrict__ bias,
                 int ntok, int d, int E, int k, int32_t* __restrict__ topk_idx,
                 float* __restrict__ topk_w, int soft) {
    pdl_enter();
    extern __shared__ float smem[];
    constexpr int kTokens = kRouterWarps / kWarpsPerToken;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = warp / kWarpsPerToken, sub = warp % kWarpsPerToken;
    const int t = blockIdx.x * kTokens + slot;
    const bool live = t < ntok;
    float* xs = smem + slot * (d + 256);
    float* logit = xs + d;

    if (live) {
        const T* xr = x + (size_t)t * d;
        for (int i = sub * 32 + lane; i < d; i += 32 * kWarpsPerToken) xs[i] = to_f32(xr[i]);
    }
    __syncthreads();

    if (live) {
        for (int e = sub; e < E; e += kWarpsPerToken) {
            const T* w = wr + (size_t)e * d;
            float s = 0.f;
            for (int i = lane * 8; i < d; i += 256) {
                float wv[8];
                load8(w + i, wv);
                const float4 xa = *reinterpret_cast<const float4*>(xs + i);
                const float4 xb = *reinterpret_cast<const float4*>(xs + i + 4);
                s = fmaf(xa.x, wv[0], s);
                s = fmaf(xa.y, wv[1], s);
                s = fmaf(xa.z, wv[2], s);
                s = fmaf(xa.w, wv[3], s);
                s = fmaf(xb.x, wv[4], s);
                s = fmaf(xb.y, wv[5], s);
                s = fmaf(xb.z, wv[6], s);
                s = fmaf(xb.w, wv[7], s);
            }
            s = warp_sum(s);
            if (lane == 0) logit[e] = bias ? s + bias[e] : s;
        }
    }
    __syncthreads();
    if (!live || sub != 0) return;

    if (soft) {
        // soft routing (k = E): every expert, in expert order, gate = the
        // softmax over all E logits (largest subtracted first)
        float m = -INFINITY;
        for (int e = lane; e < E; e += 32) m = fmaxf(m, logit[e]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float s = 0.f;
        for (int e = lane; e < E; e += 32) s += expf(logit[e] - m);
        s = warp_sum(s);
        for (int e = lane; e < E; e += 32) {
            topk_idx[(size_t)t * E + e] = e;
            topk_w[(size_t)t * E + e] = expf(logit[e] - m) / s;
        }
        return;
    }
    warp_topk_softmax(logit, E, k, lane, topk_idx + (size_t)t * k, topk_w + (size_t)t * k);
}

template <typename T, int kWarpsPerToken>
cudaError_t launch_router_t(const void* x, const void* wr, const float* bias, int ntok, int d,
                            int E, int k, int32_t* idx, float* w, cudaStream_t s, int soft) {
    constexpr int kTokens = kRouterWarps / kWarpsPerToken;
    const dim3 grid((ntok + kTokens - 1) / kTokens), block(kRouterWarps * 32);
    const size_t smem = (size_t)kTokens * (d + 256) * sizeof(float);
    auto kern = router_topk_simt<T, kWarpsPerToken>;
    smem_attr((const void*)kern, (int)smem);
    const cudaError_t e =
        launch_pdl(kern, grid, block, smem, s, (const T*)x, (const T*)wr, bias, ntok, d, E, k, idx, w,
                   soft);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool router_simt_fits(int d) { return d > 0 && (size_t)(d + 256) * 4 <= kRouterSmemMax; }

cudaError_t launch_router_simt(DType dt, const void* x, const void* wr, const float* bias,
                               int ntok, int d, int E, int k, int32_t* idx, float* w,
                               cudaStream_t s, bool soft) {
    if (ntok <= 0) return cudaSuccess;
    if (!router_simt_fits(d)) return cudaErrorInvalidValue;
    // Few tokens: spread every token over a whole CTA; many: two warps per
    // token, four tokens per CTA (70 KB of shared memory at d = 4096), unless
    // four token rows do not fit in shared memory.
    const bool small = ntok <= 256 || kRouterSmemMax < (size_t)(kRouterWarps / 2) * (d + 256) * 4;
    const int sf = soft ? 1 : 0;
    if (dt == DType::BF16)
        return small ? launch_router_t<__nv_bfloat16, kRouterWarps>(x, wr, bias, ntok, d, E, k, idx, w, s, sf)
                     : launch_router_t<__nv_bfloat16, 2>(x, wr, bias, ntok, d, E, k, idx, w, s, sf);
    return small ? launch_router_t<float, kRouterWarps>(x, wr, bias, ntok, d, E, k, idx, w, s, sf)
                 : launch_router_t<float, 2>(x, wr, bias, ntok, d, E, k, idx, w, s, sf);
}

}  // namespace colibri
