// Gather, combine, RMSNorm and the init-time weight repack.
#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "kernels.h"

namespace colibri {

namespace {

// Xp[p, :] = x[perm[p] / k, :] — the tokens of every expert as consecutive
// rows (the A operand of the grouped GEMM), in 16-byte vectors; with
// kToF16, bf16 rows are converted to f16 (the A type of the
// int8-weight GEMMs).
// A warp copies whole rows, walking p = warp, warp + (warps in the grid), ...
// with the next row's source index loaded ahead and eight 16-byte loads per
// lane in flight, so that the copy runs at memory bandwidth instead of one
// row's latency chain per CTA.
constexpr int kGatherThreads = 256;
constexpr int kGatherCtasPerSm = 8;
constexpr size_t kGatherStreamBytes = (size_t)64 << 20;

// kStream: rows stored with the streaming hint (st.global.cs), for an Xp
// too large for L2: written normally it evicts the token rows x, which every
// token's k pairs read again at k different times of the gather.
template <bool kToF16, bool kStream>
__global__ void __launch_bounds__(kGatherThreads)
gather_rows(const uint4* __restrict__ x, const int32_t* __restrict__ perm, int k, int row_vecs,
            int npairs, int src_pairs, uint4* __restrict__ xp) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nw = (int)((gridDim.x * blockDim.x) >> 5);
    // pair q = t*k + j of x's src_pairs; any other value gathers a zero row
    auto row_of = [&](int q) { return (unsigned)q < (unsigned)src_pairs ? q / k : -1; };
    int p = gw;
    int t_next = p < npairs ? row_of(perm[p]) : 0;
    for (; p < npairs; p += nw) {
        const int t = t_next;
        if (p + nw < npairs) t_next = row_of(perm[p + nw]);
        uint4* dst = xp + (size_t)p * row_vecs;
        if (t < 0) {
            for (int i = lane; i < row_vecs; i += 32) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        const uint4* src = x + (size_t)t * row_vecs;
#pragma unroll 8
        for (int i = lane; i < row_vecs; i += 32) {
            const uint4 v = __ldg(src + i);
            const uint4 w = kToF16 ? bf16x8_to_f16x8(v) : v;
            if (kStream) __stcs(dst + i, w);
            else dst[i] = w;
        }
    }
}

// Combine: y[t, c] = sum_j w[t, j] * Y[inv[t*k + j], c], j in order, float32;
// with `resid`, y[t, c] = resid[t, c] + that sum (one rounding at the end).
// zskr.cn section 3.3 stage 5 (aggregation weighted by the expert scores).
// When the down projection was split over K, Y holds `nsplit` partial slices
// `split_stride` floats apart; they are added first, in slice order.  A pair
// with inv < 0 was dropped by its expert's capacity and adds nothing.
// Four consecutive outputs in one store (8 bytes of bf16, 16 of float).
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// Each thread owns kCombineVec float4 column groups, one block stride apart
// (coalesced per group), and issues every group's loads of a row before it
// adds them, so that enough bytes are in flight.
constexpr int kCombineVec = 4;
constexpr int kCombineThreads = 128;
constexpr int kCombineSlices = 4;   // split-K slices loaded together

// Four consecutive Y values as float4: float32 rows, or bf16 rows (8 bytes).
__device__ __forceinline__ float4 load_y4(const float* row, int g) {
    return reinterpret_cast<const float4*>(row)[g];
}
__device__ __forceinline__ float4 load_y4(const __nv_bfloat16* row, int g) {
    const uint2 u = reinterpret_cast<const uint2*>(row)[g];
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// kSplit: Y holds more than one K slice (decode-sized batches, float32);
// without it the kernel keeps no slice buffers (half the registers, twice
// the resident warps for the bandwidth-bound prefill combine).  TY: the
// type Y was stored in (bf16 for prefill on the tensor cores).
template <typename T, bool kSplit, typename TY>
__global__ void combine_kernel(const TY* __restrict__ Y, const float* __restrict__ topk_w,
                               const int32_t* __restrict__ inv, int T_, int k, int d, int nsplit,
                               size_t split_stride,
                               const T* resid, T* y) {  // resid may alias y (in-place residual)
    pdl_enter();
    // tokens on grid.y, strided: gridDim.y is capped at 65535, T is not
    for (int t = blockIdx.y; t < T_; t += gridDim.y) {
    const int d4 = d / 4;
    const int g0 = blockIdx.x * kCombineThreads * kCombineVec + threadIdx.x;   // float4 index
    float4 acc[kCombineVec];
#pragma unroll
    for (int u = 0; u < kCombineVec; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int pos = inv[(size_t)t * k + j];
        if (pos < 0) continue;                      // dropped by the expert's capacity
        const float w = topk_w[(size_t)t * k + j];
        const TY* yrow = Y + (size_t)pos * d;
        float4 v[kCombineVec];
#pragma unroll
        for (int u = 0; u < kCombineVec; ++u) {
            const int g = g0 + u * kCombineThreads;
            v[u] = g < d4 ? load_y4(yrow, g) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // split-K slices, added in slice order; the loads of four slices are
        // issued before any is added
        if constexpr (kSplit) {
        static_assert(!kSplit || sizeof(TY) == 4, "K slices are float32");
        const float4* row = reinterpret_cast<const float4*>(yrow);
        for (int sp0 = 1; sp0 < nsplit; sp0 += kCombineSlices) {
            float4 p[kCombineSlices][kCombineVec];
#pragma unroll
            for (int i = 0; i < kCombineSlices; ++i) {
                const float4* prow = row + (size_t)(sp0 + i) * (split_stride / 4);
#pragma unroll
                for (int u = 0; u < kCombineVec; ++u) {
                    const int g = g0 + u * kCombineThreads;
                    p[i][u] = (sp0 + i < nsplit && g < d4) ? prow[g] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int i = 0; i < kCombineSlices; ++i) {
                if (sp0 + i >= nsplit) break;
#pragma unroll
                for (int u = 0; u < kCombineVec; ++u) {
                    v[u].x += p[i][u].x;
                    v[u].y += p[i][u].y;
                    v[u].z += p[i][u].z;
                    v[u].w += p[i][u].w;
                }
            }
        }
        }
#pragma unroll
        for (int u = 0; u < kCombineVec; ++u) {
            acc[u].x = fmaf(w, v[u].x, acc[u].x);
            acc[u].y = fmaf(w, v[u].y, acc[u].y);
            acc[u].z = fmaf(w, v[u].z, acc[u].z);
            acc[u].w = fmaf(w, v[u].w, acc[u].w);
        }
    }
#pragma unroll
    for (int u = 0; u < kCombineVec; ++u) {
        const int g = g0 + u * kCombineThreads;
        if (g >= d4) continue;
        const size_t o = (size_t)t * d + (size_t)g * 4;
        if (resid) {
            acc[u].x += to_f32(resid[o]);
            acc[u].y += to_f32(resid[o + 1]);
            acc[u].z += to_f32(resid[o + 2]);
            acc[u].w += to_f32(resid[o + 3]);
        }
        store4(y + o, acc[u]);
    }
    }
}

// RMSNorm: u = h / sqrt(mean(h^2) + eps) * gamma, float32 arithmetic, one
// warp per token (rmsnorm_row_warp), 8 tokens per CTA.
template <typename T>
__global__ void rmsnorm_kernel(const T* __restrict__ h, const T* __restrict__ gamma, int T_,
                               int d, float eps, T* __restrict__ u) {
    pdl_enter();
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T_) return;
    rmsnorm_row_warp(h + (size_t)t * d, gamma, d, eps, u + (size_t)t * d, threadIdx.x & 31);
}

// Batched transpose with a row remap, for the init-time weight repack:
// out[b][map(c)][r] = in[b][r][c] for an [R, C] matrix per batch entry b,
// map(c) = (c / blk) * period + which * blk + c % blk; with `tiled`, the
// output rows of R codes are stored tile-major (code_index).
template <typename E>
__global__ void transpose_remap(const E* __restrict__ in, E* __restrict__ out, int R, int C,
                                size_t in_batch, size_t out_batch, int blk, int period,
                                int which, int tiled) {
    __shared__ E tile[32][33];
    const int b = blockIdx.z;
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    const E* src = in + b * in_batch;
    E* dst = out + b * out_batch;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        if (r < R && c < C) tile[i][threadIdx.x] = src[(size_t)r * C + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (r < R && c < C) {
            const size_t orow = (size_t)(c / blk) * period + (size_t)which * blk + c % blk;
            dst[tiled ? code_index(orow, r, R) : orow * R + r] = tile[threadIdx.x][i];
        }
    }
}

}  // namespace

cudaError_t launch_gather(int elem_bytes, const void* x, const int32_t* perm, int k, int d,
                          int npairs, int src_pairs, void* xp, cudaStream_t s, bool to_f16) {
    if (npairs <= 0) return cudaSuccess;
    const int row_vecs = d * elem_bytes / 16;
    static int sms = 0;
    if (sms <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            sms = 1;
    }
    const int warps_per_cta = kGatherThreads / 32;
    const int grid = std::max(1, std::min((npairs + warps_per_cta - 1) / warps_per_cta,
                                          sms * kGatherCtasPerSm));
    // Xp above half of L2 streams past it (kStream); a smaller one stays for
    // the GEMM that reads it next
    const bool stream = (size_t)npairs * row_vecs * 16 > kGatherStreamBytes;
    auto kern = to_f16 ? (stream ? gather_rows<true, true> : gather_rows<true, false>)
                       : (stream ? gather_rows<false, true> : gather_rows<false, false>);
    const cudaError_t e = launch_pdl(kern, grid, kGatherThreads, 0, s, (const uint4*)x, perm, k,
                                     row_vecs, npairs, src_pairs, (uint4*)xp);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t smem_attr(const void* kernel, int bytes) {
    // keyed by (device, kernel): the attribute belongs to the kernel's
    // instance on the current device
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> done;
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t key = (reinterpret_cast<uint64_t>(kernel) << 8) ^ (uint64_t)dev;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[key] = bytes;
    return e;
}

cudaError_t launch_combine(DType dt, const float* Y, bool y_bf16, const float* topk_w,
                           const int32_t* inv, int T, int k, int d, int nsplit, size_t split_stride,
                           const void* resid, void* y, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    if (y_bf16 && (nsplit > 1 || dt != DType::BF16)) return cudaErrorInvalidValue;
    const int per_block = kCombineThreads * kCombineVec;   // float4 groups per block
    constexpr int kMaxGridY = 65535;
    const dim3 block(kCombineThreads),
        grid((d / 4 + per_block - 1) / per_block, std::min(T, kMaxGridY));
    cudaError_t e;
    const bool split = nsplit > 1;
    if (dt == DType::BF16) {
        const auto* r = (const __nv_bfloat16*)resid;
        auto* o = (__nv_bfloat16*)y;
        if (y_bf16)
            e = launch_pdl(combine_kernel<__nv_bfloat16, false, __nv_bfloat16>, grid, block, 0, s,
                           (const __nv_bfloat16*)Y, topk_w, inv, T, k, d, nsplit, split_stride, r, o);
        else if (split)
            e = launch_pdl(combine_kernel<__nv_bfloat16, true, float>, grid, block, 0, s, Y, topk_w,
                           inv, T, k, d, nsplit, split_stride, r, o);
        else
            e = launch_pdl(combine_kernel<__nv_bfloat16, false, float>, grid, block, 0, s, Y, topk_w,
                           inv, T, k, d, nsplit, split_stride, r, o);
    } else {
        const auto* r = (const float*)resid;
        auto* o = (float*)y;
        e = split ? launch_pdl(combine_kernel<float, true, float>, grid, block, 0, s, Y, topk_w, inv,
                               T, k, d, nsplit, split_stride, r, o)
                  : launch_pdl(combine_kernel<float, false, float>, grid, block, 0, s, Y, topk_w, inv,
                               T, k, d, nsplit, split_stride, r, o);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

namespace {
__global__ void invert_perm_kernel(const int32_t* __restrict__ perm, int n, int32_t* __restrict__ inv) {
    pdl_enter();
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p < n) {
        const int q = perm[p];
        if (q >= 0 && q < n) inv[q] = p;            // a value out of range is skipped
    }
}
}  // namespace

cudaError_t launch_invert_perm(const int32_t* perm, int n, int32_t* inv, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    // -1 first: a position that no perm value names reads as a dropped pair
    cudaError_t e = cudaMemsetAsync(inv, 0xff, (size_t)n * sizeof(int32_t), s);
    if (e == cudaSuccess) e = launch_pdl(invert_perm_kernel, (n + 255) / 256, 256, 0, s, perm, n, inv);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_rmsnorm(DType dt, const void* h, const void* gamma, int T, int d, float eps,
                           void* u, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int grid = (T + 7) / 8;
    cudaError_t e;
    if (dt == DType::BF16)
        e = launch_pdl(rmsnorm_kernel<__nv_bfloat16>, grid, 256, 0, s, (const __nv_bfloat16*)h,
                       (const __nv_bfloat16*)gamma, T, d, eps, (__nv_bfloat16*)u);
    else
        e = launch_pdl(rmsnorm_kernel<float>, grid, 256, 0, s, (const float*)h, (const float*)gamma,
                       T, d, eps, (float*)u);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_transpose_remap(int elem_bytes, const void* in, void* out, int batch, int R,
                                   int C, size_t in_batch, size_t out_batch, int blk, int period,
                                   int which, cudaStream_t s, bool tiled) {
    const dim3 block(32, 8), grid((C + 31) / 32, (R + 31) / 32, batch);
    const int t = tiled ? 1 : 0;
    if (elem_bytes == 1)
        transpose_remap<uint8_t><<<grid, block, 0, s>>>((const uint8_t*)in, (uint8_t*)out, R, C,
                                                        in_batch, out_batch, blk, period, which, t);
    else if (elem_bytes == 2)
        transpose_remap<uint16_t><<<grid, block, 0, s>>>((const uint16_t*)in, (uint16_t*)out, R,
                                                         C, in_batch, out_batch, blk, period,
                                                         which, t);
    else
        transpose_remap<uint32_t><<<grid, block, 0, s>>>((const uint32_t*)in, (uint32_t*)out, R,
                                                         C, in_batch, out_batch, blk, period,
                                                         which, t);
    return cudaGetLastError();
}

}  // namespace colibri
