// Weight-streaming expert SwiGLU FFN on CUDA cores (decode-sized batches and
// the float32 layer).
//
// zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析" section 3.3 stage 4
// (per expert: gate_proj, up_proj, SiLU, down_proj).  With few tokens per
// expert the FFN is a weight stream: every activated expert's weights are read
// from HBM exactly once, experts with no token are skipped entirely.
//
//   ffn_up_stream    one warp per hidden unit n: the gate row and the up row
//                    of W^T (K contiguous) are streamed in 16-byte vectors and
//                    dotted with up to kSlots token rows at a time;
//                    H[p, n] = silu(g) * u, rounded to the layer dtype.
//   ffn_down_stream  one warp per output feature c: the row c of W_down^T
//                    (contiguous over d_ff) dotted with the H rows of the
//                    expert's pairs; Y[p, c] in float32.
// Pairs p are in expert order (the dispatch permutation), so the tokens of
// one expert are consecutive rows of H and Y; an expert computes the first
// kept[e] rows of its segment (all of them unless a capacity drops some).
#include "common.cuh"
#include "kernels.h"

namespace colibri {

namespace {

constexpr int kWarps = 8;
constexpr int kSlots = 8;
// 16-byte weight chunks per lane issued before their first use: enough bytes
// in flight per warp to cover HBM latency without a shared-memory ring.
constexpr int kAhead = 4;      // x2 rows (gate, up)
constexpr int kAheadDown = 8;

// Row of the packed gate/up weight: [E][f/128][2][128][d], which = 0 gate, 1 up.
__device__ __forceinline__ size_t gu_row(int e, int n, int which, int f) {
    return ((size_t)(e * (f / 128) + n / 128) * 2 + which) * 128 + (n % 128);
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
ffn_up_stream(const T* __restrict__ x, const T* __restrict__ wgu,
              const int32_t* __restrict__ kept, const int32_t* __restrict__ offsets,
              const int32_t* __restrict__ perm, int k, int d, int f, int E, T* __restrict__ H) {
    pdl_enter();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * kWarps + warp;
    if (n >= f) return;
    for (int e = 0; e < E; ++e) {
        const int c = kept[e];
        if (c == 0) continue;
        const int off = offsets[e];
        const T* g_row = wgu + gu_row(e, n, 0, f) * d;
        const T* u_row = wgu + gu_row(e, n, 1, f) * d;
        for (int s0 = 0; s0 < c; s0 += kSlots) {
            const int ns = min(kSlots, c - s0);
            const T* xr[kSlots];
#pragma unroll
            for (int s = 0; s < kSlots; ++s)
                xr[s] = x + (size_t)(perm[off + s0 + (s < ns ? s : 0)] / k) * d;
            float ag[kSlots], au[kSlots];
#pragma unroll
            for (int s = 0; s < kSlots; ++s) ag[s] = au[s] = 0.f;
            for (int i0 = lane * 8; i0 < d; i0 += 256 * kAhead) {
                // issue every weight load of this stretch before the first use
                Raw8<T> wg[kAhead], wu[kAhead];
#pragma unroll
                for (int a = 0; a < kAhead; ++a) {
                    if (i0 + a * 256 < d) {
                        wg[a].load(g_row + i0 + a * 256);
                        wu[a].load(u_row + i0 + a * 256);
                    }
                }
#pragma unroll
                for (int a = 0; a < kAhead; ++a) {
                    const int i = i0 + a * 256;
                    if (i < d) {
#pragma unroll
                        for (int s = 0; s < kSlots; ++s) {
                            if (s < ns) {
                                float xv[8];
                                load8(xr[s] + i, xv);
                                ag[s] += wg[a].dot(xv);
                                au[s] += wu[a].dot(xv);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < kSlots; ++s) {
                if (s < ns) {
                    const float g = warp_sum(ag[s]);
                    const float u = warp_sum(au[s]);
                    if (lane == 0) H[(size_t)(off + s0 + s) * f + n] = from_f32<T>(silu(g) * u);
                }
            }
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
ffn_down_stream(const T* __restrict__ H, const T* __restrict__ wdT,
                const int32_t* __restrict__ kept, const int32_t* __restrict__ offsets, int d,
                int f, int E, float* __restrict__ Y) {
    pdl_enter();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = blockIdx.x * kWarps + warp;
    if (col >= d) return;
    for (int e = 0; e < E; ++e) {
        const int c = kept[e];
        if (c == 0) continue;
        const int off = offsets[e];
        const T* w_row = wdT + ((size_t)e * d + col) * f;
        for (int s0 = 0; s0 < c; s0 += kSlots) {
            const int ns = min(kSlots, c - s0);
            float acc[kSlots];
#pragma unroll
            for (int s = 0; s < kSlots; ++s) acc[s] = 0.f;
            for (int i0 = lane * 8; i0 < f; i0 += 256 * kAheadDown) {
                Raw8<T> w[kAheadDown];
#pragma unroll
                for (int a = 0; a < kAheadDown; ++a)
                    if (i0 + a * 256 < f) w[a].load(w_row + i0 + a * 256);
#pragma unroll
                for (int a = 0; a < kAheadDown; ++a) {
                    const int i = i0 + a * 256;
                    if (i < f) {
#pragma unroll
                        for (int s = 0; s < kSlots; ++s) {
                            if (s < ns) {
                                float hv[8];
                                load8(H + (size_t)(off + s0 + s) * f + i, hv);
                                acc[s] += w[a].dot(hv);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < kSlots; ++s) {
                if (s < ns) {
                    const float v = warp_sum(acc[s]);
                    if (lane == 0) Y[(size_t)(off + s0 + s) * d + col] = v;
                }
            }
        }
    }
}

// ------------------------------------------------------------ int8 weights
//
// Expert weights as int8 codes in 64x64 blocks, w = (q - zp) * scale
// (m.nxbn.cn section 3.1; pnsm.cn section 5.2).  A lane loads 16 consecutive
// codes of a row (one 16-byte vector, all in one block); a byte permute turns
// each code into the exact float 2^23 + 128 + q and one exact subtraction of
// 2^23 + 128 + zp leaves q - zp, so the conversion costs two instructions per
// weight; the block's scale multiplies the lane's 16-term partial sum once.
// Block scales and zero points are stored per 64-row block of the packed
// weight rows (gate/up [E][f/128][2][128] rows, down [E][d] rows), k-block
// fastest: [packed row / 64][K / 64].

constexpr int kAheadI8 = 4;   // 16-byte vectors per row in flight per lane

template <typename T>
__device__ __forceinline__ float dot16(const T* xr, const float (&t)[16]) {
    float a[8], b[8];
    load8(xr, a);
    load8(xr + 8, b);
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) s = fmaf(a[c], t[c], s);
#pragma unroll
    for (int c = 0; c < 8; ++c) s = fmaf(b[c], t[8 + c], s);
    return s;
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
ffn_up_stream_i8(const T* __restrict__ x, const int8_t* __restrict__ wq,
                 const float* __restrict__ sc, const int32_t* __restrict__ zpt,
                 const int32_t* __restrict__ kept, const int32_t* __restrict__ offsets,
                 const int32_t* __restrict__ perm, int k, int d, int f, int E, T* __restrict__ H) {
    pdl_enter();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * kWarps + warp;
    if (n >= f) return;
    const int nkb = d / 64;
    for (int e = 0; e < E; ++e) {
        const int c = kept[e];
        if (c == 0) continue;
        const int off = offsets[e];
        const size_t grow = gu_row(e, n, 0, f), urow = gu_row(e, n, 1, f);
        const size_t gb = (grow >> 6) * nkb;   // gate block row of scales
        const size_t ub = (urow >> 6) * nkb;
        for (int s0 = 0; s0 < c; s0 += kSlots) {
            const int ns = min(kSlots, c - s0);
            const T* xr[kSlots];
#pragma unroll
            for (int s = 0; s < kSlots; ++s)
                xr[s] = x + (size_t)(perm[off + s0 + (s < ns ? s : 0)] / k) * d;
            float ag[kSlots], au[kSlots];
#pragma unroll
            for (int s = 0; s < kSlots; ++s) ag[s] = au[s] = 0.f;
            for (int i0 = lane * 16; i0 < d; i0 += 512 * kAheadI8) {
                uint4 vg[kAheadI8], vu[kAheadI8];
#pragma unroll
                for (int a = 0; a < kAheadI8; ++a) {
                    if (i0 + a * 512 < d) {   // tile-major codes (code_index)
                        vg[a] = ld_stream16(wq + code_index(grow, i0 + a * 512, d));
                        vu[a] = ld_stream16(wq + code_index(urow, i0 + a * 512, d));
                    }
                }
#pragma unroll
                for (int a = 0; a < kAheadI8; ++a) {
                    const int i = i0 + a * 512;
                    if (i < d) {
                        const int kb = i >> 6;
                        const float sg = __ldg(sc + gb + kb), su = __ldg(sc + ub + kb);
                        float tg[16], tu[16];
                        dequant16(vg[a], code_offset(__ldg(zpt + gb + kb)), tg);
                        dequant16(vu[a], code_offset(__ldg(zpt + ub + kb)), tu);
#pragma unroll
                        for (int s = 0; s < kSlots; ++s) {
                            if (s < ns) {
                                ag[s] = fmaf(sg, dot16(xr[s] + i, tg), ag[s]);
                                au[s] = fmaf(su, dot16(xr[s] + i, tu), au[s]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < kSlots; ++s) {
                if (s < ns) {
                    const float g = warp_sum(ag[s]);
                    const float u = warp_sum(au[s]);
                    if (lane == 0) H[(size_t)(off + s0 + s) * f + n] = from_f32<T>(silu(g) * u);
                }
            }
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
ffn_down_stream_i8(const T* __restrict__ H, const int8_t* __restrict__ wq,
                   const float* __restrict__ sc, const int32_t* __restrict__ zpt,
                   const int32_t* __restrict__ kept, const int32_t* __restrict__ offsets, int d,
                   int f, int E, float* __restrict__ Y) {
    pdl_enter();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = blockIdx.x * kWarps + warp;
    if (col >= d) return;
    const int nkb = f / 64;
    for (int e = 0; e < E; ++e) {
        const int c = kept[e];
        if (c == 0) continue;
        const int off = offsets[e];
        const size_t wrow = (size_t)e * d + col;
        const size_t bb = (wrow >> 6) * nkb;
        for (int s0 = 0; s0 < c; s0 += kSlots) {
            const int ns = min(kSlots, c - s0);
            float acc[kSlots];
#pragma unroll
            for (int s = 0; s < kSlots; ++s) acc[s] = 0.f;
            for (int i0 = lane * 16; i0 < f; i0 += 512 * kAheadI8) {
                uint4 v[kAheadI8];
#pragma unroll
                for (int a = 0; a < kAheadI8; ++a)
                    if (i0 + a * 512 < f)   // tile-major codes (code_index)
                        v[a] = ld_stream16(wq + code_index(wrow, i0 + a * 512, f));
#pragma unroll
                for (int a = 0; a < kAheadI8; ++a) {
                    const int i = i0 + a * 512;
                    if (i < f) {
                        const int kb = i >> 6;
                        const float sw = __ldg(sc + bb + kb);
                        float t[16];
                        dequant16(v[a], code_offset(__ldg(zpt + bb + kb)), t);
#pragma unroll
                        for (int s = 0; s < kSlots; ++s)
                            if (s < ns)
                                acc[s] = fmaf(sw, dot16(H + (size_t)(off + s0 + s) * f + i, t), acc[s]);
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < kSlots; ++s) {
                if (s < ns) {
                    const float v = warp_sum(acc[s]);
                    if (lane == 0) Y[(size_t)(off + s0 + s) * d + col] = v;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_ffn_up_stream_i8(DType dt, const void* x, const int8_t* wq, const float* sc,
                                    const int32_t* zp, const int32_t* kept,
                                    const int32_t* offsets, const int32_t* perm, int k, int d,
                                    int f, int E, void* H, cudaStream_t s) {
    const dim3 block(kWarps * 32), grid((f + kWarps - 1) / kWarps);
    cudaError_t e;
    if (dt == DType::BF16)
        e = launch_pdl(ffn_up_stream_i8<__nv_bfloat16>, grid, block, 0, s, (const __nv_bfloat16*)x,
                       wq, sc, zp, kept, offsets, perm, k, d, f, E, (__nv_bfloat16*)H);
    else
        e = launch_pdl(ffn_up_stream_i8<float>, grid, block, 0, s, (const float*)x, wq, sc, zp,
                       kept, offsets, perm, k, d, f, E, (float*)H);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_ffn_down_stream_i8(DType dt, const void* H, const int8_t* wq, const float* sc,
                                      const int32_t* zp, const int32_t* kept,
                                      const int32_t* offsets, int d, int f, int E, float* Y,
                                      cudaStream_t s) {
    const dim3 block(kWarps * 32), grid((d + kWarps - 1) / kWarps);
    cudaError_t e;
    if (dt == DType::BF16)
        e = launch_pdl(ffn_down_stream_i8<__nv_bfloat16>, grid, block, 0, s,
                       (const __nv_bfloat16*)H, wq, sc, zp, kept, offsets, d, f, E, Y);
    else
        e = launch_pdl(ffn_down_stream_i8<float>, grid, block, 0, s, (const float*)H, wq, sc, zp,
                       kept, offsets, d, f, E, Y);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_ffn_up_stream(DType dt, const void* x, const void* wgu, const int32_t* kept,
                                 const int32_t* offsets, const int32_t* perm, int k, int d, int f,
                                 int E, void* H, cudaStream_t s) {
    const dim3 block(kWarps * 32), grid((f + kWarps - 1) / kWarps);
    cudaError_t e;
    if (dt == DType::BF16)
        e = launch_pdl(ffn_up_stream<__nv_bfloat16>, grid, block, 0, s, (const __nv_bfloat16*)x,
                       (const __nv_bfloat16*)wgu, kept, offsets, perm, k, d, f, E,
                       (__nv_bfloat16*)H);
    else
        e = launch_pdl(ffn_up_stream<float>, grid, block, 0, s, (const float*)x, (const float*)wgu,
                       kept, offsets, perm, k, d, f, E, (float*)H);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_ffn_down_stream(DType dt, const void* H, const void* wdT, const int32_t* kept,
                                   const int32_t* offsets, int d, int f, int E, float* Y,
                                   cudaStream_t s) {
    const dim3 block(kWarps * 32), grid((d + kWarps - 1) / kWarps);
    cudaError_t e;
    if (dt == DType::BF16)
        e = launch_pdl(ffn_down_stream<__nv_bfloat16>, grid, block, 0, s, (const __nv_bfloat16*)H,
                       (const __nv_bfloat16*)wdT, kept, offsets, d, f, E, Y);
    else
        e = launch_pdl(ffn_down_stream<float>, grid, block, 0, s, (const float*)H,
                       (const float*)wdT, kept, offsets, d, f, E, Y);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace colibri
