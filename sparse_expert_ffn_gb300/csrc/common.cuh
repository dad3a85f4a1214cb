// Shared device helpers for the MoE layer kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace colibri {

// Element types the layer runs in.
enum class DType : int { F32 = 0, BF16 = 1 };

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Load 8 consecutive elements starting at p (16-byte aligned for bf16,
// 32-byte aligned for float) and widen them to float.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(b[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Streaming (read-once) variants for weights: bypass L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// 8 elements of a weight row as raw registers (bf16: one 16-byte vector,
// float: two).
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
    uint4 a;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) { a = ld_stream16(p); }
    __device__ __forceinline__ float dot(const float (&x)[8]) const {
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&a);
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(b[i]);
            s = fmaf(x[2 * i], f.x, s);
            s = fmaf(x[2 * i + 1], f.y, s);
        }
        return s;
    }
};
template <> struct Raw8<float> {
    uint4 a, b;
    __device__ __forceinline__ void load(const float* p) {
        a = ld_stream16(p);
        b = ld_stream16(p + 4);
    }
    __device__ __forceinline__ float dot(const float (&x)[8]) const {
        float s = 0.f;
        s = fmaf(x[0], __uint_as_float(a.x), s);
        s = fmaf(x[1], __uint_as_float(a.y), s);
        s = fmaf(x[2], __uint_as_float(a.z), s);
        s = fmaf(x[3], __uint_as_float(a.w), s);
        s = fmaf(x[4], __uint_as_float(b.x), s);
        s = fmaf(x[5], __uint_as_float(b.y), s);
        s = fmaf(x[6], __uint_as_float(b.z), s);
        s = fmaf(x[7], __uint_as_float(b.w), s);
        return s;
    }
};

__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// 8 bf16 -> 8 f16 (round to nearest; exact for |v| in f16's normal range).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4& v) {
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        __half2 h = __floats2half2_rn(f.x, f.y);
        o[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Coherent 8-element load (through L2): for rows this kernel wrote itself.
__device__ __forceinline__ void load8_cg(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 u = __ldcg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(b[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8_cg(const float* p, float (&v)[8]) {
    float4 a = __ldcg(reinterpret_cast<const float4*>(p));
    float4 b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// RMSNorm of one row by one warp (Zhang & Sennrich, 2019):
// u = h / sqrt(mean(h^2) + eps) * gamma in float32.  Lane l adds the squares
// of elements 8l + 256j .. 8l + 256j + 7 in order, then the butterfly sum;
// every kernel that normalises a row uses this routine, so the result does
// not depend on which one ran.  d is a multiple of 8.
template <typename T>
__device__ __forceinline__ void rmsnorm_row_warp(const T* __restrict__ hr, const T* __restrict__ gamma,
                                                 int d, float eps, T* __restrict__ ur, int lane) {
    // (loops unrolled by 4: four rows' worth of loads in flight per lane)
    float ss = 0.f;
#pragma unroll 4
    for (int i = lane * 8; i < d; i += 256) {
        float v[8];
        load8(hr + i, v);
#pragma unroll
        for (int c = 0; c < 8; ++c) ss = fmaf(v[c], v[c], ss);
    }
    ss = warp_sum(ss);
    const float inv_rms = 1.0f / sqrtf(ss / (float)d + eps);
#pragma unroll 4
    for (int i = lane * 8; i < d; i += 256) {
        float v[8], g[8];
        load8(hr + i, v);
        load8(gamma + i, g);
#pragma unroll
        for (int c = 0; c < 8; ++c) ur[i + c] = from_f32<T>(v[c] * inv_rms * g[c]);
    }
}

// Programmatic dependent launch.  Every kernel of the layer is launched with
// programmatic stream serialization, so it may be scheduled while the kernel
// before it on the stream is still running: it sets up what touches no global
// memory (shared memory, barriers, tensor memory), then pdl_wait() blocks
// until the previous kernel has completed and its writes are visible, and only
// then does it read or write global memory.  pdl_launch_dependents() is called
// after pdl_wait(), so at most one further kernel is scheduled early.  Both
// are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_enter() {
    pdl_wait();
    pdl_launch_dependents();
}

// Launch with programmatic stream serialization (see pdl_wait); the kernel
// must call pdl_wait() before its first global memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Int8 weight codes are stored tile-major: the packed weight rows of K codes
// each are cut into tiles of 128 rows x 64 codes, tile (row / 128, k / 64) is
// 8 KB contiguous, tiles of one row block consecutive in k.  Inside a tile,
// row r takes 64 bytes and its 16-byte chunk c sits at chunk c ^ ((r >> 1) & 3)
// (the 64-byte swizzle pattern), so that one bulk copy of a tile gives a
// shared-memory image in which the 8 rows a quarter warp reads at the same
// chunk fall in 8 different bank groups.
__host__ __device__ __forceinline__ size_t code_index(size_t row, int k, int K) {
    const size_t r = row & 127;
    return ((row >> 7) * (size_t)(K >> 6) + (size_t)(k >> 6)) * 8192 + r * 64 +
           (size_t)((((k & 63) >> 4) ^ (int)((r >> 1) & 3)) << 4) + (size_t)(k & 15);
}
// Byte offset of code chunk c (16 codes) of row r inside a tile.
__device__ __forceinline__ int code_chunk_offset(int r, int c) {
    return (r & 127) * 64 + ((c ^ ((r >> 1) & 3)) << 4);
}

// Int8 weight codes (64x64 blocks, w = (q - zp) * scale).  The byte permute
// places each code, sign bit flipped (q + 128 as an unsigned byte), in the low
// mantissa byte of 2^23, which is the exact float 2^23 + 128 + q; subtracting
// 2^23 + 128 + zp leaves q - zp exactly.  Two instructions per weight.
// q - zp for the 16 codes of v, as floats.
__device__ __forceinline__ void dequant16(const uint4& v, float off, float (&t)[16]) {
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u,
                           v.w ^ 0x80808080u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        t[4 * i + 0] = __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7540)) - off;
        t[4 * i + 1] = __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7541)) - off;
        t[4 * i + 2] = __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7542)) - off;
        t[4 * i + 3] = __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7543)) - off;
    }
}

// 2^23 + 128 + zp: subtracting it from the permuted code gives q - zp exactly.
__device__ __forceinline__ float code_offset(int32_t zp) { return 8388736.0f + (float)zp; }

// The same in half precision, two codes per instruction: a byte permute puts
// two codes (sign flipped) in the low bytes of two halves 1024.0 (0x6400),
// i.e. 1024 + 128 + q each; one half2 subtraction of 1152 + zp leaves q - zp
// exactly (|q - zp| <= 254), and one half2 multiply applies the scale.
// 16 codes -> 16 halves (lo = codes 0..7, hi = codes 8..15).
__device__ __forceinline__ void dequant16_h2(const uint4& v, __half2 off2, __half2 s2, uint4& lo,
                                             uint4& hi) {
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u,
                           v.w ^ 0x80808080u};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = __byte_perm(w[i], 0x64646464u, 0x5140);   // codes 0, 1 of the word
        const uint32_t b = __byte_perm(w[i], 0x64646464u, 0x5342);   // codes 2, 3
        __half2 ha = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&a), off2), s2);
        __half2 hb = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&b), off2), s2);
        o[2 * i] = *reinterpret_cast<uint32_t*>(&ha);
        o[2 * i + 1] = *reinterpret_cast<uint32_t*>(&hb);
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Device status word values (written by kernels, read by colibri_check).
enum : int { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_BAD_INDEX = 2 };

}  // namespace colibri
