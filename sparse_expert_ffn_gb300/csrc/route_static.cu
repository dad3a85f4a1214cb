// Routing without a handle and without any device allocation.
//
// Some callers cannot call cudaMalloc: code that runs while a stream is being
// captured into a CUDA graph (an allocation there is not part of the graph
// and breaks capture), code inside a framework whose caching allocator has
// reserved the device memory (cudaMalloc fails or forces the framework to
// release its cache), and latency-critical loops that cannot take the
// device-wide synchronisation a cudaMalloc/cudaFree may imply.  For them,
// colibri_route_static runs the routing stage — router logits, top-k,
// softmax over the k, and the dispatch permutation — on the caller's own
// buffers, keeping its intermediate data (the repacked router weights, the
// pair-to-position map, the per-expert offsets and kept counts, and the
// grouped-GEMM tile list) in one file-scope device array of fixed size.
//
// The array is static device memory: every GPU that loads this library holds
// it (kStaticScratchBytes, about 4.6 MiB) until the process exits.  All calls
// on one device share it and it keeps the last call's contents, so two calls
// that overlap on the GPU (on different streams, or in one graph without an
// ordering edge) race on it.  Each call clears the one word that must start at
// zero (the device status word); everything else it reads is written earlier
// in the same call.
//
// A failure the dispatch detects on the device (an expert id outside
// 0 .. n_experts-1, which the router itself never writes) cannot be returned
// by the call, which comes back before the GPU runs; it is reported through
// the outputs instead: every counts[e] is set to -1.
#include <cuda_runtime.h>

#include <climits>
#include <mutex>

#include "colibri_moe.h"
#include "common.cuh"
#include "kernels.h"

using namespace colibri;

namespace {

constexpr int kStaticMaxRouterElems = 1 << 20;  // d_model * n_experts
constexpr int kStaticMaxPairs = 1 << 17;        // T * top_k
constexpr int kStaticTileRows = 128;
constexpr int kStaticMaxTiles = kStaticMaxPairs / kStaticTileRows + 256;

constexpr size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }
constexpr size_t kOffRouter = 0;
constexpr size_t kOffOffsets = kOffRouter + round256((size_t)kStaticMaxRouterElems * 4);
constexpr size_t kOffInv = kOffOffsets + round256(257 * 4);
constexpr size_t kOffTileExpert = kOffInv + round256((size_t)kStaticMaxPairs * 4);
constexpr size_t kOffTileRow = kOffTileExpert + round256((size_t)kStaticMaxTiles * 4);
constexpr size_t kOffTileInfo = kOffTileRow + round256((size_t)kStaticMaxTiles * 4);
constexpr size_t kOffNumTiles = kOffTileInfo + round256((size_t)kStaticMaxTiles * 4);
constexpr size_t kOffKept = kOffNumTiles + 256;
constexpr size_t kOffStatus = kOffKept + round256(256 * 4);
// per-CTA counts of the multi-CTA dispatch: at most 64 CTAs x 256 experts
constexpr size_t kOffBlockCounts = kOffStatus + 256;
constexpr int kStaticMaxDispatchBlocks = kStaticMaxPairs / 2048;
constexpr size_t kStaticScratchBytes = kOffBlockCounts + round256((size_t)kStaticMaxDispatchBlocks * 256 * 4);
// Above this many pairs the dispatch runs over many CTAs (three launches),
// as on a handle.
constexpr int kStaticMultiDispatchPairs = 12288;

static __device__ __align__(256) unsigned char g_route_scratch[kStaticScratchBytes];

// Per-device set-up: the device address of g_route_scratch (in host code the
// symbol is only a host-side stand-in) and the architecture check.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
colibri_status_t g_setup_status[kMaxDevices] = {};
bool g_setup_done[kMaxDevices] = {};

colibri_status_t scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return COLIBRI_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_setup_done[dev]) {
        cudaDeviceProp prop;
        colibri_status_t st = COLIBRI_OK;
        void* p = nullptr;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
            st = COLIBRI_ERR_CUDA;
        else if (prop.major * 10 + prop.minor != 103)
            st = COLIBRI_ERR_UNSUPPORTED;
        else if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
            st = COLIBRI_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_setup_status[dev] = st;
        g_setup_done[dev] = true;
    }
    *out = g_scratch_ptr[dev];
    return g_setup_status[dev];
}

// The dispatch's device status word, read back into the outputs: after a
// failure every count is -1 (a valid count is never negative).
__global__ void report_dispatch_status(const int* __restrict__ status, int32_t* __restrict__ counts,
                                       int E) {
    pdl_enter();
    if (*status != 0)
        for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = -1;
}

}  // namespace

extern "C" colibri_status_t colibri_route_static(const void* x, const void* w_router,
                                                 const float* router_bias, int32_t T,
                                                 int32_t d_model, int32_t n_experts,
                                                 int32_t top_k, int32_t dtype, int32_t* topk_idx,
                                                 float* topk_w, int32_t* counts, int32_t* perm,
                                                 void* stream) {
    if (!x || !w_router || !topk_idx || !topk_w || !counts || !perm) return COLIBRI_ERR_INVALID_ARG;
    if (dtype != COLIBRI_DTYPE_FP32 && dtype != COLIBRI_DTYPE_BF16) return COLIBRI_ERR_INVALID_ARG;
    if (T < 0 || d_model <= 0 || n_experts <= 0 || top_k <= 0 || top_k > n_experts)
        return COLIBRI_ERR_INVALID_ARG;
    if (n_experts > 256 || (top_k > 8 && top_k != n_experts) || d_model % 64 != 0 ||
        !router_simt_fits(d_model))
        return COLIBRI_ERR_UNSUPPORTED;
    // Sizes beyond the fixed scratch array.
    if ((int64_t)d_model * n_experts > kStaticMaxRouterElems ||
        (int64_t)T * top_k > kStaticMaxPairs)
        return COLIBRI_ERR_INVALID_ARG;
    const int esz = dtype == COLIBRI_DTYPE_BF16 ? 2 : 4;
    if (((uintptr_t)x % esz) || ((uintptr_t)w_router % esz)) return COLIBRI_ERR_INVALID_ARG;
    if (T == 0) return COLIBRI_OK;

    void* base = nullptr;
    colibri_status_t st = scratch_for_current_device(&base);
    if (st != COLIBRI_OK) return st;
    uint8_t* s = static_cast<uint8_t*>(base);
    void* wr_packed = s + kOffRouter;
    int32_t* offsets = reinterpret_cast<int32_t*>(s + kOffOffsets);
    int32_t* inv = reinterpret_cast<int32_t*>(s + kOffInv);
    int32_t* tile_expert = reinterpret_cast<int32_t*>(s + kOffTileExpert);
    int32_t* tile_row = reinterpret_cast<int32_t*>(s + kOffTileRow);
    int32_t* tile_info = reinterpret_cast<int32_t*>(s + kOffTileInfo);
    int32_t* num_tiles = reinterpret_cast<int32_t*>(s + kOffNumTiles);
    int32_t* kept = reinterpret_cast<int32_t*>(s + kOffKept);
    int* status = reinterpret_cast<int*>(s + kOffStatus);
    int32_t* block_counts = reinterpret_cast<int32_t*>(s + kOffBlockCounts);

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const DType dt = dtype == COLIBRI_DTYPE_BF16 ? DType::BF16 : DType::F32;
    const int E = n_experts, d = d_model, k = top_k;
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), cs);
    // router [d, E] -> [E, d], K contiguous per expert
    if (e == cudaSuccess)
        e = launch_transpose_remap(esz, w_router, wr_packed, 1, d, E, (size_t)d * E,
                                   (size_t)E * d, E, E, 0, cs);
    if (e == cudaSuccess)
        e = launch_router_simt(dt, x, wr_packed, router_bias, T, d, E, k, topk_idx, topk_w, cs,
                               k == E);   // top_k == n_experts: soft routing
    const int n = T * k;
    if (dispatch_blocks(n) > kStaticMaxDispatchBlocks) return COLIBRI_ERR_INVALID_ARG;  // not reached
    if (e == cudaSuccess && n > kStaticMultiDispatchPairs)
        e = launch_dispatch_multi(topk_idx, n, E, block_counts, counts, offsets, perm, inv,
                                  kStaticTileRows, tile_expert, tile_row, tile_info, num_tiles,
                                  status, INT_MAX, kept, cs);
    else if (e == cudaSuccess)
        e = launch_dispatch(topk_idx, n, E, counts, offsets, perm, inv, kStaticTileRows,
                            tile_expert, tile_row, tile_info, num_tiles, status, INT_MAX, kept,
                            cs);
    if (e == cudaSuccess) e = launch_pdl(report_dispatch_status, 1, 256, 0, cs, status, counts, E);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? COLIBRI_OK : COLIBRI_ERR_CUDA;
}
