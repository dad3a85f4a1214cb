// Host runtime of the C ABI (include/colibri_moe.h): argument checks, weight
// repack, the workspace arena, executor choice and the launch sequence.
//
// Launch sequence of one forward, all on the caller's stream, no host sync,
// no allocation (zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析" section
// 3.3 stages 2-5):
//   router_topk  -> topk_idx, topk_w
//   dispatch     -> counts, offsets, perm, inv, grouped-GEMM tile list
//   STREAM:  ffn_up_stream -> H,  ffn_down_stream -> Y
//   GROUPED: gather_rows -> Xp, tcgen05 gate/up GEMM -> H, tcgen05 down GEMM -> Y
//   combine      -> y (optionally + residual)
// The workspace is one device allocation carved into 256-byte aligned
// sub-buffers at init for max_tokens (pnsm.cn section 3.2: an arena sized
// once, no allocation on the hot path; zskr.cn section 3.2: the pool sized
// from the model and the largest batch).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "colibri_moe.h"
#include "common.cuh"
#include "gemm_tc.h"
#include "kernels.h"

using namespace colibri;

struct colibri_moe {
    colibri_moe_config_t cfg;
    DType dt;
    int esz;
    int num_sms;
    int e_pad;
    // packed weights
    void* wr = nullptr;     // [e_pad, d]
    float* bias = nullptr;  // [E] or null
    void* wgu = nullptr;    // [E][f/128][2][128][d]
    void* wdT = nullptr;    // [E][d][f]
    // int8 expert weights (colibri_init_int8): codes in the same packed
    // layouts, block scales / zero points per 64 packed rows, [rows / 64][K / 64]
    bool int8 = false;
    int8_t* q_gu = nullptr;
    int8_t* q_d = nullptr;
    void* qmeta = nullptr;            // one allocation: the four arrays below
    float* sc_gu = nullptr;
    int32_t* zp_gu = nullptr;
    float* sc_d = nullptr;
    int32_t* zp_d = nullptr;
    uint64_t weight_bytes = 0;
    // workspace
    void* ws = nullptr;
    uint64_t ws_bytes = 0;
    int32_t* topk_idx = nullptr;
    float* topk_w = nullptr;
    int32_t* counts = nullptr;
    int32_t* kept = nullptr;     // [E] pairs each expert accepted (counts capped)
    int32_t* offsets = nullptr;
    int32_t* perm = nullptr;
    int32_t* inv = nullptr;
    int32_t* tile_expert = nullptr;
    int32_t* tile_row = nullptr;
    int32_t* tile_info = nullptr;
    int32_t* num_tiles = nullptr;
    int32_t* block_counts = nullptr;  // multi-CTA dispatch: per-CTA counts, then bases
    float* route_part = nullptr;      // decode routing: partial logits [T][E][slices]
    unsigned int* route_ticket = nullptr;   // decode routing: CTA arrivals, zero at rest
    int32_t* gu_counter = nullptr;    // split gate/up: arrivals per (m-tile, n-block), zero at rest
    size_t gu_counter_bytes = 0;
    size_t y_floats = 0;              // capacity of Y (also the split gate/up partials)
    int* status = nullptr;
    void* H = nullptr;      // [max_pairs, f]
    void* xp = nullptr;     // [max_pairs, d] token rows in expert order
    float* Y = nullptr;     // [max_pairs, d]
    void* u = nullptr;      // [max_tokens, d]
    // host-buffer forwards: two staging slots of x and y ([2][max_tokens, d]),
    // an upload and a download stream, and per slot the events "x landed",
    // "layer done" and "y downloaded"
    void* x_stage = nullptr;
    void* y_stage = nullptr;
    size_t stage_bytes = 0;   // bytes of one slot
    cudaStream_t cs_in = nullptr, cs_out = nullptr;
    cudaEvent_t ev_in[2] = {nullptr, nullptr}, ev_done[2] = {nullptr, nullptr},
                ev_out[2] = {nullptr, nullptr};
    int host_slot = 0;
    int max_pairs = 0;
    int max_tiles = 0;
    int max_resident_pairs = 0;  // CTA pairs of the expert GEMMs resident at once
    bool grouped_ok = false;
    // B operands: 128-row boxes for CTA pairs, 256-row boxes for single CTAs
    CUtensorMap tm_xp, tm_wgu, tm_h, tm_wdT, tm_wr, tm_wgu1, tm_wdT1;
    TokenRowMaps tm_xp_rows, tm_h_rows;   // B of the weights-as-M GEMMs (bf16 handles)
    CUtensorMap tm_wgu_wm;  // packed gate/up, 5-D view (weights-as-M pair GEMM)
    bool wm_gate_up = false;   // the view encoded
    // decode GEMM (weights as M): token rows in 32-row boxes (bf16 weights:
    // tm_wgu / tm_wdT, 128-row boxes; int8 codes: bulk copies of tiles)
    CUtensorMap tm_xp32, tm_h32;
    uint64_t wait_limit_ns = 2000000000ull;
    bool stall_tma = false;  // failure-detection tests (COLIBRI_TEST_STALL_TMA=1)
    int last_T = 0;
    int capacity = -1;   // hard expert capacity; < 0: no limit
    uint64_t launches = 0;
    colibri_status_t sticky = COLIBRI_OK;
    // opt-in per-stage event profiling
    bool prof = false;
    struct ProfRec {
        int stage;
        cudaEvent_t a, b;
    };
    std::vector<cudaEvent_t> ev_pool;
    std::vector<ProfRec> recs;
};

namespace {

// Allocation-failure injection for tests: COLIBRI_FAIL_ALLOC_AT=n makes the
// n-th device allocation of an init fail (1-based).
struct AllocCounter {
    int n = 0;
    int fail_at = 0;
    AllocCounter() {
        const char* e = std::getenv("COLIBRI_FAIL_ALLOC_AT");
        fail_at = e ? std::atoi(e) : 0;
    }
    cudaError_t alloc(void** p, size_t bytes) {
        ++n;
        if (fail_at > 0 && n == fail_at) {
            *p = nullptr;
            return cudaErrorMemoryAllocation;
        }
        return cudaMalloc(p, bytes);
    }
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Split-K of the down projection: only for batches of at most kSplitMaxPairs
// (token, slot) pairs, into at most kMaxKSplit slices; Y holds room for them.
constexpr int kSplitMaxPairs = 2048;
// Above this many (token, slot) pairs the dispatch runs over many CTAs.
constexpr int kMultiDispatchPairs = 12288;
// Batches from this many tokens route on the tensor cores.
constexpr int kTcRouterMinTokens = 512;
// The decode routing launch gathers the token rows itself up to this many bytes.
constexpr size_t kRouteGatherBytes = 128 * 1024;
constexpr int kMaxKSplit = 16;
// K slices of the tensor-core router at most (the last slice routes the rows).
constexpr int kMaxRouterSplit = 8;
// Batches averaging at most this many (token, slot) pairs per expert run the
// decode GEMMs (weights as the MMA's M operand, 32-token tiles).
constexpr int kDecMaxPairsPerExpert = 16;
// The gate/up GEMM splits K only for batches of at most this many pairs.
constexpr int kGateUpSplitMaxPairs = 64;
// CTA-pair GEMMs run with the weights as the MMA's M operand and each tile's
// tokens as N (rounded up to 32), so an expert's last tile carries at most 31
// padding columns instead of up to 255 padding rows.  The down projection
// always; gate/up from this d_model on, where a work item's MMAs (K = d) hide
// its transposed epilogue (measured, Mixtral-shaped T = 4096: gate/up 1191 ->
// 1175 us, down 590 -> 572 us; DeepSeek-shaped T = 16384, K = 2048: gate/up
// 560 -> 718 us, the epilogue exposed).
constexpr int kWmGateUpMinK = 4096;
// Int8 weights: batches of at most this many tokens stream the codes on the
// CUDA cores (gemv_i8.cu) when the gate/up stage has at least one 64-unit
// item per SM; the tensor-core decode GEMMs take one MMA per 2 KB of codes
// whatever the token count, about 0.7 of HBM at best.  Measured, Mixtral-
// shaped layer, one forward with L2 flushed (tensor cores / CUDA cores):
// T = 1 131 / 94 us, 2 213 / 168, 3 231 / 227, 4 299 / 327, 8 399 / 721.
constexpr int kGemvMaxTokens = 3;
// Resident CTAs per SM the CUDA-core int8 items are sized for.
constexpr int kGemvCtasPerSm = 8;

// K slices of the CUDA-core int8 down projection: `units` (tile, 64-row
// group) items of nkb k-tiles; the count whose busiest SM (items spread
// evenly, every item resident) streams the fewest k-tiles, three k-tiles of
// fixed cost per item, and fewer than three items per SM penalised in
// proportion (too few loads in flight to cover HBM latency).
int choose_gemv_slices(int64_t units, int nkb, int num_sms, int max_ks) {
    int best = 1;
    double best_cost = 0.0;
    for (int ks = 1; ks <= std::max(1, std::min({max_ks, nkb, 16})); ++ks) {
        const int64_t u = units * ks;
        if (ks > 1 && u > (int64_t)num_sms * kGemvCtasPerSm) break;
        const int64_t per_sm = (u + num_sms - 1) / num_sms;
        double cost = (double)per_sm * ((nkb + ks - 1) / ks + 3);
        if (u < 3 * (int64_t)num_sms) cost *= 3.0 * num_sms / (double)u;
        if (ks == 1 || cost < best_cost) best = ks, best_cost = cost;
    }
    return best;
}

// K slices of a GEMM with `items` (m-tile, n-block) work items of kb K blocks
// each, on `units` resident work units: the count (every slice non-empty)
// that minimises the number of waves times the slice length, with two K
// blocks of fixed cost per work item (pipeline fill and epilogue).
int choose_k_splits(int64_t items, int kb, int units, int max_splits) {
    int best = 1;
    double best_cost = 0.0;
    for (int ks = 1; ks <= std::max(1, std::min(max_splits, kb)); ++ks) {
        const int per = (kb + ks - 1) / ks;
        const int eff = (kb + per - 1) / per;
        const int64_t waves = (items * eff + units - 1) / units;
        const double cost = (double)waves * (per + 2);
        if (ks == 1 || cost < best_cost) best = eff, best_cost = cost;
    }
    return best;
}

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

colibri_status_t validate_config(const colibri_moe_config_t* c) {
    if (!c) return COLIBRI_ERR_INVALID_ARG;
    if (c->n_experts <= 0 || c->top_k <= 0 || c->d_model <= 0 || c->d_ff <= 0 ||
        c->max_tokens <= 0 || c->device < 0)
        return COLIBRI_ERR_INVALID_ARG;
    if (c->top_k > c->n_experts) return COLIBRI_ERR_INVALID_ARG;
    if (c->dtype != COLIBRI_DTYPE_FP32 && c->dtype != COLIBRI_DTYPE_BF16)
        return COLIBRI_ERR_INVALID_ARG;
    if (c->executor < COLIBRI_EXEC_AUTO || c->executor > COLIBRI_EXEC_GROUPED)
        return COLIBRI_ERR_INVALID_ARG;
    if ((int64_t)c->max_tokens * c->top_k > (int64_t)1 << 30) return COLIBRI_ERR_INVALID_ARG;
    // top_k == n_experts is soft routing (every expert, softmax over all E);
    // otherwise the top-k kernels take up to 8 experts per token
    if (c->n_experts > 256 || (c->top_k > 8 && c->top_k != c->n_experts))
        return COLIBRI_ERR_UNSUPPORTED;
    if (c->d_model % 64 != 0 || c->d_ff % 128 != 0) return COLIBRI_ERR_UNSUPPORTED;
    if (!router_simt_fits(c->d_model)) return COLIBRI_ERR_UNSUPPORTED;
    if (c->executor == COLIBRI_EXEC_GROUPED && c->dtype != COLIBRI_DTYPE_BF16)
        return COLIBRI_ERR_UNSUPPORTED;
    return COLIBRI_OK;
}

bool grouped_shape_ok(const colibri_moe_config_t& c) {
    return c.dtype == COLIBRI_DTYPE_BF16 && c.d_model % 256 == 0 && c.d_ff % 128 == 0;
}

void release(colibri_moe_t* h) {
    if (!h) return;
    for (auto& r : h->recs) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    for (auto e : h->ev_pool) cudaEventDestroy(e);
    if (h->cs_in) cudaStreamSynchronize(h->cs_in);
    if (h->cs_out) cudaStreamSynchronize(h->cs_out);
    for (int i = 0; i < 2; ++i) {
        if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
        if (h->ev_done[i]) cudaEventDestroy(h->ev_done[i]);
        if (h->ev_out[i]) cudaEventDestroy(h->ev_out[i]);
    }
    if (h->cs_in) cudaStreamDestroy(h->cs_in);
    if (h->cs_out) cudaStreamDestroy(h->cs_out);
    cudaFree(h->wr);
    cudaFree(h->bias);
    cudaFree(h->wgu);
    cudaFree(h->wdT);
    cudaFree(h->q_gu);
    cudaFree(h->q_d);
    cudaFree(h->qmeta);
    cudaFree(h->ws);
    delete h;
}

colibri_status_t from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return COLIBRI_OK;
    if (e == cudaErrorMemoryAllocation) return COLIBRI_ERR_OOM;
    return COLIBRI_ERR_CUDA;
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + nb && pb < pa + na;
}

// Copy (host or device) matrices [batch][R][C] into the packed layout through
// the remapping transpose; host inputs go through a device staging buffer one
// batch entry at a time.
colibri_status_t pack(int esz, const void* src, bool src_on_device, void* dst, int batch, int R,
                      int C, size_t out_batch, int blk, int period, int which, void* staging,
                      bool tiled = false) {
    const size_t mat = (size_t)R * C * esz;
    if (src_on_device) {
        return from_cuda(launch_transpose_remap(esz, src, dst, batch, R, C, (size_t)R * C,
                                                out_batch, blk, period, which, 0, tiled));
    }
    for (int b = 0; b < batch; ++b) {
        cudaError_t e = cudaMemcpy(staging, (const uint8_t*)src + (size_t)b * mat, mat,
                                   cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return from_cuda(e);
        e = launch_transpose_remap(esz, staging, (uint8_t*)dst + (size_t)b * out_batch * esz, 1, R,
                                   C, (size_t)R * C, out_batch, blk, period, which, 0, tiled);
        if (e != cudaSuccess) return from_cuda(e);
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return from_cuda(e);
    }
    return COLIBRI_OK;
}

// The CUDA-core int8 GEMV can run this batch: int8 codes, bf16 activations,
// at most kGemvMaxTokens tokens, and its staging fits (Y holds at least 8 K
// slices of a batch this small).
bool gemv_i8_usable(const colibri_moe_t* h, int T) {
    const auto& c = h->cfg;
    return h->int8 && h->dt == DType::BF16 && T >= 1 && T <= kGemvMaxTokens &&
           gemv_i8_fits(gemv_i8_slots(T), c.d_model, c.d_ff, 8);
}

int choose_executor(const colibri_moe_t* h, int T) {
    if (h->cfg.executor != COLIBRI_EXEC_AUTO) return h->cfg.executor;
    // bf16: the TMA-fed grouped GEMM streams the active experts' weights
    // faster than the CUDA-core kernels at every batch size measured (one
    // token included, with split-K on the down projection); CUDA cores run
    // the float32 layer, shapes the tensor-core path does not take, and
    // int8 codes for a few tokens per expert.
    // (with at least one gate/up item per SM even when the tokens share
    // their experts)
    if (gemv_i8_usable(h, T) &&
        gemv_i8_items(true, h->cfg.top_k, h->cfg.d_model, h->cfg.d_ff, 1) >= h->num_sms)
        return COLIBRI_EXEC_STREAM;
    return h->grouped_ok ? COLIBRI_EXEC_GROUPED : COLIBRI_EXEC_STREAM;
}

cudaEvent_t take_event(colibri_moe_t* h) {
    if (!h->ev_pool.empty()) {
        cudaEvent_t e = h->ev_pool.back();
        h->ev_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Brackets one stage's kernel launch(es): records an event pair when
// profiling is on, counts the launches, and maps launch errors.
struct Stage {
    colibri_moe_t* h;
    int stage;
    cudaStream_t s;
    cudaEvent_t a = nullptr;
    Stage(colibri_moe_t* h_, int stage_, cudaStream_t s_) : h(h_), stage(stage_), s(s_) {
        if (h->prof && (a = take_event(h))) cudaEventRecord(a, s);
    }
    colibri_status_t done(cudaError_t e, int nlaunch) {
        h->launches += nlaunch;
        if (a) {
            cudaEvent_t b = take_event(h);
            if (b) {
                cudaEventRecord(b, s);
                h->recs.push_back({stage, a, b});
            } else {
                h->ev_pool.push_back(a);
            }
        }
        return from_cuda(e);
    }
};

// The layer on device buffers; `resid` (may equal y) adds a residual.  With
// `gamma` the layer input is u = RMSNorm(x) * gamma (written to h->u): fused
// into the small-batch routing kernel when that runs, else its own launch.
// With `r_idx` the routing is the caller's (r_k experts per row, gates r_w):
// no router runs, the rest of the layer is the same.
colibri_status_t run_layer(colibri_moe_t* h, const void* x, int T, void* y, const void* resid,
                           cudaStream_t s, const void* gamma = nullptr, float eps = 0.f,
                           const int32_t* r_idx = nullptr, const float* r_w = nullptr, int r_k = 0) {
    const auto& c = h->cfg;
    const int E = c.n_experts, k = r_idx ? r_k : c.top_k, d = c.d_model, f = c.d_ff;
    const int npairs = T * k;
    colibri_status_t st;
    const int ex = choose_executor(h, T);
    // Expert GEMMs on CTA pairs (256-row tiles) once the batch averages 128
    // rows per expert; below that most tile rows would be empty and single
    // CTAs (128-row tiles) stream the weights faster.
    const bool dec = ex == COLIBRI_EXEC_GROUPED && npairs <= kDecMaxPairsPerExpert * E;
    const bool pair = ex == COLIBRI_EXEC_GROUPED && !dec && npairs >= 128 * E && !h->int8;
    const int tile_rows = dec ? tc_gemm_dec_tile_rows() : pair ? tc_gemm_pair_rows() : tc_gemm_block_m();
    // Decode-sized batch: router, top-k, softmax, dispatch (and the gather of
    // a small batch) in one launch.  Soft routing (k == E) runs on the
    // CUDA-core router kernel.
    const bool soft = !r_idx && k == E;
    const bool fused_routing = !r_idx && !soft && route_decode_fits(T, d, E, k);
    // the gather stays in the routing launch while its rows are few: its
    // last CTA copies them alone
    const bool gather_in_route = fused_routing && (size_t)npairs * d * h->esz <= kRouteGatherBytes;
    const int cap = h->capacity < 0 ? INT_MAX : h->capacity;
    if (gamma && !fused_routing) {
        Stage g(h, COLIBRI_STAGE_RMSNORM, s);
        st = g.done(launch_rmsnorm(h->dt, x, gamma, T, d, eps, h->u, s), 1);
        if (st != COLIBRI_OK) return st;
        x = h->u;
    }
    if (r_idx) {
        // the caller's routing, into the workspace the dispatch and combine read
        Stage g(h, COLIBRI_STAGE_ROUTER, s);
        cudaError_t e = cudaMemcpyAsync(h->topk_idx, r_idx, (size_t)npairs * 4, cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(h->topk_w, r_w, (size_t)npairs * 4, cudaMemcpyDeviceToDevice, s);
        st = g.done(e, 0);
        if (st != COLIBRI_OK) return st;
    } else if (fused_routing) {
        Stage g(h, COLIBRI_STAGE_ROUTER, s);
        st = g.done(launch_route_decode(h->dt, x, h->wr, h->bias, T, d, E, k, h->route_part,
                                        h->route_ticket, h->topk_idx, h->topk_w, h->counts,
                                        h->offsets, h->perm, h->inv, tile_rows, h->tile_expert,
                                        h->tile_row, h->tile_info, h->num_tiles, h->status, cap,
                                        h->kept,
                                        ex == COLIBRI_EXEC_GROUPED && gather_in_route ? h->xp
                                                                                      : nullptr,
                                        gamma, eps, h->u, s, h->int8), 1);
        if (st != COLIBRI_OK) return st;
        if (gamma) x = h->u;
    } else if (h->grouped_ok && T >= kTcRouterMinTokens && !soft) {
        // Large batch: the router logits are a [T, d] x [d, E] GEMM on the
        // tensor cores, top-k and softmax in its epilogue.
        CUtensorMap tm_x;
        if (!make_tmap_bf16(&tm_x, x, (uint64_t)T, (uint64_t)d, 128)) return COLIBRI_ERR_CUDA;
        TcGemmArgs a{};
        a.dense_rows = T;
        a.bn_rows = h->e_pad;
        a.n_experts = E;
        a.top_k = k;
        a.bias = h->bias;
        a.topk_idx = h->topk_idx;
        a.topk_w = h->topk_w;
        a.n_blocks = 1;
        a.k_blocks = d / 64;
        a.k_splits = 1;
        a.status = h->status;
        a.wait_limit_ns = h->wait_limit_ns;
        a.stall_producer = h->stall_tma ? 1 : 0;
        // At most a quarter as many 128-token tiles as SMs, and logit rows of
        // at most 16 columns: split K (float32 partial logits in Y, one
        // arrival counter per tile and lane quarter in gu_counter).  With
        // fewer slices the fixup's latency (fence, counter, reloading the
        // partials) costs more than the shorter K loop saves (E = 64, 2
        // slices: 28 -> 35 us); with wider rows the fixup reloads every
        // slice of every 32-logit chunk (measured, 128-token tiles: 8 experts
        // at T = 4096, 27.1 us whole, 21.4 us in 4 slices; 64 experts at
        // T = 2048, 22.7 us whole, 42.5 us in 8 slices; 128 experts at
        // T = 2048, 29.8 us whole, 75.8 us in 8 slices).
        const int tiles = (T + tc_gemm_block_m() - 1) / tc_gemm_block_m();
        if (4 * tiles <= h->num_sms && h->e_pad <= 16) {
            const int fit = (int)std::min<size_t>(kMaxRouterSplit, h->y_floats / ((size_t)T * h->e_pad));
            a.k_splits = choose_k_splits(tiles, a.k_blocks, h->num_sms, fit);
            a.partial = h->Y;
            a.partial_split_stride = (size_t)T * h->e_pad;
            a.tile_counter = h->gu_counter;
        }
        const int grid = std::min(tiles * a.k_splits, h->num_sms);
        Stage g(h, COLIBRI_STAGE_ROUTER, s);
        st = g.done(launch_tc_gemm(kRouter, false, tm_x, h->tm_wr, a, grid, s), 1);
        if (st != COLIBRI_OK) return st;
    } else {
        Stage g(h, COLIBRI_STAGE_ROUTER, s);
        st = g.done(launch_router_simt(h->dt, x, h->wr, h->bias, T, d, E, k, h->topk_idx,
                                       h->topk_w, s, soft), 1);
        if (st != COLIBRI_OK) return st;
    }
    if (!fused_routing && npairs > kMultiDispatchPairs) {
        // many pairs: the counting sort over many CTAs (three launches)
        Stage g(h, COLIBRI_STAGE_DISPATCH, s);
        st = g.done(launch_dispatch_multi(h->topk_idx, npairs, E, h->block_counts, h->counts,
                                          h->offsets, h->perm, h->inv, tile_rows,
                                          h->tile_expert, h->tile_row, h->tile_info,
                                          h->num_tiles, h->status, cap, h->kept, s), 3);
        if (st != COLIBRI_OK) return st;
    } else if (!fused_routing) {
        Stage g(h, COLIBRI_STAGE_DISPATCH, s);
        st = g.done(launch_dispatch(h->topk_idx, npairs, E, h->counts, h->offsets, h->perm,
                                    h->inv, tile_rows, h->tile_expert, h->tile_row,
                                    h->tile_info, h->num_tiles, h->status, cap, h->kept, s),
                    1);
        if (st != COLIBRI_OK) return st;
    }
    int nsplit = 1;
    size_t split_stride = 0;
    bool y_bf16 = false;     // Y rows stored as bf16 by the down GEMM
    if (ex == COLIBRI_EXEC_STREAM && gemv_i8_usable(h, T)) {
        // a few tokens per expert: items of 64 weight rows, every item's
        // codes read once per pass of S token rows
        const int S = gemv_i8_slots(T);
        const GemvTiles tl{h->tile_expert, h->tile_row, h->tile_info, h->num_tiles, E, h->status,
                           h->wait_limit_ns, h->stall_tma ? 1 : 0};
        const int tiles_est = std::min(E, npairs);
        const int max_ks = (int)std::min<size_t>(kMaxKSplit, h->y_floats / ((size_t)npairs * d));
        int ks = choose_gemv_slices((int64_t)tiles_est * (d / 64), f / 64, h->num_sms, max_ks);
        while (ks < max_ks && !gemv_i8_fits(S, d, f, ks)) ++ks;   // shorter slices stage less
        const int cap_grid = h->num_sms * kGemvCtasPerSm;
        {
            Stage g(h, COLIBRI_STAGE_EXPERT_UP, s);
            const int grid = std::min(gemv_i8_items(true, tiles_est, d, f, 1), cap_grid);
            st = g.done(launch_ffn_up_gemv_i8(S, x, h->perm, k, h->q_gu, h->sc_gu,
                                              h->zp_gu, tl, d, f, grid, h->H, s),
                        1);
            if (st != COLIBRI_OK) return st;
        }
        {
            Stage g(h, COLIBRI_STAGE_EXPERT_DOWN, s);
            const int grid = std::min(gemv_i8_items(false, tiles_est, d, f, ks), cap_grid);
            st = g.done(launch_ffn_down_gemv_i8(S, h->H, h->q_d, h->sc_d, h->zp_d, tl, d,
                                                f, ks, grid, h->Y, (size_t)npairs * d, s),
                        1);
            if (st != COLIBRI_OK) return st;
        }
        nsplit = ks;
        split_stride = (size_t)npairs * d;
    } else if (ex == COLIBRI_EXEC_STREAM) {
        {
            Stage g(h, COLIBRI_STAGE_EXPERT_UP, s);
            st = g.done(h->int8 ? launch_ffn_up_stream_i8(h->dt, x, h->q_gu, h->sc_gu, h->zp_gu,
                                                          h->kept, h->offsets, h->perm, k, d, f, E,
                                                          h->H, s)
                                : launch_ffn_up_stream(h->dt, x, h->wgu, h->kept, h->offsets,
                                                       h->perm, k, d, f, E, h->H, s),
                        1);
            if (st != COLIBRI_OK) return st;
        }
        {
            Stage g(h, COLIBRI_STAGE_EXPERT_DOWN, s);
            st = g.done(h->int8 ? launch_ffn_down_stream_i8(h->dt, h->H, h->q_d, h->sc_d, h->zp_d,
                                                            h->kept, h->offsets, d, f, E, h->Y, s)
                                : launch_ffn_down_stream(h->dt, h->H, h->wdT, h->kept, h->offsets,
                                                         d, f, E, h->Y, s),
                        1);
            if (st != COLIBRI_OK) return st;
        }
    } else {
        // Expert tiles: 256 rows per CTA pair (each CTA 128), or 128 rows per CTA.
        const int tiles_ub = (npairs + tile_rows - 1) / tile_rows + std::min(E, npairs);
        // resident work units: CTA pairs, or single CTAs
        const int units = pair ? (h->max_resident_pairs > 0 ? h->max_resident_pairs : h->num_sms / 2)
                               : h->num_sms;
        const int cta_per_unit = pair ? 2 : 1;
        if (!gather_in_route) {
            // token rows in expert order (the gate/up GEMM's A operand); TMA
            // boxes of 128 consecutive rows read it far faster than per-row
            // gathers inside the GEMM
            Stage g(h, COLIBRI_STAGE_GATHER, s);
            st = g.done(launch_gather(h->esz, x, h->perm, k, d, npairs, npairs, h->xp, s, h->int8), 1);
            if (st != COLIBRI_OK) return st;
        }
        TcGemmArgs a{};
        a.tile_expert = h->tile_expert;
        a.tile_row = h->tile_row;
        a.tile_info = h->tile_info;
        a.num_tiles = h->num_tiles;
        a.status = h->status;
        a.wait_limit_ns = h->wait_limit_ns;
        a.stall_producer = h->stall_tma ? 1 : 0;
        // Work items the GEMMs will see: with at most one tile per expert,
        // an expert per distinct routed expert (exactly k for one token).
        const int64_t tiles_est = npairs <= tile_rows ? std::min(E, npairs) : tiles_ub;
        // gate/up: N = 2f in blocks of 256 rows (128 gate + 128 up), K = d.
        // A decode-sized batch leaves a fraction of a wave in the last round
        // of items: split K, the last slice to finish writes H.
        a.n_blocks = f / 128;
        a.k_blocks = d / 64;
        a.k_splits = 1;
        a.out_split_stride = 0;
        a.b_rows_per_expert = 2 * f;
        a.out = h->H;
        a.out_ld = f;
        a.q_scale = h->sc_gu;
        a.q_zp = h->zp_gu;
        a.q_codes = h->q_gu;
        if (!pair && npairs <= kGateUpSplitMaxPairs) {
            const int fit = (int)std::min<size_t>(kMaxKSplit, h->y_floats / ((size_t)npairs * 2 * f));
            a.k_splits = choose_k_splits(tiles_est * a.n_blocks, a.k_blocks, units, fit);
            a.partial = h->Y;
            a.partial_split_stride = (size_t)npairs * 2 * f;
            a.tile_counter = h->gu_counter;
        }
        {
            const int grid = cta_per_unit * (int)std::min<int64_t>(
                                                    (int64_t)tiles_ub * a.n_blocks * a.k_splits, units);
            Stage g(h, COLIBRI_STAGE_EXPERT_UP, s);
            st = g.done(dec    ? launch_tc_gemm_dec(kGateUp, h->tm_xp32, h->int8 ? h->tm_xp : h->tm_wgu,
                                                    a, grid, s, h->int8)
                        : pair && h->wm_gate_up && d >= kWmGateUpMinK
                            ? launch_tc_gemm(kGateUp, true, h->tm_wgu_wm, h->tm_xp, a, grid, s, false, true,
                                             &h->tm_xp_rows)
                        : pair ? launch_tc_gemm(kGateUp, true, h->tm_xp, h->tm_wgu, a, grid, s)
                               : launch_tc_gemm(kGateUp, false, h->tm_xp, h->tm_wgu1, a, grid, s,
                                                h->int8),
                        1);
            if (st != COLIBRI_OK) return st;
        }
        // down: N = d in blocks of 256, K = f.  Few pairs leave too few
        // (m-tile, n-block) items to fill the GPU: split K into slices whose
        // float32 partials the combine adds in slice order.
        a.n_blocks = d / (dec ? tc_gemm_dec_w_rows() : 256);
        a.k_blocks = f / 64;
        a.b_rows_per_expert = d;
        a.out = h->Y;
        a.out_ld = d;
        a.q_scale = h->sc_d;
        a.q_zp = h->zp_d;
        a.q_codes = h->q_d;
        a.k_splits = 1;
        a.partial = nullptr;
        a.partial_split_stride = 0;
        a.tile_counter = nullptr;
        if (npairs <= kSplitMaxPairs) {
            const int fit = (int)std::min<size_t>(kMaxKSplit, h->y_floats / ((size_t)npairs * d));
            a.k_splits = choose_k_splits(tiles_est * a.n_blocks, a.k_blocks, units, fit);
        }
        a.out_split_stride = (size_t)npairs * d;
        // Without K slices the token-on-M GEMM stores Y as bf16 (one
        // rounding, as H): the combine, bound by reading Y, reads half.
        a.y_bf16 = (!dec && a.k_splits == 1) ? 1 : 0;
        y_bf16 = a.y_bf16 != 0;
        {
            const int grid = cta_per_unit * (int)std::min<int64_t>(
                                                    (int64_t)tiles_ub * a.n_blocks * a.k_splits, units);
            Stage g(h, COLIBRI_STAGE_EXPERT_DOWN, s);
            st = g.done(dec    ? launch_tc_gemm_dec(kDown, h->tm_h32, h->int8 ? h->tm_h : h->tm_wdT, a,
                                                    grid, s, h->int8)
                        : pair ? launch_tc_gemm(kDown, true, h->tm_wdT, h->tm_h, a, grid, s, false,
                                                true, &h->tm_h_rows)
                               : launch_tc_gemm(kDown, false, h->tm_h, h->tm_wdT1, a, grid, s,
                                                h->int8),
                        1);
            if (st != COLIBRI_OK) return st;
        }
        nsplit = a.k_splits;
        split_stride = a.out_split_stride;
    }
    {
        Stage g(h, COLIBRI_STAGE_COMBINE, s);
        st = g.done(launch_combine(h->dt, h->Y, y_bf16, h->topk_w, h->inv, T, k, d, nsplit,
                                   split_stride, resid, y, s), 1);
        if (st != COLIBRI_OK) return st;
    }
    h->last_T = T;
    return COLIBRI_OK;
}

}  // namespace

extern "C" {

const char* colibri_status_str(colibri_status_t s) {
    switch (s) {
        case COLIBRI_OK: return "ok";
        case COLIBRI_ERR_INVALID_ARG: return "invalid argument";
        case COLIBRI_ERR_OOM: return "out of memory";
        case COLIBRI_ERR_CUDA: return "CUDA error";
        case COLIBRI_ERR_UNSUPPORTED: return "unsupported device or shape";
        case COLIBRI_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

}  // extern "C"

namespace {

// Shared by colibri_init (bf16 / fp32 expert weights) and colibri_init_int8
// (int8 blocks: qg / qu / qd non-null, w_gate / w_up / w_down unused).
colibri_status_t init_impl(const colibri_moe_config_t* cfg, const void* w_router,
                           const float* router_bias, const void* w_gate, const void* w_up,
                           const void* w_down, const colibri_int8_weights_t* qg,
                           const colibri_int8_weights_t* qu, const colibri_int8_weights_t* qd,
                           int weights_on_device, colibri_moe_t** out) {
    if (!out) return COLIBRI_ERR_INVALID_ARG;
    *out = nullptr;
    colibri_status_t st = validate_config(cfg);
    if (st != COLIBRI_OK) return st;
    const bool int8 = qg != nullptr;
    if (!w_router) return COLIBRI_ERR_INVALID_ARG;
    if (int8) {
        if (!qu || !qd) return COLIBRI_ERR_INVALID_ARG;
        for (const colibri_int8_weights_t* w : {qg, qu, qd})
            if (!w->q || !w->scale || !w->zp) return COLIBRI_ERR_INVALID_ARG;
        // code tiles hold 128 packed rows: an expert's down rows fill whole tiles
        if (cfg->d_model % 128) return COLIBRI_ERR_UNSUPPORTED;
    } else if (!w_gate || !w_up || !w_down) {
        return COLIBRI_ERR_INVALID_ARG;
    }
    if (weights_on_device != 0 && weights_on_device != 1) return COLIBRI_ERR_INVALID_ARG;

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) return COLIBRI_ERR_CUDA;
    if (cfg->device >= ndev) return COLIBRI_ERR_INVALID_ARG;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, cfg->device) != cudaSuccess) return COLIBRI_ERR_CUDA;
    if (prop.major * 10 + prop.minor != 103) return COLIBRI_ERR_UNSUPPORTED;
    DeviceGuard guard(cfg->device);
    if (!guard.ok) return COLIBRI_ERR_CUDA;

    colibri_moe_t* h = new (std::nothrow) colibri_moe;
    if (!h) return COLIBRI_ERR_OOM;
    h->cfg = *cfg;
    h->dt = cfg->dtype == COLIBRI_DTYPE_BF16 ? DType::BF16 : DType::F32;
    h->esz = cfg->dtype == COLIBRI_DTYPE_BF16 ? 2 : 4;
    h->num_sms = prop.multiProcessorCount;
    h->e_pad = (cfg->n_experts + 15) / 16 * 16;
    h->int8 = int8;
    // Failure-detection tests: a shorter bound for the device-side waits, and
    // a producer that never issues its copies (a flag that nothing sets).
    if (const char* e = std::getenv("COLIBRI_WAIT_LIMIT_NS")) h->wait_limit_ns = std::strtoull(e, nullptr, 10);
    if (const char* e = std::getenv("COLIBRI_TEST_STALL_TMA")) h->stall_tma = std::atoi(e) != 0;

    const int E = cfg->n_experts, d = cfg->d_model, f = cfg->d_ff, k = cfg->top_k;
    AllocCounter ac;
    auto fail = [&](colibri_status_t s) {
        cudaDeviceSynchronize();
        release(h);
        return s;
    };

    // ---- weights
    const size_t wr_bytes = (size_t)h->e_pad * d * h->esz;
    const size_t wsz = int8 ? 1 : (size_t)h->esz;       // expert weight element bytes
    const size_t wgu_bytes = (size_t)E * 2 * f * d * wsz;
    const size_t wd_bytes = (size_t)E * d * f * wsz;
    const size_t nblk = (size_t)(d / 64) * (f / 64);      // 64x64 blocks per matrix
    const size_t meta_bytes = int8 ? (size_t)E * 3 * nblk * 8 : 0;
    if ((st = from_cuda(ac.alloc(&h->wr, wr_bytes))) != COLIBRI_OK) return fail(st);
    if (int8) {
        if ((st = from_cuda(ac.alloc((void**)&h->q_gu, wgu_bytes))) != COLIBRI_OK) return fail(st);
        if ((st = from_cuda(ac.alloc((void**)&h->q_d, wd_bytes))) != COLIBRI_OK) return fail(st);
        if ((st = from_cuda(ac.alloc(&h->qmeta, meta_bytes))) != COLIBRI_OK) return fail(st);
        h->sc_gu = (float*)h->qmeta;
        h->zp_gu = (int32_t*)(h->sc_gu + (size_t)E * 2 * nblk);
        h->sc_d = (float*)(h->zp_gu + (size_t)E * 2 * nblk);
        h->zp_d = (int32_t*)(h->sc_d + (size_t)E * nblk);
    } else {
        if ((st = from_cuda(ac.alloc(&h->wgu, wgu_bytes))) != COLIBRI_OK) return fail(st);
        if ((st = from_cuda(ac.alloc(&h->wdT, wd_bytes))) != COLIBRI_OK) return fail(st);
    }
    if (router_bias) {
        if ((st = from_cuda(ac.alloc((void**)&h->bias, (size_t)E * 4))) != COLIBRI_OK)
            return fail(st);
        if ((st = from_cuda(cudaMemcpy(h->bias, router_bias, (size_t)E * 4, cudaMemcpyDefault))) !=
            COLIBRI_OK)
            return fail(st);
    }
    h->weight_bytes =
        wr_bytes + wgu_bytes + wd_bytes + meta_bytes + (router_bias ? (size_t)E * 4 : 0);

    void* staging = nullptr;
    if (!weights_on_device) {
        const size_t stage_bytes =
            std::max((size_t)d * f * wsz, std::max((size_t)d * E * h->esz, nblk * 4));
        if ((st = from_cuda(ac.alloc(&staging, stage_bytes))) != COLIBRI_OK) return fail(st);
    }
    auto fail_staged = [&](colibri_status_t s) {
        cudaDeviceSynchronize();
        cudaFree(staging);
        return fail(s);
    };
    const bool dev = weights_on_device != 0;
    if ((st = from_cuda(cudaMemset(h->wr, 0, wr_bytes))) != COLIBRI_OK) return fail_staged(st);
    // router [d, E] -> [E, d]
    st = pack(h->esz, w_router, dev, h->wr, 1, d, E, (size_t)h->e_pad * d, E, E, 0, staging);
    if (st != COLIBRI_OK) return fail_staged(st);
    if (!int8) {
        // gate/up [E][d][f] -> [E][f/128][2][128][d]
        st = pack(h->esz, w_gate, dev, h->wgu, E, d, f, (size_t)2 * f * d, 128, 256, 0, staging);
        if (st == COLIBRI_OK)
            st = pack(h->esz, w_up, dev, h->wgu, E, d, f, (size_t)2 * f * d, 128, 256, 1, staging);
        // down [E][f][d] -> [E][d][f]
        if (st == COLIBRI_OK)
            st = pack(h->esz, w_down, dev, h->wdT, E, f, d, (size_t)d * f, d, d, 0, staging);
    } else {
        // codes: the bf16 layouts with one-byte elements
        // codes: the bf16 packed rows, stored tile-major (code_index)
        st = pack(1, qg->q, dev, h->q_gu, E, d, f, (size_t)2 * f * d, 128, 256, 0, staging, true);
        if (st == COLIBRI_OK)
            st = pack(1, qu->q, dev, h->q_gu, E, d, f, (size_t)2 * f * d, 128, 256, 1, staging,
                      true);
        if (st == COLIBRI_OK)
            st = pack(1, qd->q, dev, h->q_d, E, f, d, (size_t)d * f, d, d, 0, staging, true);
        // block scales and zero points, one row per 64 packed weight rows:
        // gate/up [E][d/64][f/64] -> [E][f/128][2][2][d/64] (two 64-row blocks
        // of each 128-row gate or up slab), down [E][f/64][d/64] -> [E][d/64][f/64]
        const int bd = d / 64, bf = f / 64;
        const colibri_int8_weights_t* gu[2] = {qg, qu};
        for (int w = 0; w < 2 && st == COLIBRI_OK; ++w) {
            st = pack(4, gu[w]->scale, dev, h->sc_gu, E, bd, bf, 2 * nblk, 2, 4, w, staging);
            if (st == COLIBRI_OK)
                st = pack(4, gu[w]->zp, dev, h->zp_gu, E, bd, bf, 2 * nblk, 2, 4, w, staging);
        }
        if (st == COLIBRI_OK) st = pack(4, qd->scale, dev, h->sc_d, E, bf, bd, nblk, bd, bd, 0, staging);
        if (st == COLIBRI_OK) st = pack(4, qd->zp, dev, h->zp_d, E, bf, bd, nblk, bd, bd, 0, staging);
    }
    if (st != COLIBRI_OK) return fail_staged(st);
    if ((st = from_cuda(cudaDeviceSynchronize())) != COLIBRI_OK) return fail_staged(st);
    cudaFree(staging);
    staging = nullptr;

    // ---- workspace arena
    const int M = cfg->max_tokens;
    h->max_pairs = M * k;
    // the finest tiling is the decode GEMM's 32-row tiles
    h->max_tiles = (h->max_pairs + tc_gemm_dec_tile_rows() - 1) / tc_gemm_dec_tile_rows() +
                   std::min(E, h->max_pairs);
    h->grouped_ok = grouped_shape_ok(*cfg);
    if (cfg->executor == COLIBRI_EXEC_GROUPED && !h->grouped_ok) return fail(COLIBRI_ERR_UNSUPPORTED);
    const size_t P = (size_t)h->max_pairs;
    // Y: the down projection's float32 rows, or up to 8 K slices of them for
    // batches of at most kSplitMaxPairs pairs (kMaxKSplit for decode-sized
    // ones); the split gate/up partials of decode-sized batches reuse it.
    const size_t dec = std::min<size_t>(P, kGateUpSplitMaxPairs);
    const size_t y_floats =
        std::max({P * d, (size_t)8 * std::min<size_t>(P, kSplitMaxPairs) * d,
                  (size_t)kMaxKSplit * dec * std::max<size_t>(d, (size_t)2 * f)});
    const size_t gu_counter_bytes = (size_t)h->max_tiles * (f / 128) * 4;
    size_t off = 0;
    auto carve = [&](size_t bytes) {
        const size_t o = off;
        off += align256(bytes);
        return o;
    };
    const size_t o_idx = carve(P * 4), o_w = carve(P * 4), o_cnt = carve((size_t)E * 4),
                 o_kept = carve((size_t)E * 4),
                 o_off = carve((size_t)(E + 1) * 4), o_perm = carve(P * 4), o_inv = carve(P * 4),
                 o_te = carve((size_t)h->max_tiles * 4), o_tr = carve((size_t)h->max_tiles * 4),
                 o_tinfo = carve((size_t)h->max_tiles * 4), o_nt = carve(4), o_st = carve(4),
                 o_tk = carve(4), o_rp = carve(route_decode_part_floats(M, E) * 4),
                 o_bc = carve((size_t)dispatch_blocks(h->max_pairs) * E * 4),
                 o_xp = h->grouped_ok ? carve(P * d * h->esz) : 0, o_h = carve(P * f * h->esz),
                 o_y = carve(y_floats * 4), o_guc = carve(gu_counter_bytes),
                 o_u = carve((size_t)M * d * h->esz),
                 o_xs = carve((size_t)2 * M * d * h->esz), o_ys = carve((size_t)2 * M * d * h->esz);
    h->ws_bytes = off;
    if ((st = from_cuda(ac.alloc(&h->ws, off))) != COLIBRI_OK) return fail(st);
    uint8_t* b = (uint8_t*)h->ws;
    h->topk_idx = (int32_t*)(b + o_idx);
    h->topk_w = (float*)(b + o_w);
    h->counts = (int32_t*)(b + o_cnt);
    h->kept = (int32_t*)(b + o_kept);
    h->offsets = (int32_t*)(b + o_off);
    h->perm = (int32_t*)(b + o_perm);
    h->inv = (int32_t*)(b + o_inv);
    h->tile_expert = (int32_t*)(b + o_te);
    h->tile_row = (int32_t*)(b + o_tr);
    h->tile_info = (int32_t*)(b + o_tinfo);
    h->num_tiles = (int32_t*)(b + o_nt);
    h->status = (int*)(b + o_st);
    h->route_ticket = (unsigned int*)(b + o_tk);
    h->route_part = (float*)(b + o_rp);
    h->block_counts = (int32_t*)(b + o_bc);
    h->xp = h->grouped_ok ? (void*)(b + o_xp) : nullptr;
    h->H = b + o_h;
    h->Y = (float*)(b + o_y);
    h->y_floats = y_floats;
    h->gu_counter = (int32_t*)(b + o_guc);
    h->gu_counter_bytes = gu_counter_bytes;
    h->u = b + o_u;
    h->x_stage = b + o_xs;
    h->y_stage = b + o_ys;
    h->stage_bytes = (size_t)M * d * h->esz;
    if ((st = from_cuda(cudaMemset(h->ws, 0, off))) != COLIBRI_OK) return fail(st);
    // host-buffer forwards: copy streams and slot events (no timing)
    if ((st = from_cuda(cudaStreamCreateWithFlags(&h->cs_in, cudaStreamNonBlocking))) != COLIBRI_OK ||
        (st = from_cuda(cudaStreamCreateWithFlags(&h->cs_out, cudaStreamNonBlocking))) != COLIBRI_OK)
        return fail(st);
    for (int i = 0; i < 2; ++i)
        if ((st = from_cuda(cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming))) != COLIBRI_OK ||
            (st = from_cuda(cudaEventCreateWithFlags(&h->ev_done[i], cudaEventDisableTiming))) != COLIBRI_OK ||
            (st = from_cuda(cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming))) != COLIBRI_OK)
            return fail(st);

    if (h->grouped_ok) {
        // int8 handles: single-CTA tiles only, B maps over the int8 codes
        // int8 weights: Xp and H are f16 (the A type of the int8-weight GEMMs)
        bool ok = make_tmap_bf16(&h->tm_xp, h->xp, P, d, 128, int8) &&
                  make_tmap_bf16(&h->tm_h, h->H, P, f, 128, int8) &&
                  make_tmap_bf16(&h->tm_wr, h->wr, (uint64_t)h->e_pad, d, (uint32_t)h->e_pad);
        ok = ok && make_tmap_bf16(&h->tm_xp32, h->xp, P, d, (uint32_t)tc_gemm_dec_tile_rows(), int8) &&
             make_tmap_bf16(&h->tm_h32, h->H, P, f, (uint32_t)tc_gemm_dec_tile_rows(), int8);
        if (int8)
            // int8 codes are read by bulk copies of whole tiles (args.q_codes);
            // the weight tensor-map argument of those launches is not used
            h->tm_wgu1 = h->tm_xp, h->tm_wdT1 = h->tm_h;
        else
            ok = ok && make_tmap_bf16(&h->tm_wgu, h->wgu, (uint64_t)E * 2 * f, d, 128) &&
                 make_tmap_bf16(&h->tm_wdT, h->wdT, (uint64_t)E * d, f, 128) &&
                 make_tmap_bf16(&h->tm_wgu1, h->wgu, (uint64_t)E * 2 * f, d, 256) &&
                 make_tmap_bf16(&h->tm_wdT1, h->wdT, (uint64_t)E * d, f, 256) &&
                 make_tmap_token_rows(&h->tm_xp_rows, h->xp, P, d) &&
                 make_tmap_token_rows(&h->tm_h_rows, h->H, P, f);
        // the 5-D view is optional: without it gate/up stays token-on-M
        if (ok && !int8) h->wm_gate_up = make_tmap_gate_up_wm(&h->tm_wgu_wm, h->wgu, (uint64_t)E * 2 * f, d);
        if (!ok) {
            if (cfg->executor == COLIBRI_EXEC_GROUPED) return fail(COLIBRI_ERR_CUDA);
            h->grouped_ok = false;
        }
        h->max_resident_pairs = tc_gemm_max_pairs();
    }
    if ((st = from_cuda(cudaDeviceSynchronize())) != COLIBRI_OK) return fail(st);
    *out = h;
    return COLIBRI_OK;
}

}  // namespace

extern "C" {

colibri_status_t colibri_init(const colibri_moe_config_t* cfg, const void* w_router,
                              const float* router_bias, const void* w_gate, const void* w_up,
                              const void* w_down, int weights_on_device, colibri_moe_t** out) {
    return init_impl(cfg, w_router, router_bias, w_gate, w_up, w_down, nullptr, nullptr, nullptr,
                     weights_on_device, out);
}

colibri_status_t colibri_init_int8(const colibri_moe_config_t* cfg, const void* w_router,
                                   const float* router_bias, const colibri_int8_weights_t* w_gate,
                                   const colibri_int8_weights_t* w_up,
                                   const colibri_int8_weights_t* w_down, int weights_on_device,
                                   colibri_moe_t** out) {
    if (!w_gate) {
        if (out) *out = nullptr;
        return COLIBRI_ERR_INVALID_ARG;
    }
    return init_impl(cfg, w_router, router_bias, nullptr, nullptr, nullptr, w_gate, w_up, w_down,
                     weights_on_device, out);
}

colibri_status_t colibri_forward(colibri_moe_t* h, const void* x, int32_t T, void* y,
                                 void* stream) {
    if (!h || !x || !y || T < 0 || T > h->cfg.max_tokens) return COLIBRI_ERR_INVALID_ARG;
    if (((uintptr_t)x & 15) || ((uintptr_t)y & 15)) return COLIBRI_ERR_INVALID_ARG;
    const size_t bytes = (size_t)T * h->cfg.d_model * h->esz;
    if (T > 0 && ranges_overlap(x, bytes, y, bytes)) return COLIBRI_ERR_INVALID_ARG;
    if (T == 0) return COLIBRI_OK;
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return COLIBRI_ERR_CUDA;
    const colibri_status_t st = run_layer(h, x, T, y, nullptr, (cudaStream_t)stream);
    if (st != COLIBRI_OK && h->sticky == COLIBRI_OK) h->sticky = st;
    return st;
}

colibri_status_t colibri_forward_routed(colibri_moe_t* h, const void* x, int32_t T, int32_t k,
                                        const int32_t* topk_idx, const float* topk_w, void* y,
                                        void* stream) {
    if (!h || !x || !y || !topk_idx || !topk_w || T < 0 || k <= 0) return COLIBRI_ERR_INVALID_ARG;
    if ((int64_t)T * k > (int64_t)h->max_pairs) return COLIBRI_ERR_INVALID_ARG;
    if (((uintptr_t)x & 15) || ((uintptr_t)y & 15)) return COLIBRI_ERR_INVALID_ARG;
    const size_t bytes = (size_t)T * h->cfg.d_model * h->esz;
    if (T > 0 && ranges_overlap(x, bytes, y, bytes)) return COLIBRI_ERR_INVALID_ARG;
    if (T == 0) return COLIBRI_OK;
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return COLIBRI_ERR_CUDA;
    const colibri_status_t st =
        run_layer(h, x, T, y, nullptr, (cudaStream_t)stream, nullptr, 0.f, topk_idx, topk_w, k);
    if (st != COLIBRI_OK && h->sticky == COLIBRI_OK) h->sticky = st;
    return st;
}

colibri_status_t colibri_gather_rows(const void* x, int32_t x_rows, const int32_t* perm, int32_t k,
                                     int32_t npairs, int32_t d_model, int32_t dtype, void* xp,
                                     void* stream) {
    if (!x || !perm || !xp || x_rows < 0 || k <= 0 || npairs < 0 || d_model <= 0)
        return COLIBRI_ERR_INVALID_ARG;
    if ((int64_t)x_rows * k > INT32_MAX) return COLIBRI_ERR_INVALID_ARG;
    if (dtype != COLIBRI_DTYPE_FP32 && dtype != COLIBRI_DTYPE_BF16) return COLIBRI_ERR_INVALID_ARG;
    const int esz = dtype == COLIBRI_DTYPE_BF16 ? 2 : 4;
    if (((uintptr_t)x & 15) || ((uintptr_t)xp & 15) || (d_model * esz) % 16)
        return COLIBRI_ERR_INVALID_ARG;
    if (npairs == 0) return COLIBRI_OK;
    return from_cuda(
        launch_gather(esz, x, perm, k, d_model, npairs, x_rows * k, xp, (cudaStream_t)stream));
}

colibri_status_t colibri_combine_rows(const void* rows, int32_t rows_dtype, const float* topk_w,
                                      const int32_t* perm, int32_t T, int32_t k, int32_t d_model,
                                      int32_t dtype, int32_t* inv_scratch, void* y, void* stream) {
    if (!rows || !topk_w || !perm || !inv_scratch || !y || T < 0 || k <= 0 || d_model <= 0)
        return COLIBRI_ERR_INVALID_ARG;
    if (dtype != COLIBRI_DTYPE_FP32 && dtype != COLIBRI_DTYPE_BF16) return COLIBRI_ERR_INVALID_ARG;
    // float32 rows, or bf16 rows for a bf16 output
    if (rows_dtype != COLIBRI_DTYPE_FP32 && !(rows_dtype == COLIBRI_DTYPE_BF16 && dtype == COLIBRI_DTYPE_BF16))
        return COLIBRI_ERR_INVALID_ARG;
    if (((uintptr_t)rows & 15) || ((uintptr_t)y & 15) || d_model % 8) return COLIBRI_ERR_INVALID_ARG;
    if ((int64_t)T * k > INT32_MAX) return COLIBRI_ERR_INVALID_ARG;   // pair indices are int32
    if (T == 0) return COLIBRI_OK;
    const cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_invert_perm(perm, T * k, inv_scratch, s);
    if (e == cudaSuccess)
        e = launch_combine(dtype == COLIBRI_DTYPE_BF16 ? DType::BF16 : DType::F32,
                           static_cast<const float*>(rows), rows_dtype == COLIBRI_DTYPE_BF16, topk_w,
                           inv_scratch, T, k, d_model, 1, 0, nullptr, y, s);
    return from_cuda(e);
}

colibri_status_t colibri_forward_host_async(colibri_moe_t* h, const void* x_host, int32_t T,
                                            void* y_host, void* stream) {
    if (!h || !x_host || !y_host || T < 0 || T > h->cfg.max_tokens) return COLIBRI_ERR_INVALID_ARG;
    if (T == 0) return COLIBRI_OK;
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return COLIBRI_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const int slot = h->host_slot;
    h->host_slot ^= 1;
    uint8_t* xs = static_cast<uint8_t*>(h->x_stage) + slot * h->stage_bytes;
    uint8_t* ys = static_cast<uint8_t*>(h->y_stage) + slot * h->stage_bytes;
    const size_t bytes = (size_t)T * h->cfg.d_model * h->esz;
    // upload: the slot's x is free once the layer that read it two calls ago is done
    cudaError_t e = cudaStreamWaitEvent(h->cs_in, h->ev_done[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(xs, x_host, bytes, cudaMemcpyHostToDevice, h->cs_in);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_in[slot], h->cs_in);
    // the layer: x landed, and the slot's y downloaded by its previous call
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_in[slot], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_out[slot], 0);
    if (e != cudaSuccess) return from_cuda(e);
    const colibri_status_t st = run_layer(h, xs, T, ys, nullptr, s);
    if (st != COLIBRI_OK) return st;
    // download, after the layer
    e = cudaEventRecord(h->ev_done[slot], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->cs_out, h->ev_done[slot], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(y_host, ys, bytes, cudaMemcpyDeviceToHost, h->cs_out);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_out[slot], h->cs_out);
    return from_cuda(e);
}

colibri_status_t colibri_host_wait(colibri_moe_t* h) {
    if (!h) return COLIBRI_ERR_INVALID_ARG;
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return COLIBRI_ERR_CUDA;
    // every download is on cs_out and each follows its call's layer
    return from_cuda(cudaStreamSynchronize(h->cs_out));
}

colibri_status_t colibri_forward_host(colibri_moe_t* h, const void* x_host, int32_t T,
                                      void* y_host, void* stream) {
    const colibri_status_t st = colibri_forward_host_async(h, x_host, T, y_host, stream);
    if (st != COLIBRI_OK) return st;
    return colibri_host_wait(h);
}

colibri_status_t colibri_forward_stack_layer(colibri_moe_t* h, void* hidden, int32_t T,
                                             const void* gamma, float eps, void* stream) {
    if (!h || !hidden || !gamma || T < 0 || T > h->cfg.max_tokens || !(eps >= 0.0f))
        return COLIBRI_ERR_INVALID_ARG;
    if ((uintptr_t)hidden & 15) return COLIBRI_ERR_INVALID_ARG;
    if (T == 0) return COLIBRI_OK;
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return COLIBRI_ERR_CUDA;
    const colibri_status_t st =
        run_layer(h, hidden, T, hidden, hidden, (cudaStream_t)stream, gamma, eps);
    if (st != COLIBRI_OK && h->sticky == COLIBRI_OK) h->sticky = st;
    return st;
}

colibri_status_t colibri_get_routing(colibri_moe_t* h, int32_t* topk_idx, float* topk_w,
                                     int32_t* counts, int32_t* perm, void* stream) {
    if (!h) return COLIBRI_ERR_INVALID_ARG;
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return COLIBRI_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t P = (size_t)h->last_T * h->cfg.top_k;
    cudaError_t e = cudaSuccess;
    if (topk_idx && P && e == cudaSuccess)
        e = cudaMemcpyAsync(topk_idx, h->topk_idx, P * 4, cudaMemcpyDeviceToDevice, s);
    if (topk_w && P && e == cudaSuccess)
        e = cudaMemcpyAsync(topk_w, h->topk_w, P * 4, cudaMemcpyDeviceToDevice, s);
    if (counts && e == cudaSuccess)
        e = cudaMemcpyAsync(counts, h->counts, (size_t)h->cfg.n_experts * 4,
                            cudaMemcpyDeviceToDevice, s);
    if (perm && P && e == cudaSuccess)
        e = cudaMemcpyAsync(perm, h->perm, P * 4, cudaMemcpyDeviceToDevice, s);
    return from_cuda(e);
}

colibri_status_t colibri_set_executor(colibri_moe_t* h, int32_t executor) {
    if (!h || executor < COLIBRI_EXEC_AUTO || executor > COLIBRI_EXEC_GROUPED)
        return COLIBRI_ERR_INVALID_ARG;
    if (executor == COLIBRI_EXEC_GROUPED && !h->grouped_ok) return COLIBRI_ERR_UNSUPPORTED;
    h->cfg.executor = executor;
    return COLIBRI_OK;
}

colibri_status_t colibri_set_capacity(colibri_moe_t* h, int32_t capacity) {
    if (!h) return COLIBRI_ERR_INVALID_ARG;
    h->capacity = capacity < 0 ? -1 : capacity;
    return COLIBRI_OK;
}

colibri_status_t colibri_check(colibri_moe_t* h, void* stream) {
    if (!h) return COLIBRI_ERR_INVALID_ARG;
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return COLIBRI_ERR_CUDA;
    colibri_status_t st = h->sticky;
    h->sticky = COLIBRI_OK;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return COLIBRI_ERR_CUDA;
    e = cudaGetLastError();
    if (e != cudaSuccess && st == COLIBRI_OK) st = COLIBRI_ERR_CUDA;
    int dev_status = 0;
    e = cudaMemcpy(&dev_status, h->status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return COLIBRI_ERR_CUDA;
    if (dev_status != DEV_OK) {
        cudaMemset(h->status, 0, sizeof(int));
        // a launch that gave up may have left split gate/up counters armed
        cudaMemset(h->gu_counter, 0, h->gu_counter_bytes);
        cudaMemset(h->route_ticket, 0, sizeof(unsigned int));
        if (st == COLIBRI_OK) st = dev_status == DEV_TIMEOUT ? COLIBRI_ERR_TIMEOUT : COLIBRI_ERR_CUDA;
    }
    return st;
}

colibri_status_t colibri_profile_enable(colibri_moe_t* h, int enable) {
    if (!h) return COLIBRI_ERR_INVALID_ARG;
    DeviceGuard g(h->cfg.device);
    for (auto& r : h->recs) {
        cudaEventSynchronize(r.b);
        h->ev_pool.push_back(r.a);
        h->ev_pool.push_back(r.b);
    }
    h->recs.clear();
    h->prof = enable != 0;
    return COLIBRI_OK;
}

colibri_status_t colibri_profile_read(colibri_moe_t* h, double* total_ms, uint64_t* launches) {
    if (!h || !total_ms || !launches) return COLIBRI_ERR_INVALID_ARG;
    DeviceGuard g(h->cfg.device);
    for (int i = 0; i < COLIBRI_NUM_STAGES; ++i) total_ms[i] = 0.0, launches[i] = 0;
    colibri_status_t st = COLIBRI_OK;
    for (auto& r : h->recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess ||
            cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
            st = COLIBRI_ERR_CUDA;
        total_ms[r.stage] += ms;
        launches[r.stage] += 1;
        h->ev_pool.push_back(r.a);
        h->ev_pool.push_back(r.b);
    }
    h->recs.clear();
    return st;
}

colibri_status_t colibri_launch_count(const colibri_moe_t* h, uint64_t* n) {
    if (!h || !n) return COLIBRI_ERR_INVALID_ARG;
    *n = h->launches;
    return COLIBRI_OK;
}

colibri_status_t colibri_workspace_bytes(const colibri_moe_t* h, uint64_t* weights,
                                         uint64_t* workspace) {
    if (!h) return COLIBRI_ERR_INVALID_ARG;
    if (weights) *weights = h->weight_bytes;
    if (workspace) *workspace = h->ws_bytes;
    return COLIBRI_OK;
}

void colibri_free(colibri_moe_t* h) {
    if (!h) return;
    DeviceGuard g(h->cfg.device);
    cudaDeviceSynchronize();
    release(h);
}

}  // extern "C"
