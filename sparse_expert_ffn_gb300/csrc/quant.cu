// The int8 weight converter (host code): 64x64 blocks, each quantised from
// its own range.
//
// m.nxbn.cn section 3.1: the converter cuts every expert matrix into 64x64
// blocks and quantises each block on its own from its min and max into a
// weight buffer and a scale buffer.  pnsm.cn section 3.1: post-training
// min-max quantisation to [-127, 127], done on the CPU.  pnsm.cn section 5.2:
// dequantisation is (q - zp) * scale with an int32 zero point in [-127, 127].
//
// Per block: lo = min(min, 0), hi = max(max, 0); scale = float32((hi - lo) /
// 254) (1 for a block of zeros); zp = round(-127 - lo / scale); q =
// clamp(round(w / scale) + zp, -127, 127).  Every quotient is a double
// division by the float32 scale, rounded to nearest with ties to even
// (std::nearbyint in the default rounding mode): no product feeds a sum, so
// there is nothing for the compiler to contract.
#include <algorithm>
#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "colibri_moe.h"

namespace {

constexpr int kBlock = 64;
constexpr int kQMax = 127;

double weight_at(const void* w, int32_t dtype, size_t i) {
    if (dtype == COLIBRI_DTYPE_FP32) return (double)static_cast<const float*>(w)[i];
    const uint16_t b = static_cast<const uint16_t*>(w)[i];
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return (double)f;
}

}  // namespace

extern "C" colibri_status_t colibri_quantize_int8_block64(const void* w, int32_t dtype,
                                                          int32_t rows, int32_t cols, int8_t* q,
                                                          float* scale, int32_t* zp) {
    if (!w || !q || !scale || !zp) return COLIBRI_ERR_INVALID_ARG;
    if (dtype != COLIBRI_DTYPE_FP32 && dtype != COLIBRI_DTYPE_BF16) return COLIBRI_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0 || rows % kBlock || cols % kBlock) return COLIBRI_ERR_INVALID_ARG;
    if (std::fegetround() != FE_TONEAREST) return COLIBRI_ERR_INVALID_ARG;
    const size_t C = (size_t)cols;
    const int nbr = rows / kBlock, nbc = cols / kBlock;
    for (size_t i = 0; i < (size_t)rows * C; ++i)
        if (!std::isfinite(weight_at(w, dtype, i))) return COLIBRI_ERR_INVALID_ARG;
    // Blocks are independent: rows of blocks are shared out over the host
    // threads, and the result does not depend on how.
    auto rows_of_blocks = [&](int b0, int b1) {
    for (int bi = b0; bi < b1; ++bi) {
        for (int bj = 0; bj < nbc; ++bj) {
            double lo = 0.0, hi = 0.0;
            for (int r = 0; r < kBlock; ++r) {
                const size_t row = (size_t)(bi * kBlock + r) * C + (size_t)bj * kBlock;
                for (int c = 0; c < kBlock; ++c) {
                    const double v = weight_at(w, dtype, row + c);
                    lo = v < lo ? v : lo;
                    hi = v > hi ? v : hi;
                }
            }
            float s32 = 1.0f;
            int32_t z = 0;
            if (hi != lo) {
                s32 = (float)((hi - lo) / (double)(2 * kQMax));
                const double t = -(double)kQMax - lo / (double)s32;
                z = (int32_t)std::nearbyint(t);
            }
            const double s = (double)s32;
            for (int r = 0; r < kBlock; ++r) {
                const size_t row = (size_t)(bi * kBlock + r) * C + (size_t)bj * kBlock;
                for (int c = 0; c < kBlock; ++c) {
                    double code = std::nearbyint(weight_at(w, dtype, row + c) / s) + (double)z;
                    code = code < -kQMax ? -kQMax : (code > kQMax ? kQMax : code);
                    q[row + c] = (int8_t)code;
                }
            }
            scale[(size_t)bi * nbc + bj] = s32;
            zp[(size_t)bi * nbc + bj] = z;
        }
    }
    };
    const unsigned hw = std::thread::hardware_concurrency();
    const int nt = (int)std::min<unsigned>(hw ? hw : 1, (unsigned)nbr);
    if (nt <= 1 || (size_t)rows * C < ((size_t)1 << 20)) {
        rows_of_blocks(0, nbr);
        return COLIBRI_OK;
    }
    std::vector<std::thread> pool;
    const int per = (nbr + nt - 1) / nt;
    try {
        for (int t = 0; t < nt; ++t) {
            const int b0 = t * per, b1 = std::min(nbr, b0 + per);
            if (b0 < b1) pool.emplace_back(rows_of_blocks, b0, b1);
        }
    } catch (...) {
        for (auto& th : pool) th.join();
        return COLIBRI_ERR_OOM;
    }
    for (auto& th : pool) th.join();
    return COLIBRI_OK;
}
