"""Weight-only int8 expert weights: the oracle's quantiser and dequantiser
(test infrastructure only, like the rest of ``oracle``).

What the pages say about the format:

* m.nxbn.cn section 3.1 (weight format and model loading): the converter cuts
  every expert weight matrix into 64x64 blocks and quantises each block to
  int8 on its own, from the block's min and max, into a weight buffer and a
  scale buffer; the executor dequantises inside the GEMM.
* pnsm.cn section 3.1 (why FP16/INT8 mixed precision): post-training min-max
  quantisation scaled to [-127, 127], no quantisation-aware training; the
  conversion runs on the CPU.
* pnsm.cn section 5.2 ("output is all zeros"): dequantisation is
  (q - zp) * scale with an int32 zero point zp, which normally lies in
  [-127, 127].
* lmnt.cn section 3.1 (the converter's hidden details): int8 weights with a
  float32 scale, dequantised at inference time.

Readings where the pages leave a step open (also listed in the design notes):

1. Granularity: 64x64 blocks of each matrix (m.nxbn.cn), the finest of the
   pages' schemes and the one tied to the fused GEMM.  Rows and columns are
   multiples of 64, and the block grid is the same whichever way the matrix
   is stored (a transpose maps blocks onto blocks).
2. Levels: the 255 integers -127..127.  pnsm.cn states that range; its
   printed formula round((w - min) / (max - min) * 255 - 127) would give 128
   at w = max, outside both int8 and the stated range, so the step count is
   read as 254.
3. The block's range is widened to include 0: lo = min(min, 0),
   hi = max(max, 0).  Then zp = round(-127 - lo / scale) lies in [-127, 127]
   (as pnsm.cn section 5.2 expects) and w = 0 is exact.
4. scale = (hi - lo) / 254 rounded to float32 (the stored type); zp and q are
   computed from that float32 scale in float64 and rounded half to even;
   q is clamped to [-127, 127].  A block of zeros gets scale 1, zp 0.
5. Dequantised weight: (q - zp) * scale; |w - (q - zp) * scale| <= scale / 2
   (up to the float32 rounding of the scale).
"""

from __future__ import annotations

import numpy as np

BLOCK = 64
QMAX = 127


def quantize_int8_block64(w: np.ndarray):
    """[R, C] float weights -> (q int8 [R, C], scale float32 [R/64, C/64],
    zp int32 [R/64, C/64]), block by block (readings 1-4 above)."""
    w = np.asarray(w, dtype=np.float64)
    R, C = w.shape
    if R % BLOCK or C % BLOCK:
        raise ValueError("rows and columns must be multiples of 64")
    nb_r, nb_c = R // BLOCK, C // BLOCK
    q = np.empty((R, C), dtype=np.int8)
    scale = np.empty((nb_r, nb_c), dtype=np.float32)
    zp = np.empty((nb_r, nb_c), dtype=np.int32)
    for bi in range(nb_r):
        for bj in range(nb_c):
            blk = w[bi * BLOCK:(bi + 1) * BLOCK, bj * BLOCK:(bj + 1) * BLOCK]
            lo = min(float(blk.min()), 0.0)
            hi = max(float(blk.max()), 0.0)
            if hi == lo:                       # all zeros
                s32, z = np.float32(1.0), 0
            else:
                s32 = np.float32((hi - lo) / (2 * QMAX))
                z = int(np.rint(-QMAX - lo / np.float64(s32)))
            s = np.float64(s32)
            codes = np.rint(blk / s) + z
            q[bi * BLOCK:(bi + 1) * BLOCK, bj * BLOCK:(bj + 1) * BLOCK] = \
                np.clip(codes, -QMAX, QMAX).astype(np.int8)
            scale[bi, bj] = s32
            zp[bi, bj] = z
    return q, scale, zp


def dequantize_int8_block64(q: np.ndarray, scale: np.ndarray, zp: np.ndarray) -> np.ndarray:
    """(q - zp) * scale per 64x64 block, in float64 (pnsm.cn section 5.2)."""
    q = np.asarray(q).astype(np.float64)
    s = np.repeat(np.repeat(np.asarray(scale, dtype=np.float64), BLOCK, 0), BLOCK, 1)
    z = np.repeat(np.repeat(np.asarray(zp, dtype=np.float64), BLOCK, 0), BLOCK, 1)
    return (q - z) * s


def quantize_experts(w: np.ndarray):
    """[E, R, C] expert stack -> (q [E, R, C], scale [E, R/64, C/64], zp [E, R/64, C/64])."""
    parts = [quantize_int8_block64(w[e]) for e in range(w.shape[0])]
    return (np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]),
            np.stack([p[2] for p in parts]))


def dequantize_experts(q, scale, zp) -> np.ndarray:
    return np.stack([dequantize_int8_block64(q[e], scale[e], zp[e]) for e in range(q.shape[0])])
