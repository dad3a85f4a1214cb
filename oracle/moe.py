"""Plain float64 CPU oracle of one MoE layer forward (test infrastructure only).

Not part of the product: only ``tests/``, the smoke check and the benchmark's
CPU-baseline leg use it.

The layer, as the pages describe it (sources cited per function):

1. router logits      l = x . W_r (+ offset)             [T, E]
2. top-k              the k largest logits of each token
3. softmax            over the k selected logits only
4. dispatch           (token, slot) pairs grouped by expert
5. expert SwiGLU FFN  y_e = (silu(x W_g) * (x W_u)) W_d
6. combine            y[t] = sum_j g[t, j] * y_{e(t, j)}[t]

Readings where the pages are silent (each is also listed in the design notes):

* SwiGLU is ``down(silu(gate(x)) * up(x))`` with ``silu(z) = z / (1 + e^-z)``.
* Ties in top-k go to the lowest expert index; the k results come out in
  descending logit order.  NaN ranks below -inf.
* No learned router bias; an optional per-expert offset (Zipf skew or a
  -inf mask) is added to the logits before top-k and softmax.
* No capacity limit unless one is given; with a hard capacity C an expert
  accepts its pairs in token order, then slot order, up to C (capacity_keep).
* Arithmetic is float64 throughout; ``round_h`` optionally rounds the
  SwiGLU hidden activation to bfloat16 the way a bf16 tensor-core operand is.
"""

from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# bfloat16 <-> float64, written out from the format's definition
# (1 sign bit, 8 exponent bits, 7 stored mantissa bits: the upper half of an
# IEEE-754 binary32).


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exact."""
    b = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> bfloat16 bit patterns, one round-to-nearest-even step.

    A finite nonzero x is m * 2**ex with m in [0.5, 1); bfloat16 keeps 8
    significant bits, so the quantum is 2**(ex - 8), and never below the
    subnormal quantum 2**-133.  Rounding is ``np.rint`` (half to even) of the
    exactly scaled value; results of magnitude >= 2**128 become infinities.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(x) & (x != 0.0)
    out[~finite] = x[~finite]
    xf = x[finite]
    _, ex = np.frexp(xf)
    qexp = np.maximum(ex - 8, -133)
    q = np.rint(np.ldexp(xf, -qexp))
    r = np.ldexp(q, qexp)
    r[np.abs(r) >= 2.0 ** 128] = np.copysign(np.inf, xf[np.abs(r) >= 2.0 ** 128])
    out[finite] = r
    f32 = out.astype(np.float32)          # exact: r has <= 8 significant bits
    bits = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    bits[nan] = np.uint16(0x7FC0)
    return bits


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> nearest bfloat16 value (RNE), returned as float64."""
    return bf16_bits_to_f64(f64_to_bf16_bits(x))


def to_f64(t) -> np.ndarray:
    """A torch CPU tensor (float32 or bfloat16) or numpy array -> float64 numpy."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return bf16_bits_to_f64(t.view(torch.int16).numpy().view(np.uint16))
        return t.numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


# ----------------------------------------------------------------------------
# Steps 1-3: routing.


def router_logits(x: np.ndarray, w_router: np.ndarray, offset=None) -> np.ndarray:
    """Router logits l[t, e] = sum_i x[t, i] W_r[i, e] (+ offset[e]), float64.

    zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析" section 3.3, stage 2
    (routing kernel over the input and the router weights); lmnt.cn section
    2.2 (``route_tokens`` step 1, a dense layer giving [tokens, experts]);
    W_r is [hidden, experts] as in zskr.cn section 3.1's export script.
    """
    l = x @ w_router
    if offset is not None:
        l = l + np.asarray(offset, dtype=np.float64)[None, :]
    return l


def topk_select(l: np.ndarray, k: int) -> np.ndarray:
    """Indices [T, k] (int32) of the k largest logits of each row.

    lmnt.cn section 2.2 (``route_tokens`` step 2, top-k on the logits) and
    zskr.cn section 3.3 stage 2 (expert_indices [batch, top_k]).  Order: value
    descending, ties by ascending expert index, NaN below -inf.  Done by a
    full stable sort of every row: no partial selection.
    """
    T, E = l.shape
    idx = np.empty((T, k), dtype=np.int32)
    experts = np.arange(E)
    for t in range(T):
        row = l[t]
        nan = np.isnan(row)
        key = np.where(nan, 0.0, -row)
        order = np.lexsort((experts, key, nan))   # last key is primary
        idx[t] = order[:k]
    return idx


def softmax_selected(l: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Gate weights g[t, j] = softmax over the k selected logits, float64.

    lmnt.cn section 2.2 (``route_tokens`` step 3: softmax of the top-k logits,
    in place); zskr.cn section 3.3 stage 2 (expert_scores [batch, top_k]).
    The largest selected logit is subtracted first.
    """
    sel = np.take_along_axis(l, idx.astype(np.int64), axis=1)
    m = sel[:, :1]
    ex = np.exp(sel - m)
    return ex / ex.sum(axis=1, keepdims=True)


def soft_route(l: np.ndarray):
    """Dense-weighted ("soft") routing: (idx [T, E] int32, g [T, E] float64).

    m.nxbn.cn section 2.2: a Soft MoE router does not hard-select the top k
    but weights and fuses the outputs of all experts; soft_route() replaces
    hard_route() and the expert manager and executor stay as they are.
    Reading: every token goes to every expert, the j-th pair of a token is
    expert j (expert order), and the gate is the softmax over all E logits
    (the largest subtracted first).
    """
    T, E = l.shape
    idx = np.tile(np.arange(E, dtype=np.int32), (T, 1))
    m = l.max(axis=1, keepdims=True)
    ex = np.exp(l - m)
    return idx, ex / ex.sum(axis=1, keepdims=True)


# ----------------------------------------------------------------------------
# Step 4: dispatch.


def dispatch(idx: np.ndarray, n_experts: int):
    """Group the (token, slot) pairs by expert: a stable counting sort.

    zskr.cn section 3.3 stage 3 (dispatch_kernel packs every input slice of
    one expert into one mini-batch).  Pairs are numbered r = t*k + j.

    Returns ``counts[E]``, ``offsets[E+1]`` (exclusive prefix sum of counts),
    ``perm[T*k]`` with perm[p] = r for the p-th pair in expert order (pairs of
    one expert in increasing r), and ``inv[T*k]`` with inv[perm[p]] = p.
    """
    flat = idx.reshape(-1).astype(np.int64)
    counts = np.zeros(n_experts, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    for e in range(n_experts):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:-1].copy()
    perm = np.empty(flat.size, dtype=np.int64)
    for r, e in enumerate(flat):
        perm[fill[e]] = r
        fill[e] += 1
    inv = np.empty(flat.size, dtype=np.int64)
    inv[perm] = np.arange(flat.size)
    return counts, offsets, perm, inv


def capacity_keep(idx: np.ndarray, n_experts: int, capacity=None) -> np.ndarray:
    """Boolean [T, k]: the (token, slot) pairs their experts accept under a
    hard capacity of `capacity` pairs per expert (None: no limit).

    cf-1.com section 2.3 (an expert's capacity is the most tokens it handles in
    one batch) and section 4.2 (--expert-capacity is a hard limit: tokens past
    it are dropped); zskr.cn "Colibri：面向MoE架构的C语言高效推理引擎解析"
    section 2.2 (hard_capacity).  Reading: each expert accepts its pairs in
    increasing r = t*k + j (token order, then slot) until it holds `capacity`;
    a dropped pair adds nothing to its token's output and the other gates are
    left as they are.
    """
    T, k = idx.shape
    keep = np.ones((T, k), dtype=bool)
    if capacity is None:
        return keep
    held = np.zeros(n_experts, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            keep[t, j] = held[e] < capacity
            held[e] += 1
    return keep


# ----------------------------------------------------------------------------
# Step 5: the expert FFN.


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def swiglu_expert(xs: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray,
                  w_down: np.ndarray, round_h: bool = False) -> np.ndarray:
    """One expert on rows xs [n, d]: (silu(xs W_g) * (xs W_u)) W_d -> [n, d].

    zskr.cn section 3.3 stage 4 (gate_proj, up_proj, SiLU, down_proj fused
    per expert) and section 3.1 (the gate_proj / up_proj / down_proj weights
    of each expert).  W_g, W_u are [d, f]; W_d is [f, d].
    """
    h = silu(xs @ w_gate) * (xs @ w_up)
    if round_h:
        h = round_to_bf16(h)
    return h @ w_down


# ----------------------------------------------------------------------------
# Step 6: combine.


def combine(y_perm: np.ndarray, g: np.ndarray, inv: np.ndarray, keep=None) -> np.ndarray:
    """y[t] = sum_j g[t, j] * y_perm[inv[t*k + j]], j = 0..k-1 in order.

    zskr.cn section 3.3 stage 5 (aggregate_kernel adds every expert's output
    slice, weighted by its score, into the output buffer).  Pairs with
    keep[t, j] False (dropped by an expert's capacity) add nothing.
    """
    T, k = g.shape
    y = np.zeros((T, y_perm.shape[1]), dtype=np.float64)
    for j in range(k):
        rows = inv[np.arange(T) * k + j]
        w = g[:, j:j + 1] if keep is None else np.where(keep[:, j:j + 1], g[:, j:j + 1], 0.0)
        y += w * y_perm[rows]
    return y


# ----------------------------------------------------------------------------
# The whole layer.


def moe_layer(x, w_router, w_gate, w_up, w_down, top_k, offset=None,
              round_h=False, capacity=None, soft=False):
    """The full layer: logits, top-k, softmax, dispatch, experts, combine.

    pnsm.cn section 2.2 (one MoE forward: router logits, top-k indices,
    gather of the chosen experts, expert forward, gate-weighted sum) with the
    steps as zskr.cn section 3.3 stages 2-5 run them.  Arguments are float64
    arrays in the library's input layout: x [T,d], W_r [d,E],
    W_g/W_u [E,d,f], W_d [E,f,d].  `capacity` limits the pairs each expert
    accepts (capacity_keep).  `soft` routes every token to every expert
    (soft_route; top_k must equal E).
    """
    E = w_router.shape[1]
    l = router_logits(x, w_router, offset)
    if soft:
        if top_k != E:
            raise ValueError("soft routing takes every expert: top_k must equal E")
        idx, g = soft_route(l)
    else:
        idx = topk_select(l, top_k)
        g = softmax_selected(l, idx)
    counts, offsets, perm, inv = dispatch(idx, E)
    T = x.shape[0]
    y_perm = np.zeros((T * top_k, x.shape[1]), dtype=np.float64)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        rows = perm[lo:hi] // top_k
        y_perm[lo:hi] = swiglu_expert(x[rows], w_gate[e], w_up[e], w_down[e], round_h)
    keep = capacity_keep(idx, E, capacity)
    y = combine(y_perm, g, inv, keep)
    return {"logits": l, "topk_idx": idx, "topk_w": g, "counts": counts,
            "offsets": offsets, "perm": perm, "inv": inv, "keep": keep, "y": y}


def token_outputs(x_rows, idx_rows, g_rows, expert, round_h=False, keep_rows=None):
    """y for a few tokens given their routing: sum_j g_j * FFN_{idx_j}(x).

    The same sum as dispatch followed by combine, evaluated token by token,
    for checking sampled rows of a large layer.  ``expert(e)`` returns the
    float64 (W_g, W_u, W_d) of expert e; ``keep_rows`` (capacity_keep of the
    whole batch, rows of these tokens) drops pairs.
    """
    n, k = idx_rows.shape
    if keep_rows is not None:
        g_rows = np.where(keep_rows, g_rows, 0.0)
    y = np.zeros((n, x_rows.shape[1]), dtype=np.float64)
    for e in sorted(set(int(v) for v in idx_rows.reshape(-1))):
        wg, wu, wd = expert(e)
        for j in range(k):
            sel = np.nonzero(idx_rows[:, j] == e)[0]
            if sel.size:
                y[sel] += g_rows[sel, j:j + 1] * swiglu_expert(x_rows[sel], wg, wu, wd, round_h)
    return y


# ----------------------------------------------------------------------------
# Decode-step stack: RMSNorm before each MoE layer, residual add after it.


def rmsnorm(h: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """u = h / sqrt(mean(h^2) + eps) * gamma, per row (Zhang & Sennrich, 2019)."""
    ms = np.mean(h * h, axis=1, keepdims=True)
    return h / np.sqrt(ms + eps) * gamma[None, :]


def stack_layer(h_bf16, gamma, eps, w_router, w_gate, w_up, w_down, top_k,
                offset=None):
    """One layer of the decode stack: h + MoE(bf16(RMSNorm(h))), rounded to bf16.

    pnsm.cn section 2.2 (the residual add around the MoE block in the
    forward).  h is float64 holding bfloat16 values; the normalised input is
    rounded to bfloat16 (the layer's input type), the sum is formed in float64
    and rounded once to bfloat16.
    """
    u = round_to_bf16(rmsnorm(h_bf16, gamma, eps))
    out = moe_layer(u, w_router, w_gate, w_up, w_down, top_k, offset)
    out["h_out"] = round_to_bf16(h_bf16 + out["y"])
    out["u"] = u
    return out


# ----------------------------------------------------------------------------
# Parity helper: which tokens have a routing decision inside float noise.


def near_tie_tokens(x: np.ndarray, w_router: np.ndarray, l: np.ndarray, k: int,
                    rel: float = 2.0 ** -20) -> np.ndarray:
    """Boolean [T]: tokens whose top-k membership or order is a near-tie.

    Each logit gets an error radius tau[t, e] = rel * sum_i |x[t,i] W_r[i,e]|.
    With the logits sorted in descending order, a token is a near-tie when
    some adjacent pair among the first k+1 differs by less than the sum of
    their radii: float32 accumulation in another order could swap them.
    """
    tau = rel * (np.abs(x) @ np.abs(w_router))
    T, E = l.shape
    out = np.zeros(T, dtype=bool)
    m = min(k + 1, E)
    for t in range(T):
        row = np.where(np.isnan(l[t]), -np.inf, l[t])
        order = np.lexsort((np.arange(E), -row))
        for j in range(m - 1):
            a, b = order[j], order[j + 1]
            if not (np.isfinite(row[a]) and np.isfinite(row[b])):
                continue
            if abs(row[a] - row[b]) < tau[t, a] + tau[t, b]:
                out[t] = True
                break
    return out
