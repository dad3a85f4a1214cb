"""Python binding of the GB300 MoE layer library (``include/colibri_moe.h``).

Argument marshalling only: every step of the layer runs in the CUDA library
``libcolibri_moe.so`` built in-tree by ``sparse_expert_ffn_gb300.build``.
PyTorch supplies device memory and the current stream.  There is no fallback:
the library is loaded on first use, and if it is missing or fails to load that
first use raises ImportError.

The module exposes the C entry points under their C names (``colibri_init``,
``colibri_forward``, ...), each taking the same arguments as in C (ctypes
values, raw pointers), plus :class:`MoELayer`, a small owner of one handle
that accepts torch tensors.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcolibri_moe.so")

OK, ERR_INVALID_ARG, ERR_OOM, ERR_CUDA, ERR_UNSUPPORTED, ERR_TIMEOUT = range(6)
DTYPE_FP32, DTYPE_BF16 = 0, 1
EXEC_AUTO, EXEC_STREAM, EXEC_GROUPED = 0, 1, 2
_EXEC = {"auto": EXEC_AUTO, "stream": EXEC_STREAM, "grouped": EXEC_GROUPED}


class ColibriConfig(ctypes.Structure):
    _fields_ = [("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("device", ctypes.c_int32), ("executor", ctypes.c_int32)]


class ColibriInt8Weights(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("zp", ctypes.c_void_p)]


class ColibriError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {colibri_status_str(status)} (status {status})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m sparse_expert_ffn_gb300.build` "
            "(or __graft_entry__.build()); the layer has no non-CUDA implementation")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, U64P = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint64)
    sig = {
        "colibri_init": ([ctypes.POINTER(ColibriConfig), P, P, P, P, P, ctypes.c_int,
                          ctypes.POINTER(P)], I32),
        "colibri_init_int8": ([ctypes.POINTER(ColibriConfig), P, P,
                               ctypes.POINTER(ColibriInt8Weights), ctypes.POINTER(ColibriInt8Weights),
                               ctypes.POINTER(ColibriInt8Weights), ctypes.c_int, ctypes.POINTER(P)], I32),
        "colibri_quantize_int8_block64": ([P, I32, I32, I32, P, P, P], I32),
        "colibri_forward": ([P, P, I32, P, P], I32),
        "colibri_forward_host": ([P, P, I32, P, P], I32),
        "colibri_forward_host_async": ([P, P, I32, P, P], I32),
        "colibri_host_wait": ([P], I32),
        "colibri_forward_stack_layer": ([P, P, I32, P, ctypes.c_float, P], I32),
        "colibri_get_routing": ([P, P, P, P, P, P], I32),
        "colibri_set_executor": ([P, I32], I32),
        "colibri_set_capacity": ([P, I32], I32),
        "colibri_check": ([P, P], I32),
        "colibri_launch_count": ([P, U64P], I32),
        "colibri_workspace_bytes": ([P, U64P, U64P], I32),
        "colibri_profile_enable": ([P, ctypes.c_int], I32),
        "colibri_profile_read": ([P, ctypes.POINTER(ctypes.c_double), U64P], I32),
        "colibri_route_static": ([P, P, P, I32, I32, I32, I32, I32, P, P, P, P, P], I32),
        "colibri_forward_routed": ([P, P, I32, I32, P, P, P, P], I32),
        "colibri_gather_rows": ([P, I32, P, I32, I32, I32, I32, P, P], I32),
        "colibri_combine_rows": ([P, I32, P, P, I32, I32, I32, I32, P, P, P], I32),
        "colibri_free": ([P], None),
        "colibri_status_str": ([I32], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():  # noqa: B007
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = None
_C_NAMES = ("colibri_init", "colibri_init_int8", "colibri_quantize_int8_block64", "colibri_forward",
            "colibri_forward_host", "colibri_forward_host_async", "colibri_host_wait",
            "colibri_forward_stack_layer", "colibri_get_routing", "colibri_set_executor",
            "colibri_set_capacity",
            "colibri_check", "colibri_launch_count", "colibri_workspace_bytes",
            "colibri_profile_enable", "colibri_profile_read", "colibri_route_static",
            "colibri_forward_routed", "colibri_gather_rows", "colibri_combine_rows",
            "colibri_free")


def library():
    """The loaded ctypes library (loaded on first use; raises if it is not built)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def __getattr__(name):
    # The C entry points, under their C names, resolved from the library.
    if name in _C_NAMES:
        return getattr(library(), name)
    raise AttributeError(name)


def colibri_status_str(status: int) -> str:
    return library().colibri_status_str(int(status)).decode()


def _check(status: int, what: str):
    if status != OK:
        raise ColibriError(status, what)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def quantize_int8_block64(w):
    """The library's int8 converter on one [R, C] matrix or an [E, R, C] stack
    (float32 or bfloat16 torch tensor; copied to the host).  Returns CPU
    tensors (q int8, scale float32, zp int32) with scale/zp shaped
    [..., R/64, C/64] (the block format of ``colibri_init_int8``)."""
    import torch
    if w.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("weights must be float32 or bfloat16")
    wc = w.detach().to("cpu").contiguous()
    stack = wc.dim() == 3
    if not stack:
        wc = wc.unsqueeze(0)
    E, R, C = wc.shape
    q = torch.empty((E, R, C), dtype=torch.int8)
    sc = torch.empty((E, R // 64, C // 64), dtype=torch.float32)
    zp = torch.empty((E, R // 64, C // 64), dtype=torch.int32)
    dt = DTYPE_BF16 if wc.dtype == torch.bfloat16 else DTYPE_FP32
    for e in range(E):
        _check(library().colibri_quantize_int8_block64(_ptr(wc[e]), dt, R, C, _ptr(q[e]),
                                                       _ptr(sc[e]), _ptr(zp[e])),
               "colibri_quantize_int8_block64")
    if not stack:
        return q[0], sc[0], zp[0]
    return q, sc, zp


class MoELayer:
    """One MoE layer handle on one GPU.

    Weights (torch tensors, CPU or CUDA, float32 or bfloat16, all the same
    dtype) in the library's input layout: ``w_router`` [d, E],
    ``w_gate``/``w_up`` [E, d, f], ``w_down`` [E, f, d]; ``router_bias`` [E]
    float32 or None.  The library copies and repacks them; the caller may drop
    its tensors afterwards.
    """

    def __init__(self, w_router, w_gate, w_up, w_down, top_k: int, router_bias=None,
                 max_tokens: int = 4096, executor: str = "auto", device: Optional[int] = None,
                 int8=None):
        import torch
        if w_router.dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("weights must be float32 or bfloat16")
        if int8 is not None:
            # int8 expert weights: ((q, scale, zp) of gate, up, down) as made by
            # quantize_int8_block64; w_gate / w_up / w_down give only the shapes
            w_gate, w_up, w_down = (part[0] for part in int8)
            for part in int8:
                for t in part:
                    if t.device != w_router.device:
                        raise TypeError("int8 weights must be on the router's device")
        else:
            for w in (w_gate, w_up, w_down):
                if w.dtype != w_router.dtype or w.device != w_router.device:
                    raise TypeError("all weights must share dtype and device")
        E, d, f = w_gate.shape
        if tuple(w_router.shape) != (d, E) or tuple(w_up.shape) != (E, d, f) or \
                tuple(w_down.shape) != (E, f, d):
            raise ValueError("weight shapes do not match [d,E], [E,d,f], [E,d,f], [E,f,d]")
        if device is None:
            device = w_router.device.index if w_router.is_cuda else torch.cuda.current_device()
        self.device = torch.device("cuda", device)
        self.dtype = w_router.dtype
        self.E, self.d, self.f, self.k = E, d, f, int(top_k)
        self.max_tokens = int(max_tokens)
        on_dev = 1 if w_router.is_cuda else 0
        ws = [w_router.contiguous()] + ([None] * 3 if int8 is not None else
                                        [w.contiguous() for w in (w_gate, w_up, w_down)])
        bias = None
        if router_bias is not None:
            bias = router_bias.to(torch.float32).contiguous()
            if on_dev:
                bias = bias.to(self.device)
        cfg = ColibriConfig(E, self.k, d, f, self.max_tokens,
                            DTYPE_BF16 if self.dtype == torch.bfloat16 else DTYPE_FP32,
                            device, _EXEC[executor])
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            if int8 is None:
                st = library().colibri_init(ctypes.byref(cfg), _ptr(ws[0]), _ptr(bias),
                                            *[_ptr(w) for w in ws[1:]], on_dev, ctypes.byref(h))
            else:
                # int8 = ((q, scale, zp) of gate, up, down), each with the
                # float weight's layout and the router's device
                self._int8 = [tuple(t.contiguous() for t in part) for part in int8]
                iw = [ColibriInt8Weights(*[_ptr(t) for t in part]) for part in self._int8]
                st = library().colibri_init_int8(ctypes.byref(cfg), _ptr(ws[0]), _ptr(bias),
                                                 *[ctypes.byref(w) for w in iw], on_dev,
                                                 ctypes.byref(h))
                self._int8 = None
        _check(st, "colibri_init_int8" if int8 is not None else "colibri_init")
        self._h = h
        self.last_T = 0

    # -- calls -------------------------------------------------------------
    def forward(self, x, out=None, stream=None):
        """y = MoE(x) for x [T, d] on the handle's device (same dtype)."""
        import torch
        if x.dtype != self.dtype or x.device != self.device or x.dim() != 2 or x.shape[1] != self.d:
            raise ValueError("x must be [T, d_model] with the layer's dtype on its device")
        x = x.contiguous()
        if out is None:
            out = torch.empty_like(x)
        _check(library().colibri_forward(self._h, _ptr(x), x.shape[0], _ptr(out), _stream_ptr(stream)),
               "colibri_forward")
        self.last_T = x.shape[0]
        return out

    __call__ = forward

    def forward_routed(self, x, topk_idx, topk_w, out=None, stream=None):
        """y[t] = sum_j topk_w[t, j] * FFN_{topk_idx[t, j]}(x[t]) with the caller's
        routing (int32 ids of this handle's experts, float32 gates; [T] or [T, k])."""
        import torch
        if x.dtype != self.dtype or x.device != self.device or x.dim() != 2 or x.shape[1] != self.d:
            raise ValueError("x must be [T, d_model] with the layer's dtype on its device")
        T = x.shape[0]
        idx = topk_idx.reshape(T, -1).to(torch.int32).contiguous()
        w = topk_w.reshape(T, -1).to(torch.float32).contiguous()
        if idx.shape != w.shape:
            raise ValueError("topk_idx and topk_w must have the same shape")
        x = x.contiguous()
        if out is None:
            out = torch.empty_like(x)
        _check(library().colibri_forward_routed(self._h, _ptr(x), T, idx.shape[1], _ptr(idx), _ptr(w),
                                                _ptr(out), _stream_ptr(stream)),
               "colibri_forward_routed")
        return out

    def forward_host(self, x_host, y_host, stream=None):
        """The layer on host tensors (copies in, runs, copies out, waits)."""
        _check(library().colibri_forward_host(self._h, _ptr(x_host), x_host.shape[0], _ptr(y_host),
                                    _stream_ptr(stream)), "colibri_forward_host")
        self.last_T = x_host.shape[0]
        return y_host

    def forward_host_async(self, x_host, y_host, stream=None):
        """forward_host without the wait (pinned host tensors; successive calls
        overlap their copies with each other's layer).  y_host holds the result
        after host_wait(); x_host must not change before then."""
        _check(library().colibri_forward_host_async(self._h, _ptr(x_host), x_host.shape[0],
                                                    _ptr(y_host), _stream_ptr(stream)),
               "colibri_forward_host_async")
        self.last_T = x_host.shape[0]
        return y_host

    def host_wait(self):
        """Wait for every forward_host_async call on this layer."""
        _check(library().colibri_host_wait(self._h), "colibri_host_wait")

    def forward_stack_layer(self, hidden, gamma, eps: float, stream=None):
        """hidden <- hidden + MoE(RMSNorm(hidden) * gamma), in place."""
        if hidden.dtype != self.dtype or not hidden.is_contiguous():
            raise ValueError("hidden must be contiguous with the layer's dtype")
        _check(library().colibri_forward_stack_layer(self._h, _ptr(hidden), hidden.shape[0], _ptr(gamma),
                                                     float(eps), _stream_ptr(stream)),
               "colibri_forward_stack_layer")
        self.last_T = hidden.shape[0]
        return hidden

    def routing(self, stream=None):
        """The last forward's routing: dict of topk_idx, topk_w, counts, perm (device tensors)."""
        import torch
        T = self.last_T
        r = {
            "topk_idx": torch.empty((T, self.k), dtype=torch.int32, device=self.device),
            "topk_w": torch.empty((T, self.k), dtype=torch.float32, device=self.device),
            "counts": torch.empty((self.E,), dtype=torch.int32, device=self.device),
            "perm": torch.empty((T * self.k,), dtype=torch.int32, device=self.device),
        }
        _check(library().colibri_get_routing(self._h, _ptr(r["topk_idx"]), _ptr(r["topk_w"]),
                                   _ptr(r["counts"]), _ptr(r["perm"]), _stream_ptr(stream)),
               "colibri_get_routing")
        return r

    def set_executor(self, executor: str):
        _check(library().colibri_set_executor(self._h, _EXEC[executor]), "colibri_set_executor")

    def set_capacity(self, capacity: Optional[int]):
        """Hard per-expert capacity for later forwards (None: no limit)."""
        _check(library().colibri_set_capacity(self._h, -1 if capacity is None else int(capacity)),
               "colibri_set_capacity")

    def check(self, stream=None) -> int:
        """Wait for the stream; returns the library status (0 = OK)."""
        return library().colibri_check(self._h, _stream_ptr(stream))

    @property
    def launch_count(self) -> int:
        n = ctypes.c_uint64()
        _check(library().colibri_launch_count(self._h, ctypes.byref(n)), "colibri_launch_count")
        return n.value

    @property
    def bytes(self):
        w, s = ctypes.c_uint64(), ctypes.c_uint64()
        _check(library().colibri_workspace_bytes(self._h, ctypes.byref(w), ctypes.byref(s)),
               "colibri_workspace_bytes")
        return w.value, s.value

    @property
    def handle(self) -> int:
        return self._h.value

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            library().colibri_free(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
