"""ctypes binding of libnvfp4moe.so: argument marshalling only.

Every function here turns torch tensors into device pointers and sizes and
calls the C entry point of the same name; all arithmetic of the layer runs in
the library's CUDA kernels.  There is no fallback: if the library cannot be
loaded, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re

from .build import LIB, ROOT

STATUS = {
    0: "NVFP4_MOE_OK", 1: "NVFP4_MOE_ERR_INVALID_ARG", 2: "NVFP4_MOE_ERR_UNSUPPORTED_SHAPE",
    3: "NVFP4_MOE_ERR_NOT_PACKED", 4: "NVFP4_MOE_ERR_WORKSPACE", 5: "NVFP4_MOE_ERR_CUDA",
    6: "NVFP4_MOE_ERR_TIMEOUT", 7: "NVFP4_MOE_ERR_BAD_SCALE", 8: "NVFP4_MOE_ERR_NOT_IMPLEMENTED",
    9: "NVFP4_MOE_ERR_DEVICE_CHECK",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}
PATH_AUTO, PATH_DECODE, PATH_PREFILL = 0, 1, 2
SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1
HEADER = os.path.join(ROOT, "include", "nvfp4_moe.h")


class Nvfp4MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int), ("hidden", ctypes.c_int), ("inter", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("max_top_k", ctypes.c_int),
                ("decode_max_tokens", ctypes.c_int), ("logits_dtype", ctypes.c_int),
                ("device", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("num_shared_experts", ctypes.c_int)]


class LinearConfig(ctypes.Structure):
    _fields_ = [("out_features", ctypes.c_int), ("in_features", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("decode_max_tokens", ctypes.c_int), ("out_dtype", ctypes.c_int), ("device", ctypes.c_int)]


_lib = None


def header_functions():
    """Names of the functions include/nvfp4_moe.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(nvfp4_(?:moe|linear)_[a-z_0-9]+)\s*\(", text)))


def load_library(path: str | None = None):
    """Load libnvfp4moe.so (raises if it is missing or incomplete)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB
    if not os.path.exists(p):
        raise FileNotFoundError(f"{p} is missing: run __graft_entry__.build() (nvcc, sm_103a) first")
    lib = ctypes.CDLL(p)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sigs = {
        "nvfp4_moe_create": (i, [ctypes.POINTER(Config), ctypes.POINTER(vp)]),
        "nvfp4_moe_pack": (i, [vp, vp, vp, vp, vp, vp, vp]),
        "nvfp4_moe_forward": (i, [vp, vp, i, i, vp, vp, vp]),
        "nvfp4_moe_forward_host": (i, [vp, vp, i, i, vp, vp, vp]),
        "nvfp4_moe_get_status": (i, [vp, ctypes.POINTER(ctypes.c_uint32)]),
        "nvfp4_moe_set_path": (i, [vp, i]),
        "nvfp4_moe_status_string": (ctypes.c_char_p, [i]),
        "nvfp4_moe_last_error": (ctypes.c_char_p, [vp]),
        "nvfp4_moe_destroy": (None, [vp]),
        "nvfp4_moe_debug_route": (i, [vp, vp, i, i, vp, vp, vp, vp, vp]),
        "nvfp4_moe_debug_dequant": (i, [vp, i, i, vp, vp]),
        "nvfp4_moe_debug_intermediates": (i, [vp, vp, vp, vp]),
        "nvfp4_moe_debug_set_fault": (i, [vp, i]),
        "nvfp4_moe_set_profiling": (i, [vp, i]),
        "nvfp4_moe_debug_packed_blob": (i, [vp, vp, ctypes.c_size_t, vp]),
        "nvfp4_moe_forward_decode_static": (i, [vp, vp, i, i, i, vp, i, i, i, vp, vp, vp]),
        "nvfp4_moe_static_get_status": (i, [ctypes.POINTER(ctypes.c_uint32)]),
        "nvfp4_moe_static_debug_set_fault": (i, [i]),
        "nvfp4_moe_debug_poison_workspace": (i, [vp, i, vp]),
        "nvfp4_moe_decode_status_word": (i, [ctypes.c_uint32]),
        "nvfp4_moe_debug_trace": (i, [vp, ctypes.POINTER(ctypes.c_uint64), ctypes.c_size_t,
                                      ctypes.POINTER(ctypes.c_size_t)]),
        "nvfp4_moe_get_stage_times": (i, [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]),
        "nvfp4_moe_set_scoring": (i, [vp, i, i, f, vp, vp]),
        "nvfp4_moe_set_router": (i, [vp, vp, vp]),
        "nvfp4_moe_set_act_quant": (i, [vp, vp, vp]),
        "nvfp4_moe_forward_routed": (i, [vp, i, i, vp, vp, vp]),
        "nvfp4_moe_debug_logits": (i, [vp, vp, vp]),
        "nvfp4_linear_create": (i, [ctypes.POINTER(LinearConfig), ctypes.POINTER(vp)]),
        "nvfp4_linear_pack": (i, [vp, vp, vp, vp, vp]),
        "nvfp4_linear_forward": (i, [vp, i, vp, vp, vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _host_ptr(t):
    """A page-locked CPU tensor's address (the library checks that CUDA maps it)."""
    if t.is_cuda or not t.is_pinned():
        raise ValueError("expected a page-locked (pinned) CPU tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class MoELayer:
    """One handle of the library (nvfp4_moe_create ... nvfp4_moe_destroy)."""

    def __init__(self, num_experts, hidden, inter, max_tokens, max_top_k, decode_max_tokens=16,
                 logits_bf16=False, device=0, out_f32=False, num_shared_experts=0):
        self.lib = load_library()
        self.cfg = Config(num_experts, hidden, inter, max_tokens, max_top_k, decode_max_tokens,
                          1 if logits_bf16 else 0, device, 1 if out_f32 else 0, num_shared_experts)
        self.out_f32 = out_f32
        self.E, self.H, self.I = num_experts, hidden, inter
        self.S = num_shared_experts  # the shared expert is expert E of the blob
        self.device = device
        h = ctypes.c_void_p()
        st = self.lib.nvfp4_moe_create(ctypes.byref(self.cfg), ctypes.byref(h))
        if st != 0:
            raise Nvfp4MoeError(st, "nvfp4_moe_create: " + self.lib.nvfp4_moe_status_string(st).decode())
        self.h = h

    def _check(self, st, what):
        if st != 0:
            msg = self.lib.nvfp4_moe_last_error(self.h).decode()
            raise Nvfp4MoeError(st, f"{what}: {msg}")

    def close(self):
        if getattr(self, "h", None):
            self.lib.nvfp4_moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def nvfp4_moe_pack(self, w13_q, w13_s, w2_q, w2_s, gscale, stream=None):
        st = self.lib.nvfp4_moe_pack(self.h, _ptr(w13_q), _ptr(w13_s), _ptr(w2_q), _ptr(w2_s),
                                     _ptr(gscale), _stream(stream))
        self._check(st, "nvfp4_moe_pack")

    def nvfp4_moe_forward(self, logits, x, top_k, out, stream=None):
        T = x.shape[0]
        st = self.lib.nvfp4_moe_forward(self.h, _ptr(logits), T, top_k, _ptr(x), _ptr(out), _stream(stream))
        self._check(st, "nvfp4_moe_forward")
        return out

    def nvfp4_moe_forward_host(self, logits, x, top_k, out, stream=None):
        """nvfp4_moe_forward on pinned CPU tensors, read and written in place by the decode kernel."""
        T = x.shape[0]
        st = self.lib.nvfp4_moe_forward_host(self.h, _host_ptr(logits), T, top_k, _host_ptr(x), _host_ptr(out),
                                             _stream(stream))
        self._check(st, "nvfp4_moe_forward_host")
        return out

    def nvfp4_moe_forward_raw(self, logits_ptr, T, top_k, x_ptr, out_ptr, stream_handle):
        """Pointer-level call (for benchmarks that time the bare ABI)."""
        return self.lib.nvfp4_moe_forward(self.h, ctypes.c_void_p(logits_ptr), T, top_k, ctypes.c_void_p(x_ptr),
                                          ctypes.c_void_p(out_ptr), ctypes.c_void_p(stream_handle))

    def nvfp4_moe_get_status(self):
        n = ctypes.c_uint32(0)
        st = self.lib.nvfp4_moe_get_status(self.h, ctypes.byref(n))
        return st, int(n.value)

    def nvfp4_moe_set_path(self, path):
        self._check(self.lib.nvfp4_moe_set_path(self.h, path), "nvfp4_moe_set_path")

    def nvfp4_moe_debug_route(self, logits, T, top_k, stream=None):
        import torch
        dev = logits.device
        K = top_k + self.S  # slots per token; the shared expert's is last
        ids = torch.empty((T, K), dtype=torch.int32, device=dev)
        w = torch.empty((T, K), dtype=torch.float32, device=dev)
        off = torch.empty((self.E + self.S + 1,), dtype=torch.int32, device=dev)
        perm = torch.empty((T * K,), dtype=torch.int32, device=dev)
        st = self.lib.nvfp4_moe_debug_route(self.h, _ptr(logits), T, top_k, _ptr(ids), _ptr(w), _ptr(off),
                                            _ptr(perm), _stream(stream))
        self._check(st, "nvfp4_moe_debug_route")
        return ids, w, off, perm

    def nvfp4_moe_debug_trace(self):
        import numpy as np
        n = 152 * 16 * 16 * 4
        buf = (ctypes.c_uint64 * n)()
        got = ctypes.c_size_t(0)
        self._check(self.lib.nvfp4_moe_debug_trace(self.h, buf, n, ctypes.byref(got)), "nvfp4_moe_debug_trace")
        return np.frombuffer(buf, dtype=np.uint64)[:got.value].copy()

    def nvfp4_moe_debug_packed_blob(self, stream=None):
        import torch
        n = (self.E + self.S) * 3 * self.H * self.I * 9 // 16
        out = torch.empty((n,), dtype=torch.uint8, device=f"cuda:{self.device}")
        st = self.lib.nvfp4_moe_debug_packed_blob(self.h, _ptr(out), n, _stream(stream))
        self._check(st, "nvfp4_moe_debug_packed_blob")
        return out

    def nvfp4_moe_debug_dequant(self, expert, which, via_bf16=False, stream=None):
        import torch
        n, k = (self.H, self.I) if which == 2 else (self.I, self.H)
        out = torch.empty((n, k), dtype=torch.float32, device=f"cuda:{self.device}")
        st = self.lib.nvfp4_moe_debug_dequant(self.h, expert, which | (4 if via_bf16 else 0), _ptr(out),
                                              _stream(stream))
        self._check(st, "nvfp4_moe_debug_dequant")
        return out

    def nvfp4_moe_debug_intermediates(self, rows, stream=None):
        import torch
        hid = torch.empty((rows, self.I), dtype=torch.float32, device=f"cuda:{self.device}")
        y = torch.empty((rows, self.H), dtype=torch.float32, device=f"cuda:{self.device}")
        st = self.lib.nvfp4_moe_debug_intermediates(self.h, _ptr(hid), _ptr(y), _stream(stream))
        self._check(st, "nvfp4_moe_debug_intermediates")
        return hid, y

    def nvfp4_moe_set_profiling(self, on):
        self._check(self.lib.nvfp4_moe_set_profiling(self.h, 1 if on else 0), "nvfp4_moe_set_profiling")

    def nvfp4_moe_get_stage_times(self):
        ms = (ctypes.c_float * 4)()
        n = ctypes.c_int(0)
        self._check(self.lib.nvfp4_moe_get_stage_times(self.h, ms, ctypes.byref(n)), "nvfp4_moe_get_stage_times")
        return [float(v) for v in ms], int(n.value)

    def nvfp4_moe_set_scoring(self, score="softmax", renormalize=True, scale=1.0, bias=None, stream=None):
        """score: "softmax" | "sigmoid"; bias: a CUDA float32 tensor [num_experts] or None."""
        code = {"softmax": SCORE_SOFTMAX, "sigmoid": SCORE_SIGMOID}[score]
        st = self.lib.nvfp4_moe_set_scoring(self.h, code, 1 if renormalize else 0, float(scale), _ptr(bias),
                                            _stream(stream))
        self._check(st, "nvfp4_moe_set_scoring")

    def nvfp4_moe_set_act_quant(self, input_scale, stream=None):
        """input_scale: a CUDA float32 tensor [num_experts][2] (W4A4), or None (W4A16)."""
        st = self.lib.nvfp4_moe_set_act_quant(self.h, _ptr(input_scale), _stream(stream))
        self._check(st, "nvfp4_moe_set_act_quant")

    def nvfp4_moe_set_router(self, w_router, stream=None):
        """w_router: a CUDA BF16 tensor [num_experts][hidden]."""
        self._check(self.lib.nvfp4_moe_set_router(self.h, _ptr(w_router), _stream(stream)), "nvfp4_moe_set_router")

    def nvfp4_moe_forward_routed(self, x, top_k, out, stream=None):
        st = self.lib.nvfp4_moe_forward_routed(self.h, x.shape[0], top_k, _ptr(x), _ptr(out), _stream(stream))
        self._check(st, "nvfp4_moe_forward_routed")
        return out

    def nvfp4_moe_forward_routed_raw(self, T, top_k, x_ptr, out_ptr, stream_handle):
        """Pointer-level call (for benchmarks that time the bare ABI)."""
        return self.lib.nvfp4_moe_forward_routed(self.h, T, top_k, ctypes.c_void_p(x_ptr), ctypes.c_void_p(out_ptr),
                                                 ctypes.c_void_p(stream_handle))

    def nvfp4_moe_debug_logits(self, T, stream=None):
        import torch
        out = torch.empty((T, self.E), dtype=torch.float32, device=f"cuda:{self.device}")
        self._check(self.lib.nvfp4_moe_debug_logits(self.h, _ptr(out), _stream(stream)), "nvfp4_moe_debug_logits")
        return out

    def nvfp4_moe_debug_poison_workspace(self, byte=0xFF, stream=None):
        self._check(self.lib.nvfp4_moe_debug_poison_workspace(self.h, int(byte), _stream(stream)),
                    "nvfp4_moe_debug_poison_workspace")

    def nvfp4_moe_debug_set_fault(self, fault):
        self._check(self.lib.nvfp4_moe_debug_set_fault(self.h, fault), "nvfp4_moe_debug_set_fault")


class Linear(MoELayer):
    """A dense W4A16 NVFP4 linear handle (nvfp4_linear_create ... nvfp4_moe_destroy)."""

    def __init__(self, out_features, in_features, max_tokens, decode_max_tokens=16, device=0, out_f32=False):
        self.lib = load_library()
        self.cfg = LinearConfig(out_features, in_features, max_tokens, decode_max_tokens, 1 if out_f32 else 0, device)
        self.out_f32 = out_f32
        self.N, self.K = out_features, in_features
        self.device = device
        h = ctypes.c_void_p()
        st = self.lib.nvfp4_linear_create(ctypes.byref(self.cfg), ctypes.byref(h))
        if st != 0:
            raise Nvfp4MoeError(st, "nvfp4_linear_create: " + self.lib.nvfp4_moe_status_string(st).decode())
        self.h = h

    def nvfp4_linear_pack(self, w_q, w_s, gscale, stream=None):
        st = self.lib.nvfp4_linear_pack(self.h, _ptr(w_q), _ptr(w_s), _ptr(gscale), _stream(stream))
        self._check(st, "nvfp4_linear_pack")

    def nvfp4_linear_forward(self, x, out, stream=None):
        st = self.lib.nvfp4_linear_forward(self.h, x.shape[0], _ptr(x), _ptr(out), _stream(stream))
        self._check(st, "nvfp4_linear_forward")
        return out

    def nvfp4_linear_forward_raw(self, T, x_ptr, out_ptr, stream_handle):
        """Pointer-level call (for benchmarks that time the bare ABI)."""
        return self.lib.nvfp4_linear_forward(self.h, T, ctypes.c_void_p(x_ptr), ctypes.c_void_p(out_ptr),
                                             ctypes.c_void_p(stream_handle))

    def nvfp4_moe_debug_packed_blob(self, stream=None):
        import torch
        n = (self.N + 127) // 128 * 128 * self.K * 9 // 16  # rows padded to whole 128-row blocks
        out = torch.empty((n,), dtype=torch.uint8, device=f"cuda:{self.device}")
        st = self.lib.nvfp4_moe_debug_packed_blob(self.h, _ptr(out), n, _stream(stream))
        self._check(st, "nvfp4_moe_debug_packed_blob")
        return out


def nvfp4_moe_forward_decode_static(packed_experts, gscale, num_experts, hidden, inter, logits, top_k, x, out,
                                    logits_bf16=False, stream=None):
    """The allocation-free decode forward: every argument is caller memory."""
    lib = load_library()
    return lib.nvfp4_moe_forward_decode_static(_ptr(packed_experts), _ptr(gscale), num_experts, hidden, inter,
                                               _ptr(logits), 1 if logits_bf16 else 0, x.shape[0], top_k,
                                               _ptr(x), _ptr(out), _stream(stream))


def nvfp4_moe_static_get_status():
    """(status, nan_logits) of the allocation-free path on the current device
    (synchronous; reads and clears the status word)."""
    lib = load_library()
    n = ctypes.c_uint32(0)
    st = lib.nvfp4_moe_static_get_status(ctypes.byref(n))
    return st, int(n.value)


def nvfp4_moe_static_debug_set_fault(fault):
    return load_library().nvfp4_moe_static_debug_set_fault(int(fault))


def upload_layer(layer: MoELayer, weights, device="cuda:0"):
    """Copy an ExpertWeights-like set of numpy arrays to the device and pack it."""
    import torch
    t = lambda a: torch.from_numpy(a).to(device)
    layer.nvfp4_moe_pack(t(weights.w13_q), t(weights.w13_s), t(weights.w2_q), t(weights.w2_s), t(weights.gscale))
    torch.cuda.synchronize()
