"""ctypes binding of libpi.  Argument marshalling only.

Tensors are passed by ``data_ptr()``; streams by ``torch.cuda.Stream.cuda_stream``
(default: the current stream).  Output tensors the caller does not supply are
allocated with torch on the input's device; every computation happens inside
libpi's kernels.
"""
from __future__ import annotations

import ctypes as C
from pathlib import Path
from typing import Optional

import numpy as np
import torch

import os

_HERE = Path(__file__).resolve().parent
lib_path = Path(os.environ.get("PI_LIB_PATH", str(_HERE / "_lib" / "libpi.so")))

if not lib_path.exists():
    raise ImportError(
        f"libpi.so not found at {lib_path}; build it with "
        "`python activation_sparse_rank_gb300/_build.py` (no CPU fallback exists)")

lib = C.CDLL(str(lib_path))

PI_OK = 0
PI_ACT_RELU = 0
PI_ACT_REGLU = 1
PI_ACT_SWIGLU = 2
_ACTS = {"relu": PI_ACT_RELU, "reglu": PI_ACT_REGLU, "swiglu": PI_ACT_SWIGLU}
PI_MAX_BATCH = 128
PI_STACK_LAYERS_PER_LAUNCH = 32   # include/pi.h
PI_ROWS_FP16 = 0
PI_ROWS_FP8_E4M3 = 1

_p = C.c_void_p
_i32 = C.c_int32


class pi_layer_desc(C.Structure):
    _fields_ = [("d", _i32), ("ffn", _i32), ("rank", _i32), ("act", _i32),
                ("W_up", _p), ("W_gate", _p), ("b", _p), ("W_down", _p),
                ("W_p1", _p), ("W_p2", _p), ("c_p", _p), ("row_format", _i32)]


_SIG = {
    "pi_layer_create": (C.c_int, [C.POINTER(_p), C.POINTER(pi_layer_desc), _p, _p]),
    "pi_layer_destroy": (C.c_int, [_p]),
    "pi_layer_info": (C.c_int, [_p, _p, _p, _p, _p]),
    "pi_layer_perm": (C.c_int, [_p, _p]),
    "pi_layer_rows_fp8": (C.c_int, [_p, _i32, _p, _p, _p]),
    "pi_workspace_bytes": (C.c_size_t, [_p, _i32]),
    "pi_predict": (C.c_int, [_p, _p, _i32, _p, _p, _p, C.c_size_t, _p]),
    "pi_compact_active": (C.c_int, [_p, _p, _i32, _p, _p, _p]),
    "pi_sparse_ffn": (C.c_int, [_p, _p, _i32, _p, _p, _p, _p, C.c_size_t, _p]),
    "pi_sparse_ffn_noalloc": (C.c_int, [_p, _p, _i32, _p, _p, _p, _p]),
    "pi_ffn_dense_ref": (C.c_int, [_p, _p, _i32, _p, _p, C.c_size_t, _p]),
    "pi_layer_forward": (C.c_int, [_p, _p, _i32, _p, _p, _p, _p, C.c_size_t, _p]),
    "pi_stack_forward": (C.c_int, [_p, _i32, _p, _i32, _p, _p, _p, _p, C.c_size_t, _p]),
    "pi_stack_forward_chained": (C.c_int, [_p, _i32, _p, _i32, _p, _p, _p, _p, C.c_size_t, _p]),
    "pi_stack_forward_host": (C.c_int, [_p, _i32, _i32, _p, _i32, _p, _p, _p, _p, _p, _i32, _p,
                                        C.c_size_t, _p]),
    "pi_profile_activations": (C.c_int, [C.POINTER(pi_layer_desc), _p, _i32, _p, _p]),
    "pi_hot_first_perm": (C.c_int, [_p, _i32, _p]),
    "pi_device_status": (C.c_int, [_p, _p]),
    "pi_layer_set_timing_events": (C.c_int, [_p, _p, _p]),
    "pi_forward_launches": (C.c_int32, [_p, _i32]),
    "pi_layer_set_hot_count": (C.c_int, [_p, _i32]),
    "pi_last_error": (C.c_char_p, []),
    "pi_status_string": (C.c_char_p, [C.c_int]),
}
for _name, (_res, _args) in _SIG.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class PiError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = lib.pi_status_string(status).decode()
        msg = lib.pi_last_error().decode()
        super().__init__(f"{where}: {name}: {msg}")


def _check(st: int, where: str):
    if st != PI_OK:
        raise PiError(st, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _req(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def make_desc(W_up, W_gate, b, W_down, W_p1, W_p2, c_p, act, rows="fp16") -> pi_layer_desc:
    act_id = act if isinstance(act, int) else _ACTS.get(act)
    if act_id not in _ACTS.values():
        raise ValueError(f"act must be one of {sorted(_ACTS)}, not {act!r}")
    _req(W_up, torch.float16, "W_up")
    ffn, d = W_up.shape
    rank = W_p1.shape[0]
    for t, n in ((W_down, "W_down"), (W_p1, "W_p1"), (W_p2, "W_p2")):
        _req(t, torch.float16, n)
    _req(b, torch.float32, "b")
    if W_gate is not None:
        _req(W_gate, torch.float16, "W_gate")
    if c_p is not None:
        _req(c_p, torch.float32, "c_p")
    if rows not in ("fp16", "fp8"):
        raise ValueError(f"rows must be 'fp16' or 'fp8', not {rows!r}")
    return pi_layer_desc(d, ffn, rank, act_id, W_up.data_ptr(),
                         None if W_gate is None else W_gate.data_ptr(), b.data_ptr(),
                         W_down.data_ptr(), W_p1.data_ptr(), W_p2.data_ptr(),
                         None if c_p is None else c_p.data_ptr(),
                         PI_ROWS_FP8_E4M3 if rows == "fp8" else PI_ROWS_FP16)


class Layer:
    """A layer object of libpi (library-owned, permuted, neuron-major weights)."""

    def __init__(self, W_up, W_gate, b, W_down, W_p1, W_p2, c_p=None, act="relu",
                 perm=None, stream=None, rows="fp16"):
        desc = make_desc(W_up, W_gate, b, W_down, W_p1, W_p2, c_p, act, rows)
        self._h = C.c_void_p()
        perm_arr = None
        if perm is not None:
            perm_arr = np.ascontiguousarray(np.asarray(perm, dtype=np.int32))
        _check(lib.pi_layer_create(C.byref(self._h), C.byref(desc),
                                   None if perm_arr is None else perm_arr.ctypes.data_as(C.c_void_p),
                                   _stream(stream)), "pi_layer_create")
        self.d, self.ffn, self.rank = int(desc.d), int(desc.ffn), int(desc.rank)
        self.act = {v: k for k, v in _ACTS.items()}[int(desc.act)]
        self.rows = rows
        self.device = W_up.device

    @classmethod
    def from_dict(cls, t: dict, perm=None, stream=None, rows="fp16") -> "Layer":
        return cls(t["W_up"], t.get("W_gate"), t["b"], t["W_down"], t["W_p1"], t["W_p2"],
                   t.get("c_p"), t.get("act", "relu"), perm=perm, stream=stream, rows=rows)

    @property
    def handle(self) -> C.c_void_p:
        return self._h

    def close(self):
        if self._h:
            _check(lib.pi_layer_destroy(self._h), "pi_layer_destroy")
            self._h = C.c_void_p()

    def __del__(self):
        try:
            if self._h:
                lib.pi_layer_destroy(self._h)
        except Exception:
            pass

    def rows_fp8(self, matrix: int, stream=None):
        """Stored E4M3 codes (uint8 [ffn, d]) and row scales (fp32 [ffn]) of
        matrix 0 (up), 1 (gate) or 2 (down^T), in storage order."""
        codes = torch.empty(self.ffn, self.d, dtype=torch.uint8, device=self.device)
        scales = torch.empty(self.ffn, dtype=torch.float32, device=self.device)
        _check(lib.pi_layer_rows_fp8(self._h, int(matrix), _ptr(codes), _ptr(scales), _stream(stream)),
               "pi_layer_rows_fp8")
        return codes, scales

    def perm(self) -> np.ndarray:
        out = np.empty(self.ffn, dtype=np.int32)
        _check(lib.pi_layer_perm(self._h, out.ctypes.data_as(C.c_void_p)), "pi_layer_perm")
        return out

    def workspace_bytes(self, B: int) -> int:
        n = lib.pi_workspace_bytes(self._h, int(B))
        if n == 0:
            raise PiError(1, "pi_workspace_bytes")
        return int(n)

    def workspace(self, B: int) -> torch.Tensor:
        return torch.empty(self.workspace_bytes(B), dtype=torch.uint8, device=self.device)

    def _ws(self, ws, B):
        if ws is None:
            ws = self.workspace(B)
        return ws

    def predict(self, x, mask=None, logits=None, want_mask=True, want_logits=False, ws=None,
                stream=None):
        _req(x, torch.float16, "x")
        B = x.shape[0] if x.dim() == 2 else 1
        if mask is None and want_mask:
            mask = torch.empty(B, self.ffn, dtype=torch.uint8, device=x.device)
        if logits is None and want_logits:
            logits = torch.empty(B, self.ffn, dtype=torch.float32, device=x.device)
        ws = self._ws(ws, B)
        _check(lib.pi_predict(self._h, _ptr(x), B, _ptr(mask), _ptr(logits), _ptr(ws),
                              ws.numel(), _stream(stream)), "pi_predict")
        return mask, logits

    def compact(self, mask, idx=None, count=None, stream=None):
        _req(mask, torch.uint8, "mask")
        B = mask.shape[0] if mask.dim() == 2 else 1
        if idx is None:
            idx = torch.empty(self.ffn, dtype=torch.int32, device=mask.device)
        if count is None:
            count = torch.empty(1, dtype=torch.int32, device=mask.device)
        _check(lib.pi_compact_active(self._h, _ptr(mask), B, _ptr(idx), _ptr(count),
                                     _stream(stream)), "pi_compact_active")
        return idx, count

    def sparse_ffn(self, x, idx, count, y=None, ws=None, stream=None):
        _req(x, torch.float16, "x")
        B = x.shape[0] if x.dim() == 2 else 1
        if y is None:
            y = torch.empty(B, self.d, dtype=torch.float32, device=x.device)
        ws = self._ws(ws, B)
        _check(lib.pi_sparse_ffn(self._h, _ptr(x), B, _ptr(idx), _ptr(count), _ptr(y),
                                 _ptr(ws), ws.numel(), _stream(stream)), "pi_sparse_ffn")
        return y

    def dense_ref(self, x, y=None, ws=None, stream=None):
        _req(x, torch.float16, "x")
        B = x.shape[0] if x.dim() == 2 else 1
        if y is None:
            y = torch.empty(B, self.d, dtype=torch.float32, device=x.device)
        ws = self._ws(ws, B)
        _check(lib.pi_ffn_dense_ref(self._h, _ptr(x), B, _ptr(y), _ptr(ws), ws.numel(),
                                    _stream(stream)), "pi_ffn_dense_ref")
        return y

    def forward(self, x, idx=None, count=None, y=None, ws=None, stream=None):
        _req(x, torch.float16, "x")
        B = x.shape[0] if x.dim() == 2 else 1
        if idx is None:
            idx = torch.empty(self.ffn, dtype=torch.int32, device=x.device)
        if count is None:
            count = torch.empty(1, dtype=torch.int32, device=x.device)
        if y is None:
            y = torch.empty(B, self.d, dtype=torch.float32, device=x.device)
        ws = self._ws(ws, B)
        _check(lib.pi_layer_forward(self._h, _ptr(x), B, _ptr(idx), _ptr(count), _ptr(y),
                                    _ptr(ws), ws.numel(), _stream(stream)), "pi_layer_forward")
        return y, idx, count

    def set_timing_events(self, before=None, after=None):
        """Record torch.cuda.Event `before`/`after` around the main up/down kernel
        of subsequent calls (None, None switches it off)."""
        b = None if before is None else C.c_void_p(before.cuda_event)
        a = None if after is None else C.c_void_p(after.cuda_event)
        _check(lib.pi_layer_set_timing_events(self._h, b, a), "pi_layer_set_timing_events")

    def set_hot_count(self, n_hot: int):
        """Number of leading neurons of the creation order treated as hot."""
        _check(lib.pi_layer_set_hot_count(self._h, int(n_hot)), "pi_layer_set_hot_count")

    def forward_launches(self, B: int) -> int:
        return int(lib.pi_forward_launches(self._h, int(B)))

    def device_status(self, stream=None) -> int:
        """0 if no kernel flagged bad input since the last query, else the status code."""
        return int(lib.pi_device_status(self._h, _stream(stream)))


def stack_forward(layers, x, y, idx=None, count=None, ws=None, stream=None, handles=None,
                  chained=False):
    """Run layers in order on x [n_layers, B, d] fp16 into y [n_layers, B, d] fp32.
    chained: only x[0] is an input; x[l] for l >= 1 is overwritten with
    fp16(y[l-1] / RMS(y[l-1])) before layer l runs (pi_stack_forward_chained).
    `handles` may carry a prebuilt ctypes array of the layer handles."""
    n = len(layers)
    _req(x, torch.float16, "x")
    B = x.shape[1]
    if handles is None:
        handles = (C.c_void_p * n)(*[l.handle.value for l in layers])
    if ws is None:
        ws = layers[0].workspace(B)
    fn, name = ((lib.pi_stack_forward_chained, "pi_stack_forward_chained") if chained
                else (lib.pi_stack_forward, "pi_stack_forward"))
    _check(fn(handles, n, _ptr(x), B, _ptr(idx), _ptr(count), _ptr(y), _ptr(ws), ws.numel(),
              _stream(stream)), name)
    return y


def stack_forward_host(layers, x_host, y_host, x_dev, y_dev, idx=None, count=None, ws=None,
                       stream=None, handles=None, chained=False):
    """T decode steps from host buffers in one library call: x_host [T, L, B, d]
    fp16 (pinned) is copied into x_dev, each token runs through the stack, and
    y_dev is copied into y_host [T, L, B, d] fp32 (pi_stack_forward_host)."""
    if x_host.is_cuda or y_host.is_cuda:
        raise TypeError("x_host and y_host must be host tensors")
    _req(x_dev, torch.float16, "x_dev")
    _req(y_dev, torch.float32, "y_dev")
    if not (x_host.is_contiguous() and y_host.is_contiguous()):
        raise ValueError("x_host and y_host must be contiguous")
    if x_host.dtype != torch.float16 or y_host.dtype != torch.float32:
        raise TypeError("x_host must be float16 and y_host float32")
    T, n, B = int(x_host.shape[0]), len(layers), int(x_host.shape[2])
    if x_host.shape != x_dev.shape or y_host.shape != y_dev.shape or tuple(x_host.shape[:2]) != (T, n):
        raise ValueError("x_host/x_dev/y_host/y_dev must all be [T, n_layers, B, d]")
    if handles is None:
        handles = (C.c_void_p * n)(*[l.handle.value for l in layers])
    if ws is None:
        ws = layers[0].workspace(B)
    _check(lib.pi_stack_forward_host(handles, n, T, C.c_void_p(x_host.data_ptr()), B,
                                     C.c_void_p(y_host.data_ptr()), _ptr(x_dev), _ptr(y_dev), _ptr(idx),
                                     _ptr(count), 1 if chained else 0, _ptr(ws), ws.numel(), _stream(stream)),
           "pi_stack_forward_host")
    return y_host


def profile_activations(t: dict, x: torch.Tensor, counts: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """Accumulate per-neuron exact activation counts over the tokens x [T, d]
    into counts (int32 [ffn], zero-initialised if not given)."""
    desc = make_desc(t["W_up"], t.get("W_gate"), t["b"], t["W_down"], t["W_p1"], t["W_p2"],
                     t.get("c_p"), t.get("act", "relu"))
    _req(x, torch.float16, "x")
    if counts is None:
        counts = torch.zeros(desc.ffn, dtype=torch.int32, device=x.device)
    _check(lib.pi_profile_activations(C.byref(desc), _ptr(x), int(x.shape[0]), _ptr(counts),
                                      _stream(stream)), "pi_profile_activations")
    return counts


def hot_first_perm(counts) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
    out = np.empty(c.shape[0], dtype=np.int32)
    _check(lib.pi_hot_first_perm(c.ctypes.data_as(C.c_void_p), c.shape[0],
                                 out.ctypes.data_as(C.c_void_p)), "pi_hot_first_perm")
    return out
