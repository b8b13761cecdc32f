"""ctypes binding of libmoeblaze.so: the C entry points under the same names
(argument marshalling only), plus small torch helpers that allocate the
caller-owned buffers and pass their device pointers and the current stream.

Every compute step runs in the library's CUDA kernels; there is no Python or
CPU fallback.  Loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoeblaze.so")
_lib = None

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_BAD_ROUTING, ERR_WORKSPACE, ERR_TIMEOUT, ERR_CUDA = range(7)
F32, BF16 = 0, 1
SWIGLU, SILU, IDENTITY = 0, 1, 2
ACT = {"swiglu": SWIGLU, "silu": SILU, "identity": IDENTITY}
DTYPE = {torch.float32: F32, torch.bfloat16: BF16}

# names exported by include/moeblaze.h
EXPORTS = [
    "moeblaze_dispatch_meta_bytes", "moeblaze_dispatch_workspace_bytes", "moeblaze_saved_bytes",
    "moeblaze_forward_workspace_bytes", "moeblaze_backward_workspace_bytes", "moeblaze_dispatch_build",
    "moeblaze_forward", "moeblaze_backward", "moeblaze_device_error", "moeblaze_status_string",
    "moeblaze_version", "moeblaze_set_stage_events", "moeblaze_kernel_launches",
    "moeblaze_dispatch_build_static", "moeblaze_dispatch_meta_check", "moeblaze_set_fault_injection",
    "moeblaze_router_forward", "moeblaze_router_backward", "moeblaze_router_backward_workspace_bytes",
    "moeblaze_router_dispatch_workspace_bytes", "moeblaze_router_dispatch_build",
]

# fixed scratch of moeblaze_dispatch_build_static (MOEBLAZE_STATIC_SCRATCH_BYTES)
STATIC_SCRATCH_BYTES = 8 << 20


class Shape(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int64), ("d", ctypes.c_int32), ("h", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("dtype", ctypes.c_int32), ("act", ctypes.c_int32), ("flags", ctypes.c_int32)]


# moeblaze_shape.flags
RECOMPUTE_H = 1


class Dispatch(ctypes.Structure):
    _fields_ = [("expert_token_indices", ctypes.c_void_p), ("expert_token_offsets", ctypes.c_void_p),
                ("token_expert_indices", ctypes.c_void_p), ("token_index_map", ctypes.c_void_p),
                ("meta", ctypes.c_void_p)]


class MoEBlazeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib():
    """The loaded library; raises if it is missing (build it first)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libmoeblaze.so not built ({_LIB_PATH}); run "
                               "`python -m mixture_experts_atomic_gb300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        sz = ctypes.c_size_t
        P = ctypes.c_void_p
        SP = ctypes.POINTER(Shape)
        DP = ctypes.POINTER(Dispatch)
        for n in ["moeblaze_dispatch_meta_bytes", "moeblaze_dispatch_workspace_bytes", "moeblaze_saved_bytes",
                  "moeblaze_forward_workspace_bytes", "moeblaze_backward_workspace_bytes"]:
            getattr(L, n).argtypes = [SP]
            getattr(L, n).restype = sz
        L.moeblaze_dispatch_build.argtypes = [SP, P, DP, P, sz, ctypes.c_int, P]
        L.moeblaze_dispatch_build.restype = ctypes.c_int
        L.moeblaze_dispatch_build_static.argtypes = [SP, P, DP, ctypes.c_int, P]
        L.moeblaze_dispatch_build_static.restype = ctypes.c_int
        L.moeblaze_forward.argtypes = [SP, P, P, DP, P, P, P, P, P, P, sz, P]
        L.moeblaze_forward.restype = ctypes.c_int
        L.moeblaze_backward.argtypes = [SP, P, P, P, DP, P, P, P, P, P, P, P, P, P, P, sz, P]
        L.moeblaze_backward.restype = ctypes.c_int
        L.moeblaze_router_forward.argtypes = [SP, P, P, P, P, P, P]
        L.moeblaze_router_forward.restype = ctypes.c_int
        L.moeblaze_router_backward_workspace_bytes.argtypes = [SP]
        L.moeblaze_router_backward_workspace_bytes.restype = sz
        L.moeblaze_router_backward.argtypes = [SP, P, P, P, P, P, P, P, P, P, sz, P]
        L.moeblaze_router_backward.restype = ctypes.c_int
        L.moeblaze_router_dispatch_workspace_bytes.argtypes = [SP]
        L.moeblaze_router_dispatch_workspace_bytes.restype = sz
        L.moeblaze_router_dispatch_build.argtypes = [SP, P, P, P, P, P, DP, P, sz, P]
        L.moeblaze_router_dispatch_build.restype = ctypes.c_int
        L.moeblaze_device_error.argtypes = [SP, DP, ctypes.POINTER(ctypes.c_int32), P]
        L.moeblaze_device_error.restype = ctypes.c_int
        L.moeblaze_dispatch_meta_check.argtypes = [SP, P]
        L.moeblaze_dispatch_meta_check.restype = ctypes.c_int
        L.moeblaze_status_string.argtypes = [ctypes.c_int]
        L.moeblaze_status_string.restype = ctypes.c_char_p
        L.moeblaze_version.argtypes = []
        L.moeblaze_version.restype = ctypes.c_int32
        L.moeblaze_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32]
        L.moeblaze_set_stage_events.restype = None
        L.moeblaze_set_fault_injection.argtypes = [ctypes.c_int64, ctypes.c_int32]
        L.moeblaze_set_fault_injection.restype = None
        L.moeblaze_kernel_launches.argtypes = []
        L.moeblaze_kernel_launches.restype = ctypes.c_int64
        _lib = L
    return _lib


def status_string(st: int) -> str:
    return lib().moeblaze_status_string(st).decode()


# ---------------------------------------------------------------- C names

def moeblaze_dispatch_meta_bytes(shape: Shape) -> int:
    return lib().moeblaze_dispatch_meta_bytes(ctypes.byref(shape))


def moeblaze_dispatch_workspace_bytes(shape: Shape) -> int:
    return lib().moeblaze_dispatch_workspace_bytes(ctypes.byref(shape))


def moeblaze_saved_bytes(shape: Shape) -> int:
    return lib().moeblaze_saved_bytes(ctypes.byref(shape))


def moeblaze_forward_workspace_bytes(shape: Shape) -> int:
    return lib().moeblaze_forward_workspace_bytes(ctypes.byref(shape))


def moeblaze_backward_workspace_bytes(shape: Shape) -> int:
    return lib().moeblaze_backward_workspace_bytes(ctypes.byref(shape))


def moeblaze_dispatch_build(shape, topk_ids, disp, ws, ws_bytes, validate, stream) -> int:
    return lib().moeblaze_dispatch_build(ctypes.byref(shape), topk_ids, ctypes.byref(disp), ws, ws_bytes,
                                         int(validate), stream)


def moeblaze_dispatch_build_static(shape, topk_ids, disp, validate, stream) -> int:
    return lib().moeblaze_dispatch_build_static(ctypes.byref(shape), topk_ids, ctypes.byref(disp), int(validate),
                                                stream)


def moeblaze_forward(shape, x, gates, disp, W1, W2, W3, y, saved, ws, ws_bytes, stream) -> int:
    return lib().moeblaze_forward(ctypes.byref(shape), x, gates, ctypes.byref(disp), W1, W2, W3, y, saved, ws,
                                  ws_bytes, stream)


def moeblaze_backward(shape, dY, x, gates, disp, W1, W2, W3, saved, dX, dW1, dW2, dW3, dgates, ws, ws_bytes,
                      stream) -> int:
    return lib().moeblaze_backward(ctypes.byref(shape), dY, x, gates, ctypes.byref(disp), W1, W2, W3, saved, dX,
                                   dW1, dW2, dW3, dgates, ws, ws_bytes, stream)


def moeblaze_router_forward(shape, x, Wr, bias, topk_ids, gates, stream) -> int:
    return lib().moeblaze_router_forward(ctypes.byref(shape), x, Wr, bias, topk_ids, gates, stream)


def moeblaze_router_backward_workspace_bytes(shape: Shape) -> int:
    return lib().moeblaze_router_backward_workspace_bytes(ctypes.byref(shape))


def moeblaze_router_backward(shape, x, Wr, topk_ids, gates, dgates, dWr, dbias, dx, ws, ws_bytes, stream) -> int:
    return lib().moeblaze_router_backward(ctypes.byref(shape), x, Wr, topk_ids, gates, dgates, dWr, dbias, dx, ws,
                                          ws_bytes, stream)


def moeblaze_router_dispatch_workspace_bytes(shape: Shape) -> int:
    return lib().moeblaze_router_dispatch_workspace_bytes(ctypes.byref(shape))


def moeblaze_router_dispatch_build(shape, x, Wr, bias, topk_ids, gates, disp, ws, ws_bytes, stream) -> int:
    return lib().moeblaze_router_dispatch_build(ctypes.byref(shape), x, Wr, bias, topk_ids, gates, ctypes.byref(disp),
                                                ws, ws_bytes, stream)


def moeblaze_device_error(shape, disp, stream):
    code = ctypes.c_int32(0)
    st = lib().moeblaze_device_error(ctypes.byref(shape), ctypes.byref(disp), ctypes.byref(code), stream)
    return st, code.value


def moeblaze_dispatch_meta_check(shape, meta_header) -> int:
    """meta_header: a host buffer (bytes-like or ctypes pointer) holding a
    copy of the first 32 bytes of a dispatch's meta."""
    return lib().moeblaze_dispatch_meta_check(ctypes.byref(shape), meta_header)


def moeblaze_set_stage_events(events, n: int) -> None:
    lib().moeblaze_set_stage_events(events, int(n))


def moeblaze_set_fault_injection(wait_limit_ns: int, withhold: int) -> None:
    lib().moeblaze_set_fault_injection(int(wait_limit_ns), int(withhold))


def moeblaze_kernel_launches() -> int:
    return int(lib().moeblaze_kernel_launches())


# ---------------------------------------------------------------- torch helpers

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_shape(L, d, h, E, K, dtype, act, flags: int = 0) -> Shape:
    dt = DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    a = ACT[act] if isinstance(act, str) else int(act)
    return Shape(int(L), int(d), int(h), int(E), int(K), dt, a, int(flags))


_TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


def _args(*specs):
    """Check tensor arguments before their pointers go to C.  Each spec is
    (tensor, name, shape, dtype, optional); a tensor of an empty shape may
    be None, as the library takes NULL there.  Every tensor must have exactly
    that shape and dtype and a dense row-major layout (checked for all of
    them first), and live on the current CUDA device.  The C library sees
    only pointers, so a wrong tensor would otherwise be read or written out
    of bounds on the GPU."""
    for t, name, shape, dtype, optional in specs:
        if t is None:
            # an empty buffer (no tokens) may be passed as NULL
            if optional or any(int(v) == 0 for v in shape):
                continue
            raise ValueError(f"{name}: a tensor is required")
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
        want = tuple(int(v) for v in shape)
        if tuple(t.shape) != want:
            raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {want}")
        if t.dtype != dtype:
            raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name}: must be contiguous (row-major)")
    _on_device(*[(spec[0], spec[1]) for spec in specs if spec[0] is not None])


def _on_device(*named):
    for t, name in named:
        if not t.is_cuda:
            raise ValueError(f"{name}: must be a CUDA tensor")
        if t.device.index != torch.cuda.current_device():
            raise ValueError(f"{name}: on {t.device}, but the current device is cuda:{torch.cuda.current_device()}")


def _bytes_arg(t, name: str, nbytes: int):
    """A caller-provided byte buffer: at least nbytes, contiguous, on the current CUDA device."""
    if not isinstance(t, torch.Tensor) or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name}: {t.numel() * t.element_size()} bytes, needs {nbytes}")
    _on_device((t, name))


def _weight_specs(shape: Shape, W1, W2, W3, prefix: str = ""):
    """Specs of the expert weights the activation uses (the others go to C as NULL)."""
    if shape.act == IDENTITY:
        return []
    dt = _TORCH_DTYPE[shape.dtype]
    E, d, h = shape.E, shape.d, shape.h
    specs = [(W1, prefix + "W1", (E, d, h), dt, False), (W3, prefix + "W3", (E, h, d), dt, False)]
    if shape.act == SWIGLU:
        specs.append((W2, prefix + "W2", (E, d, h), dt, False))
    return specs


def _used_weights(shape: Shape, W1, W2, W3):
    if shape.act == IDENTITY:
        return None, None, None
    return W1, (W2 if shape.act == SWIGLU else None), W3


def _check_dispatch_bufs(shape: Shape, bufs: "DispatchBuffers"):
    LK = shape.L * shape.K
    for name in ("expert_token_indices", "token_expert_indices", "token_index_map"):
        _bytes_arg(getattr(bufs, name), name, 4 * LK)
    _bytes_arg(bufs.expert_token_offsets, "expert_token_offsets", 4 * (shape.E + 1))
    _bytes_arg(bufs.meta, "meta", moeblaze_dispatch_meta_bytes(shape))


def _check(st: int, where: str):
    if st != OK:
        raise MoEBlazeError(st, where)


@dataclass
class DispatchBuffers:
    shape: Shape
    expert_token_indices: torch.Tensor
    expert_token_offsets: torch.Tensor
    token_expert_indices: torch.Tensor
    token_index_map: torch.Tensor
    meta: torch.Tensor
    ws: torch.Tensor

    def struct(self) -> Dispatch:
        return Dispatch(self.expert_token_indices.data_ptr(), self.expert_token_offsets.data_ptr(),
                        self.token_expert_indices.data_ptr(), self.token_index_map.data_ptr(), self.meta.data_ptr())


def _bytes(n: int, device) -> torch.Tensor:
    # 256-byte aligned device buffer of at least n bytes (torch allocations are)
    return torch.empty(max(int(n), 16), dtype=torch.uint8, device=device)


def alloc_dispatch(shape: Shape, device="cuda") -> DispatchBuffers:
    LK = shape.L * shape.K
    i32 = dict(dtype=torch.int32, device=device)
    return DispatchBuffers(
        shape,
        torch.empty(max(LK, 4), **i32),
        torch.empty(shape.E + 1 + 3, **i32),
        torch.empty(max(LK, 4), **i32),
        torch.empty(max(LK, 4), **i32),
        _bytes(moeblaze_dispatch_meta_bytes(shape), device),
        _bytes(moeblaze_dispatch_workspace_bytes(shape), device),
    )


def dispatch_build(shape: Shape, topk_ids: torch.Tensor, bufs: Optional[DispatchBuffers] = None,
                   validate: bool = False, stream=None) -> DispatchBuffers:
    """Run the three-step dispatch build; returns the buffers holding the
    index structures (views: [:L*K], [:E+1])."""
    _args((topk_ids, "topk_ids", (shape.L, shape.K), torch.int32, False))
    if bufs is None:
        bufs = alloc_dispatch(shape, topk_ids.device)
    _check_dispatch_bufs(shape, bufs)
    d = bufs.struct()
    st = moeblaze_dispatch_build(shape, _ptr(topk_ids), d, _ptr(bufs.ws), bufs.ws.numel(), validate, _stream(stream))
    _check(st, "moeblaze_dispatch_build")
    return bufs


def index_views(shape: Shape, bufs: DispatchBuffers):
    LK = shape.L * shape.K
    return (bufs.expert_token_indices[:LK], bufs.expert_token_offsets[:shape.E + 1],
            bufs.token_expert_indices[:LK].view(shape.L, shape.K), bufs.token_index_map[:LK].view(shape.L, shape.K))


@dataclass
class LayerBuffers:
    saved: torch.Tensor
    fwd_ws: torch.Tensor
    bwd_ws: torch.Tensor


def alloc_layer(shape: Shape, device="cuda") -> LayerBuffers:
    return LayerBuffers(_bytes(moeblaze_saved_bytes(shape), device),
                        _bytes(moeblaze_forward_workspace_bytes(shape), device),
                        _bytes(moeblaze_backward_workspace_bytes(shape), device))


def forward(shape: Shape, x, gates, disp: DispatchBuffers, W1, W2, W3, y, layer: LayerBuffers, stream=None):
    dt = _TORCH_DTYPE[shape.dtype]
    _args((x, "x", (shape.L, shape.d), dt, False), (gates, "gates", (shape.L, shape.K), torch.float32, False),
          (y, "y", (shape.L, shape.d), dt, False), *_weight_specs(shape, W1, W2, W3))
    W1, W2, W3 = _used_weights(shape, W1, W2, W3)
    _check_dispatch_bufs(shape, disp)
    _bytes_arg(layer.saved, "saved", moeblaze_saved_bytes(shape))
    st = moeblaze_forward(shape, _ptr(x), _ptr(gates), disp.struct(), _ptr(W1), _ptr(W2), _ptr(W3), _ptr(y),
                          _ptr(layer.saved), _ptr(layer.fwd_ws), layer.fwd_ws.numel(), _stream(stream))
    _check(st, "moeblaze_forward")
    return y


def backward(shape: Shape, dY, x, gates, disp: DispatchBuffers, W1, W2, W3, layer: LayerBuffers, dX, dW1, dW2, dW3,
             dgates=None, stream=None):
    dt = _TORCH_DTYPE[shape.dtype]
    _args((dY, "dY", (shape.L, shape.d), dt, False), (x, "x", (shape.L, shape.d), dt, False),
          (gates, "gates", (shape.L, shape.K), torch.float32, False), (dX, "dX", (shape.L, shape.d), dt, False),
          (dgates, "dgates", (shape.L, shape.K), torch.float32, True),
          *_weight_specs(shape, W1, W2, W3), *_weight_specs(shape, dW1, dW2, dW3, prefix="d"))
    W1, W2, W3 = _used_weights(shape, W1, W2, W3)
    dW1, dW2, dW3 = _used_weights(shape, dW1, dW2, dW3)
    _check_dispatch_bufs(shape, disp)
    _bytes_arg(layer.saved, "saved", moeblaze_saved_bytes(shape))
    st = moeblaze_backward(shape, _ptr(dY), _ptr(x), _ptr(gates), disp.struct(), _ptr(W1), _ptr(W2), _ptr(W3),
                           _ptr(layer.saved), _ptr(dX), _ptr(dW1), _ptr(dW2), _ptr(dW3), _ptr(dgates),
                           _ptr(layer.bwd_ws), layer.bwd_ws.numel(), _stream(stream))
    _check(st, "moeblaze_backward")


class StageEvents:
    """CUDA events the library records at its stage boundaries (see
    moeblaze_set_stage_events); use as a context manager around one call."""

    def __init__(self, n: int):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in self.events:  # torch creates the CUDA event on its first record
            e.record()
        torch.cuda.current_stream().synchronize()
        self._arr = (ctypes.c_void_p * n)(*[ctypes.c_void_p(e.cuda_event) for e in self.events])

    def __enter__(self):
        moeblaze_set_stage_events(self._arr, len(self.events))
        return self

    def __exit__(self, *exc):
        moeblaze_set_stage_events(None, 0)
        return False

    def elapsed_ms(self):
        return [self.events[i].elapsed_time(self.events[i + 1]) for i in range(len(self.events) - 1)]


def router_forward(shape: Shape, x, Wr, bias, topk_ids, gates, stream=None):
    """Token-choice top-K softmax router: fills topk_ids (L,K) int32 and gates (L,K) fp32."""
    _args((x, "x", (shape.L, shape.d), _TORCH_DTYPE[shape.dtype], False),
          (Wr, "Wr", (shape.d, shape.E), torch.float32, False), (bias, "bias", (shape.E,), torch.float32, True),
          (topk_ids, "topk_ids", (shape.L, shape.K), torch.int32, False),
          (gates, "gates", (shape.L, shape.K), torch.float32, False))
    st = moeblaze_router_forward(shape, _ptr(x), _ptr(Wr), _ptr(bias), _ptr(topk_ids), _ptr(gates), _stream(stream))
    _check(st, "moeblaze_router_forward")


def router_dispatch_build(shape: Shape, x, Wr, bias, topk_ids, gates, bufs: Optional["DispatchBuffers"] = None,
                          ws=None, stream=None) -> "DispatchBuffers":
    """The router fused with the dispatch build's first step: fills topk_ids
    (L,K) int32, gates (L,K) fp32 and the dispatch buffers in one call.  `ws`
    is a device byte tensor of moeblaze_router_dispatch_workspace_bytes(shape)
    bytes (allocated here when None)."""
    _args((x, "x", (shape.L, shape.d), _TORCH_DTYPE[shape.dtype], False),
          (Wr, "Wr", (shape.d, shape.E), torch.float32, False), (bias, "bias", (shape.E,), torch.float32, True),
          (topk_ids, "topk_ids", (shape.L, shape.K), torch.int32, False),
          (gates, "gates", (shape.L, shape.K), torch.float32, False))
    if bufs is None:
        bufs = alloc_dispatch(shape, Wr.device)
    _check_dispatch_bufs(shape, bufs)
    n = moeblaze_router_dispatch_workspace_bytes(shape)
    if n == 0:
        raise MoEBlazeError(ERR_UNSUPPORTED, "moeblaze_router_dispatch_workspace_bytes")
    if ws is None:
        ws = _bytes(n, Wr.device)
    _bytes_arg(ws, "ws", n)
    st = moeblaze_router_dispatch_build(shape, _ptr(x), _ptr(Wr), _ptr(bias), _ptr(topk_ids), _ptr(gates),
                                        bufs.struct(), _ptr(ws), n, _stream(stream))
    _check(st, "moeblaze_router_dispatch_build")
    return bufs


def router_backward(shape: Shape, x, Wr, topk_ids, gates, dgates, dWr, dbias, dx, ws=None, stream=None):
    """Router gradients from the gate gradients: fills dWr (d,E) fp32, dbias (E) fp32 and dx (L,d) (dbias and dx
    may be None).  `ws` is a device byte tensor of moeblaze_router_backward_workspace_bytes(shape) bytes
    (allocated here when None)."""
    _args((x, "x", (shape.L, shape.d), _TORCH_DTYPE[shape.dtype], False),
          (Wr, "Wr", (shape.d, shape.E), torch.float32, False),
          (topk_ids, "topk_ids", (shape.L, shape.K), torch.int32, False),
          (gates, "gates", (shape.L, shape.K), torch.float32, False),
          (dgates, "dgates", (shape.L, shape.K), torch.float32, False),
          (dWr, "dWr", (shape.d, shape.E), torch.float32, False),
          (dbias, "dbias", (shape.E,), torch.float32, True),
          (dx, "dx", (shape.L, shape.d), _TORCH_DTYPE[shape.dtype], True))
    n = moeblaze_router_backward_workspace_bytes(shape)
    if ws is None:
        ws = _bytes(n, Wr.device)
    _bytes_arg(ws, "ws", n)
    st = moeblaze_router_backward(shape, _ptr(x), _ptr(Wr), _ptr(topk_ids), _ptr(gates), _ptr(dgates), _ptr(dWr),
                                  _ptr(dbias), _ptr(dx), _ptr(ws), n, _stream(stream))
    _check(st, "moeblaze_router_backward")


def device_error(shape: Shape, disp: DispatchBuffers, stream=None) -> int:
    """The device error word of a dispatch (0: every kernel since its build
    finished normally; bits 1 bad routing, 2 timeout, 4 shape mismatch)."""
    st, code = moeblaze_device_error(shape, disp.struct(), _stream(stream))
    if st not in (OK, ERR_BAD_ROUTING, ERR_TIMEOUT) and not (st == ERR_INVALID_ARG and code & 4):
        raise MoEBlazeError(st, "moeblaze_device_error")
    return code


def padded_rows(shape: Shape) -> int:
    """Rows of the expert-major row space: L*K plus each expert's padding to
    a multiple of 256 rows, at most."""
    r = shape.L * shape.K + shape.E * 255
    return (r + 255) // 256 * 256


def saved_views(shape: Shape, layer: LayerBuffers, dtype):
    """(A, B) views of the saved checkpoint: (padded_rows, h) each (B None for
    SiLU).  After a bf16 backward they hold dA and dB."""
    es = 4 if dtype == torch.float32 else 2
    h = shape.h
    nb = 2 if shape.act == SWIGLU else 1
    rows = padded_rows(shape)
    t = layer.saved[: rows * nb * h * es].view(dtype).view(nb, rows, h)
    return t[0], (t[1] if nb == 2 else None)


def meta_arrays(shape: Shape, disp: DispatchBuffers):
    """Host copies of (num_m_tiles, n_e, pad_off, order) from the meta buffer."""
    m = disp.meta.view(torch.int32).cpu()
    E = shape.E
    n_e = m[8:8 + E]
    pad = m[8 + E:8 + 2 * E + 1]
    order = m[8 + 2 * E + 1:8 + 3 * E + 1]
    return int(m[1]), n_e, pad, order
