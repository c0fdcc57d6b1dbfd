"""Python binding of the GB300 resolvent-operator causal head (libresolvent.so).

Argument marshalling only: every step of the computation runs in the CUDA kernels behind the
C ABI declared in include/resolvent.h. PyTorch supplies device memory and the current
stream. There is no CPU path: if the library is missing the calls raise.

Functions mirror the C entry points:
  gate_prep(u, theta, g)                        -> dict of gate outputs
  head_forward(q, k, u, theta, v, beta, qk, g)  -> (O_re, O_im)
  chain_scan(u, theta, g, b)                    -> (y_re, y_im)
  status_sync(status)                           -> raises NonFinite / DeviceTimeout
  debug_path_product(u, theta, g)               -> G (complex64) for tests
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Union

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libresolvent.so")
BLOCK = 128

RS_OK, RS_ERR_NONFINITE, RS_ERR_SHAPE, RS_ERR_UNSUPPORTED = 0, 1, 2, 3
RS_ERR_ALIGN, RS_ERR_WORKSPACE, RS_ERR_CUDA, RS_ERR_TIMEOUT = 4, 5, 6, 7
RS_F32, RS_BF16 = 0, 1

Switch = Union[float, Sequence[float]]


class ResolventError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (rs_status {code})")
        self.code = code


class NonFinite(ResolventError):
    """The pages' NonFinite refusal, raised when the device status word says so."""


class DeviceTimeout(ResolventError):
    """A bounded device-side wait ran out."""


class _Switches(ctypes.Structure):
    _fields_ = [("beta", ctypes.POINTER(ctypes.c_float)), ("qk", ctypes.POINTER(ctypes.c_float)),
                ("g", ctypes.POINTER(ctypes.c_float)), ("count", ctypes.c_int)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """The loaded C library. Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
                "g.build()'); there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        L.resolvent_gate_prep.argtypes = [_P, _P, _Switches, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]
        L.resolvent_gate_prep.restype = _I
        L.resolvent_head_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, _I]
        L.resolvent_head_workspace_bytes.restype = _SZ
        L.resolvent_head_forward.argtypes = [_P, _P, _P, _P, _P, _Switches, _I, _I, _I, _I, _I, _I,
                                             _P, _P, _P, _SZ, _P, _P]
        L.resolvent_head_forward.restype = _I
        L.resolvent_operator_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
        L.resolvent_operator_workspace_bytes.restype = _SZ
        L.resolvent_operator.argtypes = [_P, _P, _P, _P, _Switches, _I, _I, _I, _I, _I, _P, _P, _P,
                                         _SZ, _P, _P]
        L.resolvent_operator.restype = _I
        L.resolvent_position_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
        L.resolvent_position_workspace_bytes.restype = _SZ
        L.resolvent_position_head.argtypes = [_P, _P, _Switches, _I, _I, _I, _I, _I, _P, _P, _SZ,
                                              _P, _P]
        L.resolvent_position_head.restype = _I
        L.resolvent_chain_workspace_bytes.argtypes = [_I, _I, _I, _I]
        L.resolvent_chain_workspace_bytes.restype = _SZ
        L.resolvent_chain_scan.argtypes = [_P, _P, _Switches, _P, _I, _I, _I, _I, _P, _P, _P, _SZ,
                                           _P, _P]
        L.resolvent_chain_scan.restype = _I
        L.resolvent_chain_scan_carry.argtypes = [_P, _P, _Switches, _P, _I, _I, _I, _I, _P, _P, _P,
                                                 _P, _P, _SZ, _P, _P]
        L.resolvent_chain_scan_carry.restype = _I
        L.resolvent_chain_scan_noalloc.argtypes = [_P, _P, _Switches, _P, _I, _I, _I, _I, _P, _P,
                                                   _P, _P]
        L.resolvent_chain_scan_noalloc.restype = _I
        L.resolvent_status_sync.argtypes = [_P, _P]
        L.resolvent_status_sync.restype = _I
        L.resolvent_status_string.argtypes = [_I]
        L.resolvent_status_string.restype = ctypes.c_char_p
        L.resolvent_last_launch_count.argtypes = []
        L.resolvent_last_launch_count.restype = _I
        L.resolvent_debug_path_product.argtypes = [_P, _P, _Switches, _I, _I, _I, _P, _P, _SZ, _P, _P]
        L.resolvent_debug_path_product.restype = _I
        L.resolvent_test_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.resolvent_test_set_wait_limit_ns.restype = None
        L.resolvent_test_set_chain_withhold.argtypes = [_I]
        L.resolvent_test_set_chain_withhold.restype = None
        L.resolvent_test_set_position_withhold.argtypes = [_I]
        L.resolvent_test_set_position_withhold.restype = None
        L.resolvent_test_set_head_withhold.argtypes = [_I]
        L.resolvent_test_set_head_withhold.restype = None
        L.resolvent_test_set_operator_withhold.argtypes = [_I, _I]
        L.resolvent_test_set_operator_withhold.restype = None
        L.resolvent_profile_enable.argtypes = [_I]
        L.resolvent_profile_enable.restype = _I
        L.resolvent_profile_collect.argtypes = [ctypes.POINTER(ctypes.c_float), _I]
        L.resolvent_profile_collect.restype = _I
        L.resolvent_profile_collect_kinds.argtypes = [ctypes.POINTER(ctypes.c_float),
                                                      ctypes.POINTER(ctypes.c_int), _I]
        L.resolvent_profile_collect_kinds.restype = _I
        _lib = L
    return _lib


def _raise(rc: int):
    if rc == RS_OK:
        return
    msg = lib().resolvent_status_string(rc).decode()
    if rc == RS_ERR_NONFINITE:
        raise NonFinite(rc, msg)
    if rc == RS_ERR_TIMEOUT:
        raise DeviceTimeout(rc, msg)
    raise ResolventError(rc, msg)


def _switches(H: int, beta: Switch, qk: Switch, g: Switch):
    def arr(x):
        if hasattr(x, "tolist"):
            x = x.tolist()
        return [float(v) for v in x] if isinstance(x, (list, tuple)) else [float(x)]

    b, q, gg = arr(beta), arr(qk), arr(g)
    count = max(len(b), len(q), len(gg))
    if count not in (1, H) or any(len(v) not in (1, count) for v in (b, q, gg)):
        raise ResolventError(RS_ERR_SHAPE, "switches must have 1 or H values")
    b, q, gg = [(v * count if len(v) == 1 else v) for v in (b, q, gg)]
    keep = [(ctypes.c_float * count)(*v) for v in (b, q, gg)]
    sw = _Switches(*[ctypes.cast(x, ctypes.POINTER(ctypes.c_float)) for x in keep], count)
    return sw, keep


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dev(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not t.is_cuda:
        raise ResolventError(RS_ERR_SHAPE, f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ResolventError(RS_ERR_SHAPE, f"{name} must be {dtype}")
    return t.contiguous()


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word for the calls below."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def status_sync(status: torch.Tensor, stream=None) -> None:
    """Synchronises the stream, reads and clears the status word, raises on a refusal."""
    _raise(lib().resolvent_status_sync(_ptr(status), _stream(stream)))


def last_launch_count() -> int:
    """Kernels the last call on this thread enqueued."""
    return int(lib().resolvent_last_launch_count())


def gate_prep_outputs(B, H, n, device) -> dict:
    """Output buffers of gate_prep: m, theta_p [B,H,n]; gate, prefix, suffix [B,H,n,2];
    carry [B,H,ceil(n/128),2] (fp32, complex values as (re, im) pairs)."""
    nb = (n + BLOCK - 1) // BLOCK
    return {"m": torch.empty(B, H, n, device=device), "theta_p": torch.empty(B, H, n, device=device),
            "gate": torch.empty(B, H, n, 2, device=device),
            "prefix": torch.empty(B, H, n, 2, device=device),
            "suffix": torch.empty(B, H, n, 2, device=device),
            "carry": torch.empty(B, H, nb, 2, device=device)}


def gate_prep(u: torch.Tensor, theta: torch.Tensor, g: Switch, *, out=None, status=None,
              stream=None, sync: bool = True) -> dict:
    """Blended gates and block products of every head; u, theta fp32 [B,H,n]. `out` (from
    gate_prep_outputs) receives them; entries set to None are not written."""
    u = _dev(u, "u", torch.float32)
    theta = _dev(theta, "theta", torch.float32)
    B, H, n = u.shape
    sw, keep = _switches(H, 0.0, 0.0, g)
    dev = u.device
    if out is None:
        out = gate_prep_outputs(B, H, n, dev)
    st = status if status is not None else new_status(dev)
    _raise(lib().resolvent_gate_prep(_ptr(u), _ptr(theta), sw, B, H, n, *[
        _ptr(out.get(k)) for k in ("m", "theta_p", "gate", "prefix", "suffix", "carry")],
        _ptr(st), _stream(stream)))
    if sync and status is None:
        status_sync(st, stream)
    return out


def head_workspace_bytes(B, H, n, d, dv, dtype: torch.dtype) -> int:
    return int(lib().resolvent_head_workspace_bytes(B, H, n, d, dv,
                                                     RS_F32 if dtype == torch.float32 else RS_BF16))


def head_forward(q, k, u, theta, v, beta: Switch, qk: Switch, g: Switch, *, out=None,
                 workspace=None, status=None, stream=None, sync: bool = True):
    """O = W V for every head; q, k [B,H,n,d], v [B,H,n,dv] (bf16 or fp32), u, theta fp32
    [B,H,n]. Returns (O_re, O_im) fp32 [B,H,n,dv]."""
    if q.dtype not in (torch.bfloat16, torch.float32) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ResolventError(RS_ERR_UNSUPPORTED, "q, k, v must all be bf16 or all fp32")
    q, k, v = _dev(q, "q"), _dev(k, "k"), _dev(v, "v")
    u = _dev(u, "u", torch.float32)
    theta = _dev(theta, "theta", torch.float32)
    B, H, n, d = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or u.shape != (B, H, n) or theta.shape != u.shape:
        raise ResolventError(RS_ERR_SHAPE, "shape mismatch")
    dt = RS_F32 if q.dtype == torch.float32 else RS_BF16
    sw, keep = _switches(H, beta, qk, g)
    dev = q.device
    if out is None:
        out = (torch.empty(B, H, n, dv, device=dev), torch.empty(B, H, n, dv, device=dev))
    wsb = int(lib().resolvent_head_workspace_bytes(B, H, n, d, dv, dt))
    if workspace is None:
        workspace = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    st = status if status is not None else new_status(dev)
    _raise(lib().resolvent_head_forward(_ptr(q), _ptr(k), _ptr(u), _ptr(theta), _ptr(v), sw, B, H,
                                        n, d, dv, dt, _ptr(out[0]), _ptr(out[1]), _ptr(workspace),
                                        workspace.numel(), _ptr(st), _stream(stream)))
    if sync and status is None:
        status_sync(st, stream)
    return out


def operator_workspace_bytes(B, H, n, d, dtype: torch.dtype) -> int:
    return int(lib().resolvent_operator_workspace_bytes(
        B, H, n, d, RS_F32 if dtype == torch.float32 else RS_BF16))


def chain_workspace_bytes(B, H, n, dv) -> int:
    return int(lib().resolvent_chain_workspace_bytes(B, H, n, dv))


def chain_scan(u, theta, g: Switch, b, *, out=None, workspace=None, status=None, stream=None,
               sync: bool = True, carry_in=None, carry_out=None):
    """y_0 = b_0, y_i = a_i y_{i-1} + b_i; b fp32 [B,H,n,dv]. Returns (y_re, y_im).

    carry_in / carry_out (complex64 [B,H,dv] on the device, optional): continue from y at the
    end of a previous segment (then y_0 = a_0 y_{-1} + b_0) and receive y at token n-1
    (resolvent_chain_scan_carry)."""
    u = _dev(u, "u", torch.float32)
    theta = _dev(theta, "theta", torch.float32)
    b = _dev(b, "b", torch.float32)
    B, H, n, dv = b.shape
    if u.shape != (B, H, n) or theta.shape != u.shape:
        raise ResolventError(RS_ERR_SHAPE, "shape mismatch")
    sw, keep = _switches(H, 0.0, 0.0, g)
    dev = b.device
    if out is None:
        out = (torch.empty(B, H, n, dv, device=dev), torch.empty(B, H, n, dv, device=dev))
    wsb = chain_workspace_bytes(B, H, n, dv)
    if workspace is None:
        workspace = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    st = status if status is not None else new_status(dev)
    if carry_in is None and carry_out is None:
        _raise(lib().resolvent_chain_scan(_ptr(u), _ptr(theta), sw, _ptr(b), B, H, n, dv,
                                          _ptr(out[0]), _ptr(out[1]), _ptr(workspace),
                                          workspace.numel(), _ptr(st), _stream(stream)))
    else:
        def carry(c, name):
            if c is None:
                return None
            if c.dtype != torch.complex64 or c.shape != (B, H, dv) or not c.is_contiguous() \
                    or c.device != dev:
                raise ResolventError(RS_ERR_SHAPE, f"{name}: complex64 [B,H,dv] on {dev}")
            return ctypes.c_void_p(torch.view_as_real(c).data_ptr())
        _raise(lib().resolvent_chain_scan_carry(_ptr(u), _ptr(theta), sw, _ptr(b), B, H, n, dv,
                                                carry(carry_in, "carry_in"),
                                                carry(carry_out, "carry_out"), _ptr(out[0]),
                                                _ptr(out[1]), _ptr(workspace), workspace.numel(),
                                                _ptr(st), _stream(stream)))
    if sync and status is None:
        status_sync(st, stream)
    return out


def operator(q, k, u, theta, beta: Switch, qk: Switch, g: Switch, *, out=None, workspace=None,
             status=None, stream=None, sync: bool = True):
    """W [B,H,n,n] complex64 (section "Object"); q, k [B,H,n,d] bf16 or fp32."""
    if q.dtype not in (torch.bfloat16, torch.float32) or k.dtype != q.dtype:
        raise ResolventError(RS_ERR_UNSUPPORTED, "q, k must both be bf16 or both fp32")
    dt = RS_F32 if q.dtype == torch.float32 else RS_BF16
    q, k = _dev(q, "q"), _dev(k, "k")
    u = _dev(u, "u", torch.float32)
    theta = _dev(theta, "theta", torch.float32)
    B, H, n, d = q.shape
    if k.shape != q.shape or u.shape != (B, H, n) or theta.shape != u.shape:
        raise ResolventError(RS_ERR_SHAPE, "shape mismatch")
    sw, keep = _switches(H, beta, qk, g)
    dev = q.device
    if out is None:
        out = (torch.empty(B, H, n, n, device=dev), torch.empty(B, H, n, n, device=dev))
    wsb = int(lib().resolvent_operator_workspace_bytes(B, H, n, d, dt))
    if workspace is None:
        workspace = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    st = status if status is not None else new_status(dev)
    _raise(lib().resolvent_operator(_ptr(q), _ptr(k), _ptr(u), _ptr(theta), sw, B, H, n, d, dt,
                                    _ptr(out[0]), _ptr(out[1]), _ptr(workspace), workspace.numel(),
                                    _ptr(st), _stream(stream)))
    if sync and status is None:
        status_sync(st, stream)
    return out


def position_workspace_bytes(B, H, n, dv, dtype: torch.dtype) -> int:
    return int(lib().resolvent_position_workspace_bytes(
        B, H, n, dv, RS_F32 if dtype == torch.float32 else RS_BF16))


def position_head(a, v, beta: Switch, qk: Switch, *, out=None, workspace=None, status=None,
                  stream=None, sync: bool = True):
    """O [B,H,n,dv] fp32 of position-only heads: logits qk * a[h, i - j] (a [H,n] fp32);
    v [B,H,n,dv] bf16 or fp32; g = 0 ("A position-only causal softmax head is a causal
    convolution divided by a prefix normalizer")."""
    if v.dtype not in (torch.bfloat16, torch.float32):
        raise ResolventError(RS_ERR_UNSUPPORTED, "v must be bf16 or fp32")
    dt = RS_F32 if v.dtype == torch.float32 else RS_BF16
    v = _dev(v, "v")
    a = _dev(a, "a", torch.float32)
    B, H, n, dv = v.shape
    if a.shape != (H, n):
        raise ResolventError(RS_ERR_SHAPE, "a must be [H, n]")
    sw, keep = _switches(H, beta, qk, 0.0)
    dev = v.device
    if out is None:
        out = torch.empty(B, H, n, dv, device=dev)
    wsb = int(lib().resolvent_position_workspace_bytes(B, H, n, dv, dt))
    if workspace is None:
        workspace = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    st = status if status is not None else new_status(dev)
    _raise(lib().resolvent_position_head(_ptr(a), _ptr(v), sw, B, H, n, dv, dt, _ptr(out),
                                         _ptr(workspace), workspace.numel(), _ptr(st),
                                         _stream(stream)))
    if sync and status is None:
        status_sync(st, stream)
    return out


def debug_path_product(u, theta, g: Switch, *, stream=None) -> torch.Tensor:
    """G [B,H,n,n] complex64 as the head kernel factors it (tests only; n <= 4096)."""
    u = _dev(u, "u", torch.float32)
    theta = _dev(theta, "theta", torch.float32)
    B, H, n = u.shape
    sw, keep = _switches(H, 0.0, 0.0, g)
    dev = u.device
    G = torch.empty(B, H, n, n, 2, device=dev)
    wsb = int(lib().resolvent_head_workspace_bytes(B, H, n, 8, 8, RS_BF16))
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    st = new_status(dev)
    _raise(lib().resolvent_debug_path_product(_ptr(u), _ptr(theta), sw, B, H, n, _ptr(G), _ptr(ws),
                                              ws.numel(), _ptr(st), _stream(stream)))
    status_sync(st, stream)
    return torch.view_as_complex(G)


def test_set_wait_limit_ns(ns: int) -> None:
    lib().resolvent_test_set_wait_limit_ns(int(ns))


def test_set_chain_withhold(ticket: int) -> None:
    lib().resolvent_test_set_chain_withhold(int(ticket))


def test_set_position_withhold(block: int) -> None:
    lib().resolvent_test_set_position_withhold(int(block))


def test_set_head_withhold(block: int) -> None:
    lib().resolvent_test_set_head_withhold(int(block))


def test_set_operator_withhold(launch: int, block: int) -> None:
    """launch 0: the row statistics, 1: the write of W; block -1 turns the knob off."""
    lib().resolvent_test_set_operator_withhold(int(launch), int(block))


def profile_enable(on: bool = True) -> None:
    """Record CUDA events around the main kernel of every following call."""
    _raise(lib().resolvent_profile_enable(1 if on else 0))


PROF_HEAD_GATED, PROF_HEAD_REAL, PROF_READOUT, PROF_CHAIN = 0, 1, 2, 3
PROF_OPERATOR, PROF_POSITION, PROF_GATE_PREP = 4, 5, 6


def profile_collect(max_pairs: int = 4096, kinds: bool = False) -> list:
    """Durations (ms) of the launches recorded since profiling was enabled or last collected;
    with kinds=True, (ms, class) pairs (PROF_* above)."""
    buf = (ctypes.c_float * max_pairs)()
    kb = (ctypes.c_int * max_pairs)()
    k = lib().resolvent_profile_collect_kinds(buf, kb, max_pairs)
    if k < 0:
        raise ResolventError(RS_ERR_CUDA, "profile collection failed")
    if kinds:
        return [(float(buf[i]), int(kb[i])) for i in range(k)]
    return [float(buf[i]) for i in range(k)]
