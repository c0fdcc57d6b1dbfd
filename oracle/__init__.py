"""Plain fp64 CPU oracle of the resolvent-operator causal head.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` import this package; the CUDA library never loads it and shares no code
with it. The arithmetic lives in ``resolvent_oracle.c`` (plain C, fp64, explicit descending
path products); this module compiles it with gcc and marshals numpy arrays through ctypes.

Every routine follows "Resolvent Operator" (teerth.dev/Aether-Lang/integrated/resolvent/),
section "Object" and section "Evaluation and refusals". Inputs are passed as fp32 arrays
holding the same stored values the GPU reads (bf16 and fp32 both widen to fp64 exactly).

Parity status: every regime is pinned by the CPU tests; for beta strictly inside (0,1), where
the pages give no value, by the closed forms of constant logits and W(beta) Z^beta = W(0).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "resolvent_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libresolvent_oracle.so")
_lock = threading.Lock()
_lib = None

RO_OK, RO_NONFINITE, RO_SHAPE = 0, 1, 2

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64 = ctypes.c_int64
_f64 = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the library path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-shared", "-fPIC",
            "-I", _HERE, _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.ro_blend.argtypes = [_f64, _f64, _f64, _f64p, _f64p]
            L.ro_blend.restype = ctypes.c_int
            L.ro_gate.argtypes = [_f64, _f64, _f64p, _f64p]
            L.ro_gate.restype = None
            L.ro_path_product.argtypes = [_f64p, _f64p, _i64, _f64p, _f64p]
            L.ro_path_product.restype = None
            L.ro_operator.argtypes = [_f32p, _f32p, _f32p, _f32p, _i64, _i64, _f64, _f64,
                                      _f64, _f64p, _f64p]
            L.ro_operator.restype = ctypes.c_int
            L.ro_readout.argtypes = [_f64p, _f64p, _f32p, _i64, _i64, _f64p, _f64p]
            L.ro_readout.restype = None
            L.ro_chain.argtypes = [_f64p, _f64p, _f32p, _i64, _i64, _f64p, _f64p, _f64p]
            L.ro_chain.restype = None
            L.ro_head_rows.argtypes = [_f32p, _f32p, _f32p, _f32p, _f32p, _i64, _i64, _i64,
                                       _i64, _f64p, _f64p, _f64p, _i64p, _i64, _f64p, _f64p,
                                       _i32p, ctypes.c_int]
            L.ro_head_rows.restype = ctypes.c_int
            L.ro_gate_prep.argtypes = [_f32p, _f32p, _f64p, _i64, _i64, _i64] + [_f64p] * 10 \
                + [_i32p]
            L.ro_gate_prep.restype = ctypes.c_int
            L.ro_chain_heads.argtypes = [_f32p, _f32p, _f64p, _f32p, _i64, _i64, _i64, _f64p,
                                         _f64p, _f64p, _i32p, ctypes.c_int]
            L.ro_chain_heads.restype = ctypes.c_int
            L.ro_position_head.argtypes = [_f32p, _f32p, _i64, _i64, _f64, _f64, _f64p]
            L.ro_position_head.restype = ctypes.c_int
            L.ro_position_heads.argtypes = [_f32p, _f32p, _i64, _i64, _i64, _i64, _f64p, _f64p,
                                            _f64p, _i32p, ctypes.c_int]
            L.ro_position_heads.restype = ctypes.c_int
            L.ro_position_rows.argtypes = [_f32p, _f32p, _i64, _i64, _f64, _f64, _i64p, _i64,
                                           _f64p]
            L.ro_position_rows.restype = ctypes.c_int
            L.ro_operator_rows.argtypes = [_f32p, _f32p, _f32p, _f32p, _i64, _i64, _f64, _f64,
                                           _f64, _i64p, _i64, _f64p, _f64p]
            L.ro_operator_rows.restype = ctypes.c_int
            L.ro_max_threads.argtypes = []
            L.ro_max_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _f32(x):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return a, a.ctypes.data_as(_f32p)


def _f64a(x):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return a, a.ctypes.data_as(_f64p)


def _ptr64(a):
    return None if a is None else a.ctypes.data_as(_f64p)


class NonFinite(Exception):
    """The pages' NonFinite refusal."""


class ShapeError(Exception):
    """Shape mismatch or head_dim = 0 with n > 0 (the pages' Rust module panics)."""


def _raise(rc):
    if rc == RO_NONFINITE:
        raise NonFinite()
    if rc == RO_SHAPE:
        raise ShapeError()


def max_threads() -> int:
    return int(lib().ro_max_threads())


# ------------------------------------------------------------------ scalar / single head

def blend(u: float, theta: float, g: float):
    m, t = ctypes.c_double(), ctypes.c_double()
    _raise(lib().ro_blend(u, theta, g, ctypes.byref(m), ctypes.byref(t)))
    return m.value, t.value


def gate(m: float, theta_p: float) -> complex:
    re, im = ctypes.c_double(), ctypes.c_double()
    lib().ro_gate(m, theta_p, ctypes.byref(re), ctypes.byref(im))
    return complex(re.value, im.value)


def path_product(a) -> np.ndarray:
    """G [n,n] complex from gates a [n] complex."""
    a = np.asarray(a, dtype=np.complex128).reshape(-1)
    n = a.shape[0]
    ar, par = _f64a(a.real)
    ai, pai = _f64a(a.imag)
    Gr = np.zeros((n, n)); Gi = np.zeros((n, n))
    lib().ro_path_product(par, pai, n, _ptr64(Gr), _ptr64(Gi))
    return Gr + 1j * Gi


def operator(q, k, u, theta, beta: float, qk: float, g: float) -> np.ndarray:
    """W [n,n] complex for one head; q, k [n,d]; u, theta [n]."""
    q = np.asarray(q, dtype=np.float32)
    n = q.shape[0]
    d = q.shape[1] if q.ndim == 2 else 0
    qa, pq = _f32(q); ka, pk = _f32(k); ua, pu = _f32(u); ta, pt = _f32(theta)
    if ka.size != n * d or ua.size != n or ta.size != n:
        raise ShapeError()
    Wr = np.zeros((n, n)); Wi = np.zeros((n, n))
    _raise(lib().ro_operator(pq, pk, pu, pt, n, d, beta, qk, g, _ptr64(Wr), _ptr64(Wi)))
    return Wr + 1j * Wi


def readout(W, v) -> np.ndarray:
    """O [n,dv] complex from W [n,n] complex and real v [n,dv]."""
    W = np.asarray(W, dtype=np.complex128)
    n = W.shape[0]
    va, pv = _f32(v)
    dv = va.shape[1]
    Wr, pWr = _f64a(W.real); Wi, pWi = _f64a(W.imag)
    Or = np.zeros((n, dv)); Oi = np.zeros((n, dv))
    lib().ro_readout(pWr, pWi, pv, n, dv, _ptr64(Or), _ptr64(Oi))
    return Or + 1j * Oi


def chain(a, b, with_envelope: bool = False):
    """y [n,dv] complex: y_0 = b_0, y_i = a_i y_{i-1} + b_i."""
    a = np.asarray(a, dtype=np.complex128).reshape(-1)
    ba, pb = _f32(b)
    if ba.ndim == 1:
        ba = ba.reshape(-1, 1)
        pb = ba.ctypes.data_as(_f32p)
    n, dv = ba.shape
    ar, par = _f64a(a.real); ai, pai = _f64a(a.imag)
    yr = np.zeros((n, dv)); yi = np.zeros((n, dv)); env = np.zeros((n, dv))
    lib().ro_chain(par, pai, pb, n, dv, _ptr64(yr), _ptr64(yi), _ptr64(env))
    y = yr + 1j * yi
    return (y, env) if with_envelope else y


# ------------------------------------------------------------------ batched

def _per_head(x, BH):
    x = np.asarray(x, dtype=np.float64).reshape(-1)
    if x.size == 1:
        x = np.full(BH, x[0])
    if x.size != BH:
        raise ShapeError()
    return np.ascontiguousarray(x)


def head_rows(q, k, u, theta, v, beta, qk, g, rows, threads: int = 0):
    """O at selected rows for every head.

    q, k [BH,n,d]; v [BH,n,dv]; u, theta [BH,n]; beta/qk/g scalars or [BH].
    Returns (O [BH,nrows,dv] complex, status [BH] int32)."""
    qa, pq = _f32(q); ka, pk = _f32(k); va, pv = _f32(v)
    ua, pu = _f32(u); ta, pt = _f32(theta)
    BH, n, d = qa.shape
    dv = va.shape[2]
    b_, pb_ = _f64a(_per_head(beta, BH)); q_, pq_ = _f64a(_per_head(qk, BH))
    g_, pg_ = _f64a(_per_head(g, BH))
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    Or = np.zeros((BH, r.size, dv)); Oi = np.zeros((BH, r.size, dv))
    st = np.zeros(BH, dtype=np.int32)
    rc = lib().ro_head_rows(pq, pk, pu, pt, pv, BH, n, d, dv, pb_, pq_, pg_,
                            r.ctypes.data_as(_i64p), r.size, _ptr64(Or), _ptr64(Oi),
                            st.ctypes.data_as(_i32p), int(threads))
    if rc == RO_SHAPE:
        raise ShapeError()
    return Or + 1j * Oi, st


def gate_prep(u, theta, g, block: int = 128):
    """Gates and block products for every head; u, theta [BH,n]; g scalar or [BH].

    Returns a dict of m, theta_p [BH,n]; gate, prefix, suffix [BH,n] complex;
    carry [BH,nb] complex; status [BH]."""
    ua, pu = _f32(u); ta, pt = _f32(theta)
    BH, n = ua.shape
    g_, pg_ = _f64a(_per_head(g, BH))
    nb = (n + block - 1) // block
    out = {k: np.zeros((BH, n)) for k in
           ("m", "theta_p", "a_re", "a_im", "p_re", "p_im", "s_re", "s_im")}
    out["c_re"] = np.zeros((BH, nb)); out["c_im"] = np.zeros((BH, nb))
    st = np.zeros(BH, dtype=np.int32)
    rc = lib().ro_gate_prep(pu, pt, pg_, BH, n, block, *[_ptr64(out[k]) for k in (
        "m", "theta_p", "a_re", "a_im", "p_re", "p_im", "s_re", "s_im", "c_re", "c_im")],
        st.ctypes.data_as(_i32p))
    if rc == RO_SHAPE:
        raise ShapeError()
    return {"m": out["m"], "theta_p": out["theta_p"],
            "gate": out["a_re"] + 1j * out["a_im"],
            "prefix": out["p_re"] + 1j * out["p_im"],
            "suffix": out["s_re"] + 1j * out["s_im"],
            "carry": out["c_re"] + 1j * out["c_im"], "status": st}


def chain_heads(u, theta, g, b, threads: int = 0):
    """Chain per head with gates from (u, theta, g); b [BH,n,dv].

    Returns (y [BH,n,dv] complex, envelope [BH,n,dv], status [BH])."""
    ua, pu = _f32(u); ta, pt = _f32(theta); ba, pb = _f32(b)
    BH, n, dv = ba.shape
    g_, pg_ = _f64a(_per_head(g, BH))
    yr = np.zeros((BH, n, dv)); yi = np.zeros((BH, n, dv)); env = np.zeros((BH, n, dv))
    st = np.zeros(BH, dtype=np.int32)
    rc = lib().ro_chain_heads(pu, pt, pg_, pb, BH, n, dv, _ptr64(yr), _ptr64(yi),
                              _ptr64(env), st.ctypes.data_as(_i32p), int(threads))
    if rc == RO_SHAPE:
        raise ShapeError()
    return yr + 1j * yi, env, st


def operator_rows(q, k, u, theta, beta: float, qk: float, g: float, rows) -> np.ndarray:
    """Rows `rows` of W (same arithmetic as operator): [len(rows), n] complex."""
    q = np.asarray(q, dtype=np.float32)
    n = q.shape[0]
    d = q.shape[1] if q.ndim == 2 else 0
    qa, pq = _f32(q); ka, pk = _f32(k); ua, pu = _f32(u); ta, pt = _f32(theta)
    if ka.size != n * d or ua.size != n or ta.size != n:
        raise ShapeError()
    rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    Wr = np.zeros((rr.size, n)); Wi = np.zeros((rr.size, n))
    _raise(lib().ro_operator_rows(pq, pk, pu, pt, n, d, beta, qk, g, rr.ctypes.data_as(_i64p),
                                  rr.size, _ptr64(Wr), _ptr64(Wi)))
    return Wr + 1j * Wi


def position_head(a, v, beta: float, qk: float) -> np.ndarray:
    """O [n,dv] real of one position-only head: logits qk * a(i - j) (a [n], one per offset),
    v [n,dv] (proofs.blah.dev's theorem pos-head-is-causal-convolution, left-hand side, with
    the switches at g = 0)."""
    aa, pa = _f32(a)
    va, pv = _f32(v)
    n = aa.size
    if va.ndim != 2 or va.shape[0] != n:
        raise ShapeError()
    O = np.zeros((n, va.shape[1]))
    _raise(lib().ro_position_head(pa, pv, n, va.shape[1], float(beta), float(qk), _ptr64(O)))
    return O


def position_rows(a, v, beta: float, qk: float, rows) -> np.ndarray:
    """Rows `rows` of one position-only head (same arithmetic as position_head): a [n],
    v [n,dv]; returns O [len(rows), dv]."""
    aa, pa = _f32(a)
    va, pv = _f32(v)
    n = aa.size
    if va.ndim != 2 or va.shape[0] != n:
        raise ShapeError()
    rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    O = np.zeros((rr.size, va.shape[1]))
    _raise(lib().ro_position_rows(pa, pv, n, va.shape[1], float(beta), float(qk),
                                  rr.ctypes.data_as(_i64p), rr.size, _ptr64(O)))
    return O


def position_heads(a, v, beta, qk, threads: int = 0):
    """Position-only heads: a [H,n] (head h of every batch reads row h), v [BH,n,dv];
    beta/qk scalars or [BH]. Returns (O [BH,n,dv], status [BH])."""
    aa, pa = _f32(a)
    va, pv = _f32(v)
    BH, n, dv = va.shape
    H = aa.shape[0]
    if aa.ndim != 2 or aa.shape[1] != n:
        raise ShapeError()
    b_, pb_ = _f64a(_per_head(beta, BH)); q_, pq_ = _f64a(_per_head(qk, BH))
    O = np.zeros((BH, n, dv))
    st = np.zeros(BH, dtype=np.int32)
    rc = lib().ro_position_heads(pa, pv, BH, H, n, dv, pb_, pq_, _ptr64(O),
                                 st.ctypes.data_as(_i32p), int(threads))
    if rc == RO_SHAPE:
        raise ShapeError()
    return O, st
