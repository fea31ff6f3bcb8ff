"""ctypes front end of the float64 C oracle (test infrastructure only).

Builds ``liboracle.so`` next to ``fa_oracle.c`` with the host gcc (no CUDA,
no architecture-specific flags, so it builds the same on x86-64 and aarch64)
and exposes numpy-returning wrappers.  Inputs that carry bfloat16 data may be
given as torch ``bfloat16`` tensors or as numpy ``uint16`` bit arrays; they
are passed to C as raw bits and widened there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)


def library_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into liboracle.so (if missing or older than the source)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # The pin suite's mutation check runs the pins against deliberately
        # broken copies of the oracle; it points this variable at one.
        override = os.environ.get("FA_ORACLE_LIB_OVERRIDE")
        if override:
            lib = ctypes.CDLL(override)
        else:
            build()
            lib = ctypes.CDLL(_LIB)
        lib.oracle_softmax_naive.argtypes = [_dp, ctypes.c_int, _dp]
        lib.oracle_softmax_safe.argtypes = [_dp, ctypes.c_int, _dp]
        lib.oracle_online_softmax_trace.argtypes = [_dp, ctypes.c_int, _dp, _dp]
        lib.oracle_block_state.argtypes = [_dp, _dp, ctypes.c_int, ctypes.c_int, _dp, _dp, _dp]
        lib.oracle_state_merge.argtypes = [ctypes.c_double, ctypes.c_double, _dp,
                                           ctypes.c_double, ctypes.c_double, _dp,
                                           ctypes.c_int, _dp, _dp, _dp]
        lib.oracle_lse_reduce.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, _dp, _dp]
        lib.oracle_attend_scores.argtypes = [_dp, _dp, ctypes.c_int, ctypes.c_int, _dp, _dp]
        lib.oracle_sdpa_rows.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_double, _i32p, _i64p, ctypes.c_int64,
                                         _dp, _dp, ctypes.c_int]
        lib.oracle_sdpa_rows.restype = ctypes.c_int
        lib.oracle_sdpa_forward.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, _i32p, _dp, _dp, ctypes.c_int]
        lib.oracle_sdpa_forward.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [_u16p, _u16p, _u16p, _i32p, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_double, _dp, _dp,
                                      ctypes.c_int]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_decode_paged.argtypes = [_u16p, _u16p, _u16p, _i32p, ctypes.c_int, _i32p, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, _dp, _dp, ctypes.c_int]
        lib.oracle_decode_paged.restype = ctypes.c_int
        lib.oracle_sdpa_forward_f64.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_double, _i32p, _dp, _dp]
        lib.oracle_sdpa_forward_f64.restype = ctypes.c_int
        lib.oracle_sdpa_backward.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_double, _i32p,
                                             _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int]
        lib.oracle_sdpa_backward.restype = ctypes.c_int
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.POINTER(ctypes.c_uint8), ctypes.c_int64, _dp]
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
        return lib


# ---------------------------------------------------------------- marshalling

def _f64(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return a


def _ptr(a: np.ndarray, typ):
    return a.ctypes.data_as(typ)


def _bf16_bits(x) -> np.ndarray:
    """bfloat16 data as a contiguous uint16 numpy array of raw bits."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy bf16 inputs must be uint16 bit arrays")
        return np.ascontiguousarray(x)
    import torch  # only for tensor inputs
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16:
        raise TypeError("expected a torch.bfloat16 tensor or a numpy uint16 array")
    t = x.detach()
    if t.device.type != "cpu":
        t = t.cpu()
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32(x):
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _threads(n):
    return max_threads() if n is None else int(n)


# ------------------------------------------------------------------ pins API

def softmax_naive(x):
    x = _f64(x)
    y = np.empty_like(x)
    _load().oracle_softmax_naive(_ptr(x, _dp), x.size, _ptr(y, _dp))
    return y


def softmax_safe(x):
    x = _f64(x)
    y = np.empty_like(x)
    _load().oracle_softmax_safe(_ptr(x, _dp), x.size, _ptr(y, _dp))
    return y


def online_softmax_trace(x):
    """Running (m_j, d_j) of the element-wise online softmax."""
    x = _f64(x)
    m = np.empty_like(x)
    d = np.empty_like(x)
    _load().oracle_online_softmax_trace(_ptr(x, _dp), x.size, _ptr(m, _dp), _ptr(d, _dp))
    return m, d


def block_state(x, V):
    """(m, l, u) of one block of scores x with value rows V [n, dv]."""
    x = _f64(x)
    V = _f64(V)
    V = V.reshape(x.size, V.shape[-1] if V.ndim > 1 else 1)
    dv = V.shape[1]
    m = ctypes.c_double()
    l_ = ctypes.c_double()
    u = np.empty(dv)
    _load().oracle_block_state(_ptr(x, _dp), _ptr(V, _dp), x.size, dv,
                               ctypes.byref(m), ctypes.byref(l_), _ptr(u, _dp))
    return m.value, l_.value, u


def state_merge(a, b):
    """Merge two (m, l, u) states."""
    ma, la, ua = a
    mb, lb, ub = b
    ua = _f64(ua)
    ub = _f64(ub)
    dv = ua.size
    m = ctypes.c_double()
    l_ = ctypes.c_double()
    u = np.empty(dv)
    _load().oracle_state_merge(float(ma), float(la), _ptr(ua, _dp), float(mb), float(lb),
                               _ptr(ub, _dp), dv, ctypes.byref(m), ctypes.byref(l_), _ptr(u, _dp))
    return m.value, l_.value, u


def lse_reduce(m_k, l_k, O_k):
    """Flash-Decoding reduction of per-chunk (m_k, l_k, O_k); returns (O, L)."""
    m_k = _f64(m_k)
    l_k = _f64(l_k)
    O_k = _f64(O_k).reshape(m_k.size, -1)
    dv = O_k.shape[1]
    O = np.empty(dv)
    L = ctypes.c_double()
    _load().oracle_lse_reduce(_ptr(m_k, _dp), _ptr(l_k, _dp), _ptr(O_k, _dp), m_k.size, dv,
                              _ptr(O, _dp), ctypes.byref(L))
    return O, L.value


def attend_scores(x, V):
    """Stable-softmax attention of one query over explicit scores; returns (O, L)."""
    x = _f64(x)
    V = _f64(V)
    V = V.reshape(x.size, V.shape[-1] if V.ndim > 1 else 1)
    dv = V.shape[1]
    O = np.empty(dv)
    L = ctypes.c_double()
    _load().oracle_attend_scores(_ptr(x, _dp), _ptr(V, _dp), x.size, dv, _ptr(O, _dp),
                                 ctypes.byref(L))
    return O, L.value


# -------------------------------------------------------------- attention API

def _shape4(x):
    shp = tuple(x.shape)
    if len(shp) != 4:
        raise ValueError("expected a [B, H, N, d] tensor")
    return shp


def sdpa_rows(Q, K, V, rows, causal=False, scale=None, key_len=None, nthreads=None):
    """Selected query rows of exact attention.

    ``rows`` holds flat row indices (b * H + h) * Nq + i.  Returns O [n, d]
    and L [n] in float64.
    """
    B, H, Nq, d = _shape4(Q)
    _, _, Nk, _ = _shape4(K)
    q = _bf16_bits(Q)
    k = _bf16_bits(K)
    v = _bf16_bits(V)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kl = _i32(key_len)
    O = np.empty((rows.size, d))
    L = np.empty(rows.size)
    rc = _load().oracle_sdpa_rows(_ptr(q, _u16p), _ptr(k, _u16p), _ptr(v, _u16p), B, H, Nq, Nk,
                                  d, int(bool(causal)), float(scale),
                                  None if kl is None else _ptr(kl, _i32p),
                                  _ptr(rows, _i64p), rows.size, _ptr(O, _dp), _ptr(L, _dp),
                                  _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_sdpa_rows rejected its arguments")
    return O, L


def sdpa_forward(Q, K, V, causal=False, scale=None, key_len=None, nthreads=None):
    """Every row of exact attention: O [B,H,N,d] and L [B,H,N] in float64."""
    B, H, N, d = _shape4(Q)
    q = _bf16_bits(Q)
    k = _bf16_bits(K)
    v = _bf16_bits(V)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kl = _i32(key_len)
    O = np.empty((B, H, N, d))
    L = np.empty((B, H, N))
    rc = _load().oracle_sdpa_forward(_ptr(q, _u16p), _ptr(k, _u16p), _ptr(v, _u16p), B, H, N, d,
                                     int(bool(causal)), float(scale),
                                     None if kl is None else _ptr(kl, _i32p),
                                     _ptr(O, _dp), _ptr(L, _dp), _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_sdpa_forward rejected its arguments")
    return O, L


def decode(q, Kc, Vc, seqlens, scale=None, nthreads=None):
    """Single-query attention over the first seqlens[b] cached keys (no split).

    q: [B, H, d]; Kc, Vc: [B, H, Lmax, d].  Returns O [B, H, d], L [B, H].
    """
    B, H, d = tuple(q.shape)
    _, _, Lmax, _ = _shape4(Kc)
    qb = _bf16_bits(q)
    kb = _bf16_bits(Kc)
    vb = _bf16_bits(Vc)
    sl = _i32(seqlens)
    if sl is None or sl.size != B:
        raise ValueError("seqlens must hold B entries")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    O = np.empty((B, H, d))
    L = np.empty((B, H))
    rc = _load().oracle_decode(_ptr(qb, _u16p), _ptr(kb, _u16p), _ptr(vb, _u16p),
                               _ptr(sl, _i32p), B, H, Lmax, d, float(scale), _ptr(O, _dp),
                               _ptr(L, _dp), _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments")
    return O, L


def decode_paged(q, Kpool, Vpool, block_table, seqlens, scale=None, nthreads=None):
    """Single-query attention through a block table (no split).

    q: [B, H, d]; Kpool, Vpool: [num_blocks, H, block_size, d];
    block_table: int32 [B, max_blocks].  Returns O [B, H, d], L [B, H].
    """
    B, H, d = tuple(q.shape)
    nblk, H2, bs, d2 = tuple(Kpool.shape)
    if H2 != H or d2 != d:
        raise ValueError("pool must be [num_blocks, H, block_size, d]")
    qb = _bf16_bits(q)
    kb = _bf16_bits(Kpool)
    vb = _bf16_bits(Vpool)
    bt = _i32(block_table)
    if bt.ndim != 2 or bt.shape[0] != B:
        raise ValueError("block_table must be [B, max_blocks]")
    sl = _i32(seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    O = np.empty((B, H, d))
    L = np.empty((B, H))
    rc = _load().oracle_decode_paged(_ptr(qb, _u16p), _ptr(kb, _u16p), _ptr(vb, _u16p),
                                     _ptr(np.ascontiguousarray(bt), _i32p), bt.shape[1],
                                     _ptr(sl, _i32p), B, H, nblk, bs, d, float(scale),
                                     _ptr(O, _dp), _ptr(L, _dp), _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode_paged rejected its arguments (table entry out of range?)")
    return O, L



def _as_f64_4d(x):
    """float64 copy of a [B, H, N, d] input (torch tensors of any float dtype are widened exactly)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if a.ndim != 4:
        raise ValueError("expected a [B, H, N, d] array")
    return a


def sdpa_forward_f64(Q, K, V, causal=False, scale=None, key_len=None):
    """Exact attention on float64 inputs: O [B,H,N,d], L [B,H,N] (single thread)."""
    q, k, v = _as_f64_4d(Q), _as_f64_4d(K), _as_f64_4d(V)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kl = _i32(key_len)
    O = np.empty((B, H, N, d))
    L = np.empty((B, H, N))
    rc = _load().oracle_sdpa_forward_f64(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), B, H, N, d,
                                         int(bool(causal)), float(scale),
                                         None if kl is None else _ptr(kl, _i32p), _ptr(O, _dp), _ptr(L, _dp))
    if rc != 0:
        raise ValueError("oracle_sdpa_forward_f64 rejected its arguments")
    return O, L


def sdpa_backward(Q, K, V, dO, causal=False, scale=None, key_len=None, magnitudes=False, nthreads=None):
    """Gradients of exact attention with respect to Q, K, V for upstream gradient dO.

    All inputs [B, H, N, d] (bf16 tensors are widened exactly).  Returns a
    dict with dQ, dK, dV [B,H,N,d], D and L [B,H,N] in float64, and with
    magnitudes=True also M_dQ, M_dK, M_dV: per-element sums of the terms'
    magnitudes (see fa_oracle.c) for rounding-error bounds.
    """
    q, k, v, g = _as_f64_4d(Q), _as_f64_4d(K), _as_f64_4d(V), _as_f64_4d(dO)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kl = _i32(key_len)
    dQ = np.empty((B, H, N, d))
    dK = np.empty((B, H, N, d))
    dV = np.empty((B, H, N, d))
    D = np.empty((B, H, N))
    L = np.empty((B, H, N))
    mag = np.empty((3, B, H, N, d)) if magnitudes else None
    rc = _load().oracle_sdpa_backward(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(g, _dp), B, H, N, d,
                                      int(bool(causal)), float(scale), None if kl is None else _ptr(kl, _i32p),
                                      _ptr(dQ, _dp), _ptr(dK, _dp), _ptr(dV, _dp), _ptr(D, _dp), _ptr(L, _dp),
                                      None if mag is None else _ptr(mag, _dp), _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_sdpa_backward rejected its arguments")
    out = dict(dQ=dQ, dK=dK, dV=dV, D=D, L=L)
    if magnitudes:
        out.update(M_dV=mag[0], M_dK=mag[1], M_dQ=mag[2])
    return out


def e4m3_to_f64(x):
    """Exact float64 values of E4M3 codes (a uint8 numpy array or a torch float8_e4m3fn/uint8 tensor)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            t = x.detach().cpu().contiguous()
            if t.dtype != torch.uint8:
                t = t.view(torch.uint8)
            x = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(np.asarray(x, dtype=np.uint8))
    out = np.empty(a.shape, dtype=np.float64)
    _load().oracle_e4m3_to_f64(a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), a.size, _ptr(out, _dp))
    return out


def sdpa_forward_e4m3(Q8, K8, V8, causal=False, scale=None, key_len=None):
    """Exact attention on E4M3 inputs (codes decoded exactly): O [B,H,N,d], L [B,H,N]."""
    return sdpa_forward_f64(e4m3_to_f64(Q8), e4m3_to_f64(K8), e4m3_to_f64(V8), causal=causal, scale=scale,
                            key_len=key_len)
