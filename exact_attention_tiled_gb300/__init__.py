"""GB300-native exact tiled attention: Python binding of libfa.so.

This module only marshals arguments: it checks that tensors are CUDA bf16 and
contiguous, allocates outputs with torch, and passes raw device pointers and
the current CUDA stream to the C ABI declared in ``include/fa.h``.  Every step
of the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and the calls raise if ``libfa.so`` is missing.

    fa_forward(Q, K, V, causal=False, scale=None, key_len=None) -> (O, L)
    fa_decode(q, Kcache, Vcache, seqlens, num_splits=0, ...)   -> (O, L)
    fa_decode_paged(q, Kpool, Vpool, block_table, seqlens, ...) -> (O, L)
    fa_backward(Q, K, V, O, dO, L, causal=False, ...)           -> (dQ, dK, dV)
    fa_forward_fp8(Q8, K8, V8, causal=False, ...)               -> (O, L)
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["fa_forward", "fa_forward_host", "fa_forward_host_workspace_bytes", "fa_forward_fp8", "fa_backward", "fa_backward_workspace_bytes", "fa_decode", "fa_decode_paged", "fa_decode_plan", "fa_decode_workspace_bytes",
           "fa_device_error", "fa_get_last_device_error", "fa_shutdown", "FaError", "library", "library_path", "STATUS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfa.so")
_lock = threading.Lock()
_lib = None

STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA",
          4: "FA_ERR_WORKSPACE", 5: "FA_ERR_DEVICE_TIMEOUT"}

_vp = ctypes.c_void_p
_i = ctypes.c_int


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def library():
    """Load libfa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"{_LIB_PATH} is missing: build it with exact_attention_tiled_gb300.build.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        lib.fa_forward.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _vp, _vp]
        lib.fa_forward.restype = _i
        lib.fa_forward_count_tiles.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _vp,
                                               _vp, _vp]
        lib.fa_forward_count_tiles.restype = _i
        lib.fa_forward_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _vp, _i,
                                        _vp, ctypes.c_size_t, _vp]
        lib.fa_forward_host.restype = _i
        lib.fa_forward_host_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
        lib.fa_forward_host_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, ctypes.c_float, _i,
                                  _vp, ctypes.c_size_t, _vp]
        lib.fa_decode.restype = _i
        lib.fa_backward.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                    ctypes.c_float, _vp, _vp, ctypes.c_size_t, _vp]
        lib.fa_backward.restype = _i
        lib.fa_backward_workspace_bytes.argtypes = [_i, _i, _i, _i]
        lib.fa_backward_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_backward_atomic_dq.argtypes = lib.fa_backward.argtypes
        lib.fa_backward_atomic_dq.restype = _i
        lib.fa_backward_atomic_dq_workspace_bytes.argtypes = [_i, _i, _i, _i]
        lib.fa_backward_atomic_dq_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_forward_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_float, _vp, _vp,
                                        ctypes.c_size_t, _vp]
        lib.fa_forward_fp8.restype = _i
        lib.fa_forward_fp8_workspace_bytes.argtypes = [_i, _i, _i, _i]
        lib.fa_forward_fp8_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_decode_paged.argtypes = [_vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                         ctypes.c_float, _i, _vp, ctypes.c_size_t, _vp]
        lib.fa_decode_paged.restype = _i
        lib.fa_decode_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, ctypes.c_float,
                                          _i, _vp]
        lib.fa_decode_noalloc.restype = _i
        lib.fa_decode_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
        lib.fa_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_decode_workspace_bytes_for_lengths.argtypes = [_i, _i, _i, _i, _i, _vp]
        lib.fa_decode_workspace_bytes_for_lengths.restype = ctypes.c_size_t
        lib.fa_decode_plan.argtypes = [_i, _i, _i, _i, _i, _vp, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)]
        lib.fa_decode_plan.restype = _i
        lib.fa_status_string.argtypes = [_i]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_device_error.argtypes = [_i, ctypes.POINTER(_i)]
        lib.fa_device_error.restype = _i
        lib.fa_get_last_device_error.argtypes = []
        lib.fa_get_last_device_error.restype = _i
        lib.fa_version.restype = _i
        lib.fa_shutdown.argtypes = []
        lib.fa_shutdown.restype = _i
        lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_uint, _vp]
        lib.fa_selftest_wait_timeout.restype = _i
        _lib = lib
        return lib


def _torch():
    import torch
    return torch


def _check_bf16(name, t, ndim):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor")


def _stream_handle(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _host_i32(x):
    """(ctypes buffer, keep-alive) of a host int32 array, or (None, None)."""
    if x is None:
        return None, None
    torch = _torch()
    if isinstance(x, torch.Tensor):
        vals = [int(v) for v in x.detach().cpu().tolist()]
    else:
        vals = [int(v) for v in x]
    buf = (ctypes.c_int32 * len(vals))(*vals)
    return ctypes.cast(buf, ctypes.c_void_p), buf


def fa_forward(Q, K, V, causal=False, scale=None, key_len=None, out=None, lse=None,
               return_lse=True, stream=None, tile_counts=None):
    """Exact attention forward.  Q, K, V: CUDA bf16 [B, H, N, d]; returns (O, L).

    key_len: optional CUDA int32 [B] key-padding lengths.  L is float32
    [B, H, N] (None when return_lse=False and no `lse` buffer is given).
    tile_counts: optional CUDA int32 [B, H, 2]; when given, the call goes
    through fa_forward_count_tiles and the tensor receives the number of S
    and P V tile products issued per (batch, head).
    """
    torch = _torch()
    for n, t in (("Q", Q), ("K", K), ("V", V)):
        _check_bf16(n, t, 4)
    if K.shape != Q.shape or V.shape != Q.shape:
        raise ValueError("Q, K, V must share the shape [B, H, N, d]")
    B, H, N, d = Q.shape
    if out is None:
        out = torch.empty_like(Q)
    else:
        _check_bf16("out", out, 4)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), device=Q.device, dtype=torch.float32)
    if key_len is not None:
        if key_len.dtype != torch.int32 or not key_len.is_cuda or key_len.numel() != B:
            raise TypeError("key_len must be a CUDA int32 tensor with B entries")
        key_len = key_len.contiguous()
    sc = float(scale) if scale is not None else 0.0
    if tile_counts is not None:
        if (tile_counts.dtype != torch.int32 or not tile_counts.is_cuda or tuple(tile_counts.shape) != (B, H, 2)
                or not tile_counts.is_contiguous()):
            raise TypeError("tile_counts must be a contiguous CUDA int32 tensor [B, H, 2]")
        st = library().fa_forward_count_tiles(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), _ptr(lse), B, H, N, d,
                                              int(bool(causal)), sc, _ptr(key_len), _ptr(tile_counts),
                                              _stream_handle(stream))
        if st != 0:
            raise FaError(st, "fa_forward_count_tiles")
        return out, lse
    st = library().fa_forward(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), _ptr(lse), B, H, N, d,
                              int(bool(causal)), sc, _ptr(key_len), _stream_handle(stream))
    if st != 0:
        raise FaError(st, "fa_forward")
    return out, lse


def _check_host_bf16(name, t):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) bfloat16 tensor")
    if t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 4-D tensor")


def fa_forward_host_workspace_bytes(B, H, N, d, heads_per_group=0):
    """Device scratch bytes fa_forward_host needs (0 for an invalid shape)."""
    return int(library().fa_forward_host_workspace_bytes(B, H, N, d, heads_per_group))


def fa_forward_host(Q, K, V, causal=False, scale=None, key_len=None, out=None, lse=None, return_lse=True,
                    heads_per_group=0, workspace=None, stream=None, device=None):
    """fa_forward over HOST bf16 tensors [B, H, N, d]; returns host (O, L).

    The library copies groups of heads to the device, runs the forward on each and
    copies the results back, overlapping the copies of one group with the work of
    the others.  Pinned inputs (and outputs: allocated pinned when Q is pinned) let
    the copies run asynchronously; the results are complete once `stream` (the
    current stream of `device` by default) is synchronised.  key_len: optional
    host int32 [B]; workspace: optional CUDA uint8 scratch.
    """
    torch = _torch()
    for n, t in (("Q", Q), ("K", K), ("V", V)):
        _check_host_bf16(n, t)
    if K.shape != Q.shape or V.shape != Q.shape:
        raise ValueError("Q, K, V must share the shape [B, H, N, d]")
    B, H, N, d = Q.shape
    pin = Q.is_pinned()
    if out is None:
        out = torch.empty(Q.shape, dtype=torch.bfloat16, pin_memory=pin)
    else:
        _check_host_bf16("out", out)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    if lse is not None and (lse.is_cuda or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise TypeError("lse must be a contiguous host float32 tensor")
    kl = None
    if key_len is not None:
        kl = torch.as_tensor(key_len, dtype=torch.int32).cpu().contiguous()
        if kl.numel() != B:
            raise ValueError("key_len must have B entries")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    need = library().fa_forward_host_workspace_bytes(B, H, N, d, heads_per_group)
    if need == 0:
        raise FaError(1, "fa_forward_host (shape or heads_per_group)")
    if workspace is None:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    with torch.cuda.device(dev):
        st = library().fa_forward_host(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), _ptr(lse), B, H, N, d,
                                       int(bool(causal)), float(scale) if scale is not None else 0.0, _ptr(kl),
                                       int(heads_per_group), _ptr(workspace), workspace.numel(),
                                       _stream_handle(stream))
    if st != 0:
        raise FaError(st, "fa_forward_host")
    return out, lse


def _check_e4m3(name, t):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"{name} must be a CUDA float8_e4m3fn (or uint8 E4M3 code) tensor")
    if t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 4-D tensor")


def fa_forward_fp8(Q8, K8, V8, causal=False, scale=None, key_len=None, out=None, lse=None, return_lse=True,
                   workspace=None, stream=None):
    """Exact attention over E4M3 inputs [B, H, N, 128]; returns (O bf16, L float32)."""
    torch = _torch()
    for n, t in (("Q8", Q8), ("K8", K8), ("V8", V8)):
        _check_e4m3(n, t)
        if t.shape != Q8.shape:
            raise ValueError(f"{n} must have the shape of Q8")
    B, H, N, d = Q8.shape
    if out is None:
        out = torch.empty((B, H, N, d), device=Q8.device, dtype=torch.bfloat16)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), device=Q8.device, dtype=torch.float32)
    if key_len is not None:
        if key_len.dtype != torch.int32 or not key_len.is_cuda or key_len.numel() != B:
            raise TypeError("key_len must be a CUDA int32 tensor with B entries")
        key_len = key_len.contiguous()
    need = library().fa_forward_fp8_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), device=Q8.device, dtype=torch.uint8)
    st = library().fa_forward_fp8(_ptr(Q8), _ptr(K8), _ptr(V8), _ptr(out), _ptr(lse), B, H, N, d,
                                  int(bool(causal)), float(scale) if scale is not None else 0.0, _ptr(key_len),
                                  _ptr(workspace), workspace.numel(), _stream_handle(stream))
    if st != 0:
        raise FaError(st, "fa_forward_fp8")
    return out, lse


def fa_forward_fp8_workspace_bytes(B, H, N, d):
    return int(library().fa_forward_fp8_workspace_bytes(B, H, N, d))


def fa_backward_workspace_bytes(B, H, N, d):
    return int(library().fa_backward_workspace_bytes(B, H, N, d))


def fa_backward(Q, K, V, O, dO, L, causal=False, scale=None, key_len=None, dQ=None, dK=None, dV=None,
                workspace=None, stream=None, atomic_dq=False):
    """Gradients (dQ, dK, dV) of exact attention; all bf16 [B, H, N, d] on the GPU.

    O and L are the outputs of fa_forward for the same Q, K, V, causal, scale
    and key_len; dO is the upstream gradient of O.  atomic_dq=True (d = 64)
    calls fa_backward_atomic_dq: dQ accumulated by fp32 atomics, less work,
    dQ not bitwise reproducible.
    """
    torch = _torch()
    for n, t in (("Q", Q), ("K", K), ("V", V), ("O", O), ("dO", dO)):
        _check_bf16(n, t, 4)
        if t.shape != Q.shape:
            raise ValueError(f"{n} must have the shape of Q")
    B, H, N, d = Q.shape
    if L is None or L.dtype != torch.float32 or not L.is_cuda or tuple(L.shape) != (B, H, N):
        raise TypeError("L must be a CUDA float32 tensor [B, H, N]")
    L = L.contiguous()
    if key_len is not None:
        if key_len.dtype != torch.int32 or not key_len.is_cuda or key_len.numel() != B:
            raise TypeError("key_len must be a CUDA int32 tensor with B entries")
        key_len = key_len.contiguous()
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(Q) if dK is None else dK
    dV = torch.empty_like(Q) if dV is None else dV
    for n, t in (("dQ", dQ), ("dK", dK), ("dV", dV)):
        _check_bf16(n, t, 4)
    lib = library()
    need = (lib.fa_backward_atomic_dq_workspace_bytes if atomic_dq else lib.fa_backward_workspace_bytes)(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), device=Q.device, dtype=torch.uint8)
    fn, name = (lib.fa_backward_atomic_dq, "fa_backward_atomic_dq") if atomic_dq else (lib.fa_backward, "fa_backward")
    st = fn(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L), _ptr(dQ), _ptr(dK), _ptr(dV), B, H, N, d,
            int(bool(causal)), float(scale) if scale is not None else 0.0, _ptr(key_len), _ptr(workspace),
            workspace.numel(), _stream_handle(stream))
    if st != 0:
        raise FaError(st, name)
    return dQ, dK, dV


def fa_decode_plan(B, H, Lmax, d, num_splits=0, seqlens_host=None, num_sms=0):
    """(chunk_len, max_chunks) of the split plan fa_decode would use."""
    hp, keep = _host_i32(seqlens_host)
    c, m = _i(), _i()
    st = library().fa_decode_plan(B, H, Lmax, d, num_splits, hp, num_sms, ctypes.byref(c), ctypes.byref(m))
    del keep
    if st != 0:
        raise FaError(st, "fa_decode_plan")
    return c.value, m.value


def fa_decode_workspace_bytes(B, H, Lmax, d, num_splits=0, seqlens_host=None):
    """Decode workspace bytes: without seqlens_host the bound for any lengths,
    with it the exact size of that call on the current device."""
    if seqlens_host is None:
        return int(library().fa_decode_workspace_bytes(B, H, Lmax, d, num_splits))
    hp, keep = _host_i32(seqlens_host)
    n = library().fa_decode_workspace_bytes_for_lengths(B, H, Lmax, d, num_splits, hp)
    del keep
    return int(n)


def fa_decode(q, Kcache, Vcache, seqlens, num_splits=0, scale=None, seqlens_host=None,
              out=None, lse=None, return_lse=True, workspace=None, stream=None):
    """Split-KV single-query attention.  q: [B, H, d]; caches [B, H, Lmax, d].

    seqlens: CUDA int32 [B].  seqlens_host: optional host copy used for the
    split plan (defaults to a host copy of seqlens, which synchronises).
    Returns (O [B, H, d] bf16, L [B, H] float32).
    """
    torch = _torch()
    _check_bf16("q", q, 3)
    _check_bf16("Kcache", Kcache, 4)
    _check_bf16("Vcache", Vcache, 4)
    B, H, Lmax, d = Kcache.shape
    if Vcache.shape != Kcache.shape or tuple(q.shape) != (B, H, d):
        raise ValueError("q must be [B, H, d] and the caches [B, H, Lmax, d]")
    if seqlens.dtype != torch.int32 or not seqlens.is_cuda or seqlens.numel() != B:
        raise TypeError("seqlens must be a CUDA int32 tensor with B entries")
    seqlens = seqlens.contiguous()
    if seqlens_host is None:
        seqlens_host = seqlens.cpu()
    hp, keep = _host_i32(seqlens_host)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H), device=q.device, dtype=torch.float32)
    need = library().fa_decode_workspace_bytes_for_lengths(B, H, Lmax, d, num_splits, hp)
    if workspace is None:
        workspace = torch.empty(max(need, 256), device=q.device, dtype=torch.uint8)
    st = library().fa_decode(_ptr(q), _ptr(Kcache), _ptr(Vcache), _ptr(seqlens), hp, _ptr(out),
                             _ptr(lse), B, H, Lmax, d, float(scale) if scale is not None else 0.0,
                             int(num_splits), _ptr(workspace), workspace.numel(), _stream_handle(stream))
    del keep
    if st != 0:
        raise FaError(st, "fa_decode")
    return out, lse


def fa_decode_paged(q, Kpool, Vpool, block_table, seqlens, num_splits=0, scale=None, seqlens_host=None,
                    out=None, lse=None, return_lse=True, workspace=None, stream=None):
    """Split-KV decode over a paged cache.  q: [B, H, d]; pools [num_blocks, H, block_size, d].

    block_table: CUDA int32 [B, max_blocks]; token t of sequence b is row
    t % block_size of pool block block_table[b, t // block_size].
    Returns (O [B, H, d] bf16, L [B, H] float32).
    """
    torch = _torch()
    _check_bf16("q", q, 3)
    _check_bf16("Kpool", Kpool, 4)
    _check_bf16("Vpool", Vpool, 4)
    num_blocks, H, bs, d = Kpool.shape
    B = q.shape[0]
    if Vpool.shape != Kpool.shape or tuple(q.shape) != (B, H, d):
        raise ValueError("q must be [B, H, d] and the pools [num_blocks, H, block_size, d]")
    if (block_table.dtype != torch.int32 or not block_table.is_cuda or block_table.dim() != 2
            or block_table.shape[0] != B):
        raise TypeError("block_table must be a CUDA int32 tensor [B, max_blocks]")
    block_table = block_table.contiguous()
    max_blocks = block_table.shape[1]
    if seqlens.dtype != torch.int32 or not seqlens.is_cuda or seqlens.numel() != B:
        raise TypeError("seqlens must be a CUDA int32 tensor with B entries")
    seqlens = seqlens.contiguous()
    if seqlens_host is None:
        seqlens_host = seqlens.cpu()
    hp, keep = _host_i32(seqlens_host)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H), device=q.device, dtype=torch.float32)
    need = library().fa_decode_workspace_bytes_for_lengths(B, H, max_blocks * bs, d, num_splits, hp)
    if workspace is None:
        workspace = torch.empty(max(need, 256), device=q.device, dtype=torch.uint8)
    st = library().fa_decode_paged(_ptr(q), _ptr(Kpool), _ptr(Vpool), _ptr(block_table), max_blocks,
                                   _ptr(seqlens), hp, _ptr(out), _ptr(lse), B, H, num_blocks, bs, d,
                                   float(scale) if scale is not None else 0.0, int(num_splits),
                                   _ptr(workspace), workspace.numel(), _stream_handle(stream))
    del keep
    if st != 0:
        raise FaError(st, "fa_decode_paged")
    return out, lse


def fa_device_error(clear=True):
    """(status, site) of the device error word; synchronises the device."""
    site = _i()
    st = library().fa_device_error(int(bool(clear)), ctypes.byref(site))
    return st, site.value


def fa_get_last_device_error():
    """Status of the device error word, which is then reset; synchronises the device."""
    return int(library().fa_get_last_device_error())


def fa_shutdown():
    """Release the library's streams, events and per-device lookups (status code).

    Call with no other library call running; the next call sets them up again.
    """
    return int(library().fa_shutdown())
