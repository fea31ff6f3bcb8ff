"""fa_decode_noalloc: split-KV decode without a caller-provided workspace.

For callers that cannot allocate device memory while they decode, the
library keeps the split partials in one fixed array of its own.  These tests
call that entry point through the C ABI, twice in a row on different inputs,
and compare it with fa_decode (which takes the caller's workspace) within the
parity tolerances.  The file is named so that it is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_tiled_gb300 import workloads
from gpu_util import O_TOL, L_TOL

pytestmark = pytest.mark.gpu

FA_ERR_WORKSPACE = 4
NOALLOC_MAX_BYTES = 8 << 20


def _lib():
    import exact_attention_tiled_gb300 as fa
    return fa.library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _host(vals):
    buf = (ctypes.c_int32 * len(vals))(*[int(v) for v in vals])
    return ctypes.cast(buf, ctypes.c_void_p), buf


def _run_pair(B, H, Lmax, d, lens, splits, seed):
    lib = _lib()
    dev = torch.device("cuda")
    q, Kc, Vc = workloads.decode_inputs(B, H, Lmax, d, seed, device=dev)
    seqlens = torch.tensor(lens, dtype=torch.int32, device=dev)
    hp, keep = _host(lens)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    scale = ctypes.c_float(0.0)

    O_na = torch.empty_like(q)
    L_na = torch.empty((B, H), device=dev, dtype=torch.float32)
    st = lib.fa_decode_noalloc(_p(q), _p(Kc), _p(Vc), _p(seqlens), hp, _p(O_na), _p(L_na), B, H, Lmax, d,
                               scale, splits, stream)
    assert st == 0, f"fa_decode_noalloc returned {st}"

    need = lib.fa_decode_workspace_bytes_for_lengths(B, H, Lmax, d, splits, hp)
    assert 0 < need <= NOALLOC_MAX_BYTES
    ws = torch.empty(need, device=dev, dtype=torch.uint8)
    O_ref = torch.empty_like(q)
    L_ref = torch.empty((B, H), device=dev, dtype=torch.float32)
    st = lib.fa_decode(_p(q), _p(Kc), _p(Vc), _p(seqlens), hp, _p(O_ref), _p(L_ref), B, H, Lmax, d, scale,
                       splits, _p(ws), ctypes.c_size_t(need), stream)
    assert st == 0, f"fa_decode returned {st}"
    torch.cuda.synchronize()
    del keep
    eo = (O_na.float() - O_ref.float()).abs().max().item()
    el = (L_na - L_ref).abs().max().item()
    assert np.isfinite(eo) and eo <= O_TOL, f"max|dO| {eo}"
    assert np.isfinite(el) and el <= L_TOL, f"max|dL| {el}"


def test_noalloc_matches_workspace_entry_point_twice():
    # two calls in a row on different shapes: the second reuses the shared array
    _run_pair(B=4, H=8, Lmax=3000, d=128, lens=[3000, 1, 1777, 640], splits=0, seed=61)
    _run_pair(B=3, H=4, Lmax=1000, d=64, lens=[999, 64, 500], splits=5, seed=62)


# d = 64 and 25 * 31 * 41 = 31775 partial slots: 31775 * 64 * 4 bytes of O_k plus
# 31775 * 8 bytes of (m_k, l_k), each rounded up to 256 bytes, fill the array exactly.
EDGE = dict(B=25, H=31, Lmax=41 * 64, d=64, splits=41)


def test_noalloc_request_that_fills_the_array_exactly():
    lib = _lib()
    e = EDGE
    assert lib.fa_decode_workspace_bytes_for_lengths(e["B"], e["H"], e["Lmax"], e["d"], e["splits"], None) \
        == NOALLOC_MAX_BYTES
    lens = np.random.default_rng(63).integers(1, e["Lmax"] + 1, e["B"]).tolist()
    lens[0] = e["Lmax"]
    _run_pair(B=e["B"], H=e["H"], Lmax=e["Lmax"], d=e["d"], lens=lens, splits=e["splits"], seed=63)


def test_noalloc_rejects_requests_beyond_its_array():
    lib = _lib()
    e = EDGE
    # one more chunk per sequence than the exact fit; null pointers: the size
    # check comes first, and fa_decode would reject null pointers before a launch
    need = lib.fa_decode_workspace_bytes_for_lengths(e["B"], e["H"], e["Lmax"], e["d"], e["splits"] + 1, None)
    assert need > NOALLOC_MAX_BYTES
    st = lib.fa_decode_noalloc(None, None, None, None, None, None, None, e["B"], e["H"], e["Lmax"], e["d"],
                               ctypes.c_float(0.0), e["splits"] + 1, None)
    assert st == FA_ERR_WORKSPACE
    B, H, Lmax, d, splits = 64, 64, 65536, 128, 64
    assert lib.fa_decode_workspace_bytes_for_lengths(B, H, Lmax, d, splits, None) > NOALLOC_MAX_BYTES
    st = lib.fa_decode_noalloc(None, None, None, None, None, None, None, B, H, Lmax, d, ctypes.c_float(0.0),
                               splits, None)
    assert st == FA_ERR_WORKSPACE
