"""Host-side checks of the C ABI (no GPU needed).

The library loads without a GPU, exports every entry point include/fa.h
declares, rejects bad arguments before touching CUDA, and plans decode splits
with pure host arithmetic.
"""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_tiled_gb300 import build
    build.build()
    import exact_attention_tiled_gb300 as fa
    return fa.library()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    return sorted(set(re.findall(r"FA_API\s+[\w\s\*]*?\b(fa_\w+)\s*\(", text)))


def test_header_declares_the_api():
    names = _declared_symbols()
    # the boundary's calls, by the names the scope table gives them
    assert {"fa_forward", "fa_decode", "fa_decode_workspace_bytes", "fa_status_string",
            "fa_get_last_device_error"} <= set(names)
    # and this library's additions
    assert {"fa_decode_plan", "fa_decode_workspace_bytes_for_lengths", "fa_device_error", "fa_version",
            "fa_decode_paged", "fa_backward", "fa_forward_fp8", "fa_forward_host",
            "fa_decode_noalloc", "fa_shutdown", "fa_backward_atomic_dq"} <= set(names)


def test_boundary_signatures(lib):
    """Each boundary call, through ctypes, with the argument list the header gives it."""
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    flat = " ".join(text.split())
    assert "size_t fa_decode_workspace_bytes(int B, int H, int Lmax, int d, int num_splits);" in flat
    assert "fa_status fa_get_last_device_error(void);" in flat
    assert ("fa_status fa_forward(const void *Q, const void *K, const void *V, void *O, float *L, int B, int H, "
            "int N, int d, int causal, float scale, const int32_t *key_len, fa_stream_t stream);") in flat
    f = lib.fa_decode_workspace_bytes
    f.argtypes = [ctypes.c_int] * 5
    f.restype = ctypes.c_size_t
    assert f(1, 32, 32768, 128, 8) > 0
    assert f(1, 32, 32768, 96, 8) == 0
    g = lib.fa_get_last_device_error
    g.argtypes = []
    g.restype = ctypes.c_int
    # without a GPU the device cannot be queried: a CUDA error, never a crash
    import torch
    if not torch.cuda.is_available():
        assert g() == 3


def test_shutdown_with_nothing_cached_touches_no_device(lib):
    """fa_shutdown before any call that caches state: FA_OK, even without a GPU, and twice."""
    lib.fa_shutdown.argtypes = []
    lib.fa_shutdown.restype = ctypes.c_int
    assert lib.fa_shutdown() == 0
    assert lib.fa_shutdown() == 0


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), f"libfa.so does not export {name}"


def test_status_strings(lib):
    for code, name in [(0, b"FA_OK"), (1, b"FA_ERR_INVALID_ARG"), (2, b"FA_ERR_UNSUPPORTED"),
                       (3, b"FA_ERR_CUDA"), (4, b"FA_ERR_WORKSPACE"), (5, b"FA_ERR_DEVICE_TIMEOUT")]:
        assert lib.fa_status_string(code) == name
    assert lib.fa_version() >= 100


FAKE = 0x100000  # a 16-byte aligned, never-dereferenced address


def _fwd(lib, **kw):
    a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, L=None, B=1, H=1, N=16, d=64, causal=0, scale=0.0,
             key_len=None)
    a.update(kw)
    return lib.fa_forward(a["Q"], a["K"], a["V"], a["O"], a["L"], a["B"], a["H"], a["N"], a["d"],
                          a["causal"], ctypes.c_float(a["scale"]), a["key_len"], None)


def test_forward_rejects_bad_arguments_before_cuda(lib):
    assert _fwd(lib, Q=None) == 1
    assert _fwd(lib, O=None) == 1
    assert _fwd(lib, N=0) == 1
    assert _fwd(lib, B=0) == 1
    assert _fwd(lib, H=-3) == 1
    assert _fwd(lib, causal=2) == 1
    assert _fwd(lib, K=FAKE + 8) == 1          # not 16-byte aligned
    assert _fwd(lib, L=FAKE + 2) == 1          # not 4-byte aligned
    assert _fwd(lib, key_len=FAKE + 1) == 1
    assert _fwd(lib, scale=float("nan")) == 1
    assert _fwd(lib, d=96) == 2
    assert _fwd(lib, d=256) == 2
    assert _fwd(lib, B=70000) == 1


def _dec(lib, **kw):
    a = dict(q=FAKE, K=FAKE, V=FAKE, sl=FAKE, slh=None, O=FAKE, L=None, B=2, H=2, Lmax=128, d=128,
             scale=0.0, splits=4, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    return lib.fa_decode(a["q"], a["K"], a["V"], a["sl"], a["slh"], a["O"], a["L"], a["B"], a["H"],
                         a["Lmax"], a["d"], ctypes.c_float(a["scale"]), a["splits"], a["ws"], a["wsb"],
                         None)


def test_decode_rejects_bad_arguments_before_cuda(lib):
    assert _dec(lib, q=None) == 1
    assert _dec(lib, sl=None) == 1
    assert _dec(lib, Lmax=0) == 1
    assert _dec(lib, V=FAKE + 4) == 1
    assert _dec(lib, d=80) == 2
    # fixed splits: the workspace check needs no device
    assert _dec(lib, ws=None) == 4
    assert _dec(lib, wsb=16) == 4
    assert _dec(lib, ws=FAKE + 16) == 4        # workspace must be 256-byte aligned


def _ws_bytes(B, H, smax, d):
    up = lambda v: (v + 255) // 256 * 256
    slots = B * H * smax
    return up(slots * d * 4) + up(slots * 2 * 4)


def test_workspace_bytes_fixed_splits(lib):
    B, H, Lmax, d, S = 3, 5, 1000, 128, 7
    assert lib.fa_decode_workspace_bytes(B, H, Lmax, d, S) == _ws_bytes(B, H, S, d)
    assert lib.fa_decode_workspace_bytes_for_lengths(B, H, Lmax, d, S, None) == _ws_bytes(B, H, S, d)
    assert lib.fa_decode_workspace_bytes(B, H, Lmax, 96, S) == 0
    assert lib.fa_decode_workspace_bytes(0, H, Lmax, d, S) == 0
    assert lib.fa_decode_workspace_bytes_for_lengths(0, H, Lmax, d, S, None) == 0


def test_workspace_bound_covers_every_automatic_plan(lib):
    """The five-argument size is enough for the plan of any lengths on any SM count."""
    import random
    import exact_attention_tiled_gb300 as fa
    rng = random.Random(7)
    for _ in range(300):
        B, H = rng.randint(1, 40), rng.choice([1, 2, 8, 32, 64])
        Lmax = rng.choice([1, 63, 64, 65, 255, 257, 1000, 4096, 32768, 65536, 300000])
        d = rng.choice([64, 128])
        kind = rng.random()
        if kind < 0.3:
            lens = [Lmax] * B
        elif kind < 0.5:
            lens = [rng.randint(1, Lmax)] * B
        else:
            lens = [rng.randint(0, Lmax) for _ in range(B)]
        bound = lib.fa_decode_workspace_bytes(B, H, Lmax, d, 0)
        for sms in (1, 8, 152, 2000):
            for hp in (lens, None):
                _, smax = fa.fa_decode_plan(B, H, Lmax, d, 0, hp, sms)
                assert _ws_bytes(B, H, smax, d) <= bound, (B, H, Lmax, d, sms, hp is None)


def _plan(B, H, Lmax, d, splits, seqlens=None, sms=152):
    import exact_attention_tiled_gb300 as fa
    return fa.fa_decode_plan(B, H, Lmax, d, splits, seqlens, sms)


def test_plan_fixed_splits():
    for splits in (1, 8, 32, 128):
        c, m = _plan(1, 32, 32768, 128, splits)
        assert m == splits
        assert c % 64 == 0 and c * splits >= 32768 and c == -(-(32768 // splits) // 64) * 64
    # short sequence with many splits: chunks are at least one granule
    c, m = _plan(1, 1, 100, 128, 128, [100])
    assert c == 64 and m == 128


def test_plan_auto_uniform_one_wave():
    slots = 152 * 3
    c, m = _plan(1, 32, 32768, 128, 0)
    assert c % 64 == 0 and m * c >= 32768 and (m - 1) * c < 32768
    # equal lengths: one wave, the most chunks per sequence whose CTAs fit in 85 % of the slots
    assert 32 * m <= 0.85 * slots < 32 * (m + 1), (c, m)
    # chunks stay at least 256 tokens long
    c, m = _plan(1, 1, 1000, 128, 0)
    assert c >= 256 and m == math.ceil(1000 / c)
    # more sequences than 85 % of the slots: whole waves of short chunks (cost model
    # waves x (chunk + per-CTA overhead)); here one or two chunks per sequence
    c, m = _plan(64, 32, 2048, 128, 0)
    assert m in (1, 2) and c * m >= 2048 and c % 64 == 0


def test_plan_auto_mixed_lengths():
    import torch
    g = torch.Generator().manual_seed(5)
    lens = torch.randint(1024, 65537, (16,), generator=g, dtype=torch.int32).tolist()
    c, m = _plan(16, 32, 65536, 128, 0, lens)
    assert c % 64 == 0 and 256 <= c <= 65536
    assert m == math.ceil(max(lens) / c)
    total_ctas = sum(32 * math.ceil(L / c) for L in lens)
    assert total_ctas >= 4 * 152 * 2   # several waves, so the tail is short


def test_plan_empty_and_clamped():
    c, m = _plan(2, 2, 500, 64, 0, [0, 0])
    assert m == 1
    c2, m2 = _plan(2, 2, 500, 64, 0, [10_000, -5])   # clamped to [0, Lmax]
    assert m2 * c2 >= 500


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import exact_attention_tiled_gb300 as fa
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        fa.library()


def _paged(lib, **kw):
    a = dict(q=FAKE, K=FAKE, V=FAKE, bt=FAKE, mb=8, sl=FAKE, slh=None, O=FAKE, L=None, B=2, H=2, nb=16,
             bs=16, d=128, scale=0.0, splits=4, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    return lib.fa_decode_paged(a["q"], a["K"], a["V"], a["bt"], a["mb"], a["sl"], a["slh"], a["O"], a["L"],
                               a["B"], a["H"], a["nb"], a["bs"], a["d"], ctypes.c_float(a["scale"]),
                               a["splits"], a["ws"], a["wsb"], None)


def test_paged_decode_rejects_bad_arguments_before_cuda(lib):
    assert _paged(lib, bt=None) == 1
    assert _paged(lib, bt=FAKE + 2) == 1       # table must be 4-byte aligned
    assert _paged(lib, mb=0) == 1
    assert _paged(lib, nb=0) == 1
    assert _paged(lib, bs=0) == 1
    assert _paged(lib, bs=65537) == 1
    assert _paged(lib, mb=1 << 20, bs=4096) == 2   # more than 2^30 tokens per sequence
    assert _paged(lib, K=FAKE + 8) == 1
    assert _paged(lib, d=96) == 2
    assert _paged(lib, ws=None) == 4
    assert _paged(lib, ws=FAKE + 16) == 4


def test_paged_inputs_structure():
    from exact_attention_tiled_gb300 import workloads
    lens = [100, 0, 16, 33]
    q, Kp, Vp, table, sl = workloads.paged_inputs(4, 2, 16, 64, lens, seed=3, spare_blocks=4)
    need = [7, 0, 1, 3]
    assert tuple(Kp.shape) == (sum(need) + 4, 2, 16, 64) and Vp.shape == Kp.shape
    assert tuple(table.shape) == (4, 7) and table.dtype.is_signed
    used = []
    for b, n in enumerate(need):
        assert (table[b, n:] == -1).all()
        used += table[b, :n].tolist()
    assert len(set(used)) == len(used) and all(0 <= u < Kp.shape[0] for u in used)
    assert used != sorted(used)                # blocks are scattered, not in logical order
    assert sl.tolist() == lens


def _bwd(lib, **kw):
    a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, dO=FAKE, L=FAKE, dQ=FAKE, dK=FAKE, dV=FAKE, B=1, H=2, N=256, d=64,
             causal=0, scale=0.0, kl=None, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    return lib.fa_backward(a["Q"], a["K"], a["V"], a["O"], a["dO"], a["L"], a["dQ"], a["dK"], a["dV"], a["B"],
                           a["H"], a["N"], a["d"], a["causal"], ctypes.c_float(a["scale"]), a["kl"], a["ws"],
                           a["wsb"], None)


def test_backward_rejects_bad_arguments_before_cuda(lib):
    assert _bwd(lib, dO=None) == 1
    assert _bwd(lib, L=None) == 1
    assert _bwd(lib, dK=FAKE + 8) == 1
    assert _bwd(lib, L=FAKE + 2) == 1
    assert _bwd(lib, N=0) == 1
    assert _bwd(lib, causal=3) == 1
    assert _bwd(lib, scale=float("inf")) == 1
    assert _bwd(lib, d=32) == 2
    assert _bwd(lib, ws=None) == 4
    assert _bwd(lib, wsb=16) == 4
    assert lib.fa_backward_workspace_bytes(2, 3, 1000, 128) == (2 * 3 * 1000 * 4 + 255) // 256 * 256
    assert lib.fa_backward_workspace_bytes(2, 3, 1000, 96) == 0


def test_backward_atomic_dq_rejects_bad_arguments_before_cuda(lib):
    f = lib.fa_backward_atomic_dq
    f.restype = ctypes.c_int
    wsb = lib.fa_backward_atomic_dq_workspace_bytes
    wsb.argtypes = [ctypes.c_int] * 4
    wsb.restype = ctypes.c_size_t

    def call(**kw):
        a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, dO=FAKE, L=FAKE, dQ=FAKE, dK=FAKE, dV=FAKE, B=1, H=2, N=256,
                 d=64, causal=0, scale=0.0, kl=None, ws=FAKE, wsb=1 << 20)
        a.update(kw)
        return f(a["Q"], a["K"], a["V"], a["O"], a["dO"], a["L"], a["dQ"], a["dK"], a["dV"], a["B"], a["H"],
                 a["N"], a["d"], a["causal"], ctypes.c_float(a["scale"]), a["kl"], a["ws"], a["wsb"], None)

    assert call(dQ=None) == 1
    assert call(causal=2) == 1
    assert call(d=128) == 2      # the dQ accumulator fits in TMEM at d = 64 only
    assert call(d=32) == 2
    # D, then the fp32 dQ accumulator: the plain backward's workspace is too small
    need = wsb(1, 2, 256, 64)
    assert need == lib.fa_backward_workspace_bytes(1, 2, 256, 64) + 1 * 2 * 256 * 64 * 4
    assert call(wsb=lib.fa_backward_workspace_bytes(1, 2, 256, 64)) == 4
    assert call(wsb=need - 1) == 4
    assert wsb(1, 2, 256, 128) == 0 and wsb(0, 2, 256, 64) == 0


def test_forward_fp8_rejects_bad_arguments_before_cuda(lib):
    def f8(**kw):
        a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, L=None, B=1, H=2, N=256, d=128, causal=0, scale=0.0, kl=None,
                 ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return lib.fa_forward_fp8(a["Q"], a["K"], a["V"], a["O"], a["L"], a["B"], a["H"], a["N"], a["d"],
                                  a["causal"], ctypes.c_float(a["scale"]), a["kl"], a["ws"], a["wsb"], None)
    assert f8(Q=None) == 1
    assert f8(V=FAKE + 4) == 1
    assert f8(N=0) == 1
    assert f8(d=64) == 2
    assert f8(ws=None) == 4
    assert f8(wsb=1024) == 4
    assert lib.fa_forward_fp8_workspace_bytes(1, 2, 300, 128) == (2 * 300 * 128 * 2 + 255) // 256 * 256
    assert lib.fa_forward_fp8_workspace_bytes(1, 2, 300, 64) == 0


def test_forward_host_rejects_bad_arguments_before_cuda(lib):
    def fh(**kw):
        a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, L=None, B=2, H=6, N=300, d=64, causal=0, scale=0.0, kl=None,
                 hpg=0, ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return lib.fa_forward_host(a["Q"], a["K"], a["V"], a["O"], a["L"], a["B"], a["H"], a["N"], a["d"],
                                   a["causal"], ctypes.c_float(a["scale"]), a["kl"], a["hpg"], a["ws"], a["wsb"],
                                   None)
    assert fh(Q=None) == 1
    assert fh(O=None) == 1
    assert fh(N=0) == 1
    assert fh(causal=2) == 1
    assert fh(d=96) == 2
    assert fh(hpg=4) == 1          # does not divide H = 6
    assert fh(hpg=7) == 1
    assert fh(ws=None) == 4
    assert fh(ws=FAKE + 16) == 4   # not 256-byte aligned
    assert fh(wsb=1024) == 4


def test_forward_host_workspace_plan(lib):
    ws = lib.fa_forward_host_workspace_bytes
    ws.restype = ctypes.c_size_t
    a256 = lambda v: (v + 255) // 256 * 256
    # automatic groups: the largest divisor of H whose Q slice is at most 16 MiB
    head = 8192 * 128 * 2                       # 2 MiB per head
    slot = 4 * a256(8 * head) + a256(8 * 8192 * 4)
    assert ws(1, 32, 8192, 128, 0) == 3 * slot + 256
    # explicit groups; fewer groups than slots use fewer slots
    slot1 = 4 * a256(300 * 64 * 2) + a256(300 * 4)
    assert ws(2, 6, 300, 64, 1) == 3 * slot1 + 256
    slot6 = 4 * a256(6 * 300 * 64 * 2) + a256(6 * 300 * 4)
    assert ws(1, 6, 300, 64, 6) == 1 * slot6 + 256
    assert ws(2, 6, 300, 64, 6) == 2 * slot6 + 256
    assert ws(2, 6, 300, 64, 4) == 0
    assert ws(2, 6, 300, 96, 0) == 0
