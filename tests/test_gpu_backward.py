"""Parity of the attention backward (fa_backward through the C ABI) with the float64 oracle.

Tolerance, from the arithmetic: P and dS are rounded to bf16 before the second
GEMMs (relative error 2^-9 each), D comes from the bf16 O (error <= 2^-9 sum|dO||O|),
the accumulations are fp32 and the outputs are rounded to bf16 (2^-9 relative).
With M the oracle's per-element sum of term magnitudes (M_dV = sum_i P_ij |dO_ic|;
M_dK, M_dQ = scale sum P (|dP| + A) |Q| or |K|, A_i = |D_i| + sum_c |dO_ic||O_ic|)
those roundings stay below 2^-8 M + 2^-9 |ref|; the test allows 2^-6 M + 2^-8 |ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_tiled_gb300 import workloads

pytestmark = pytest.mark.gpu


def fa():
    import exact_attention_tiled_gb300 as m
    m.library()
    return m


def _inputs(B, H, N, d, seed, amp=1.0):
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed, amp)
    g = torch.Generator().manual_seed(seed + 1000)
    dO = torch.randn((B, H, N, d), generator=g).to(torch.bfloat16)
    return Q, K, V, dO


def _gpu_backward(Q, K, V, dO, causal, key_len=None):
    dev = torch.device("cuda")
    Qd, Kd, Vd, dOd = (t.to(dev) for t in (Q, K, V, dO))
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device=dev)
    O, L = fa().fa_forward(Qd, Kd, Vd, causal=causal, key_len=kl)
    dQ, dK, dV = fa().fa_backward(Qd, Kd, Vd, O, dOd, L, causal=causal, key_len=kl)
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    return {n: t.float().cpu().numpy() for n, t in (("dQ", dQ), ("dK", dK), ("dV", dV))}


def _check(name, got, ref):
    for g in ("dQ", "dK", "dV"):
        a, r, m = got[g], ref[g], ref["M_" + g]
        assert np.all(np.isfinite(a)), f"{name} {g}: non-finite"
        bound = 2.0 ** -6 * m + 2.0 ** -8 * np.abs(r) + 1e-6
        excess = np.abs(a - r) - bound
        worst = np.unravel_index(np.argmax(excess), excess.shape)
        assert excess.max() <= 0, (f"{name} {g}: |err| {np.abs(a - r)[worst]:.3e} > bound {bound[worst]:.3e} "
                                   f"at {worst} (ref {r[worst]:.3e})")


# 64: exactly one half-step; 192: the second tile's second half is empty; 300: a 44-row
# tail inside the first half; 640: five steps, so the two- and three-stage rings wrap
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [64, 128, 192, 300, 640])
def test_backward_small(d, causal, N):
    Q, K, V, dO = _inputs(2, 2, N, d, seed=300 + N + d)
    got = _gpu_backward(Q, K, V, dO, causal)
    ref = oracle.sdpa_backward(Q, K, V, dO, causal=causal, magnitudes=True)
    _check(f"bwd N{N} d{d} c{int(causal)}", got, ref)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_key_padding_and_empty_rows(d):
    Q, K, V, dO = _inputs(3, 2, 260, d, seed=400 + d)
    key_len = [260, 77, 0]
    got = _gpu_backward(Q, K, V, dO, False, key_len)
    ref = oracle.sdpa_backward(Q, K, V, dO, key_len=key_len, magnitudes=True)
    _check(f"bwd keypad d{d}", got, ref)
    # masked keys and key-less rows carry exactly zero gradient
    assert np.all(got["dK"][1, :, 77:] == 0) and np.all(got["dV"][1, :, 77:] == 0)
    assert np.all(got["dQ"][2] == 0) and np.all(got["dK"][2] == 0) and np.all(got["dV"][2] == 0)


def test_backward_single_token():
    Q, K, V, dO = _inputs(1, 3, 1, 64, seed=410)
    got = _gpu_backward(Q, K, V, dO, True)
    # one key: P = 1, so dQ = dK = 0 up to rounding, and dV = dO exactly (P rounds to 1 in bf16)
    ref = oracle.sdpa_backward(Q, K, V, dO, causal=True, magnitudes=True)
    assert np.all(ref["dQ"] == 0) and np.all(ref["dK"] == 0)
    _check("bwd single token", got, ref)
    np.testing.assert_array_equal(got["dV"], dO.float().numpy())


def test_backward_batched_d64_sampled_heads():
    """B8 H16 N2048 d64 (x0.5), the batched prefill shape; oracle on sampled heads."""
    B, H, N, d = 8, 16, 2048, 64
    Q, K, V, dO = _inputs(B, H, N, d, seed=3, amp=0.5)
    got = _gpu_backward(Q, K, V, dO, False)
    for b, h in ((0, 0), (3, 7), (7, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.sdpa_backward(Q[sl], K[sl], V[sl], dO[sl], magnitudes=True)
        _check(f"bwd batched b{b}h{h}", {k: v[sl] for k, v in got.items()}, ref)
    # shifting all keys of a head by one vector leaves the softmax unchanged: sum_j dK_j = 0
    s = np.abs(got["dK"].astype(np.float64).sum(axis=2))
    assert np.all(s <= 2.0 ** -6 * np.abs(got["dK"]).sum(axis=2) + 1e-4)


def test_backward_causal_d128_sampled_heads():
    B, H, N, d = 1, 8, 2048, 128
    Q, K, V, dO = _inputs(B, H, N, d, seed=2)
    got = _gpu_backward(Q, K, V, dO, True)
    for h in (0, 5):
        sl = (slice(0, 1), slice(h, h + 1))
        ref = oracle.sdpa_backward(Q[sl], K[sl], V[sl], dO[sl], causal=True, magnitudes=True)
        _check(f"bwd causal h{h}", {k: v[sl] for k, v in got.items()}, ref)


@pytest.mark.slow
def test_backward_causal_8k_d128_bench_shape_sampled_heads():
    """B1 H32 N8192 d128 causal (the bench's causal backward, same launch: 64 key tiles and 64
    query tiles per head in the grouped grid); the oracle on the first and the last head,
    every element of dQ, dK, dV (about 30 s of host time per head)."""
    B, H, N, d = 1, 32, 8192, 128
    Q, K, V, dO = _inputs(B, H, N, d, seed=2)
    got = _gpu_backward(Q, K, V, dO, True)
    for h in (0, H - 1):
        sl = (slice(0, 1), slice(h, h + 1))
        ref = oracle.sdpa_backward(Q[sl], K[sl], V[sl], dO[sl], causal=True, magnitudes=True)
        _check(f"bwd causal 8k h{h}", {k: v[sl] for k, v in got.items()}, ref)


def test_backward_is_deterministic():
    """Every gradient element is written by one CTA (no atomics): two runs agree bit for bit."""
    Q, K, V, dO = _inputs(2, 4, 1000, 64, seed=420)
    dev = torch.device("cuda")
    Qd, Kd, Vd, dOd = (t.to(dev) for t in (Q, K, V, dO))
    O, L = fa().fa_forward(Qd, Kd, Vd, causal=True)
    a = fa().fa_backward(Qd, Kd, Vd, O, dOd, L, causal=True)
    b = fa().fa_backward(Qd, Kd, Vd, O, dOd, L, causal=True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
