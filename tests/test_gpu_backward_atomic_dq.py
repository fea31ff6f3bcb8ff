"""fa_backward_atomic_dq: the backward with dQ accumulated across key tiles by fp32
atomics in the dK/dV thread blocks ("Infra: Flash Attention", "Blocked gradient
computation": dQ_i = scale sum_j dS_ij K_j, summed here in another order).

Against the float64 oracle with the per-element bound of the backward tests
(2^-6 M + 2^-8 |ref| + 1e-6, M the oracle's sum of term magnitudes); dK and dV
come out of the same products as in fa_backward, so they must be the same bits.
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


def _both(Q, K, V, dO, causal, key_len=None):
    dev = torch.device("cuda")
    Qd, Kd, Vd, dOd = (t.to(dev) for t in (Q, K, V, dO))
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device=dev)
    O, L = fa().fa_forward(Qd, Kd, Vd, causal=causal, key_len=kl)
    det = fa().fa_backward(Qd, Kd, Vd, O, dOd, L, causal=causal, key_len=kl)
    atm = fa().fa_backward(Qd, Kd, Vd, O, dOd, L, causal=causal, key_len=kl, atomic_dq=True)
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    # dK and dV: the same products in the same order as the deterministic path
    assert torch.equal(det[1], atm[1]) and torch.equal(det[2], atm[2])
    return {n: t.float().cpu().numpy() for n, t in zip(("dQ", "dK", "dV"), atm)}


def _check(name, got, ref):
    for g in ("dQ", "dK", "dV"):
        a, r, m = got[g], ref[g], ref["M_" + g]
        assert np.all(np.isfinite(a)), f"{name} {g}: non-finite"
        bound = 2.0 ** -6 * m + 2.0 ** -8 * np.abs(r) + 1e-6
        excess = np.abs(a - r) - bound
        worst = np.unravel_index(np.argmax(excess), excess.shape)
        assert excess.max() <= 0, (f"{name} {g}: |err| {np.abs(a - r)[worst]:.3e} > bound {bound[worst]:.3e} "
                                   f"at {worst} (ref {r[worst]:.3e})")


# 64: one half-step; 192: an empty second half; 300: a 44-row tail; 640: the rings wrap
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [64, 128, 192, 300, 640])
def test_atomic_dq_small(causal, N):
    Q, K, V, dO = _inputs(2, 2, N, 64, seed=1300 + N)
    got = _both(Q, K, V, dO, causal)
    ref = oracle.sdpa_backward(Q, K, V, dO, causal=causal, magnitudes=True)
    _check(f"atomic dQ N{N} c{int(causal)}", got, ref)


def test_atomic_dq_key_padding_and_empty_rows():
    Q, K, V, dO = _inputs(3, 2, 260, 64, seed=1400)
    key_len = [260, 77, 0]
    got = _both(Q, K, V, dO, False, key_len)
    ref = oracle.sdpa_backward(Q, K, V, dO, key_len=key_len, magnitudes=True)
    _check("atomic dQ keypad", got, ref)
    assert np.all(got["dQ"][2] == 0)


@pytest.mark.parametrize("N,key_len", [(300, [300, 129, 1]), (640, [500, 128, 640])])
def test_atomic_dq_causal_with_key_padding(N, key_len):
    Q, K, V, dO = _inputs(3, 2, N, 64, seed=1450 + N)
    got = _both(Q, K, V, dO, True, key_len)
    ref = oracle.sdpa_backward(Q, K, V, dO, causal=True, key_len=key_len, magnitudes=True)
    _check(f"atomic dQ causal keypad N{N}", got, ref)


def test_atomic_dq_batched_sampled_heads():
    """B8 H16 N2048 d64 (x0.5), the batched prefill shape; oracle on sampled heads."""
    B, H, N, d = 8, 16, 2048, 64
    Q, K, V, dO = _inputs(B, H, N, d, seed=3, amp=0.5)
    got = _both(Q, K, V, dO, False)
    for b, h in ((0, 0), (4, 9), (7, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.sdpa_backward(Q[sl], K[sl], V[sl], dO[sl], magnitudes=True)
        _check(f"atomic dQ batched b{b}h{h}", {k: v[sl] for k, v in got.items()}, ref)


def test_atomic_dq_rejects_d128():
    dev = torch.device("cuda")
    Q, K, V, dO = (t.to(dev) for t in _inputs(1, 1, 128, 128, seed=1500))
    O, L = fa().fa_forward(Q, K, V)
    with pytest.raises(fa().FaError) as e:
        fa().fa_backward(Q, K, V, O, dO, L, atomic_dq=True)
    assert e.value.status == 2   # FA_ERR_UNSUPPORTED
