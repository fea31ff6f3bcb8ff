"""Pins of the oracle's backward ("Infra: Flash Attention", "Backward and recomputation" and
"Blocked gradient computation"; CMU 10-423 Lecture 18 notes, section 5.3).

The backward oracle is checked against things other than its own formulas:
central finite differences of the forward, torch.autograd in float64 (a library
routine), closed forms (one valid key, zero upstream gradient, all-zero keys), and
invariants (the key gradients sum to zero, D_i = dO_i . O_i).  The float64-input
forward it is differentiated against is itself pinned to the bf16 oracle forward.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed, amp=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * amp


def _loss(Q, K, V, G, causal, key_len, scale):
    O, _ = oracle.sdpa_forward_f64(Q, K, V, causal=causal, scale=scale, key_len=key_len)
    return float((O * G).sum())


@pytest.mark.parametrize("causal,key_len", [(False, None), (True, None), (False, [4, 6])])
def test_backward_matches_central_differences(causal, key_len):
    B, H, N, d = 2, 2, 6, 4
    Q, K, V, G = (_rand((B, H, N, d), s) for s in (1, 2, 3, 4))
    scale = 0.7
    r = oracle.sdpa_backward(Q, K, V, G, causal=causal, scale=scale, key_len=key_len)
    eps = 1e-6
    for name, X in (("dQ", Q), ("dK", K), ("dV", V)):
        num = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args = {"Q": Q, "K": K, "V": V}
            key = name[1]
            args[key] = Xp
            lp = _loss(args["Q"], args["K"], args["V"], G, causal, key_len, scale)
            args[key] = Xm
            lm = _loss(args["Q"], args["K"], args["V"], G, causal, key_len, scale)
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(r[name], num, atol=2e-8, rtol=1e-6, err_msg=name)


def test_backward_matches_torch_autograd_float64():
    B, H, N, d = 1, 3, 97, 16
    g = torch.Generator().manual_seed(11)
    Q, K, V, G = (torch.randn(B, H, N, d, generator=g, dtype=torch.float64) for _ in range(4))
    for causal in (False, True):
        q, k, v = (t.clone().requires_grad_(True) for t in (Q, K, V))
        out = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal)
        out.backward(G)
        r = oracle.sdpa_backward(Q, K, V, G, causal=causal)
        for name, t in (("dQ", q), ("dK", k), ("dV", v)):
            np.testing.assert_allclose(r[name], t.grad.numpy(), atol=1e-12, rtol=1e-10, err_msg=name)


def test_backward_key_padding_matches_masked_autograd():
    B, H, N, d = 2, 2, 33, 8
    g = torch.Generator().manual_seed(12)
    Q, K, V, G = (torch.randn(B, H, N, d, generator=g, dtype=torch.float64) for _ in range(4))
    key_len = [20, 33]
    mask = torch.zeros(B, 1, N, N, dtype=torch.bool)
    for b, n in enumerate(key_len):
        mask[b, :, :, :n] = True
    q, k, v = (t.clone().requires_grad_(True) for t in (Q, K, V))
    torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask).backward(G)
    r = oracle.sdpa_backward(Q, K, V, G, key_len=key_len)
    for name, t in (("dQ", q), ("dK", k), ("dV", v)):
        np.testing.assert_allclose(r[name], t.grad.numpy(), atol=1e-12, rtol=1e-10, err_msg=name)
    # keys past key_len get no gradient
    assert np.all(r["dK"][0, :, 20:] == 0) and np.all(r["dV"][0, :, 20:] == 0)


def test_backward_single_valid_key_closed_form():
    # one valid key: P = 1 for every row, so the scores carry no gradient
    B, H, N, d = 1, 2, 7, 5
    Q, K, V, G = (_rand((B, H, N, d), s) for s in (21, 22, 23, 24))
    r = oracle.sdpa_backward(Q, K, V, G, key_len=[1])
    assert np.abs(r["dQ"]).max() < 1e-15
    assert np.abs(r["dK"]).max() < 1e-15
    np.testing.assert_allclose(r["dV"][:, :, 0], G.sum(axis=2), atol=1e-14)
    assert np.all(r["dV"][:, :, 1:] == 0)
    # causal row 0 sees only key 0 as well: its dQ is zero
    rc = oracle.sdpa_backward(Q, K, V, G, causal=True)
    assert np.abs(rc["dQ"][:, :, 0]).max() < 1e-15


def test_backward_zero_upstream_and_zero_keys():
    B, H, N, d = 1, 1, 9, 4
    Q, K, V = (_rand((B, H, N, d), s) for s in (31, 32, 33))
    r = oracle.sdpa_backward(Q, K, V, np.zeros((B, H, N, d)))
    for name in ("dQ", "dK", "dV"):
        assert np.all(r[name] == 0)
    # all-zero keys: uniform P, dQ = scale * sum_j dS_ij K_j = 0
    G = _rand((B, H, N, d), 34)
    r = oracle.sdpa_backward(Q, np.zeros((B, H, N, d)), V, G)
    assert np.abs(r["dQ"]).max() < 1e-15
    # uniform P = 1/N: dV_j = mean over rows of G
    np.testing.assert_allclose(r["dV"][0, 0], np.tile(G[0, 0].sum(axis=0) / N, (N, 1)), atol=1e-14)


def test_backward_invariants():
    B, H, N, d = 2, 3, 40, 8
    Q, K, V, G = (_rand((B, H, N, d), s) for s in (41, 42, 43, 44))
    for causal in (False, True):
        r = oracle.sdpa_backward(Q, K, V, G, causal=causal)
        # shifting every key by the same vector leaves each softmax row unchanged
        assert np.abs(r["dK"].sum(axis=2)).max() < 1e-12
        # D_i = dO_i . O_i (the identity the pages use to avoid a pass over P)
        O, L = oracle.sdpa_forward_f64(Q, K, V, causal=causal)
        np.testing.assert_allclose(r["D"], (G * O).sum(axis=-1), atol=1e-12)
        np.testing.assert_allclose(r["L"], L, atol=1e-13)
        # magnitudes bound the gradients
        m = oracle.sdpa_backward(Q, K, V, G, causal=causal, magnitudes=True)
        for name in ("dQ", "dK", "dV"):
            assert np.all(np.abs(m[name]) <= m["M_" + name] + 1e-12)


def test_f64_forward_equals_bf16_oracle_on_bf16_values():
    g = torch.Generator().manual_seed(51)
    Q, K, V = (torch.randn(2, 2, 37, 16, generator=g).to(torch.bfloat16) for _ in range(3))
    for causal, kl in ((False, None), (True, None), (False, [10, 37])):
        O1, L1 = oracle.sdpa_forward(Q, K, V, causal=causal, key_len=kl)
        O2, L2 = oracle.sdpa_forward_f64(Q, K, V, causal=causal, key_len=kl)
        np.testing.assert_array_equal(O1, O2)
        np.testing.assert_array_equal(L1, L2)


# ---------------------------------------------------------------------------
# The magnitude arrays M_dV, M_dK, M_dQ set the per-element tolerance of every
# GPU gradient comparison, so they are pinned on their own: to the gradient
# they bound where that bound is attained exactly, to a closed form with one
# valid key, and to a from-scratch 50-digit evaluation of their definition.
# ---------------------------------------------------------------------------

def test_magnitude_dV_equals_dV_of_absolute_upstream_gradient():
    # dV_j = sum_i P_ij dO_i ("Blocked gradient computation": dV = P^T dO), and
    # P >= 0, so with |dO| as the upstream gradient every term is nonnegative:
    # the sum of term magnitudes for dO equals the gradient for |dO| exactly.
    # That gradient is taken from torch.autograd in float64, not from the oracle.
    B, H, N, d = 1, 2, 23, 6
    g = torch.Generator().manual_seed(61)
    Q, K, V, G = (torch.randn(B, H, N, d, generator=g, dtype=torch.float64) for _ in range(4))
    for causal in (False, True):
        v = V.clone().requires_grad_(True)
        torch.nn.functional.scaled_dot_product_attention(Q, K, v, is_causal=causal).backward(G.abs())
        m = oracle.sdpa_backward(Q, K, V, G, causal=causal, magnitudes=True)
        np.testing.assert_allclose(m["M_dV"], v.grad.numpy(), rtol=1e-12, atol=1e-14)


def test_magnitudes_one_valid_key_closed_form():
    # One valid key (key_len = 1): P_i0 = 1, O_i = V_0, dP_i0 = dO_i . V_0 and
    # D_i = dP_i0.  So A_i = |D_i| + sum_c |dO_ic| |V_0c| and
    #   M_dV[0]   = sum_i |dO_i|
    #   M_dK[0,c] = scale sum_i (|dP_i0| + A_i) |Q_ic|
    #   M_dQ[i,c] = scale (|dP_i0| + A_i) |K_0c|
    # while every other key has all-zero magnitudes.
    B, H, N, d = 1, 2, 6, 4
    Q, K, V, G = (_rand((B, H, N, d), s) for s in (71, 72, 73, 74))
    scale = 0.45
    m = oracle.sdpa_backward(Q, K, V, G, scale=scale, key_len=[1], magnitudes=True)
    for h in range(H):
        q, k0, v0, g = Q[0, h], K[0, h, 0], V[0, h, 0], G[0, h]
        dp = g @ v0                              # [N]
        A = np.abs(dp) + np.abs(g) @ np.abs(v0)  # |D| = |dP| here
        w = np.abs(dp) + A
        np.testing.assert_allclose(m["M_dV"][0, h, 0], np.abs(g).sum(axis=0), rtol=1e-13)
        np.testing.assert_allclose(m["M_dK"][0, h, 0], scale * (w[:, None] * np.abs(q)).sum(axis=0), rtol=1e-13)
        np.testing.assert_allclose(m["M_dQ"][0, h], scale * w[:, None] * np.abs(k0)[None, :], rtol=1e-13)
        for name in ("M_dV", "M_dK"):
            assert np.all(m[name][0, h, 1:] == 0), name


def test_magnitudes_match_50_digit_evaluation():
    # Tiny inputs (N <= 7): every quantity the magnitudes are made of (scores,
    # the softmax P, dP = dO V^T, D = rowsum(dO o O), O = P V) is recomputed in
    # 50-digit arithmetic straight from the inputs, then the three sums.
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    B, H, N, d = 2, 1, 7, 3
    Q, K, V, G = (_rand((B, H, N, d), s, amp=1.3) for s in (81, 82, 83, 84))
    scale = 0.6
    for causal, key_len in ((False, None), (True, None), (False, [5, 7])):
        m = oracle.sdpa_backward(Q, K, V, G, causal=causal, scale=scale, key_len=key_len, magnitudes=True)
        for b in range(B):
            q, k, v, g = (X[b, 0] for X in (Q, K, V, G))
            MdV = [[mp.mpf(0)] * d for _ in range(N)]
            MdK = [[mp.mpf(0)] * d for _ in range(N)]
            MdQ = [[mp.mpf(0)] * d for _ in range(N)]
            for i in range(N):
                keys = [j for j in range(N) if (key_len is None or j < key_len[b]) and (not causal or j <= i)]
                s = {j: mp.mpf(scale) * mp.fsum(mp.mpf(q[i, c]) * mp.mpf(k[j, c]) for c in range(d)) for j in keys}
                den = mp.fsum(mp.exp(x) for x in s.values())
                P = {j: mp.exp(s[j]) / den for j in keys}
                dP = {j: mp.fsum(mp.mpf(g[i, c]) * mp.mpf(v[j, c]) for c in range(d)) for j in keys}
                O = [mp.fsum(P[j] * mp.mpf(v[j, c]) for j in keys) for c in range(d)]
                D = mp.fsum(mp.mpf(g[i, c]) * O[c] for c in range(d))
                A = abs(D) + mp.fsum(abs(mp.mpf(g[i, c])) * abs(O[c]) for c in range(d))
                for j in keys:
                    w = P[j] * (abs(dP[j]) + A)
                    for c in range(d):
                        MdV[j][c] += P[j] * abs(mp.mpf(g[i, c]))
                        MdK[j][c] += mp.mpf(scale) * w * abs(mp.mpf(q[i, c]))
                        MdQ[i][c] += mp.mpf(scale) * w * abs(mp.mpf(k[j, c]))
            for name, M in (("M_dV", MdV), ("M_dK", MdK), ("M_dQ", MdQ)):
                exact = np.array([[float(x) for x in row] for row in M])
                np.testing.assert_allclose(m[name][b, 0], exact, rtol=1e-13, atol=1e-15,
                                           err_msg=f"{name} causal={causal} key_len={key_len}")
