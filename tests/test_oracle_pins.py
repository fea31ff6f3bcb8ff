"""Pins of the float64 oracle against what the pages and the mathematics fix.

None of these compare the oracle with itself: each check uses a printed value
from the pages (fixtures under tests/golden/), a closed form, an invariant, a
library routine (torch float64 softmax), or an independent brute force in
50-digit arithmetic on tiny inputs.  tests/test_oracle_mutants.py re-runs this
file against deliberately broken copies of the oracle to show that a dropped
term, a wrong sign, a wrong index or a missing scale is caught.
"""
import json
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16(shape, seed, amp=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * amp).to(torch.bfloat16)


# ---------------------------------------------------------------- worked example

def test_worked_example_blocks_and_merge():
    """Flash Attention page, 'Accumulating the weighted sum': exps 1,2,4,8, V = 1..4."""
    g = _golden("worked_example_online_softmax.json")
    x = np.log([1.0, 2.0, 4.0, 8.0])
    V = np.array(g["V"], dtype=float).reshape(4, 1)
    pr, dv = g["printed"], g["derived_from_definitions"]

    mA, lA, uA = oracle.block_state(x[:2], V[:2])
    mB, lB, uB = oracle.block_state(x[2:], V[2:])
    assert mA == pytest.approx(math.log(2), abs=1e-15)
    assert mB == pytest.approx(math.log(8), abs=1e-15)
    assert lA == pytest.approx(dv["l_A"], abs=1e-15)
    assert uA[0] == pytest.approx(dv["u_A"], abs=1e-15)
    assert lB == pytest.approx(dv["l_B"], abs=1e-15)
    assert uB[0] == pytest.approx(dv["u_B"], abs=1e-15)
    # the left block is rescaled by exp(log 2 - log 8) = 1/4
    assert math.exp(mA - max(mA, mB)) == pytest.approx(pr["alpha_left_block"], abs=1e-15)

    m, l_, u = oracle.state_merge((mA, lA, uA), (mB, lB, uB))
    assert l_ == pytest.approx(pr["l_merged"], abs=1e-15)
    assert u[0] == pytest.approx(pr["u_merged"], abs=1e-15)
    assert u[0] / l_ == pytest.approx(pr["O_num"] / pr["O_den"], abs=1e-15)
    # merge is commutative on the example
    m2, l2, u2 = oracle.state_merge((mB, lB, uB), (mA, lA, uA))
    assert (m2, l2) == pytest.approx((m, l_), abs=1e-15) and u2[0] == pytest.approx(u[0], abs=1e-15)


def test_worked_example_direct_attention():
    g = _golden("worked_example_online_softmax.json")
    x = np.log([1.0, 2.0, 4.0, 8.0])
    V = np.array(g["V"], dtype=float).reshape(4, 1)
    O, L = oracle.attend_scores(x, V)
    assert O[0] == pytest.approx(49.0 / 15.0, abs=1e-15)
    assert L == pytest.approx(math.log(15.0), abs=1e-15)


def test_averaging_block_outputs_is_wrong():
    """The page warns that the two blocks' own outputs cannot just be averaged."""
    x = np.log([1.0, 2.0, 4.0, 8.0])
    V = np.arange(1.0, 5.0).reshape(4, 1)
    OA, _ = oracle.attend_scores(x[:2], V[:2])
    OB, _ = oracle.attend_scores(x[2:], V[2:])
    assert abs(0.5 * (OA[0] + OB[0]) - 49.0 / 15.0) > 0.1


# ---------------------------------------------------------------- online softmax

def test_online_softmax_row_trace():
    """Lecture 18 section 2.2: row [1,3,2,6,4,5]; invariant of Exercise 1."""
    mp = pytest.importorskip("mpmath")
    g = _golden("online_softmax_row.json")
    x = g["x"]
    m, d = oracle.online_softmax_trace(x)
    assert list(m) == g["m_trace"]
    changes = [j for j in range(1, len(x)) if m[j] != m[j - 1]]
    assert changes == g["base_changes_at_index"]
    mp.mp.dps = 50
    for j in range(len(x)):
        closed = mp.fsum(mp.exp(x[k] - max(x[: j + 1])) for k in range(j + 1))
        assert d[j] == pytest.approx(float(closed), rel=1e-15)
    # after the whole row, d_N is the safe-softmax denominator
    y = oracle.softmax_safe(x)
    assert y[0] == pytest.approx(math.exp(x[0] - m[-1]) / d[-1], rel=1e-15)


def test_softmax_forms_agree_and_naive_overflows():
    rng = np.random.default_rng(7)
    for n in (1, 2, 5, 16, 33):
        x = rng.normal(size=n) * 3
        a = oracle.softmax_naive(x)
        b = oracle.softmax_safe(x)
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=0)
        assert abs(b.sum() - 1.0) < 1e-15 * n + 1e-15
        m, d = oracle.online_softmax_trace(x)
        np.testing.assert_allclose(np.exp(x - m[-1]) / d[-1], b, rtol=1e-13, atol=0)
    # exp(1000) overflows: the naive form breaks, the safe form does not
    x = np.array([1000.0, 999.0, 0.0])
    assert not np.all(np.isfinite(oracle.softmax_naive(x)))
    y = oracle.softmax_safe(x)
    assert np.all(np.isfinite(y))
    assert y[0] == pytest.approx(1.0 / (1.0 + math.exp(-1.0) + math.exp(-1000.0)), rel=1e-15)


# ---------------------------------------------------------------- merge algebra

def _blocks_state(x, V, nb):
    size = len(x) // nb
    return [oracle.block_state(x[i * size:(i + 1) * size], V[i * size:(i + 1) * size])
            for i in range(nb)]


def _fold(states):
    acc = states[0]
    for s in states[1:]:
        acc = oracle.state_merge(acc, s)
    return acc


def _pairwise(states):
    while len(states) > 1:
        nxt = [oracle.state_merge(states[i], states[i + 1]) for i in range(0, len(states) - 1, 2)]
        if len(states) % 2:
            nxt.append(states[-1])
        states = nxt
    return states[0]


def test_merge_orders_match_direct_softmax():
    """Lecture 18 section 2.3: 64 scores in 8 blocks, four merge orders."""
    mp = pytest.importorskip("mpmath")
    rng = np.random.default_rng(64)
    x = rng.normal(size=64) * 2.0
    V = rng.normal(size=(64, 3))
    states = _blocks_state(x, V, 8)
    shuffled = list(states)
    random.Random(5).shuffle(shuffled)
    orders = {
        "left_to_right": _fold(states),
        "right_to_left": _fold(states[::-1]),
        "pairwise": _pairwise(states),
        "shuffled": _fold(shuffled),
    }
    mp.mp.dps = 50
    den = mp.fsum(mp.exp(xi) for xi in x)
    exact = [float(mp.fsum(mp.exp(x[j]) * V[j, c] for j in range(64)) / den) for c in range(3)]
    O_direct, L_direct = oracle.attend_scores(x, V)
    np.testing.assert_allclose(O_direct, exact, rtol=0, atol=1e-14)
    assert L_direct == pytest.approx(float(mp.log(den)), abs=1e-14)
    for name, (m, l_, u) in orders.items():
        np.testing.assert_allclose(u / l_, exact, rtol=0, atol=1e-14, err_msg=name)
        assert m + math.log(l_) == pytest.approx(float(mp.log(den)), abs=1e-14), name


def test_cheating_blockwise_softmax_differs():
    """Lecture 18 section 1.4: 12 scores, 3 blocks softmaxed separately sum to 3."""
    rng = np.random.default_rng(12)
    x = rng.normal(size=12) * 2.0
    parts = np.concatenate([oracle.softmax_safe(x[i * 4:(i + 1) * 4]) for i in range(3)])
    assert parts.sum() == pytest.approx(3.0, abs=1e-14)
    assert np.max(np.abs(parts - oracle.softmax_safe(x))) > 1e-2


def test_merge_with_empty_state_is_identity():
    rng = np.random.default_rng(3)
    x = rng.normal(size=5)
    V = rng.normal(size=(5, 2))
    s = oracle.block_state(x, V)
    e = (-math.inf, 0.0, np.zeros(2))
    for a, b in ((s, e), (e, s)):
        m, l_, u = oracle.state_merge(a, b)
        assert m == s[0] and l_ == pytest.approx(s[1], rel=1e-15)
        np.testing.assert_allclose(u, s[2], rtol=1e-15)


def test_lse_reduce_matches_unsplit_attention():
    """Flash-Decoding step 3: chunk partials (m_k, l_k, O_k) reduce to the unsplit result."""
    mp = pytest.importorskip("mpmath")
    rng = np.random.default_rng(11)
    n, dv = 1000, 4
    x = rng.normal(size=n) * 3
    V = rng.normal(size=(n, dv))
    bounds = [0, 1, 130, 130, 517, 999, 1000]      # includes an empty chunk
    m_k, l_k, O_k = [], [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        m, l_, u = oracle.block_state(x[a:b], V[a:b])
        m_k.append(m)
        l_k.append(l_)
        O_k.append(u / l_ if l_ > 0 else np.zeros(dv))
    O, L = oracle.lse_reduce(m_k, l_k, np.array(O_k))
    mp.mp.dps = 40
    den = mp.fsum(mp.exp(xi) for xi in x)
    exact = [float(mp.fsum(mp.exp(x[j]) * V[j, c] for j in range(n)) / den) for c in range(dv)]
    np.testing.assert_allclose(O, exact, rtol=0, atol=1e-13)
    assert L == pytest.approx(float(mp.log(den)), abs=1e-13)
    # reduction is order-invariant
    perm = [3, 0, 5, 1, 4, 2]
    O2, L2 = oracle.lse_reduce(np.array(m_k)[perm], np.array(l_k)[perm], np.array(O_k)[perm])
    np.testing.assert_allclose(O2, O, rtol=0, atol=1e-14)
    assert L2 == pytest.approx(L, abs=1e-14)


# ---------------------------------------------------------------- whole forward

def _mp_attention(Q, K, V, causal, scale, key_len):
    """Brute force in 50-digit arithmetic, naive softmax (no max shift needed)."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    q = Q.double().numpy()
    k = K.double().numpy()
    v = V.double().numpy()
    B, H, N, d = q.shape
    Nk = k.shape[2]
    O = np.zeros((B, H, N, d))
    L = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                keys = [j for j in range(Nk)
                        if (key_len is None or j < key_len[b]) and (not causal or j <= i)]
                if not keys:
                    O[b, h, i] = 0.0
                    L[b, h, i] = -math.inf
                    continue
                e = {j: mp.exp(mp.mpf(scale) * mp.fsum(mp.mpf(q[b, h, i, c]) * mp.mpf(k[b, h, j, c])
                                                      for c in range(d))) for j in keys}
                den = mp.fsum(e.values())
                for c in range(d):
                    O[b, h, i, c] = float(mp.fsum(e[j] * mp.mpf(v[b, h, j, c]) for j in keys) / den)
                L[b, h, i] = float(mp.log(den))
    return O, L


@pytest.mark.parametrize("causal,key_len", [(False, None), (True, None), (False, [3, 7]),
                                            (True, [5, 1])])
def test_sdpa_brute_force_tiny(causal, key_len):
    B, H, N, d = 2, 2, 7, 5
    Q = _bf16((B, H, N, d), 1, 1.5)
    K = _bf16((B, H, N, d), 2, 1.5)
    V = _bf16((B, H, N, d), 3)
    scale = 1.0 / math.sqrt(d)
    O, L = oracle.sdpa_forward(Q, K, V, causal=causal, scale=scale, key_len=key_len)
    Oe, Le = _mp_attention(Q, K, V, causal, scale, key_len)
    np.testing.assert_allclose(O, Oe, rtol=0, atol=1e-14)
    np.testing.assert_allclose(L, Le, rtol=0, atol=1e-14)


def test_sdpa_matches_torch_float64_softmax():
    """Special case reducing to a library routine: torch float64 softmax(S) V."""
    B, H, N, d = 2, 3, 97, 32
    Q = _bf16((B, H, N, d), 10)
    K = _bf16((B, H, N, d), 11)
    V = _bf16((B, H, N, d), 12)
    key_len = torch.tensor([97, 40], dtype=torch.int32)
    scale = 0.17
    for causal in (False, True):
        O, L = oracle.sdpa_forward(Q, K, V, causal=causal, scale=scale, key_len=key_len)
        S = torch.matmul(Q.double(), K.double().transpose(-1, -2)) * scale
        mask = torch.zeros(B, 1, N, N, dtype=torch.bool)
        for b in range(B):
            mask[b, :, :, int(key_len[b]):] = True
        if causal:
            mask |= torch.triu(torch.ones(N, N, dtype=torch.bool), 1)
        S = S.masked_fill(mask, -math.inf)
        Oref = torch.softmax(S, dim=-1) @ V.double()
        Lref = torch.logsumexp(S, dim=-1)
        np.testing.assert_allclose(O, Oref.numpy(), rtol=0, atol=1e-13)
        np.testing.assert_allclose(L, Lref.numpy(), rtol=0, atol=1e-13)


def test_sdpa_closed_forms():
    B, H, N, d = 2, 2, 33, 16
    Q = _bf16((B, H, N, d), 20)
    V = _bf16((B, H, N, d), 21)
    Kz = torch.zeros((B, H, N, d), dtype=torch.bfloat16)
    key_len = torch.tensor([33, 9], dtype=torch.int32)
    v = V.double().numpy()
    # all-zero keys: uniform weights over the valid keys
    for causal in (False, True):
        O, L = oracle.sdpa_forward(Q, Kz, V, causal=causal, key_len=key_len)
        for b in range(B):
            for i in range(N):
                n = min(int(key_len[b]), i + 1 if causal else N)
                np.testing.assert_allclose(O[b, :, i], v[b, :, :n].mean(axis=1), atol=1e-14)
                np.testing.assert_allclose(L[b, :, i], math.log(n), atol=1e-14)
    # causal row 0 sees only key 0: O_0 = V_0, L_0 = S_00
    K = _bf16((B, H, N, d), 22)
    scale = 1.0 / math.sqrt(d)
    O, L = oracle.sdpa_forward(Q, K, V, causal=True, scale=scale)
    np.testing.assert_array_equal(O[:, :, 0], v[:, :, 0])
    s00 = (Q.double()[:, :, 0] * K.double()[:, :, 0]).sum(-1).numpy() * scale
    np.testing.assert_allclose(L[:, :, 0], s00, atol=1e-14)
    # key_len = 1: every row returns V_0
    O, L = oracle.sdpa_forward(Q, K, V, causal=False, key_len=[1, 1])
    for i in range(N):
        np.testing.assert_array_equal(O[:, :, i], v[:, :, 0])


def test_sdpa_invariants():
    B, H, N, d = 1, 2, 40, 8
    Q = _bf16((B, H, N, d), 30, 2.0)
    K = _bf16((B, H, N, d), 31, 2.0)
    V = _bf16((B, H, N, d), 32)
    scale = 1.0 / math.sqrt(d)
    O, L = oracle.sdpa_forward(Q, K, V, causal=False, scale=scale)
    # joint permutation of keys and values changes nothing (non-causal)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(4))
    O2, L2 = oracle.sdpa_forward(Q, K[:, :, perm], V[:, :, perm], causal=False, scale=scale)
    np.testing.assert_allclose(O2, O, atol=1e-14)
    np.testing.assert_allclose(L2, L, atol=1e-14)
    # convex combination bounds, and max S <= L <= max S + log N
    v = V.double().numpy()
    assert np.all(O <= v.max(axis=2, keepdims=True) + 1e-14)
    assert np.all(O >= v.min(axis=2, keepdims=True) - 1e-14)
    S = (Q.double() @ K.double().transpose(-1, -2) * scale).numpy()
    assert np.all(L >= S.max(-1) - 1e-14) and np.all(L <= S.max(-1) + math.log(N) + 1e-14)
    # duplicating key 0 adds exp(S_i0) to the partition sum
    K3 = torch.cat([K, K[:, :, :1]], dim=2)
    V3 = torch.cat([V, V[:, :, :1]], dim=2)
    rows = np.arange(B * H * N)
    O3, L3 = oracle.sdpa_rows(Q, K3, V3, rows)
    L3 = L3.reshape(B, H, N)
    np.testing.assert_allclose(L3, np.logaddexp(L, S[..., 0]), atol=1e-13)
    # selected rows equal the full forward
    pick = [0, 5, 41, 79]
    Or, Lr = oracle.sdpa_rows(Q, K, V, pick, scale=scale)
    np.testing.assert_allclose(Or, O.reshape(-1, d)[pick], atol=0)
    np.testing.assert_allclose(Lr, L.reshape(-1)[pick], atol=0)


def test_attend_shift_invariance_and_empty_row():
    rng = np.random.default_rng(9)
    x = rng.normal(size=20)
    V = rng.normal(size=(20, 3))
    O, L = oracle.attend_scores(x, V)
    O2, L2 = oracle.attend_scores(x + 123.5, V)
    np.testing.assert_allclose(O2, O, atol=1e-14)
    assert L2 == pytest.approx(L + 123.5, abs=1e-12)
    O0, L0 = oracle.attend_scores(np.zeros(0), np.zeros((0, 3)))
    assert np.all(O0 == 0) and L0 == -math.inf


def test_decode_oracle_brute_force_and_cache_tail_ignored():
    B, H, Lmax, d = 3, 2, 12, 6
    q = _bf16((B, H, d), 40, 1.5)
    Kc = _bf16((B, H, Lmax, d), 41, 1.5)
    Vc = _bf16((B, H, Lmax, d), 42)
    seqlens = [12, 5, 1]
    O, L = oracle.decode(q, Kc, Vc, seqlens)
    for b in range(B):
        n = seqlens[b]
        Oe, Le = _mp_attention(q[b:b + 1, :, None, :], Kc[b:b + 1, :, :n], Vc[b:b + 1, :, :n],
                               False, 1.0 / math.sqrt(d), None)
        np.testing.assert_allclose(O[b], Oe[0, :, 0], atol=1e-14)
        np.testing.assert_allclose(L[b], Le[0, :, 0], atol=1e-14)
    # seqlen 1: the output is v_0 exactly
    np.testing.assert_array_equal(O[2], Vc[2, :, 0].double().numpy())
    # whatever sits past seqlens[b] in the cache is never read
    K2 = Kc.clone()
    V2 = Vc.clone()
    K2[1, :, 5:] = 100.0
    V2[1, :, 5:] = -100.0
    O2, L2 = oracle.decode(q, K2, V2, seqlens)
    np.testing.assert_array_equal(O2, O)
    np.testing.assert_array_equal(L2, L)


def test_causal_tile_count_closed_form():
    """Lecture 18 Exercise 4: T(T+1)/2 of T^2 tiles; T = 32 gives 33/64."""
    g = _golden("causal_tile_count.json")
    T = g["T"]
    # count the tiles a causal query tile i visits: key tiles 0..i
    tiles = sum(1 for i in range(T) for j in range(T) if j <= i)
    assert tiles == g["tiles"]
    assert tiles * g["ratio_den"] == T * T * g["ratio_num"]


# ---------------------------------------------------------------- paged decode

def _pool_from_contiguous(Kc, table, bs, nblk):
    """Scatter a contiguous cache [B, H, L, d] into a pool [nblk, H, bs, d] via table."""
    B, H, L, d = Kc.shape
    pool = torch.full((nblk, H, bs, d), 7.0, dtype=torch.bfloat16)   # junk everywhere else
    for b in range(B):
        for i in range(table.shape[1]):
            lo = i * bs
            if lo >= L:
                break
            n = min(bs, L - lo)
            pool[table[b, i], :, :n] = Kc[b, :, lo:lo + n]
    return pool


def test_paged_decode_lecture_example_matches_contiguous():
    """Lecture 18 section 7.3: 12 physical blocks of 4 tokens; request B's table is 1 -> 4 -> 5.
    Keys fetched through the table are the request's own; attention equals the contiguous one."""
    H, d, bs, nblk = 2, 8, 4, 12
    q = _bf16((1, H, d), 50)
    Kc = _bf16((1, H, 12, d), 51)
    Vc = _bf16((1, H, 12, d), 52)
    table = torch.tensor([[1, 4, 5]], dtype=torch.int32)
    Kp = _pool_from_contiguous(Kc, table, bs, nblk)
    Vp = _pool_from_contiguous(Vc, table, bs, nblk)
    for n in (12, 10, 5, 1):     # a partly filled last block wastes at most bs - 1 slots
        Op, Lp = oracle.decode_paged(q, Kp, Vp, table, [n])
        Oc, Lc = oracle.decode(q, Kc, Vc, [n])
        np.testing.assert_array_equal(Op, Oc)
        np.testing.assert_array_equal(Lp, Lc)


def test_paged_decode_scrambled_pool_and_unused_slots():
    B, H, d, bs, L = 3, 2, 16, 16, 80
    nblk = 3 * (L // bs) + 4
    q = _bf16((B, H, d), 60)
    Kc = _bf16((B, H, L, d), 61)
    Vc = _bf16((B, H, L, d), 62)
    perm = torch.randperm(nblk, generator=torch.Generator().manual_seed(6))[:B * (L // bs)]
    table = perm.reshape(B, L // bs).to(torch.int32)
    Kp = _pool_from_contiguous(Kc, table, bs, nblk)
    Vp = _pool_from_contiguous(Vc, table, bs, nblk)
    seqlens = [80, 33, 1]
    Op, Lp = oracle.decode_paged(q, Kp, Vp, table, seqlens)
    Oc, Lc = oracle.decode(q, Kc, Vc, seqlens)
    np.testing.assert_array_equal(Op, Oc)
    np.testing.assert_array_equal(Lp, Lc)
    # brute force on one row
    Oe, Le = _mp_attention(q[1:2, :, None, :], Kc[1:2, :, :33], Vc[1:2, :, :33], False,
                           1.0 / math.sqrt(d), None)
    np.testing.assert_allclose(Op[1], Oe[0, :, 0], atol=1e-14)
    np.testing.assert_allclose(Lp[1], Le[0, :, 0], atol=1e-14)
    # an out-of-range table entry is rejected
    bad = table.clone()
    bad[0, 0] = nblk
    with pytest.raises(ValueError):
        oracle.decode_paged(q, Kp, Vp, bad, seqlens)


def test_paged_decode_shared_prompt_blocks():
    """Lecture 18 section 7.5: one 200-token prompt, 4 answers of 100 tokens, blocks of 16.
    Without sharing the answers take 76 blocks, sharing the prompt takes 40; the prompt's
    last block (200 is not a multiple of 16) is copied on write.  Attention through the
    shared table equals attention over each answer's own contiguous cache."""
    from exact_attention_tiled_gb300 import workloads
    n, P, G, bs, H, d = 4, 200, 100, 16, 2, 16
    q, Kp, Vp, table, seqlens = workloads.shared_prompt_inputs(n, P, G, bs, H, d, seed=70)
    assert n * math.ceil((P + G) / bs) == 76
    assert Kp.shape[0] == 40 and len(set(table.flatten().tolist())) == 40
    assert all((table[i, :P // bs] == table[0, :P // bs]).all() for i in range(n))
    Kc = torch.stack([Kp[table[i].long()].permute(1, 0, 2, 3).reshape(H, -1, d) for i in range(n)])
    Vc = torch.stack([Vp[table[i].long()].permute(1, 0, 2, 3).reshape(H, -1, d) for i in range(n)])
    # every answer sees the same 200 prompt keys, including the copied tail rows
    for i in range(1, n):
        assert torch.equal(Kc[i, :, :P], Kc[0, :, :P]) and torch.equal(Vc[i, :, :P], Vc[0, :, :P])
    Op, Lp = oracle.decode_paged(q, Kp, Vp, table, seqlens)
    Oc, Lc = oracle.decode(q, Kc, Vc, seqlens)
    np.testing.assert_array_equal(Op, Oc)
    np.testing.assert_array_equal(Lp, Lc)
