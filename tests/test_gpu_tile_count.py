"""Causal tile skipping, observed on the GPU ("CMU 10-423 Lecture 18", section 4.3
and exercise 4; "Infra: Flash Attention", the causal figure of "Symbols and
boundary conditions").

fa_forward_count_tiles counts, per (batch, head), the 128 x 128 tile products
the kernel issues.  A tile product is needed exactly when its query tile and
key tile share at least one unmasked (query, key) pair; the expected count is
that definition evaluated pair by pair on the host.  For a causal sequence cut
into T tiles it is T(T+1)/2 of the T^2 tiles: 528 for T = 32, the lecture's
exercise (tests/golden/causal_tile_count.json).
"""
import json
import os

import numpy as np
import pytest
import torch

from exact_attention_tiled_gb300 import workloads

pytestmark = pytest.mark.gpu

TILE = 128
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "causal_tile_count.json")


def _needed_tiles(N, causal, key_len):
    """Tile pairs (query tile, key tile) holding at least one unmasked score."""
    T = -(-N // TILE)
    kl = N if key_len is None else max(0, min(N, key_len))
    count = 0
    for qt in range(T):
        q_last = min(N, (qt + 1) * TILE) - 1          # last query row of the tile
        for kt in range(T):
            k_first = kt * TILE                          # first key of the tile
            if k_first < kl and (not causal or k_first <= q_last):
                count += 1
    return count


def _run(B, H, N, d, causal, key_len=None, seed=0):
    import exact_attention_tiled_gb300 as fa
    dev = torch.device("cuda")
    Q, K, V = (t.to(dev) for t in workloads.prefill_inputs(B, H, N, d, seed=seed))
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device=dev)
    counts = torch.full((B, H, 2), -1, dtype=torch.int32, device=dev)
    O, L = fa.fa_forward(Q, K, V, causal=causal, key_len=kl, tile_counts=counts)
    O2, L2 = fa.fa_forward(Q, K, V, causal=causal, key_len=kl)
    torch.cuda.synchronize()
    # counting leaves the results bit for bit as they are
    assert torch.equal(O.view(torch.int16), O2.view(torch.int16))
    assert torch.equal(L, L2)
    assert fa.fa_device_error() == (0, 0)
    return counts.cpu().numpy()


def test_golden_exercise_causal_T32():
    g = json.load(open(GOLDEN))
    assert g["T"] == 32 and _needed_tiles(32 * TILE, True, None) == g["tiles"]
    for d in (64, 128):
        c = _run(1, 3, 32 * TILE, d, True, seed=d)
        assert (c[..., 0] == g["tiles"]).all(), c[..., 0]     # S = Q K^T products
        assert (c[..., 1] == g["tiles"]).all(), c[..., 1]     # P V products
        assert g["tiles"] * g["ratio_den"] == g["ratio_num"] * 32 * 32


def test_non_causal_visits_every_tile():
    for d in (64, 128):
        c = _run(2, 2, 32 * TILE, d, False, seed=10 + d)
        assert (c == 32 * 32).all(), c


@pytest.mark.parametrize("B,H,N,d,causal,key_len", [
    (3, 2, 4000, 64, False, [4000, 1, 2000]),    # key padding: ceil(key_len / 128) * T
    (3, 2, 4000, 128, False, [129, 128, 0]),
    (2, 2, 3900, 128, True, [3900, 700]),        # causal and key padding, odd tile count
    (1, 2, 3900, 64, True, None),
    (1, 1, 1, 64, True, None),
    (2, 1, 300, 128, True, [300, 5]),
])
def test_counts_match_the_needed_tiles(B, H, N, d, causal, key_len):
    c = _run(B, H, N, d, causal, key_len, seed=N + d)
    for b in range(B):
        want = _needed_tiles(N, causal, None if key_len is None else key_len[b])
        assert (c[b, :, 0] == want).all(), (b, c[b, :, 0], want)
        assert (c[b, :, 1] == want).all(), (b, c[b, :, 1], want)
    if key_len is None and not causal:
        T = -(-N // TILE)
        assert (c == T * T).all()


def test_headline_shape_counts_2080():
    """The causal B1 H32 N8192 d128 prefill: T = 64 tiles a side, T(T+1)/2 = 2080 tile
    products per (b, h) instead of 4096."""
    T = 8192 // TILE
    assert _needed_tiles(8192, True, None) == T * (T + 1) // 2 == 2080
    c = _run(1, 32, 8192, 128, True, seed=2)
    assert (c == 2080).all(), c
