"""Key padding without causal masking, batches with many and with unequal key
lengths ("Infra: Flash Attention", "Attention and its scope": keys j >= key_len[b]
masked).

Items of one batch element cost ceil(key_len[b] / 128) KV steps, so these cases
give CTAs of the persistent forward very different loads: equal lengths (ties),
zero lengths (O = 0, L = -inf), 128 and 130 batch elements of one head each.
Every row must match the float64 oracle, and the tile products issued per
(b, h) must be exactly those the lengths need.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_tiled_gb300 import workloads
from gpu_util import compare

pytestmark = pytest.mark.gpu


def fa():
    import exact_attention_tiled_gb300 as m
    m.library()
    return m


def _run(B, H, N, d, key_len, seed):
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed)
    dev = torch.device("cuda")
    kl = torch.tensor(key_len, dtype=torch.int32, device=dev)
    O, L = fa().fa_forward(Q.to(dev), K.to(dev), V.to(dev), causal=False, key_len=kl)
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    Oref, Lref = oracle.sdpa_forward(Q, K, V, causal=False, key_len=key_len)
    return O.float().cpu().numpy(), L.cpu().numpy(), Oref, Lref


@pytest.mark.parametrize("d", [64, 128])
def test_ties_and_empty_batches(d):
    # 3, 1, 3, 0, 2, 1 KV steps per item
    key_len = [300, 5, 300, 0, 129, 5]
    O, L, Oref, Lref = _run(6, 3, 300, d, key_len, seed=1700 + d)
    compare(f"keypad order d{d}", O, L, Oref, Lref)
    assert np.all(O[3] == 0) and np.all(np.isneginf(L[3]))


@pytest.mark.parametrize("B", [128, 130])
def test_many_batch_elements(B):
    g = torch.Generator().manual_seed(1800 + B)
    key_len = torch.randint(0, 200, (B,), generator=g).tolist()
    O, L, Oref, Lref = _run(B, 1, 190, 64, key_len, seed=1810 + B)
    compare(f"keypad order B{B}", O, L, Oref, Lref)


def test_tile_counts_follow_the_key_lengths():
    """Each (b, h) issues ceil(key_len[b] / 128) S and P V tile products per query tile."""
    B, H, N, d = 5, 2, 384, 64
    key_len = [384, 1, 257, 0, 128]
    Q, K, V = (t.cuda() for t in workloads.prefill_inputs(B, H, N, d, seed=1900))
    kl = torch.tensor(key_len, dtype=torch.int32, device="cuda")
    counts = torch.full((B, H, 2), -1, dtype=torch.int32, device="cuda")
    fa().fa_forward(Q, K, V, causal=False, key_len=kl, tile_counts=counts)
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    counts = counts.cpu().numpy()
    T = (N + 127) // 128
    for b in range(B):
        want = T * ((key_len[b] + 127) // 128)
        for h in range(H):
            assert tuple(int(x) for x in counts[b, h]) == (want, want), (b, h, counts[b, h])
