"""Parity of the split-KV decode path (through the C ABI) with the float64 oracle."""
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


def _run(q, Kc, Vc, seqlens, splits):
    dev = torch.device("cuda")
    O, L = fa().fa_decode(q.to(dev), Kc.to(dev), Vc.to(dev), seqlens.to(dev), num_splits=splits)
    torch.cuda.synchronize()
    return O.float().cpu().numpy(), L.cpu().numpy()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [0, 1, 2, 7, 64])
def test_decode_small_ragged(d, splits):
    q, Kc, Vc = workloads.decode_inputs(3, 4, 1000, d, seed=100 + d)
    seqlens = torch.tensor([1000, 1, 333], dtype=torch.int32)
    O, L = _run(q, Kc, Vc, seqlens, splits)
    Oref, Lref = oracle.decode(q, Kc, Vc, seqlens)
    compare(f"decode d{d} s{splits}", O, L, Oref, Lref)
    # seqlen 1: the output is the first cached value row (exact up to bf16 of v itself)
    np.testing.assert_array_equal(O[1], Vc[1, :, 0].float().numpy())


def test_decode_empty_sequence():
    q, Kc, Vc = workloads.decode_inputs(2, 2, 256, 128, seed=7)
    seqlens = torch.tensor([0, 200], dtype=torch.int32)
    O, L = _run(q, Kc, Vc, seqlens, 0)
    assert np.all(O[0] == 0) and np.all(np.isneginf(L[0]))
    Oref, Lref = oracle.decode(q, Kc, Vc, seqlens)
    compare("decode empty", O, L, Oref, Lref)


def test_decode_long_context_split_sweep():
    """B1 H32 over a 32768-token cache, chunk counts 1, 8, 32, 128 and automatic."""
    w = workloads.WORKLOADS["decode_b1h32_l32768_d128"]
    inp = workloads.make(w.name)
    Oref, Lref = oracle.decode(inp["q"], inp["Kc"], inp["Vc"], inp["seqlens"])
    outs = {}
    for splits in tuple(w.splits) + (0,):
        O, L = _run(inp["q"], inp["Kc"], inp["Vc"], inp["seqlens"], splits)
        compare(f"decode 32k s{splits}", O, L, Oref, Lref)
        outs[splits] = O
    # the split count changes only the rounding order
    for s, O in outs.items():
        assert np.abs(O - outs[1]).max() <= 2e-2


def test_decode_variable_length_batch_sampled():
    """B16 H32, lengths U[1024, 65536], automatic per-sequence chunking; sampled (b, h)."""
    w = workloads.WORKLOADS["decode_varlen_b16h32_d128"]
    inp = workloads.make(w.name, device="cuda")
    seqlens = inp["seqlens"]
    O, L = fa().fa_decode(inp["q"], inp["Kc"], inp["Vc"], seqlens.cuda(), num_splits=0)
    torch.cuda.synchronize()
    O = O.float().cpu().numpy()
    L = L.cpu().numpy()
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    lens = seqlens.tolist()
    # the longest and the shortest sequence, every sequence at least once (each has its own
    # chunk count), and seeded (b, h) pairs up to 64 of the 512
    picks = {(int(np.argmax(lens)), 0), (int(np.argmin(lens)), 31)}
    rng = np.random.default_rng(5)
    for b in range(len(lens)):
        picks.add((b, int(rng.integers(32))))
    while len(picks) < 64:
        picks.add((int(rng.integers(16)), int(rng.integers(32))))
    for b, h in sorted(picks):
        n = lens[b]
        q = inp["q"][b:b + 1, h:h + 1].cpu()
        Kc = inp["Kc"][b:b + 1, h:h + 1, :n].cpu()
        Vc = inp["Vc"][b:b + 1, h:h + 1, :n].cpu()
        Oref, Lref = oracle.decode(q, Kc, Vc, torch.tensor([n], dtype=torch.int32))
        compare(f"varlen b{b} h{h} len{n}", O[b, h][None, None], L[b, h][None, None], Oref, Lref)


def test_decode_equals_last_row_of_causal_prefill():
    """One query over N cached keys = the last row of causal attention over those keys."""
    B, H, N, d = 2, 3, 700, 128
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed=9)
    dev = torch.device("cuda")
    m = fa()
    Of, Lf = m.fa_forward(Q.to(dev), K.to(dev), V.to(dev), causal=True)
    q = Q[:, :, N - 1].contiguous()
    Od, Ld = m.fa_decode(q.to(dev), K.to(dev), V.to(dev), torch.full((B,), N, dtype=torch.int32, device=dev),
                         num_splits=5)
    torch.cuda.synchronize()
    Oref, Lref = oracle.decode(q, K, V, torch.full((B,), N, dtype=torch.int32))
    compare("decode vs oracle", Od.float().cpu().numpy(), Ld.cpu().numpy(), Oref, Lref)
    compare("decode vs prefill", Od.float().cpu().numpy(), Ld.cpu().numpy(),
            Of[:, :, N - 1].float().cpu().numpy(), Lf[:, :, N - 1].cpu().numpy())


def test_decode_no_device_error_recorded():
    st, site = fa().fa_device_error(clear=True)
    assert st == 0, f"bounded wait ran out at site {site:#x}"
