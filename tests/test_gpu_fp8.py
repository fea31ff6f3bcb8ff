"""FP8 (E4M3) forward (fa_forward_fp8 through the C ABI) against the float64 oracle.

The parity tests feed both sides the same E4M3 values: the oracle decodes the codes exactly,
and since every product of two E4M3 values is exact in fp32, the kernel's rounding is that of
the bf16 forward (P to bf16, fp32 accumulation, O to bf16), so the bf16 tolerances apply.
test_fp8_quantisation_error measures what quantising N(0,1) inputs to E4M3 costs against the
oracle on the unquantised (bf16) inputs: the separate evaluation the pages ask for.
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


def _e4m3_inputs(B, H, N, d, seed, amp=1.0):
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed, amp)
    return tuple(t.float().to(torch.float8_e4m3fn) for t in (Q, K, V)), (Q, K, V)


def _run(Q8, K8, V8, causal, key_len=None):
    dev = torch.device("cuda")
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device=dev)
    O, L = fa().fa_forward_fp8(Q8.to(dev), K8.to(dev), V8.to(dev), causal=causal, key_len=kl)
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    return O.float().cpu().numpy(), L.cpu().numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 300, 1000])
def test_fp8_forward_small(causal, N):
    (Q8, K8, V8), _ = _e4m3_inputs(2, 2, N, 128, seed=500 + N)
    O, L = _run(Q8, K8, V8, causal)
    Oref, Lref = oracle.sdpa_forward_e4m3(Q8, K8, V8, causal=causal)
    compare(f"fp8 N{N} c{int(causal)}", O, L, Oref, Lref)


def test_fp8_forward_key_padding_and_empty_rows():
    (Q8, K8, V8), _ = _e4m3_inputs(3, 2, 260, 128, seed=510)
    key_len = [260, 33, 0]
    O, L = _run(Q8, K8, V8, False, key_len)
    Oref, Lref = oracle.sdpa_forward_e4m3(Q8, K8, V8, key_len=key_len)
    compare("fp8 keypad", O, L, Oref, Lref)
    assert np.all(O[2] == 0) and np.all(np.isneginf(L[2]))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_masked_keys_with_huge_scores_do_not_set_the_row_max(causal):
    """As in the bf16 forward: masked keys (padding, or causal future keys of the diagonal
    tile) with scores ~250 log2 units above every valid score must not move the row max."""
    B, H, N, d = 2, 2, 640, 128
    Q, K, _V = workloads.prefill_inputs(B, H, N, d, seed=93)
    Qf = Q.float() * 0.5 + 1.0
    Kf = K.float() * 0.5
    key_len = None
    if causal:
        Kf[:, :, 127::128] = 16.0
    else:
        key_len = [400, 577]
        for b, kl in enumerate(key_len):
            Kf[b, :, kl:] = 16.0
    Q8, K8, V8 = (t.to(torch.float8_e4m3fn) for t in (Qf, Kf, _V.float()))
    O, L = _run(Q8, K8, V8, causal, key_len)
    Oref, Lref = oracle.sdpa_forward_e4m3(Q8, K8, V8, causal=causal, key_len=key_len)
    compare(f"fp8 masked huge keys c{int(causal)}", O, L, Oref, Lref)


def test_fp8_forward_equals_bf16_forward_of_the_same_values():
    """E4M3 values are bf16 values: the FP8 path must match fa_forward on them (S differs only
    in fp32 summation order)."""
    (Q8, K8, V8), _ = _e4m3_inputs(1, 4, 1024, 128, seed=520)
    O8, L8 = _run(Q8, K8, V8, True)
    dev = torch.device("cuda")
    Ob, Lb = fa().fa_forward(*(t.to(torch.bfloat16).to(dev) for t in (Q8, K8, V8)), causal=True)
    torch.cuda.synchronize()
    assert np.abs(O8 - Ob.float().cpu().numpy()).max() <= 2e-2
    assert np.abs(L8 - Lb.cpu().numpy()).max() <= 1e-3


def test_fp8_forward_causal_long_sampled_rows():
    """B1 H32 N8192 d128 causal (the headline shape); oracle on sampled rows (the E4M3 values
    are given to the bf16 oracle, which holds them exactly)."""
    B, H, N, d = 1, 32, 8192, 128
    (Q8, K8, V8), _ = _e4m3_inputs(B, H, N, d, seed=2)
    O, L = _run(Q8, K8, V8, True)
    rows = workloads.sample_indices(B * H * N, 512, seed=9)
    Qb, Kb, Vb = (t.to(torch.bfloat16) for t in (Q8, K8, V8))
    Oref, Lref = oracle.sdpa_rows(Qb, Kb, Vb, rows, causal=True)
    r = rows.numpy()
    compare("fp8 8k sampled", O.reshape(-1, d)[r], L.reshape(-1)[r], Oref, Lref)


def test_fp8_quantisation_error():
    """What E4M3 inputs cost: FP8 forward on quantised N(0,1) inputs vs the oracle on the bf16
    inputs.  Bounds are loose sanity limits; the measured numbers are in the design notes."""
    (Q8, K8, V8), (Q, K, V) = _e4m3_inputs(1, 4, 2048, 128, seed=530)
    O, L = _run(Q8, K8, V8, True)
    Oref, Lref = oracle.sdpa_forward(Q, K, V, causal=True)
    eo = np.abs(O - Oref)
    el = np.abs(L - Lref)
    rel_rms = np.sqrt((eo ** 2).mean() / (Oref ** 2).mean())
    print(f"\nfp8 quantisation: O max {eo.max():.3e} mean {eo.mean():.3e} rel-rms {rel_rms:.3e}; "
          f"L max {el.max():.3e} mean {el.mean():.3e}")
    assert rel_rms < 0.1 and el.max() < 0.5
