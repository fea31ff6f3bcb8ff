"""Optional outputs and caller streams of the entry points (include/fa.h).

L may be NULL in fa_forward, fa_forward_fp8, fa_decode and fa_decode_paged: the
kernels then write O only, and O must be the same bits as with L requested.
Each call also takes a stream; on a side stream (ordered after the inputs'
stream) the results must again be the same bits as on the current stream.
"""
import pytest
import torch

from exact_attention_tiled_gb300 import workloads

pytestmark = pytest.mark.gpu


def fa():
    import exact_attention_tiled_gb300 as m
    m.library()
    return m


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16)) if a.dtype == torch.bfloat16 else torch.equal(a, b)


@pytest.mark.parametrize("d,causal,key_len", [(64, False, None), (64, True, [300, 5]), (128, True, None),
                                              (128, False, [300, 0])])
def test_forward_without_lse_and_on_a_side_stream(d, causal, key_len):
    dev = torch.device("cuda")
    Q, K, V = (t.to(dev) for t in workloads.prefill_inputs(2, 3, 300, d, seed=800 + d))
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device=dev)
    O, L = fa().fa_forward(Q, K, V, causal=causal, key_len=kl)
    O2, L2 = fa().fa_forward(Q, K, V, causal=causal, key_len=kl, return_lse=False)
    assert L2 is None
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        O3, L3 = fa().fa_forward(Q, K, V, causal=causal, key_len=kl, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    assert _same(O, O2) and _same(O, O3) and _same(L, L3)


def test_fp8_forward_without_lse():
    dev = torch.device("cuda")
    Q, K, V = workloads.prefill_inputs(2, 2, 300, 128, seed=820)
    Q8, K8, V8 = (t.float().to(torch.float8_e4m3fn).to(dev) for t in (Q, K, V))
    O, L = fa().fa_forward_fp8(Q8, K8, V8, causal=True)
    O2, L2 = fa().fa_forward_fp8(Q8, K8, V8, causal=True, return_lse=False)
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    assert L2 is None and _same(O, O2)


@pytest.mark.parametrize("splits", [0, 1, 6])
def test_decode_without_lse_and_on_a_side_stream(splits):
    dev = torch.device("cuda")
    q, Kc, Vc = (t.to(dev) for t in workloads.decode_inputs(2, 4, 900, 128, seed=840 + splits))
    seqlens = torch.tensor([900, 77], dtype=torch.int32, device=dev)
    O, L = fa().fa_decode(q, Kc, Vc, seqlens, num_splits=splits)
    O2, L2 = fa().fa_decode(q, Kc, Vc, seqlens, num_splits=splits, return_lse=False)
    assert L2 is None
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        O3, L3 = fa().fa_decode(q, Kc, Vc, seqlens, num_splits=splits, seqlens_host=seqlens.cpu(), stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    assert _same(O, O2) and _same(O, O3) and _same(L, L3)


def test_paged_decode_without_lse():
    dev = torch.device("cuda")
    q, Kp, Vp, table, seqlens = workloads.paged_inputs(2, 4, 16, 64, [500, 31], seed=860, spare_blocks=2)
    args = (q.to(dev), Kp.to(dev), Vp.to(dev), table.to(dev), seqlens.to(dev))
    O, L = fa().fa_decode_paged(*args)
    O2, L2 = fa().fa_decode_paged(*args, return_lse=False)
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    assert L2 is None and _same(O, O2)
