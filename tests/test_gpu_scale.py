"""A softmax scale passed by the caller reaches every kernel.

"Infra: Flash Attention", "Attention and its scope": S = scale * Q K^T, with
scale = 1/sqrt(d) in the definition; the C ABI takes the scale as an argument
(<= 0 selects 1/sqrt(d)).  Every other parity test uses that default.  Here each
entry point runs with scales well away from it -- 0.02 (flat rows) and 0.5
(peaked rows, so the exponent base moves more often) -- against the oracle at the
same scale.  Each case also checks that the result is far from the oracle's
default-scale result, so a kernel that fell back to 1/sqrt(d) could not pass.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_tiled_gb300 import workloads
from gpu_util import O_TOL, compare

pytestmark = pytest.mark.gpu

SCALES = [0.02, 0.5]   # the default is 0.125 at d = 64 and 0.088 at d = 128


def fa():
    import exact_attention_tiled_gb300 as m
    m.library()
    return m


def _far_from_default(name, O, O_default_ref):
    gap = np.abs(np.asarray(O, dtype=np.float64) - np.asarray(O_default_ref, dtype=np.float64)).max()
    assert gap > 5 * O_TOL, f"{name}: result within {gap:.3e} of the default-scale oracle"


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("d,causal,key_len", [
    (64, False, None),
    (64, True, [300, 77]),
    (128, True, None),
    (128, False, [1, 300]),
])
def test_forward_scale(scale, d, causal, key_len):
    Q, K, V = workloads.prefill_inputs(2, 2, 300, d, seed=700 + d)
    dev = torch.device("cuda")
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device=dev)
    O, L = fa().fa_forward(Q.to(dev), K.to(dev), V.to(dev), causal=causal, scale=scale, key_len=kl)
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    On, Ln = O.float().cpu().numpy(), L.cpu().numpy()
    Oref, Lref = oracle.sdpa_forward(Q, K, V, causal=causal, scale=scale, key_len=key_len)
    name = f"forward d{d} c{int(causal)} kl{key_len} scale {scale}"
    compare(name, On, Ln, Oref, Lref)
    Odef, _ = oracle.sdpa_forward(Q, K, V, causal=causal, key_len=key_len)
    _far_from_default(name, On, Odef)


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("d", [64, 128])
def test_decode_scale(scale, d):
    q, Kc, Vc = workloads.decode_inputs(2, 4, 700, d, seed=720 + d)
    seqlens = torch.tensor([700, 129], dtype=torch.int32)
    Oref, Lref = oracle.decode(q, Kc, Vc, seqlens, scale=scale)
    Odef, _ = oracle.decode(q, Kc, Vc, seqlens)
    for splits in (0, 5):
        O, L = fa().fa_decode(q.cuda(), Kc.cuda(), Vc.cuda(), seqlens.cuda(), num_splits=splits, scale=scale)
        torch.cuda.synchronize()
        assert fa().fa_device_error() == (0, 0)
        name = f"decode d{d} s{splits} scale {scale}"
        On = O.float().cpu().numpy()
        compare(name, On, L.cpu().numpy(), Oref, Lref)
        _far_from_default(name, On, Odef)


@pytest.mark.parametrize("scale", SCALES)
def test_paged_decode_scale(scale):
    lens = [600, 45]
    q, Kp, Vp, table, seqlens = workloads.paged_inputs(2, 4, 16, 128, lens, seed=740, spare_blocks=3)
    O, L = fa().fa_decode_paged(q.cuda(), Kp.cuda(), Vp.cuda(), table.cuda(), seqlens.cuda(), scale=scale)
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    Oref, Lref = oracle.decode_paged(q, Kp, Vp, table, seqlens, scale=scale)
    Odef, _ = oracle.decode_paged(q, Kp, Vp, table, seqlens)
    On = O.float().cpu().numpy()
    compare(f"paged decode scale {scale}", On, L.cpu().numpy(), Oref, Lref)
    _far_from_default(f"paged decode scale {scale}", On, Odef)


@pytest.mark.parametrize("scale", SCALES)
def test_fp8_forward_scale(scale):
    Q, K, V = workloads.prefill_inputs(2, 2, 300, 128, seed=760)
    Q8, K8, V8 = (t.float().to(torch.float8_e4m3fn) for t in (Q, K, V))
    dev = torch.device("cuda")
    O, L = fa().fa_forward_fp8(Q8.to(dev), K8.to(dev), V8.to(dev), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    Oref, Lref = oracle.sdpa_forward_e4m3(Q8, K8, V8, causal=True, scale=scale)
    Odef, _ = oracle.sdpa_forward_e4m3(Q8, K8, V8, causal=True)
    On = O.float().cpu().numpy()
    compare(f"fp8 scale {scale}", On, L.cpu().numpy(), Oref, Lref)
    _far_from_default(f"fp8 scale {scale}", On, Odef)


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_backward_scale(scale, d, causal):
    """Gradients at the same scale, within the per-element bound of the backward tests
    (2^-6 M + 2^-8 |ref| + 1e-6, M the oracle's sum of term magnitudes)."""
    Q, K, V = workloads.prefill_inputs(2, 2, 300, d, seed=780 + d)
    g = torch.Generator().manual_seed(781 + d)
    dO = torch.randn((2, 2, 300, d), generator=g).to(torch.bfloat16)
    dev = torch.device("cuda")
    Qd, Kd, Vd, dOd = (t.to(dev) for t in (Q, K, V, dO))
    O, L = fa().fa_forward(Qd, Kd, Vd, causal=causal, scale=scale)
    dQ, dK, dV = fa().fa_backward(Qd, Kd, Vd, O, dOd, L, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    got = {n: t.float().cpu().numpy() for n, t in (("dQ", dQ), ("dK", dK), ("dV", dV))}
    ref = oracle.sdpa_backward(Q, K, V, dO, causal=causal, scale=scale, magnitudes=True)
    ref_def = oracle.sdpa_backward(Q, K, V, dO, causal=causal)
    for gname in ("dQ", "dK", "dV"):
        a, r, m = got[gname], ref[gname], ref["M_" + gname]
        assert np.all(np.isfinite(a)), gname
        bound = 2.0 ** -6 * m + 2.0 ** -8 * np.abs(r) + 1e-6
        excess = np.abs(a - r) - bound
        worst = np.unravel_index(np.argmax(excess), excess.shape)
        assert excess.max() <= 0, (f"bwd d{d} scale {scale} {gname}: |err| {np.abs(a - r)[worst]:.3e} "
                                   f"> bound {bound[worst]:.3e} at {worst}")
        # the default scale gives other gradients by far more than the bound
        assert (np.abs(a - ref_def[gname]) - bound).max() > 0, f"bwd d{d} scale {scale} {gname}: default-like"
