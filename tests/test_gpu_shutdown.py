"""fa_shutdown between calls (include/fa.h).

fa_shutdown releases fa_forward_host's streams and events and forgets the
per-device lookups (error word and no-allocation array addresses, SM count,
decode CTAs per SM).  Here every kind of that state is in use before the call,
a host-buffer forward is still queued when it runs, and afterwards each entry
point sets its state up again and returns the same bits as before.
"""
import ctypes

import pytest
import torch

import exact_attention_tiled_gb300 as fa
from exact_attention_tiled_gb300 import workloads

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(q, Kc, Vc, seqlens, lens):
    lib = fa.library()
    B, H, Lmax, d = Kc.shape
    hp = (ctypes.c_int32 * len(lens))(*lens)
    O = torch.empty_like(q)
    L = torch.empty((B, H), device=q.device, dtype=torch.float32)
    st = lib.fa_decode_noalloc(_p(q), _p(Kc), _p(Vc), _p(seqlens), ctypes.cast(hp, ctypes.c_void_p), _p(O), _p(L),
                               B, H, Lmax, d, ctypes.c_float(0.0), 0,
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    return O, L


def _all_calls(Qh, Kh, Vh, dec):
    dev = torch.device("cuda")
    Q, K, V = (t.to(dev) for t in (Qh, Kh, Vh))
    out = {}
    out["forward"] = fa.fa_forward(Q, K, V, causal=True)
    out["host"] = fa.fa_forward_host(Qh, Kh, Vh, causal=True, heads_per_group=1)
    q, Kc, Vc, seqlens, lens = dec
    out["decode"] = fa.fa_decode(q, Kc, Vc, seqlens, seqlens_host=seqlens.cpu())
    out["noalloc"] = _noalloc(q, Kc, Vc, seqlens, lens)
    torch.cuda.synchronize()
    return out


def _same(a, b):
    return all(torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y) for x, y in zip(a, b))


def test_shutdown_then_every_entry_point_again():
    dev = torch.device("cuda")
    Qh, Kh, Vh = (t.pin_memory() for t in workloads.prefill_inputs(1, 4, 300, 128, seed=900))
    q, Kc, Vc = workloads.decode_inputs(2, 4, 800, 128, seed=901, device=dev)
    lens = [800, 33]
    dec = (q, Kc, Vc, torch.tensor(lens, dtype=torch.int32, device=dev), lens)

    before = _all_calls(Qh, Kh, Vh, dec)
    # a host-buffer forward still in flight: fa_shutdown waits for it before its streams go
    Oh, Lh = fa.fa_forward_host(Qh, Kh, Vh, causal=True, heads_per_group=1)
    assert fa.fa_shutdown() == 0
    torch.cuda.synchronize()
    assert _same((Oh, Lh), before["host"])
    assert fa.fa_shutdown() == 0            # nothing left to release
    after = _all_calls(Qh, Kh, Vh, dec)
    for name in before:
        assert _same(before[name], after[name]), name
    assert fa.fa_device_error() == (0, 0)
