"""fa_forward_host: the forward over host buffers, copies pipelined by head groups.

Every (batch, head) is computed by the same kernel code as fa_forward, so the host
path must reproduce fa_forward bit for bit, whatever the grouping; one case is also
checked against the oracle directly.
"""
import numpy as np
import pytest
import torch

import exact_attention_tiled_gb300 as fa
from exact_attention_tiled_gb300 import workloads
from oracle import oracle

pytestmark = pytest.mark.gpu


def _device_reference(Q, K, V, causal, key_len):
    dev = torch.device("cuda")
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device=dev)
    O, L = fa.fa_forward(Q.to(dev), K.to(dev), V.to(dev), causal=causal, key_len=kl)
    torch.cuda.synchronize()
    return O.cpu(), L.cpu()


@pytest.mark.parametrize("B,H,N,d,causal,key_len,hpg,pin", [
    (2, 6, 300, 64, True, [300, 177], 2, True),     # 6 groups: every slot reused
    (2, 6, 300, 64, False, None, 1, False),          # pageable host memory, 12 groups
    (1, 4, 1000, 128, False, None, 0, True),         # automatic grouping (one group)
    (3, 2, 520, 128, True, [1, 520, 0], 1, True),    # a batch without keys, a single-key batch
])
def test_host_forward_matches_device_forward_bitwise(B, H, N, d, causal, key_len, hpg, pin):
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed=700 + N + d)
    if pin:
        Q, K, V = Q.pin_memory(), K.pin_memory(), V.pin_memory()
    O, L = fa.fa_forward_host(Q, K, V, causal=causal, key_len=key_len, heads_per_group=hpg)
    torch.cuda.synchronize()
    Od, Ld = _device_reference(Q, K, V, causal, key_len)
    assert torch.equal(O.view(torch.int16), Od.view(torch.int16))
    assert torch.equal(L, Ld)
    assert fa.fa_device_error() == (0, 0)


def test_host_forward_without_lse_and_against_the_oracle():
    B, H, N, d = 1, 3, 200, 64
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed=41)
    O, L = fa.fa_forward_host(Q.pin_memory(), K.pin_memory(), V.pin_memory(), causal=True, return_lse=False,
                              heads_per_group=1)
    torch.cuda.synchronize()
    assert L is None
    ref_O, _ = oracle.sdpa_forward(Q, K, V, causal=True)
    err = np.abs(O.float().numpy() - np.asarray(ref_O)).max()
    assert err <= 2e-2, err


def test_host_forward_is_ordered_on_the_callers_stream():
    # work queued on the stream before the call finishes first; the stream waits for the call
    B, H, N, d = 1, 8, 512, 128
    Q, K, V = (t.pin_memory() for t in workloads.prefill_inputs(B, H, N, d, seed=43))
    s = torch.cuda.Stream()
    buf = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(s):
        buf.fill_(1)
        O, L = fa.fa_forward_host(Q, K, V, heads_per_group=2, stream=s)
        done = torch.cuda.Event()
        done.record(s)
    done.synchronize()
    Od, Ld = _device_reference(Q, K, V, False, None)
    assert torch.equal(O.view(torch.int16), Od.view(torch.int16))
    assert torch.equal(L, Ld)


def test_host_forward_from_two_host_threads():
    # two host threads share the device's internal streams and events; each call
    # enqueues its whole pipeline under the device's lock, so both results stay
    # identical to fa_forward
    import threading
    cases = [workloads.prefill_inputs(2, 4, 384, 64, seed=51), workloads.prefill_inputs(1, 6, 640, 128, seed=52)]
    cases = [tuple(t.pin_memory() for t in c) for c in cases]
    refs = [_device_reference(*c, True, None) for c in cases]
    results, errors = {}, []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            outs = []
            for _ in range(4):
                O, L = fa.fa_forward_host(*cases[i], causal=True, heads_per_group=1, stream=s)
                outs.append((O, L))
            s.synchronize()
            results[i] = outs
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not errors, errors
    for i, (Od, Ld) in enumerate(refs):
        for O, L in results[i]:
            assert torch.equal(O.view(torch.int16), Od.view(torch.int16))
            assert torch.equal(L, Ld)
    assert fa.fa_device_error() == (0, 0)
