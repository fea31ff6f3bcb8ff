"""The bounded-wait failure path on the GPU: a wait that runs out reports a
status the host reads, and the context stays usable afterwards.  Nothing here
faults, traps or hangs the GPU: the waiting kernel gives up after 20 ms."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_attention_tiled_gb300 import workloads
from gpu_util import compare

pytestmark = pytest.mark.gpu

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_DEVICE_TIMEOUT = 0, 1, 5
SITE_SELFTEST = 0x301


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    import exact_attention_tiled_gb300 as fa
    lib = fa.library()
    st, _ = fa.fa_device_error(clear=True)
    assert st == FA_OK
    assert lib.fa_selftest_wait_timeout(0, None) == FA_ERR_INVALID_ARG
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.fa_selftest_wait_timeout(20000, stream) == FA_OK
    st, site = fa.fa_device_error(clear=True)
    assert st == FA_ERR_DEVICE_TIMEOUT and site == SITE_SELFTEST
    st, site = fa.fa_device_error(clear=True)
    assert st == FA_OK
    # the same through fa_get_last_device_error, which reads and resets the word
    assert lib.fa_selftest_wait_timeout(2000, stream) == FA_OK
    assert fa.fa_get_last_device_error() == FA_ERR_DEVICE_TIMEOUT
    assert fa.fa_get_last_device_error() == FA_OK
    # the context still computes correctly
    Q, K, V = workloads.prefill_inputs(1, 2, 300, 64, seed=21)
    O, L = fa.fa_forward(Q.cuda(), K.cuda(), V.cuda(), causal=True)
    torch.cuda.synchronize()
    Oref, Lref = oracle.sdpa_forward(Q, K, V, causal=True)
    compare("after timeout", O.float().cpu().numpy(), L.cpu().numpy(), Oref, Lref)
