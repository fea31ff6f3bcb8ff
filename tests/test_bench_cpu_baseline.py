"""Host-side pieces of the CPU baseline that bench.py reports beside the GPU
numbers: the host description and the oracle's decode rate (GB/s of cached K
and V attended per second), on a small cache."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def test_host_cpu_fields():
    import bench
    info = bench.host_cpu()
    assert isinstance(info["cpu_model"], str) and info["cpu_model"]
    assert info["affinity_cores"] >= 1
    assert info["machine"]


def test_oracle_decode_rate_small_cache():
    import bench
    from exact_attention_tiled_gb300 import workloads
    q, Kc, Vc = workloads.decode_inputs(2, 3, 512, 64, seed=7)
    seqlens = workloads.decode_seqlens(2, 512, seed=7, seqlen_range=(100, 512))
    one = bench.oracle_decode_rate(q, Kc, Vc, seqlens, 1)
    two = bench.oracle_decode_rate(q, Kc, Vc, seqlens, 2)
    assert one > 0 and two > 0
    # the byte count is the algorithmic one: K and V rows of the valid tokens only
    assert bench.decode_bytes(3, [int(n) for n in seqlens], 64) == pytest.approx(
        2 * 3 * 64 * 2 * float(seqlens.sum()))
