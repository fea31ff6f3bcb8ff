"""Parity of the tcgen05 prefill path (through the C ABI) with the float64 oracle."""
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


def _fwd(Q, K, V, causal, key_len=None):
    dev = torch.device("cuda")
    kl = None if key_len is None else torch.as_tensor(key_len, dtype=torch.int32).to(dev)
    O, L = fa().fa_forward(Q.to(dev), K.to(dev), V.to(dev), causal=causal, key_len=kl)
    torch.cuda.synchronize()
    return O.float().cpu().numpy(), L.cpu().numpy()


def test_tiny_workload_full():
    """B1 H1 N256 d64, non-causal, seed 0: every element against the oracle."""
    inp = workloads.make("tiny_n256_d64")
    O, L = _fwd(inp["Q"], inp["K"], inp["V"], False)
    Oref, Lref = oracle.sdpa_forward(inp["Q"], inp["K"], inp["V"], causal=False)
    compare("tiny", O, L, Oref, Lref)


CASES = [
    # B, H, N, d, causal, key_len
    (2, 3, 1000, 128, True, None),
    (2, 2, 777, 64, False, None),
    (1, 2, 1, 64, False, None),
    (1, 1, 127, 128, True, None),
    (1, 2, 129, 64, True, None),
    (1, 1, 256, 128, False, None),
    (1, 1, 640, 64, True, None),
    (2, 2, 300, 128, False, [1, 300]),
    (2, 2, 300, 64, True, [150, 7]),
    (3, 1, 384, 128, False, [0, 384, 200]),
    (2, 1, 513, 128, True, [513, 1]),
]


@pytest.mark.parametrize("B,H,N,d,causal,key_len", CASES)
def test_small_ragged_full(B, H, N, d, causal, key_len):
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed=N + d + B)
    O, L = _fwd(Q, K, V, causal, key_len)
    Oref, Lref = oracle.sdpa_forward(Q, K, V, causal=causal, key_len=key_len)
    compare(f"B{B} H{H} N{N} d{d} c{int(causal)} kl{key_len}", O, L, Oref, Lref)


def test_causal_first_row_is_first_value():
    Q, K, V = workloads.prefill_inputs(1, 4, 512, 128, seed=3)
    O, _ = _fwd(Q, K, V, True)
    np.testing.assert_array_equal(O[:, :, 0], V[:, :, 0].float().numpy())


def test_single_valid_key_returns_that_value():
    Q, K, V = workloads.prefill_inputs(2, 2, 300, 64, seed=4)
    O, _ = _fwd(Q, K, V, False, [1, 1])
    for i in (0, 77, 299):
        np.testing.assert_array_equal(O[:, :, i], V[:, :, 0].float().numpy())


def _sampled(name, nrows, seed, use_key_len=True):
    inp = workloads.make(name)
    Q, K, V, causal = inp["Q"], inp["K"], inp["V"], inp["causal"]
    kl = inp.get("key_len") if use_key_len else None
    O, L = _fwd(Q, K, V, causal, kl)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    B, H, N, d = Q.shape
    rows = workloads.sample_indices(B * H * N, nrows, seed).numpy()
    # plus the rows at 128-row tile edges (and at the edges of 256-row work items) of the
    # first, a middle and the last (batch, head) unit and of three more seeded ones; under
    # causal masking the items holding rows 0..255 are the lightest, dealt in the last round
    units = {0, (B * H) // 2, B * H - 1}
    units.update(int(u) for u in workloads.sample_indices(B * H, 3, seed + 1).numpy())
    edges = [r for r in (0, 1, 127, 128, 129, 255, 256, 511, 512, N - 257, N - 256, N - 129, N - 128, N - 1)
             if 0 <= r < N]
    extra = [u * N + r for u in sorted(units) for r in edges]
    rows = np.unique(np.concatenate([rows, np.asarray(extra, dtype=rows.dtype)]))
    Oref, Lref = oracle.sdpa_rows(Q, K, V, rows, causal=causal, key_len=kl)
    compare(name, O.reshape(-1, d)[rows], L.reshape(-1)[rows], Oref, Lref)


@pytest.mark.slow
def test_batched_d64_sampled():
    """B8 H16 N2048 d64 (x0.5), non-causal, no padding; 2048 sampled rows."""
    _sampled("prefill_b8h16_n2048_d64", 2048, 31, use_key_len=False)


@pytest.mark.slow
def test_batched_d64_key_padding_sampled():
    """Same workload with per-batch key lengths U[N/2, N]."""
    _sampled("prefill_b8h16_n2048_d64", 2048, 32)


@pytest.mark.slow
def test_causal_8k_d128_sampled():
    """B1 H32 N8192 d128 causal; 1024 sampled rows."""
    _sampled("prefill_causal_b1h32_n8192_d128", 1024, 33)


def test_prefill_no_device_error_recorded():
    st, site = fa().fa_device_error(clear=True)
    assert st == 0, f"bounded wait ran out at site {site:#x}"


@pytest.mark.parametrize("d,causal", [(128, False), (64, True), (128, True)])
def test_late_max_jump_rebases_and_rescales(d, causal):
    """Keys in later KV tiles with much larger scores force the exponent base to
    move after the first tile (the recompute-and-rescale path of the softmax)."""
    B, H, N = 1, 2, 700
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed=77)
    K = K.float()
    K[:, :, 300:420] *= 6.0          # scores ~6x larger from the third KV tile on
    K[:, :, 600:] *= 12.0            # and again in the last tile
    K = K.to(torch.bfloat16)
    O, L = _fwd(Q, K, V, causal)
    Oref, Lref = oracle.sdpa_forward(Q, K, V, causal=causal)
    compare(f"max jump d{d} c{int(causal)}", O, L, Oref, Lref)


@pytest.mark.parametrize("d,causal", [(64, False), (128, False), (64, True), (128, True)])
def test_masked_keys_with_huge_scores_do_not_set_the_row_max(d, causal):
    """Masked keys whose scores exceed every valid score by ~150 log2 units or more:
    padded keys beyond key_len, or, causal, the last key of every 128-key tile, a
    future key for the other rows of its tile.  The TMEM load's row maximum covers
    the masked columns too, so a tile with masked entries must take its maximum over
    the masked row; with the load's maximum every valid weight of such a row would
    underflow to zero and O, L would be wrong."""
    B, H, N = 2, 2, 640
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed=91)
    Qf = Q.float() * 0.5 + 1.0     # a positive mean along every dimension
    Kf = K.float() * 0.5
    key_len = None
    if causal:
        Kf[:, :, 127::128] = 16.0
    else:
        key_len = [400, 577]
        for b, kl in enumerate(key_len):
            Kf[b, :, kl:] = 16.0
    Q, K = Qf.to(torch.bfloat16), Kf.to(torch.bfloat16)
    O, L = _fwd(Q, K, V, causal, key_len)
    Oref, Lref = oracle.sdpa_forward(Q, K, V, causal=causal, key_len=key_len)
    compare(f"masked huge keys d{d} c{int(causal)}", O, L, Oref, Lref)


def test_many_short_items_persistent_rounds():
    """B16 H32 N384: 1536 work items over the persistent grid (several rounds per CTA); every
    row of a few heads against the oracle."""
    B, H, N, d = 16, 32, 384, 64
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed=77)
    for causal in (False, True):
        O, L = _fwd(Q, K, V, causal)
        for b, h in ((0, 0), (7, 13), (15, 31)):
            sl = (slice(b, b + 1), slice(h, h + 1))
            Oref, Lref = oracle.sdpa_forward(Q[sl], K[sl], V[sl], causal=causal)
            compare(f"many items b{b}h{h} c{int(causal)}", O[sl], L[sl], Oref, Lref)


@pytest.mark.parametrize("causal", [False, True])
def test_many_items_d128_shared_output_staging(causal):
    """B8 H32 N384 d128: 384 work items, so every CTA runs several items and both query
    tiles of each item hand their output tile through the one shared-memory staging
    buffer in turn; whole heads against the oracle."""
    B, H, N, d = 8, 32, 384, 128
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed=79)
    O, L = _fwd(Q, K, V, causal)
    for b, h in ((0, 0), (3, 17), (7, 31)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        Oref, Lref = oracle.sdpa_forward(Q[sl], K[sl], V[sl], causal=causal)
        compare(f"d128 items b{b}h{h} c{int(causal)}", O[sl], L[sl], Oref, Lref)


def test_forward_is_deterministic():
    Q, K, V = workloads.prefill_inputs(1, 8, 2048, 128, seed=78)
    a = _fwd(Q, K, V, True)
    b = _fwd(Q, K, V, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("B,H,N,causal,key_len", [
    (1, 2, 128, False, None),          # one query tile: the second tile of the pair has no work
    (2, 1, 200, True, [200, 0]),       # a partial second tile; a batch with no valid key
    (1, 3, 256, True, None),           # two tiles with 1 and 2 KV steps
    (2, 2, 1536, True, [1536, 700]),   # long causal items, uneven steps, key padding mid-item
])
def test_d64_schedule_edges(B, H, N, causal, key_len):
    """d = 64 runs its own schedule (S of the next KV tile issued while the softmax of the
    current one runs, P in separate tensor-memory columns, two issuing warps): items whose
    two query tiles have different numbers of KV steps, a single tile, and empty rows."""
    Q, K, V = workloads.prefill_inputs(B, H, N, 64, seed=N + 5 * B + H)
    O, L = _fwd(Q, K, V, causal, key_len)
    Oref, Lref = oracle.sdpa_forward(Q, K, V, causal=causal, key_len=key_len)
    compare(f"d64 edges B{B} H{H} N{N} c{int(causal)} kl{key_len}", O, L, Oref, Lref)


def test_d64_long_causal_many_rounds():
    """B2 H16 N4096 d64 causal: 256 items of up to 32 KV steps over the persistent grid,
    several rounds per CTA with heavy and light items mixed; whole heads against the oracle."""
    B, H, N, d = 2, 16, 4096, 64
    Q, K, V = workloads.prefill_inputs(B, H, N, d, seed=91)
    O, L = _fwd(Q, K, V, True)
    for b, h in ((0, 0), (1, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        Oref, Lref = oracle.sdpa_forward(Q[sl], K[sl], V[sl], causal=True)
        compare(f"d64 long causal b{b}h{h}", O[sl], L[sl], Oref, Lref)
