"""Paged-KV decode (fa_decode_paged through the C ABI) against the float64 oracle.

The cache is a pool of fixed-size blocks reached through a per-sequence block
table ("CMU 10-423 Lecture 18", section 7, PagedAttention).  Three checks:
element-wise parity with oracle.decode_paged, bit-for-bit equality with the
contiguous-cache decode over the same tokens gathered in logical order (the
two paths differ only in how the copies are addressed), and the device error
word for a table entry outside the pool.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_tiled_gb300 import workloads
from gpu_util import compare

pytestmark = pytest.mark.gpu

FA_ERR_INVALID_ARG = 1
SITE_DECODE_TABLE = 0x104


def fa():
    import exact_attention_tiled_gb300 as m
    m.library()
    return m


def _gather(pool, table, seqlens, bs):
    """Contiguous [B, H, Lmax, d] cache holding each sequence's tokens in logical order."""
    B = table.shape[0]
    Lmax = table.shape[1] * bs
    num_blocks, H, _, d = pool.shape
    out = torch.zeros((B, H, Lmax, d), dtype=pool.dtype, device=pool.device)
    for b in range(B):
        n = int(seqlens[b])
        for i in range((n + bs - 1) // bs):
            out[b, :, i * bs:(i + 1) * bs] = pool[int(table[b, i])]
    return out


def _paged(q, Kp, Vp, table, seqlens, splits):
    dev = torch.device("cuda")
    O, L = fa().fa_decode_paged(q.to(dev), Kp.to(dev), Vp.to(dev), table.to(dev), seqlens.to(dev),
                                num_splits=splits)
    torch.cuda.synchronize()
    return O, L


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [1, 16, 48, 64, 256])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_paged_small_ragged(d, bs, splits):
    lens = [1000, 1, 333, 0]
    q, Kp, Vp, table, seqlens = workloads.paged_inputs(4, 3, bs, d, lens, seed=200 + bs + d, spare_blocks=5)
    O, L = _paged(q, Kp, Vp, table, seqlens, splits)
    assert fa().fa_device_error() == (0, 0)
    On, Ln = O.float().cpu().numpy(), L.cpu().numpy()
    Oref, Lref = oracle.decode_paged(q, Kp, Vp, table, seqlens)
    compare(f"paged d{d} bs{bs} s{splits}", On, Ln, Oref, Lref)
    assert np.all(On[3] == 0) and np.all(np.isneginf(Ln[3]))
    # a one-token sequence returns that token's value row
    np.testing.assert_array_equal(On[1], Vp[int(table[1, 0]), :, 0].float().numpy())
    # the contiguous path over the gathered cache computes the same numbers in the same order
    Kc, Vc = _gather(Kp, table, seqlens, bs), _gather(Vp, table, seqlens, bs)
    Oc, Lc = fa().fa_decode(q.cuda(), Kc.cuda(), Vc.cuda(), seqlens.cuda(), num_splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(O, Oc) and torch.equal(L, Lc)


def test_paged_long_context_block16_matches_contiguous_and_oracle():
    """B1 H32 over 32768 tokens in blocks of 16 (2048 scattered blocks), automatic split."""
    bs, d, n = 16, 128, 32768
    q, Kp, Vp, table, seqlens = workloads.paged_inputs(1, 32, bs, d, [n], seed=210, device="cuda")
    O, L = fa().fa_decode_paged(q, Kp, Vp, table.cuda(), seqlens.cuda())
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    Kc = Kp[table[0].long().cuda()].permute(1, 0, 2, 3).reshape(1, 32, n, d).contiguous()
    Vc = Vp[table[0].long().cuda()].permute(1, 0, 2, 3).reshape(1, 32, n, d).contiguous()
    Oc, Lc = fa().fa_decode(q, Kc, Vc, seqlens.cuda())
    torch.cuda.synchronize()
    assert torch.equal(O, Oc) and torch.equal(L, Lc)
    Oref, Lref = oracle.decode(q.cpu(), Kc.cpu(), Vc.cpu(), seqlens)
    compare("paged 32k bs16", O.float().cpu().numpy(), L.cpu().numpy(), Oref, Lref)


def test_paged_variable_lengths_sampled():
    """B8 H8 d128, lengths U[1, 20000], block 32, spare blocks in the pool; sampled heads."""
    g = torch.Generator().manual_seed(9)
    lens = torch.randint(1, 20001, (8,), generator=g, dtype=torch.int32)
    q, Kp, Vp, table, seqlens = workloads.paged_inputs(8, 8, 32, 128, lens, seed=211, spare_blocks=100,
                                                       device="cuda")
    O, L = fa().fa_decode_paged(q, Kp, Vp, table.cuda(), seqlens.cuda())
    torch.cuda.synchronize()
    assert fa().fa_device_error() == (0, 0)
    for b in range(8):
        h = b % 8
        On = O[b:b + 1, h:h + 1].float().cpu().numpy()
        Ln = L[b:b + 1, h:h + 1].cpu().numpy()
        Oref, Lref = oracle.decode_paged(q[b:b + 1, h:h + 1].cpu(), Kp[:, h:h + 1].cpu(), Vp[:, h:h + 1].cpu(),
                                         table[b:b + 1], seqlens[b:b + 1])
        compare(f"paged varlen b{b}", On, Ln, Oref, Lref)


def test_table_entry_outside_pool_is_reported_not_dereferenced():
    bs, d = 16, 64
    q, Kp, Vp, table, seqlens = workloads.paged_inputs(2, 2, bs, d, [100, 50], seed=212)
    fa().fa_device_error()                                 # start from a clear word
    bad = table.clone()
    bad[0, 3] = Kp.shape[0] + 7                            # block 3 holds tokens 48..63 of sequence 0
    O, L = _paged(q, Kp, Vp, bad, seqlens, 0)
    assert fa().fa_device_error() == (FA_ERR_INVALID_ARG, SITE_DECODE_TABLE)
    # sequence 1 is untouched by the bad entry and still matches the oracle
    Oref, Lref = oracle.decode_paged(q[1:], Kp, Vp, table[1:], seqlens[1:])
    compare("paged after bad entry", O[1:].float().cpu().numpy(), L[1:].cpu().numpy(), Oref, Lref)
    # the context stays usable: a valid call afterwards is clean and correct
    O2, L2 = _paged(q, Kp, Vp, table, seqlens, 0)
    assert fa().fa_device_error() == (0, 0)
    Oref, Lref = oracle.decode_paged(q, Kp, Vp, table, seqlens)
    compare("paged after recovery", O2.float().cpu().numpy(), L2.cpu().numpy(), Oref, Lref)


def test_paged_shared_prompt_blocks_parallel_sampling():
    """4 answers of 100 tokens share one 200-token prompt in blocks of 16 (40 pool blocks)."""
    q, Kp, Vp, table, seqlens = workloads.shared_prompt_inputs(4, 200, 100, 16, 8, 128, seed=213)
    O, L = _paged(q, Kp, Vp, table, seqlens, 0)
    assert fa().fa_device_error() == (0, 0)
    Oref, Lref = oracle.decode_paged(q, Kp, Vp, table, seqlens)
    compare("paged shared prompt", O.float().cpu().numpy(), L.cpu().numpy(), Oref, Lref)
    Kc, Vc = _gather(Kp, table, seqlens, 16), _gather(Vp, table, seqlens, 16)
    Oc, Lc = fa().fa_decode(q.cuda(), Kc.cuda(), Vc.cuda(), seqlens.cuda())
    torch.cuda.synchronize()
    assert torch.equal(O, Oc) and torch.equal(L, Lc)
