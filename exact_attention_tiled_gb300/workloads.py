"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle.

This module only draws random tensors; it holds none of the attention
arithmetic.  Both sides of every parity check consume the very same tensors
produced here (the oracle gets host copies of the bf16 bits).

Recipe (the pages' example shapes, see the workload table below):
  * a ``torch.Generator`` on the target device seeded with the workload seed;
  * Q, then K, then V drawn as float32 standard normals in [B, H, N, d] order
    (decode: q [B, H, d], then the K cache, then the V cache, each
    [B, H, Lmax, d], drawn one batch entry at a time to bound temporaries),
    multiplied by the workload amplitude in float32, then rounded to bf16;
  * key lengths / sequence lengths from a separate CPU generator.

CPU and CUDA generators are different engines: the same seed gives different
values on the two devices.  That never matters, because a parity check always
feeds one set of tensors to both implementations.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                  # "prefill" or "decode"
    B: int
    H: int
    N: int                     # prefill sequence length, or decode cache capacity Lmax
    d: int
    seed: int
    causal: bool = False
    amp: float = 1.0
    key_len_seed: int | None = None        # prefill key-padding variant
    seqlen_range: tuple | None = None      # decode: per-sequence lengths U[lo, hi]
    splits: tuple = field(default_factory=tuple)


# The five workloads: one tiny correctness case, two prefill shapes and two
# decode shapes, all shaped like the pages' examples (N = 8192, d = 128,
# 32 heads; decode over a 32768-token cache).
WORKLOADS = {
    "tiny_n256_d64": Workload("tiny_n256_d64", "prefill", 1, 1, 256, 64, seed=0),
    "prefill_causal_b1h32_n8192_d128": Workload(
        "prefill_causal_b1h32_n8192_d128", "prefill", 1, 32, 8192, 128, seed=2, causal=True),
    "prefill_b8h16_n2048_d64": Workload(
        "prefill_b8h16_n2048_d64", "prefill", 8, 16, 2048, 64, seed=3, amp=0.5, key_len_seed=31),
    "decode_b1h32_l32768_d128": Workload(
        "decode_b1h32_l32768_d128", "decode", 1, 32, 32768, 128, seed=4, splits=(1, 8, 32, 128)),
    "decode_varlen_b16h32_d128": Workload(
        "decode_varlen_b16h32_d128", "decode", 16, 32, 65536, 128, seed=5,
        seqlen_range=(1024, 65536)),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def prefill_inputs(B, H, N, d, seed, amp=1.0, device="cpu"):
    """bf16 Q, K, V of shape [B, H, N, d], N(0, amp^2) before rounding."""
    g = _gen(device, seed)
    out = []
    for _ in range(3):
        x = torch.randn((B, H, N, d), generator=g, device=device, dtype=torch.float32)
        if amp != 1.0:
            x = x * amp
        out.append(x.to(torch.bfloat16))
    return tuple(out)


def key_lengths(B, N, seed):
    """Per-batch valid key count, uniform in [N/2, N] (so every row keeps >= 1 key)."""
    g = _gen("cpu", seed)
    return torch.randint(N // 2, N + 1, (B,), generator=g, dtype=torch.int32)


def decode_seqlens(B, Lmax, seed, seqlen_range=None):
    """Per-sequence cache lengths: all Lmax, or uniform in [lo, hi] (inclusive)."""
    if seqlen_range is None:
        return torch.full((B,), Lmax, dtype=torch.int32)
    lo, hi = seqlen_range
    g = _gen("cpu", seed)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int32)


def decode_inputs(B, H, Lmax, d, seed, amp=1.0, device="cpu"):
    """bf16 q [B, H, d] and caches K, V [B, H, Lmax, d]."""
    g = _gen(device, seed)
    q = torch.randn((B, H, d), generator=g, device=device, dtype=torch.float32)
    if amp != 1.0:
        q = q * amp
    q = q.to(torch.bfloat16)
    caches = []
    for _ in range(2):
        c = torch.empty((B, H, Lmax, d), device=device, dtype=torch.bfloat16)
        for b in range(B):
            x = torch.randn((H, Lmax, d), generator=g, device=device, dtype=torch.float32)
            if amp != 1.0:
                x = x * amp
            c[b].copy_(x)
            del x
        caches.append(c)
    return q, caches[0], caches[1]


def paged_inputs(B, H, bs, d, seqlens, seed, spare_blocks=0, amp=1.0, device="cpu"):
    """Inputs of a paged-cache decode: (q, Kpool, Vpool, block_table, seqlens).

    q is bf16 [B, H, d]; the pools are bf16 [num_blocks, H, bs, d] with
    num_blocks = sum_b ceil(seqlens[b] / bs) + spare_blocks.  Sequence b
    owns ceil(seqlens[b] / bs) physical blocks taken from a seeded random
    permutation of the pool, so logically adjacent blocks are scattered;
    block_table is int32 [B, max_blocks] (max_blocks = the largest block
    count, at least 1) with -1 in the slots a sequence does not use.  The
    table and seqlens are CPU tensors; q and the pools live on `device`.
    """
    seqlens = torch.as_tensor(seqlens, dtype=torch.int32).cpu()
    nblk = [(int(n) + bs - 1) // bs for n in seqlens.tolist()]
    max_blocks = max(1, max(nblk))
    num_blocks = max(1, sum(nblk) + int(spare_blocks))
    g = _gen(device, seed)
    q = torch.randn((B, H, d), generator=g, device=device, dtype=torch.float32)
    if amp != 1.0:
        q = q * amp
    q = q.to(torch.bfloat16)
    pools = []
    step = max(1, (1 << 26) // (H * bs * d))   # blocks drawn per batch, bounds the fp32 temporary
    for _ in range(2):
        pool = torch.empty((num_blocks, H, bs, d), device=device, dtype=torch.bfloat16)
        for b0 in range(0, num_blocks, step):
            b1 = min(num_blocks, b0 + step)
            x = torch.randn((b1 - b0, H, bs, d), generator=g, device=device, dtype=torch.float32)
            if amp != 1.0:
                x = x * amp
            pool[b0:b1].copy_(x)
            del x
        pools.append(pool)
    perm = torch.randperm(num_blocks, generator=_gen("cpu", seed + 1)).to(torch.int32)
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    return q, pools[0], pools[1], table, seqlens


def shared_prompt_inputs(n_samples, prompt_len, gen_len, bs, H, d, seed, device="cpu"):
    """Paged inputs of parallel sampling: n_samples answers of gen_len tokens to one prompt.

    The prompt's full blocks are stored once and every answer's block table
    points at them; the prompt's last, partly filled block is copied on
    write (each answer but the last gets its own copy holding the same
    prompt rows, the last answer writes into the original).  Returns
    (q, Kpool, Vpool, block_table, seqlens) like paged_inputs, with the
    physical block ids permuted; the pool has
    prompt_len // bs + n_samples * (ceil((prompt_len + gen_len) / bs) - prompt_len // bs)
    blocks.
    """
    full = prompt_len // bs
    tail = prompt_len % bs
    total = prompt_len + gen_len
    per_seq = (total + bs - 1) // bs
    own = per_seq - full
    num_blocks = full + n_samples * own
    g = _gen(device, seed)
    q = torch.randn((n_samples, H, d), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    perm = torch.randperm(num_blocks, generator=_gen("cpu", seed + 1))
    pools = []
    for _ in range(2):
        logical = torch.randn((num_blocks, H, bs, d), generator=g, device=device,
                              dtype=torch.float32).to(torch.bfloat16)
        if tail:
            orig = full + (n_samples - 1) * own       # the last answer keeps the original tail block
            for i in range(n_samples - 1):
                logical[full + i * own, :, :tail] = logical[orig, :, :tail]
        pool = torch.empty_like(logical)
        pool[perm.to(device)] = logical
        pools.append(pool)
    table = torch.empty((n_samples, per_seq), dtype=torch.int32)
    for i in range(n_samples):
        ids = list(range(full)) + [full + i * own + k for k in range(own)]
        table[i] = perm[torch.tensor(ids)].to(torch.int32)
    seqlens = torch.full((n_samples,), total, dtype=torch.int32)
    return q, pools[0], pools[1], table, seqlens


def make(name, device="cpu"):
    """All inputs of a named workload as a dict."""
    w = WORKLOADS[name]
    if w.kind == "prefill":
        Q, K, V = prefill_inputs(w.B, w.H, w.N, w.d, w.seed, w.amp, device)
        out = dict(Q=Q, K=K, V=V, causal=w.causal)
        if w.key_len_seed is not None:
            out["key_len"] = key_lengths(w.B, w.N, w.key_len_seed)
        return out
    q, Kc, Vc = decode_inputs(w.B, w.H, w.N, w.d, w.seed, w.amp, device)
    seqlens = decode_seqlens(w.B, w.N, w.seed, w.seqlen_range)
    return dict(q=q, Kc=Kc, Vc=Vc, seqlens=seqlens)


def sample_indices(total, count, seed):
    """`count` distinct indices in [0, total), always including 0 and total-1."""
    g = _gen("cpu", seed)
    count = min(count, total)
    idx = torch.randperm(total, generator=g)[:count]
    idx = torch.unique(torch.cat([idx, torch.tensor([0, total - 1])]))
    return idx.to(torch.int64)
