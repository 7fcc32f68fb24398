"""Seeded synthetic inputs for the O = f(A.B).C workloads.

The one module both the CUDA path's tests/bench and the oracle read inputs
from.  It holds workload shapes and random draws only -- none of the
method's arithmetic.

Seeds: workload k (1-based, in the order of ``WORKLOADS``) draws with seed
``1000*k + offset``, offsets Q/X +0, K/W1 +1, V/W2 +2, dO +3.  Values are
drawn in fp32 (``torch.randn``) and rounded to bf16 (round-to-nearest-even)
where the workload is bf16, to the nearest e4m3 value where it is e4m3.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

OFF_Q, OFF_K, OFF_V, OFF_DO = 0, 1, 2, 3


@dataclass(frozen=True)
class Workload:
    key: str
    index: int  # 1-based, fixes the seed base
    kind: str  # "attn_fwd" | "mlp_fwd" | "relayout+attn_fwd" | "attn_bwd" | "attn_fwd+attn_bwd"
    dims: dict = field(default_factory=dict)

    @property
    def seed(self) -> int:
        return 1000 * self.index


# Shapes of the method's long-sequence workloads (d = 128 heads as in the
# Llama-family models the AutoSP write-up trains; sequence lengths of the
# "hundreds of thousands of tokens" regime of the Ulysses write-up).
WORKLOADS = {
    "tiny_attn_fp32": Workload("tiny_attn_fp32", 1, "attn_fwd",
                               dict(BH=1, n=256, d=64, causal=False, dtype="f32")),
    "gelu_mlp": Workload("gelu_mlp", 2, "mlp_fwd",
                         dict(M=4096, K=1024, N=4096, P=1024, dtype="bf16")),
    "causal_attn_32k": Workload("causal_attn_32k", 3, "attn_fwd",
                                dict(BH=32, n=32768, d=128, causal=True, dtype="bf16")),
    "ulysses_128k": Workload("ulysses_128k", 4, "relayout+attn_fwd",
                             dict(p=4, n_loc=32768, H=32, d=128, g=0, causal=True,
                                  dtype="bf16")),
    "causal_bwd_64k": Workload("causal_bwd_64k", 5, "attn_bwd",
                               dict(BH=16, n=65536, d=128, causal=True, dtype="bf16")),
    # the causal 32k forward with Q, K, V stored as e4m3 (fp32 draws rounded
    # to the nearest e4m3 value)
    "causal_attn_32k_e4m3": Workload("causal_attn_32k_e4m3", 6, "attn_fwd",
                                     dict(BH=32, n=32768, d=128, causal=True, dtype="e4m3")),
    # grouped-query attention: 32 query heads over 8 K/V heads at n = 32768
    "gqa_32k": Workload("gqa_32k", 7, "attn_fwd+attn_bwd",
                        dict(BH=32, BHkv=8, n=32768, d=128, causal=True, dtype="bf16")),
    # sequences of mixed lengths (see varlen_lengths) packed end to end into
    # 131072 positions, 16 heads
    "varlen_128k": Workload("varlen_128k", 8, "attn_fwd+attn_bwd",
                            dict(total=131072, H=16, d=128, causal=True, dtype="bf16",
                                 min_len=1024, max_len=16384)),
}


def varlen_lengths(total: int, min_len: int, max_len: int, seed: int):
    """Sequence lengths drawn uniformly from [min_len, max_len] (seeded) until
    they cover `total` positions; the last one is cut to fit."""
    g = torch.Generator().manual_seed(int(seed))
    lens = []
    left = total
    while left > 0:
        n = int(torch.randint(min_len, max_len + 1, (1,), generator=g))
        n = min(n, left)
        lens.append(n)
        left -= n
    return lens


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, std: float = 1.0, dtype=torch.bfloat16, device="cpu"):
    """N(0, std^2) draw in fp32 from ``seed``, then cast to ``dtype`` (RNE)."""
    x = torch.randn(*shape, generator=_gen(seed, device), dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def attn_inputs(BH: int, n: int, d: int, seed: int, dtype=torch.bfloat16, device="cpu",
                with_do: bool = False, dv: int | None = None):
    """Q, K [BH, n, d], V [BH, n, dv] ~ N(0,1); optionally dO [BH, n, dv]."""
    dv = d if dv is None else dv
    q = normal((BH, n, d), seed + OFF_Q, dtype=dtype, device=device)
    k = normal((BH, n, d), seed + OFF_K, dtype=dtype, device=device)
    v = normal((BH, n, dv), seed + OFF_V, dtype=dtype, device=device)
    if with_do:
        do = normal((BH, n, dv), seed + OFF_DO, dtype=dtype, device=device)
        return q, k, v, do
    return q, k, v


def mlp_inputs(M: int, K: int, N: int, P: int, seed: int, dtype=torch.bfloat16, device="cpu"):
    """X [M,K] ~ N(0,1); W1 [K,N], W2 [N,P] ~ N(0, 1/fan_in) (std = fan_in^-1/2)."""
    x = normal((M, K), seed + OFF_Q, dtype=dtype, device=device)
    w1 = normal((K, N), seed + OFF_K, std=1.0 / math.sqrt(K), dtype=dtype, device=device)
    w2 = normal((N, P), seed + OFF_V, std=1.0 / math.sqrt(N), dtype=dtype, device=device)
    return x, w1, w2


def shard_inputs(p: int, n_loc: int, H: int, d: int, seed: int, dtype=torch.bfloat16,
                 device="cpu"):
    """Sequence shards [p, n_loc, H, d] ~ N(0,1) (one tensor: Q, K or V)."""
    return normal((p, n_loc, H, d), seed, dtype=dtype, device=device)


def iota16(shape, device="cpu"):
    """int16 pattern whose value is the element's linear index mod 2^16, so
    a misplaced element is visible."""
    numel = math.prod(shape)
    x = torch.arange(numel, dtype=torch.int32, device=device).remainder_(65536)
    return x.to(torch.int32).sub_(32768).to(torch.int16).reshape(shape)


def sample_rows(BH: int, n: int, per_head: int, seed: int, full_heads=()):
    """(bh, i) pairs: every row of ``full_heads``; elsewhere ``per_head``
    seeded rows always including 0, 1, 127, 128 and n-1 (those that exist)."""
    g = torch.Generator().manual_seed(int(seed))
    out = []
    fixed = sorted({r for r in (0, 1, 127, 128, n - 1) if 0 <= r < n})
    for bh in range(BH):
        if bh in full_heads:
            rows = list(range(n))
        else:
            k = max(0, min(per_head, n) - len(fixed))
            extra = torch.randint(0, n, (k,), generator=g).tolist() if k else []
            rows = sorted(set(fixed) | set(extra))
        out.extend((bh, r) for r in rows)
    return torch.tensor(out, dtype=torch.int64)
