"""Seeded synthetic workloads for chunked Q8_0-KV causal prefill attention.

This module only draws random inputs and describes problem sizes; it holds none
of the method's arithmetic, so both the GPU path and the CPU oracle can take
their inputs from it.

The five workloads are single-layer prefill problems with 32 heads of
dimension 64 and a causal mask, computed chunk by chunk over the KV:

  name       B x M          KV chunk   draw (seed)
  m512       1 x 512        128        Q ~ N(0,1) fp16; K, V ~ N(0,1) fp32      (0)
  m2k_out    1 x 2048       256        as m512, K channels 3 and 35 scaled x20  (1)
  b8_m2k     8 x 2048       512        Q ~ N(0,1); K, V ~ N(0, 0.5^2)           (2)
  m64k       1 x 65536      8192       as m512                                  (3)
  m1m        1 x 1048576    131072     as m512                                  (4)

and one head_dim 128 problem (an extension beyond the pages' head_dim 64):

  m16k_d128  1 x 16384      4096       32 heads x 128, as m512                  (6)

The pages measure no public dataset; these draws stand in for the activations
of a prefill pass.  Inputs are drawn with a torch generator on the device they
are created on, in the fixed order Q, then K, then V.

Mode B (speculative burst verification) has workloads of its own:

  burst_m1m  64 candidate queries at positions M .. M+63 against an
             M = 1,048,576-token context, 32 heads x 64, rectangular
             full-context mask; Q ~ N(0,1) fp16, K, V ~ N(0,1) fp32 (seed 5);
             the context's keys are folded in parallel key ranges whose
             count makes the launch a whole number of waves on the device
             (q8attn.split_keys_for: 19 ranges of 55,296 keys on 152 SMs).
  burst_m1m_gqa8  the same with 32 query heads on 8 K/V heads (seed 7):
             grouped-query attention, an extension beyond the pages.
"""

from dataclasses import dataclass

import torch

HEADS = 32
HEAD_DIM = 64


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    tokens: int
    chunk: int
    seed: int
    kv_sigma: float = 1.0
    outlier_channels: tuple = ()
    outlier_scale: float = 1.0
    heads: int = HEADS
    head_dim: int = HEAD_DIM

    @property
    def n_chunks(self):
        return -(-self.tokens // self.chunk)

    @property
    def causal_pairs(self):
        """Unmasked (query, key) pairs: B * H * M (M + 1) / 2."""
        return self.batch * self.heads * self.tokens * (self.tokens + 1) // 2

    @property
    def causal_flops(self):
        """Algorithmic flops: 2*D for q.k plus 2*D for p*v per unmasked pair."""
        return 4 * self.head_dim * self.causal_pairs

    def describe(self):
        return (f"{self.name}: B={self.batch} M={self.tokens} H={self.heads} D={self.head_dim} "
                f"causal, KV chunks of {self.chunk} ({self.n_chunks} chunks), seed {self.seed}")


WORKLOADS = {
    w.name: w for w in [
        Workload("m512", 1, 512, 128, 0),
        Workload("m2k_out", 1, 2048, 256, 1, outlier_channels=(3, 35), outlier_scale=20.0),
        Workload("b8_m2k", 8, 2048, 512, 2, kv_sigma=0.5),
        Workload("m64k", 1, 65536, 8192, 3),
        Workload("m1m", 1, 1048576, 131072, 4),
        Workload("m16k_d128", 1, 16384, 4096, 6, head_dim=128),
    ]
}


@dataclass(frozen=True)
class Burst:
    name: str
    context: int
    queries: int
    split_keys: int   # 0: sized to whole waves on the device (q8attn.split_keys_for)
    seed: int
    heads: int = HEADS
    head_dim: int = HEAD_DIM
    kv_heads: int = 0   # K/V heads (grouped-query attention); 0: as many as query heads

    @property
    def kv_h(self):
        return self.kv_heads or self.heads

    @property
    def kv_bytes(self):
        """Q8_0 K and V of the context: 2 * H_kv * M * (D / 32 * 34) bytes."""
        return 2 * self.kv_h * self.context * (self.head_dim // 32 * 34)

    @property
    def flops(self):
        """4*D flops per (candidate, context key) pair."""
        return 4 * self.head_dim * self.heads * self.queries * self.context

    def describe(self):
        return (f"{self.name}: {self.queries} candidate queries after a {self.context}-token context, "
                f"H={self.heads}" + (f" on {self.kv_h} K/V heads" if self.kv_h != self.heads else "")
                + f" D={self.head_dim}, rectangular mask, key ranges "
                + (f"of {self.split_keys}" if self.split_keys else "sized to whole waves")
                + f", seed {self.seed}")


BURSTS = {b.name: b for b in [Burst("burst_m1m", 1048576, 64, 0, 5),
                              Burst("burst_m1m_gqa8", 1048576, 64, 0, 7, kv_heads=8)]}


def make_burst_inputs(b, device="cpu", context=None):
    """Draw (Q fp16 [1, queries, H, D], K fp32 [1, M, H_kv, D], V fp32), in that order."""
    M = b.context if context is None else context
    g = torch.Generator(device=device)
    g.manual_seed(b.seed)
    q = torch.randn((1, b.queries, b.heads, b.head_dim), generator=g, device=device,
                    dtype=torch.float32).to(torch.float16)
    k = torch.randn((1, M, b.kv_h, b.head_dim), generator=g, device=device, dtype=torch.float32)
    v = torch.randn((1, M, b.kv_h, b.head_dim), generator=g, device=device, dtype=torch.float32)
    return q, k, v


def make_inputs(w, device="cpu", batch=None, tokens=None):
    """Draw (Q fp16, K fp32, V fp32), each [B, M, H, D] token-major.

    `batch`/`tokens` override the sizes (for reduced-size cases) while keeping
    the workload's distributions and seed.
    """
    B = w.batch if batch is None else batch
    M = w.tokens if tokens is None else tokens
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    shape = (B, M, w.heads, w.head_dim)
    q = torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.float16)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if w.kv_sigma != 1.0:
        k.mul_(w.kv_sigma)
        v.mul_(w.kv_sigma)
    for c in w.outlier_channels:
        k[..., c].mul_(w.outlier_scale)
    return q, k, v


def sampled_rows(w, n=4096, seed=None):
    """Query rows checked on the largest problem: row 0, row M-1, the rows on
    both sides of every chunk boundary, then rows drawn uniformly (seeded) until
    there are n distinct rows.  Returns a sorted int64 tensor."""
    M = w.tokens
    fixed = {0, M - 1}
    for c in range(1, w.n_chunks):
        b = c * w.chunk
        if b < M:
            fixed.update({b - 1, b})
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    rows = set(fixed)
    n = min(n, M)
    while len(rows) < n:
        cand = torch.randint(0, M, (2 * n,), generator=g).tolist()
        for r in cand:
            rows.add(r)
            if len(rows) >= n:
                break
    return torch.tensor(sorted(rows), dtype=torch.int64)
