"""Seeded synthetic workloads for the attention forward pass.

This module only draws inputs: it holds no attention arithmetic, and it is the
one module that both the CUDA-path tests and the CPU oracle's callers share.

The workloads mirror the lecture's demo (random q, k, v with B=4, H=8, D=64;
a numerical check at L=256 and a sequence-length sweep), plus causal
prefill, long-context and single-query decode shapes:

    mha_l256_d64     B=4  H=8  Lq=Lk=256     D=64   seed 0  non-causal
    sweep_d64_L{L}   B=4  H=8  Lq=Lk=L       D=64   seed 1  non-causal, L = 64..8192
    causal_l8k_d128  B=2  H=32 Lq=Lk=8192    D=128  seed 2  causal (j <= i)
    causal_l64k_d128 B=1  H=32 Lq=Lk=65536   D=128  seed 3  causal, q,k drawn x3
    decode_l128k_d128 B=16 H=32 Lq=1 Lk=131072 D=128 seed 4 non-causal,
                     1 % of the keys of every head scaled x8 (outlier logits)

Recipe (the same on any device, deterministic for a device):
  * every (tensor t in q=0,k=1,v=2; batch index b) gets its own generator,
    seeded (seed << 20) | (b << 2) | t, on the device the tensors are made on;
  * x = randn(H, L, D) in fp32 from it; q and k are multiplied by `qk_std`;
    the result is cast to bf16 (round to nearest even);
  * outliers (decode workload): for batch index b a generator seeded
    (seed << 20) | (1 << 19) | b draws, for each head h in order,
    randperm(Lk)[:floor(frac * Lk)]; those key rows are multiplied by 8,
    which is exact in bf16;
  * sampled query rows (long-context check): a generator seeded
    (seed << 20) | (1 << 18) draws, for each head in order,
    randperm(Lq)[:n-2]; rows 0 and Lq-1 are always added.
The CPU and CUDA torch generators give different streams, so a test makes its
inputs once and hands the same bf16 tensors to both sides.

Paged single-query decode (PagedWorkload, make_paged_inputs): B sequences, H
heads, pages of page_size positions, lengths up to max_len.
  * lengths: a generator seeded (seed << 20) | (1 << 17) draws randint in
    [1, max_len] per sequence (or `lengths` gives them);
  * pages: sequence b needs ceil(len_b / page_size) pages; all pages are
    numbered by a randperm from a generator seeded (seed << 20) | (1 << 16)
    and handed out in sequence order; unused page-table entries are -1;
  * q [B, H, D], then the caches [num_pages, page_size, H, D] (k, then v):
    randn in fp32 from generators seeded (seed << 20) | t (t = 0, 1, 2),
    cast to bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "SWEEP_LENGTHS", "sweep", "make_inputs",
           "sample_rows", "outlier_rows", "PagedWorkload", "PAGED_WORKLOADS",
           "make_paged_inputs"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Lq: int
    Lk: int
    D: int
    causal: bool
    seed: int
    qk_std: float = 1.0
    outlier_frac: float = 0.0
    outlier_mul: float = 8.0
    sample_rows: int = 0          # rows per head the oracle checks (0 = all)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """4*B*H*Lq*Lk*D (two matrix products), halved when causal."""
        f = 4.0 * self.B * self.H * self.Lq * self.Lk * self.D
        return f / 2 if self.causal else f

    @property
    def bytes(self) -> int:
        """Algorithmic HBM bytes: q, k, v read once, O (bf16) and LSE (fp32)
        written once."""
        bh = self.B * self.H
        return (bh * (self.Lq + 2 * self.Lk) * self.D * 2
                + bh * self.Lq * self.D * 2 + bh * self.Lq * 4)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


SWEEP_LENGTHS = (64, 128, 256, 512, 1024, 2048, 4096, 8192)


def sweep(L: int) -> Workload:
    return Workload(f"sweep_d64_L{L}", 4, 8, L, L, 64, False, 1)


WORKLOADS = {
    "mha_l256_d64": Workload("mha_l256_d64", 4, 8, 256, 256, 64, False, 0),
    "causal_l8k_d128": Workload("causal_l8k_d128", 2, 32, 8192, 8192, 128, True, 2),
    "causal_l64k_d128": Workload("causal_l64k_d128", 1, 32, 65536, 65536, 128, True, 3,
                                 qk_std=3.0, sample_rows=512),
    "decode_l128k_d128": Workload("decode_l128k_d128", 16, 32, 1, 131072, 128, False, 4,
                                  outlier_frac=0.01),
}
for _L in SWEEP_LENGTHS:
    WORKLOADS[f"sweep_d64_L{_L}"] = sweep(_L)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def outlier_rows(w: Workload, b: int, device="cpu"):
    """Per head h, the key rows of batch index b that get the x8 outlier."""
    n = int(math.floor(w.outlier_frac * w.Lk))
    if n == 0:
        return [torch.empty(0, dtype=torch.long, device=device) for _ in range(w.H)]
    g = _gen(device, (w.seed << 20) | (1 << 19) | b)
    return [torch.randperm(w.Lk, generator=g, device=device)[:n] for _ in range(w.H)]


def make_inputs(w: Workload, device="cpu", batches: Optional[range] = None):
    """q [B,Lq], k, v [B,Lk] as bf16 tensors of shape [nb, H, L, D] on `device`.

    `batches` restricts generation to some batch indices (the values of a
    batch index do not depend on which others are generated).
    """
    device = torch.device(device)
    bs = list(range(w.B)) if batches is None else list(batches)
    out = []
    for t, L in enumerate((w.Lq, w.Lk, w.Lk)):
        x = torch.empty((len(bs), w.H, L, w.D), dtype=torch.bfloat16, device=device)
        for n, b in enumerate(bs):
            g = _gen(device, (w.seed << 20) | (b << 2) | t)
            f = torch.randn((w.H, L, w.D), generator=g, device=device, dtype=torch.float32)
            if t < 2 and w.qk_std != 1.0:
                f.mul_(w.qk_std)
            x[n].copy_(f)
            del f
        out.append(x)
    q, k, v = out
    if w.outlier_frac > 0:
        for n, b in enumerate(bs):
            for h, idx in enumerate(outlier_rows(w, b, device)):
                k[n, h, idx] = k[n, h, idx] * w.outlier_mul
    return q, k, v


def sample_rows(w: Workload, n: Optional[int] = None):
    """Per head, the sorted query rows the long-context check compares:
    rows 0 and Lq-1 plus n-2 drawn without replacement (CPU generator)."""
    n = w.sample_rows if n is None else n
    if n == 0 or n >= w.Lq:
        return [torch.arange(w.Lq) for _ in range(w.H * w.B)]
    g = _gen("cpu", (w.seed << 20) | (1 << 18))
    rows = []
    for _ in range(w.B * w.H):
        inner = torch.randperm(w.Lq - 2, generator=g)[: n - 2] + 1
        r = torch.cat([torch.tensor([0, w.Lq - 1]), inner])
        rows.append(torch.sort(r).values)
    return rows


@dataclass(frozen=True)
class PagedWorkload:
    name: str
    B: int
    H: int
    D: int
    page_size: int
    max_len: int
    seed: int
    lengths: Optional[tuple] = None   # fixed lengths instead of drawn ones

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def max_pages(self) -> int:
        return (self.max_len + self.page_size - 1) // self.page_size


PAGED_WORKLOADS = {
    # 16 sequences of up to 128K cached positions, 16-position pages
    "decode_paged_128k_d128": PagedWorkload("decode_paged_128k_d128", 16, 32, 128, 16, 131072, 5),
}


def paged_lengths(w: PagedWorkload) -> torch.Tensor:
    if w.lengths is not None:
        return torch.tensor(w.lengths, dtype=torch.int32)
    g = _gen("cpu", (w.seed << 20) | (1 << 17))
    return torch.randint(1, w.max_len + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)


def make_paged_inputs(w: PagedWorkload, device="cpu"):
    """q [B,H,D], k_cache, v_cache [num_pages, page_size, H, D] (bf16),
    block_table [B, max_pages] and seq_lens [B] (int32), all on `device`."""
    device = torch.device(device)
    lens = paged_lengths(w)
    need = [min(w.max_pages, (max(int(L), 0) + w.page_size - 1) // w.page_size) for L in lens.tolist()]
    num_pages = max(1, sum(need))
    g = _gen("cpu", (w.seed << 20) | (1 << 16))
    order = torch.randperm(num_pages, generator=g)
    table = torch.full((w.B, w.max_pages), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = order[at:at + n].to(torch.int32)
        at += n
    out = []
    for t, shape in enumerate(((w.B, w.H, w.D), (num_pages, w.page_size, w.H, w.D),
                               (num_pages, w.page_size, w.H, w.D))):
        x = torch.empty(shape, dtype=torch.bfloat16, device=device)
        gg = _gen(device, (w.seed << 20) | t)
        flat = x.view(-1, shape[-1])
        step = 1 << 20   # rows per draw, bounds the fp32 temporary
        for r0 in range(0, flat.shape[0], step):
            r1 = min(flat.shape[0], r0 + step)
            flat[r0:r1].copy_(torch.randn((r1 - r0, shape[-1]), generator=gg, device=device,
                                          dtype=torch.float32))
        out.append(x)
    q, kc, vc = out
    return q, kc, vc, table.to(device), lens.to(device)
