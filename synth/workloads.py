"""Workload recipes: shapes, value distributions and step counts of the synthetic
ZeRO shard-step workloads, and helpers that materialise their inputs on a CUDA device
with the seeded generator. Input recipes only: nothing here computes the step.

Every workload follows the same recipe. Per step and per logical rank k, rank k's fp16
gradient for the whole flat buffer is an independent draw of N(0, grad_sigma) times the
loss scale (Irwin-Hall(8) stand-in, see ``synth``), rounded to fp16; flat indices past
the real parameters (the partition padding) are 0. The fp32 master weights are
N(0, master_sigma); the momentum is N(0, m_sigma) or 0; the variance is
|N(0, v_sigma)| or 0. The fp16 parameter copy starts as fp16(master).
"""
from __future__ import annotations

from dataclasses import dataclass, field

from . import (EXP_AVG, EXP_AVG_SQ, GRAD, MASTER, SHARD16, fill, inject_index, stream_key)


@dataclass(frozen=True)
class Workload:
    name: str
    cfg: int                 # stream id of the workload in the generator
    n: int                   # real parameters N
    nd: int                  # logical data-parallel ranks
    align: int
    stage: int
    r0: int                  # span of logical ranks processed on this device
    r1: int
    loss_scale: float
    grad_sigma: float        # of the unscaled gradient
    clip: float              # <= 0: no clipping
    steps: int
    master_sigma: float = 0.02
    m_sigma: float = 0.0
    v_sigma: float = 0.0
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    inject: tuple = ()       # ((step, rank, value_bits, where), ...), where: "seeded" or int
    layers: tuple = ()       # ZeRO-3 gather: layer offsets into the flat buffer
    shard_sigma: float = 0.02
    seed: int = 0

    def hparams(self) -> dict:
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay)

    def layout(self) -> tuple[int, int]:
        unit = self.nd * self.align
        np_ = -(-self.n // unit) * unit
        return np_, np_ // self.nd

    def span(self) -> tuple[int, int, int]:
        """(first flat index, span length, real parameters in the span)."""
        _, s = self.layout()
        first = self.r0 * s
        n_span = (self.r1 - self.r0) * s
        return first, n_span, max(0, min(n_span, self.n - first))

    def injections(self, step: int) -> list[tuple[int, int, int]]:
        """(rank, span-relative index, fp16 bits) planted into this step's gradients."""
        out = []
        first, n_span, n_valid = self.span()
        for st, rank, bits, where in self.inject:
            if st != step:
                continue
            i = inject_index(self.seed, self.cfg, step, rank, self.n) if where == "seeded" else where
            if first <= i < first + n_span:
                out.append((rank, i - first, bits))
        return out


# fp16 bit patterns
POS_INF = 0x7C00
NEG_INF = 0xFC00
QNAN = 0x7E00

WORKLOADS = {
    w.name: w for w in [
        # tiny ZeRO-2 step, all four ranks on the device
        Workload("zero2_tiny_1m_nd4", cfg=0, n=1_048_576, nd=4, align=8, stage=2, r0=0, r1=4,
                 loss_scale=1024.0, grad_sigma=1e-3, clip=0.0, steps=3),
        # GPT-2-small-sized flat buffer, 128-element alignment, random moments, clipping
        Workload("gpt2_small_flat_nd8", cfg=1, n=124_439_808, nd=8, align=128, stage=2, r0=0,
                 r1=8, loss_scale=65536.0, grad_sigma=1e-3, clip=1.0, steps=10,
                 m_sigma=1e-3, v_sigma=1e-6),
        # 1.3B flat buffer, 16 ranks; the third step (index 2) gets one +inf in rank 5
        Workload("flat_1p3b_nd16_inf", cfg=2, n=1_300_000_000, nd=16, align=8, stage=2, r0=0,
                 r1=16, loss_scale=4096.0, grad_sigma=1e-3, clip=1.0, steps=8,
                 inject=((2, 5, POS_INF, "seeded"),)),
        # 7B ZeRO-2: this device is rank 0 and owns S = 875M parameters
        Workload("zero2_7b_rank0_nd8", cfg=3, n=7_000_000_000, nd=8, align=8, stage=2, r0=0,
                 r1=1, loss_scale=1024.0, grad_sigma=1e-3, clip=1.0, steps=5),
        # the GPT-2-small recipe on a 32M-parameter buffer (1 GB on the device): a case
        # small enough for detailed profiler captures, still far larger than L2
        Workload("flat_32m_nd8", cfg=5, n=33_554_432, nd=8, align=128, stage=2, r0=0, r1=8,
                 loss_scale=65536.0, grad_sigma=1e-3, clip=1.0, steps=3,
                 m_sigma=1e-3, v_sigma=1e-6),
        # the 13B ZeRO-3 recipe at a tenth of the size (40 layers of 32.5M, 5.2 GB of shards
        # and layers): a case for detailed profiler captures of the gather
        Workload("zero3_1p3b_rank0_nd64", cfg=6, n=1_300_000_000, nd=64, align=8, stage=3,
                 r0=0, r1=1, loss_scale=1024.0, grad_sigma=1e-3, clip=1.0, steps=5,
                 layers=tuple(l * 32_500_000 for l in range(41))),
        # 13B, 40 layers of 325M, ZeRO-3: rank 0's step over S ~ 203M, then the gather of
        # all 64 fp16 shards into the 40 layer buffers
        Workload("zero3_13b_rank0_nd64", cfg=4, n=13_000_000_000, nd=64, align=8, stage=3, r0=0,
                 r1=1, loss_scale=1024.0, grad_sigma=1e-3, clip=1.0, steps=5,
                 layers=tuple(l * 325_000_000 for l in range(41))),
    ]
}


def key(w: Workload, kind: int, step: int = 0, rank: int = 0) -> int:
    return stream_key(w.seed, kind, w.cfg, step, rank)


def make_state(w: Workload, device="cuda"):
    """(master, exp_avg, exp_avg_sq, param16, workspace) for the span, on the device."""
    import torch
    first, n_span, _ = w.span()
    master = torch.empty(n_span, dtype=torch.float32, device=device)
    m = torch.zeros(n_span, dtype=torch.float32, device=device)
    v = torch.zeros(n_span, dtype=torch.float32, device=device)
    fill(master, key(w, MASTER), w.master_sigma, start=first, n_valid=w.n)
    if w.m_sigma > 0:
        fill(m, key(w, EXP_AVG), w.m_sigma, start=first, n_valid=w.n)
    if w.v_sigma > 0:
        fill(v, key(w, EXP_AVG_SQ), -w.v_sigma, start=first, n_valid=w.n)
    p16 = master.to(torch.float16)
    ws = torch.empty(n_span, dtype=torch.float32, device=device)
    return master, m, v, p16, ws


def fill_grads(w: Workload, step: int, out: list) -> None:
    """Write step ``step``'s nd fp16 gradient contributions into ``out`` (span-relative)."""
    import torch
    first, n_span, _ = w.span()
    for k, t in enumerate(out):
        assert t.dtype == torch.float16 and t.numel() == n_span
        fill(t, key(w, GRAD, step, k), w.grad_sigma * w.loss_scale, start=first, n_valid=w.n)
    for rank, idx, bits in w.injections(step):
        out[rank].view(torch.int16)[idx] = bits - 65536 if bits >= 32768 else bits


def make_grads(w: Workload, step: int, device="cuda") -> list:
    import torch
    _, n_span, _ = w.span()
    out = [torch.empty(n_span, dtype=torch.float16, device=device) for _ in range(w.nd)]
    fill_grads(w, step, out)
    return out


def make_shards(w: Workload, shard0, device="cuda") -> list:
    """The nd fp16 shards for the gather: rank 0's is ``shard0`` (the step's output), the
    others are seeded N(0, shard_sigma) values of their own flat indices."""
    import torch
    _, s = w.layout()
    shards = [shard0]
    for r in range(1, w.nd):
        t = torch.empty(s, dtype=torch.float16, device=device)
        fill(t, key(w, SHARD16, 0, r), w.shard_sigma, start=r * s, n_valid=w.n)
        shards.append(t)
    return shards


def span_shards(w: Workload, span16, device="cuda") -> list:
    """The nd fp16 shards for the gather after a step over the span [r0, r1): the span's
    own shards are slices of ``span16`` (the step's fp16 output, (r1 - r0) * S elements),
    the other ranks' are seeded N(0, shard_sigma) values of their own flat indices."""
    import torch
    _, s = w.layout()
    shards = []
    for r in range(w.nd):
        if w.r0 <= r < w.r1:
            shards.append(span16[(r - w.r0) * s:(r - w.r0 + 1) * s])
            continue
        t = torch.empty(s, dtype=torch.float16, device=device)
        fill(t, key(w, SHARD16, 0, r), w.shard_sigma, start=r * s, n_valid=w.n)
        shards.append(t)
    return shards
