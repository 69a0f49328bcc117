"""Seeded synthetic attention workloads.

This module only draws inputs: shapes, seeds and random tensors.  It holds none
of the attention arithmetic, so both the CUDA path and the CPU oracle may be fed
from it.

Recipe (every workload): a CPU ``torch.Generator`` seeded with the workload's
seed draws fp32 ``randn`` tensors of shape [B, H, N, d] in the order Q, K, V
(then dO for the backward workload); each is rounded to bf16 (round to nearest
even).  The "K x 3" workload multiplies K by 3 in fp32 before the rounding, so
that rows are close to one-hot and the running max is exercised.  The causal and
non-causal runs of one workload share inputs; scale = 1/sqrt(d).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    seed: int
    causal_modes: tuple = (True,)
    k_scale: float = 1.0
    backward: bool = False
    sampled_rows: int = 0  # 0 = every query row is checkable in full
    note: str = ""

    @property
    def BH(self) -> int:
        return self.B * self.H

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def shape(self):
        return (self.B, self.H, self.N, self.d)


# The five workloads: sizes, seeds, value distributions.
WORKLOADS = {
    "single_head_256": Workload(
        "single_head_256", 1, 1, 256, 64, seed=0, causal_modes=(False, True),
        note="single-head fwd B=1 H=1 N=256 d=64, non-causal and causal"),
    "fwd_2k_d64": Workload(
        "fwd_2k_d64", 4, 16, 2048, 64, seed=1, causal_modes=(False, True),
        note="fwd B=4 H=16 N=2048 d=64, non-causal and causal"),
    "fwd_8k_d128_kx3": Workload(
        "fwd_8k_d128_kx3", 2, 16, 8192, 128, seed=2, causal_modes=(True,), k_scale=3.0,
        note="fwd B=2 H=16 N=8192 d=128, K rows scaled by 3, causal"),
    "fwd_32k_d128": Workload(
        "fwd_32k_d128", 1, 32, 32768, 128, seed=3, causal_modes=(True,), sampled_rows=512,
        note="long-context fwd B=1 H=32 N=32768 d=128, causal, 512 sampled rows per head"),
    "fwdbwd_4k_d128": Workload(
        "fwdbwd_4k_d128", 4, 16, 4096, 128, seed=4, causal_modes=(True,), backward=True,
        note="fwd+bwd B=4 H=16 N=4096 d=128, causal, dO iid N(0,1)"),
}


def make_inputs(w: Workload, device="cpu", B=None, H=None, N=None, d=None, seed=None):
    """Draw Q, K, V (and dO when the workload has a backward) as bf16 [B,H,N,d].

    Overrides (B, H, N, d, seed) let tests draw the same distribution at other
    sizes.  Returns a dict of tensors on ``device``."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    N = w.N if N is None else N
    d = w.d if d is None else d
    seed = w.seed if seed is None else seed
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if w.k_scale != 1.0:
        k = k * w.k_scale
    out = {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}
    if w.backward:
        out["do"] = torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return {n: t.to(device) for n, t in out.items()}


def make_inputs_device(B, H, N, d, seed, device, backward=True):
    """Q, K, V (and dO) as iid N(0, 1) bf16 [B, H, N, d], drawn by PyTorch's
    generator on ``device`` (seeded, in that order): for sizes near the 2^31
    element limit, where the host generator of make_inputs would take minutes.
    The same recipe otherwise; the values differ from make_inputs' for a seed."""
    g = torch.Generator(device=device).manual_seed(seed)
    names = ("q", "k", "v", "do") if backward else ("q", "k", "v")
    return {n: torch.randn((B, H, N, d), generator=g, device=device, dtype=torch.float32)
            .to(torch.bfloat16) for n in names}


def random_bf16(shape, seed: int, scale: float = 1.0, device="cpu"):
    """One bf16 tensor of iid N(0, scale^2) values from a seeded CPU generator."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    t = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if scale != 1.0:
        t = t * scale
    return t.to(torch.bfloat16).to(device)


def sampled_rows(w: Workload, count=None, BH=None, N=None):
    """Per head (b, h): ``count`` distinct query rows drawn without replacement
    from a generator seeded ``seed + 1000 + b*H + h``; rows 0 and N-1 are always
    included.  Returns a sorted int64 array [BH, count]."""
    count = w.sampled_rows if count is None else count
    BH = w.BH if BH is None else BH
    N = w.N if N is None else N
    if count >= N:
        return np.tile(np.arange(N, dtype=np.int64), (BH, 1))
    rows = np.empty((BH, count), dtype=np.int64)
    for bh in range(BH):
        g = torch.Generator(device="cpu").manual_seed(w.seed + 1000 + bh)
        inner = torch.randperm(N - 2, generator=g)[: count - 2].numpy().astype(np.int64) + 1
        rows[bh] = np.sort(np.concatenate([[0, N - 1], inner]))
    return rows


def worked_example_inputs(d: int = 64, device="cpu"):
    """The 3-score example (scores [0, ln2, ln3], V = [1, 2, 4]) encoded as
    attention inputs with N = 3, d = 64, scale = 1: every query is (1, 1, 0, ...),
    key j is (hi_j, lo_j, 0, ...) where hi_j = bf16(s_j) and lo_j = bf16(s_j - hi_j),
    so q . k_j = hi_j + lo_j reproduces s_j to about 2^-16; V[:, 0] = (1, 2, 4)
    and the other value columns are 0.  Returns bf16 tensors [1, 1, 3, d]."""
    s = torch.tensor([0.0, math.log(2.0), math.log(3.0)], dtype=torch.float64)
    hi = s.to(torch.bfloat16)
    lo = (s - hi.to(torch.float64)).to(torch.bfloat16)
    q = torch.zeros(1, 1, 3, d, dtype=torch.bfloat16)
    q[..., 0] = 1.0
    q[..., 1] = 1.0
    k = torch.zeros(1, 1, 3, d, dtype=torch.bfloat16)
    k[0, 0, :, 0] = hi
    k[0, 0, :, 1] = lo
    v = torch.zeros(1, 1, 3, d, dtype=torch.bfloat16)
    v[0, 0, :, 0] = torch.tensor([1.0, 2.0, 4.0]).to(torch.bfloat16)
    return {"q": q.to(device), "k": k.to(device), "v": v.to(device)}


def sign_bits(seed: int, d: int = 128) -> np.ndarray:
    """Random signs for the FP8 path's Hadamard rotation, as d/32 uint32 words
    (bit j set: s_j = -1): d fair coin flips from a CPU generator seeded
    ``seed``."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    flips = torch.randint(0, 2, (d,), generator=g).numpy().astype(np.uint64)
    words = np.zeros(d // 32, dtype=np.uint64)
    for j in range(d):
        words[j // 32] |= flips[j] << np.uint64(j % 32)
    return words.astype(np.uint32)


def outlier_inputs(B: int, H: int, N: int, d: int, seed: int, kind: str = "entries",
                   device="cpu"):
    """Q, K, V with simulated outlier features (bf16 [B,H,N,d]).

    kind "entries": every entry is N(0, 1) plus, with probability 0.001, an
    extra N(0, 10^2) term (independently in Q, K and V).
    kind "channels": N(0, 1) entries, except that 4 feature channels (drawn
    once per seed, the same for Q and K and for every head and row) have
    standard deviation 5 in Q and K; V is plain N(0, 1)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if kind == "entries":
        for t in (q, k, v):
            hit = torch.rand(shape, generator=g) < 0.001
            t += hit * torch.randn(shape, generator=g, dtype=torch.float32) * 10.0
    elif kind == "channels":
        ch = torch.randperm(d, generator=g)[:4]
        q[..., ch] *= 5.0
        k[..., ch] *= 5.0
    else:
        raise ValueError(f"unknown outlier kind {kind!r}")
    return {n: t.to(torch.bfloat16).to(device) for n, t in (("q", q), ("k", k), ("v", v))}


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bf16 bit patterns of a tensor as a uint16 numpy array [BH, N, d]."""
    t = t.detach().to("cpu").contiguous()
    assert t.dtype == torch.bfloat16
    a = t.view(torch.int16).numpy().view(np.uint16)
    return a.reshape(-1, t.shape[-2], t.shape[-1])
