"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds no attention arithmetic: it only draws random tensors and
rounds them to the storage type.  Both the CUDA path and the fp64 oracle are
fed the *rounded* 16-bit values, so the two sides see identical inputs.

Recipe (one per workload): every tensor is drawn on the CPU with its own
``torch.Generator`` seeded as listed, as i.i.d. N(0, 1) in float32, multiplied
by the workload's value scale, then rounded to nearest-even into fp16/bf16.
"""
from __future__ import annotations

import dataclasses
import math

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, storage type, mask and input recipe."""

    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str  # "fp16" | "bf16"
    causal: bool
    value_scale: float = 1.0  # multiplies Q, K, V after the N(0,1) draw
    seeds: tuple = (0, 1, 2, 3)  # Q, K, V, dO
    backward: bool = True
    H_kv: int | None = None  # key/value heads (grouped-query attention); None means H
    N_k: int | None = None   # key/value rows; None means N
    softmax_scale: float | None = None  # None means 1/sqrt(d)

    @property
    def kv_heads(self) -> int:
        return self.H if self.H_kv is None else self.H_kv

    @property
    def kv_len(self) -> int:
        return self.N if self.N_k is None else self.N_k

    @property
    def scale(self) -> float:
        """Softmax scale (1/sqrt(d) unless set), rounded to float32 as the kernels receive it."""
        s = 1.0 / math.sqrt(self.d) if self.softmax_scale is None else self.softmax_scale
        return float(torch.tensor(s, dtype=torch.float32))

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the method's evaluation, by shape.
TINY = Workload("tiny_B1_H1_N256_d64_fp16", 1, 1, 256, 64, "fp16", False, 1.0, (0, 1, 2, 3), False)
TRAIN = Workload("train_B4_H16_N2048_d64_fp16", 4, 16, 2048, 64, "fp16", False, 1.0, (10, 11, 12, 13))
LONG = Workload("long_B2_H16_N8192_d128_bf16_causal", 2, 16, 8192, 128, "bf16", True, 0.5, (20, 21, 22, 23))
D256 = Workload("d256_B8_H8_N4096_d256_bf16", 8, 8, 4096, 256, "bf16", False, 1.0, (30, 31, 32, 33))
CTX32K = Workload("ctx32k_B1_H32_N32768_d128_bf16_causal", 1, 32, 32768, 128, "bf16", True, 1.0, (40, 41, 42, 43), False)

WORKLOADS = {w.name: w for w in (TINY, TRAIN, LONG, D256, CTX32K)}


def draw(shape, seed: int, dtype: str, value_scale: float = 1.0) -> torch.Tensor:
    """i.i.d. N(0,1) float32 on the CPU from ``seed``, times ``value_scale``, rounded to ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if value_scale != 1.0:
        x = x * value_scale
    return x.to(DTYPES[dtype])


def make_inputs(w: Workload, with_dout: bool | None = None):
    """Return CPU tensors ``(q, k, v, dout)`` in the storage type: q and dout
    [B, H, N, d], k and v [B, H_kv, N_k, d].

    ``dout`` is drawn unscaled (N(0,1)); it is ``None`` when not requested.
    """
    shape = (w.B, w.H, w.N, w.d)
    kv_shape = (w.B, w.kv_heads, w.kv_len, w.d)
    q = draw(shape, w.seeds[0], w.dtype, w.value_scale)
    k = draw(kv_shape, w.seeds[1], w.dtype, w.value_scale)
    v = draw(kv_shape, w.seeds[2], w.dtype, w.value_scale)
    want = w.backward if with_dout is None else with_dout
    do = draw(shape, w.seeds[3], w.dtype, 1.0) if want else None
    return q, k, v, do


def sample_heads(w: Workload, count: int = 4, seed: int = 1234):
    """Fixed sample of (b, h) pairs: the first, the last and ``count-2`` seeded others."""
    BH = w.B * w.H
    picks = [0, BH - 1]
    g = torch.Generator().manual_seed(seed)
    while len(set(picks)) < min(count, BH):
        picks.append(int(torch.randint(0, BH, (1,), generator=g)))
    out = []
    for i in sorted(set(picks)):
        out.append((i // w.H, i % w.H))
    return out


def sample_rows(N: int, count: int, seed: int = 99):
    """Sorted query rows to check: the first, the last, tile edges and seeded others."""
    rows = {0, N - 1}
    for e in (127, 128, 255, 256):
        if e < N:
            rows.add(e)
    g = torch.Generator().manual_seed(seed)
    extra = torch.randint(0, N, (count,), generator=g).tolist()
    rows.update(extra)
    return sorted(rows)
