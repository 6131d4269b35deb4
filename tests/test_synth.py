"""The seeded input generators both sides consume (CPU only).

They hold no attention arithmetic, but the parity tests, the bench and the smoke
check all rely on them: the same workload must give the same rounded tensors on
every call, in the storage type, with the shapes and value scales the recipe
states, and the softmax scale the kernels receive must be the fp32 value.
"""
import math

import numpy as np
import pytest
import torch

from exact_attention_37_gb300 import synth
from exact_attention_37_gb300.synth import Workload


def test_inputs_are_reproducible_and_in_the_storage_type():
    w = Workload("w", 2, 3, 50, 64, "bf16", True, 1.0, (5, 6, 7, 8))
    a = synth.make_inputs(w, with_dout=True)
    b = synth.make_inputs(w, with_dout=True)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    # distinct seeds give distinct tensors
    assert not torch.equal(a[0], a[1])


def test_each_tensor_is_its_seed_drawn_in_fp32_then_rounded():
    w = Workload("w", 1, 2, 40, 128, "fp16", False, 0.5, (11, 12, 13, 14))
    q, k, v, do = synth.make_inputs(w, with_dout=True)
    for t, seed, scale in ((q, 11, 0.5), (k, 12, 0.5), (v, 13, 0.5), (do, 14, 1.0)):
        g = torch.Generator().manual_seed(seed)
        x = torch.randn(1, 2, 40, 128, generator=g, dtype=torch.float32) * scale
        assert t.dtype == torch.float16
        assert torch.equal(t, x.to(torch.float16))  # round to nearest even, once


def test_grouped_and_unequal_shapes():
    w = Workload("w", 2, 8, 30, 64, "fp16", True, 1.0, (1, 2, 3, 4), True, 2, 70)
    q, k, v, do = synth.make_inputs(w)
    assert q.shape == do.shape == (2, 8, 30, 64)
    assert k.shape == v.shape == (2, 2, 70, 64)
    assert synth.make_inputs(w.with_(backward=False))[3] is None


@pytest.mark.parametrize("d", [64, 128, 256])
def test_softmax_scale_is_the_fp32_value_the_kernels_receive(d):
    w = Workload("w", 1, 1, 8, d, "bf16", False)
    assert w.scale == float(np.float32(1.0 / math.sqrt(d)))
    assert w.with_(softmax_scale=0.3).scale == float(np.float32(0.3))
    assert w.with_(softmax_scale=0.3).scale != 0.3  # 0.3 is not an fp32 value


def test_the_five_workloads_match_their_names():
    for name, w in synth.WORKLOADS.items():
        _, b, h, n, d, dtype, *mask = name.split("_")  # e.g. train_B4_H16_N2048_d64_fp16
        assert (b, h, n, d) == (f"B{w.B}", f"H{w.H}", f"N{w.N}", f"d{w.d}") and dtype == w.dtype
        assert w.causal == (mask == ["causal"])


def test_sampled_heads_and_rows_include_the_edges():
    w = synth.D256
    heads = synth.sample_heads(w, count=4)
    assert heads[0] == (0, 0) and heads[-1] == (w.B - 1, w.H - 1) and len(heads) == 4
    rows = synth.sample_rows(4096, 8)
    assert rows == sorted(set(rows)) and {0, 127, 128, 255, 256, 4095} <= set(rows)
    assert synth.sample_rows(100, 3)[-1] == 99 and max(synth.sample_rows(100, 3)) < 100
