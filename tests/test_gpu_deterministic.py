"""Bitwise repeatability of the backward pass at every head dimension (no atomics:
each gradient row is summed in a fixed order inside one CTA): repeated calls on
the same inputs give identical dQ, dK, dV.
"""
import pytest
import torch

import exact_attention_37_gb300 as fa
from exact_attention_37_gb300.synth import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_attention_37_gb300 import build

    build.build()
    fa.load()


@pytest.mark.parametrize(
    "w",
    [
        Workload("det_mha", 2, 4, 1000, 128, "bf16", False, 1.0, (501, 502, 503, 504)),
        Workload("det_mha_causal", 2, 4, 1000, 128, "bf16", True, 1.0, (505, 506, 507, 508)),
        Workload("det_gqa_unequal", 1, 4, 700, 128, "fp16", True, 1.0, (509, 510, 511, 512), True, 2, 1000),
        Workload("det_d64", 2, 3, 900, 64, "fp16", True, 1.0, (513, 514, 515, 516)),
        Workload("det_d64_mqa", 1, 4, 500, 64, "bf16", False, 1.0, (517, 518, 519, 520), True, 1, 777),
        Workload("det_d256", 2, 3, 1000, 256, "bf16", False, 1.0, (521, 522, 523, 524)),
        Workload("det_d256_causal", 2, 3, 1000, 256, "bf16", True, 1.0, (525, 526, 527, 528)),
        Workload("det_d256_gqa_unequal", 1, 4, 700, 256, "fp16", True, 1.0, (529, 530, 531, 532), True, 2, 1000),
    ],
    ids=lambda w: w.name,
)
def test_backward_is_bitwise_repeatable(w):
    q, k, v, do = (x.cuda() for x in make_inputs(w, with_dout=True))
    o, lse = fa.forward(q, k, v, scale=w.scale, causal=w.causal)
    first = fa.backward(q, k, v, o, lse, do, scale=w.scale, causal=w.causal)
    for _ in range(3):
        again = fa.backward(q, k, v, o, lse, do, scale=w.scale, causal=w.causal)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    fa.fa_check_device_status()
