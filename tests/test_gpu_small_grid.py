"""The forward's CTA shape on both sides of its one-wave boundary.

At d = 64 and 128 a forward CTA takes two 128-row query sub-tiles, unless that grid
(B*H*ceil(N/256) CTAs) would fill less than one wave of SMs: then it takes one
sub-tile with two score buffers (twice the CTAs).  These cases put the grid one CTA
below and exactly at the SM count of the device they run on, so each side is run
with the same heads and row counts, and sampled rows (first, a sub-tile boundary,
the ragged last ones) are compared with the oracle.
"""
import pytest
import torch

from exact_attention_37_gb300.synth import Workload

from . import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import exact_attention_37_gb300 as fa
    from exact_attention_37_gb300 import build

    build.build()
    fa.load()


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("below", [True, False], ids=["one_subtile", "two_subtiles"])
@pytest.mark.parametrize("d,dtype", [(64, "fp16"), (128, "bf16")])
def test_forward_at_the_one_wave_boundary(d, dtype, below, causal):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = sms - 1 if below else sms  # one 256-row block per head: the grid has H CTAs
    w = Workload(f"wave_d{d}_H{H}", 1, H, 200, d, dtype, causal, 1.0, (951, 952, 953, 954), False)
    parity.check_forward_sampled(w, [(0, 0), (0, H // 2), (0, H - 1)], [0, 1, 127, 128, 198, 199])
