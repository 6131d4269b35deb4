"""The device-buffer entry points inside a captured CUDA graph.

A training loop that is launch-bound captures its step once and replays it, so the
forward and backward calls must be capturable: no synchronizing call, allocation or
host read on their path once the library has been used on the device.  Each case
runs forward + backward eagerly, captures the same calls on static buffers, replays
the graph, and requires the replay to give bitwise the eager results (the kernels
are deterministic); it then copies new inputs into the captured buffers, replays
again and compares with eager calls on those inputs.
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


CASES = [
    Workload("graph_d64_fp16", 2, 4, 700, 64, "fp16", False, 1.0, (901, 902, 903, 904)),
    Workload("graph_d128_bf16_causal_gqa", 1, 4, 1000, 128, "bf16", True, 1.0, (905, 906, 907, 908), True, 2, 1000),
    Workload("graph_d256_bf16_causal", 1, 2, 513, 256, "bf16", True, 1.0, (909, 910, 911, 912)),
]


def eager(w, q, k, v, do):
    o, lse = fa.forward(q, k, v, scale=w.scale, causal=w.causal)
    return (o, lse, *fa.backward(q, k, v, o, lse, do, scale=w.scale, causal=w.causal))


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_forward_backward_replay_matches_eager(w):
    q, k, v, do = (x.cuda() for x in make_inputs(w, with_dout=True))
    ref = eager(w, q, k, v, do)
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capture stream, as torch recommends
        eager(w, q, k, v, do)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = eager(w, q, k, v, do)
    g.replay()
    torch.cuda.synchronize()
    fa.fa_check_device_status()
    for name, a, b in zip(("O", "L", "dQ", "dK", "dV"), out, ref):
        assert torch.equal(a, b), f"{w.name}: {name} of the replay differs from the eager call"

    # new inputs in the captured buffers
    q2, k2, v2, do2 = (x.cuda() for x in make_inputs(
        Workload(w.name + "_2", w.B, w.H, w.N, w.d, w.dtype, w.causal, w.value_scale,
                 tuple(s + 100 for s in w.seeds), True, w.H_kv, w.N_k), with_dout=True))
    for dst, src in zip((q, k, v, do), (q2, k2, v2, do2)):
        dst.copy_(src)
    g.replay()
    torch.cuda.synchronize()
    ref2 = eager(w, q2, k2, v2, do2)
    torch.cuda.synchronize()
    fa.fa_check_device_status()
    for name, a, b in zip(("O", "L", "dQ", "dK", "dV"), out, ref2):
        assert torch.equal(a, b), f"{w.name}: {name} of the second replay differs from the eager call"
