"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small problems are compared element by element over every head; they span
several 128-row tiles and a ragged tail.  The five workloads of the method's
evaluation are run at full size in the launch configuration the bench uses and
checked on sampled heads and rows.  Tolerances are in tests/parity.py.
"""
import numpy as np
import pytest
import torch

import exact_attention_37_gb300 as fa
import oracle
from exact_attention_37_gb300 import synth
from exact_attention_37_gb300.synth import Workload

from . import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_attention_37_gb300 import build

    build.build()
    fa.load()


def small(N, d, dtype, causal, B=1, H=2, scale=1.0, seeds=(101, 102, 103, 104)):
    return Workload(f"small_N{N}_d{d}_{dtype}_{'c' if causal else 'nc'}", B, H, N, d, dtype, causal, scale, seeds)


# --------------------------------------------------------------------- forward, exact over all elements
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_small(d, dtype, causal):
    parity.check_forward_full(small(300, d, dtype, causal))


@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 256, 257, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_ragged_lengths(N, causal):
    parity.check_forward_full(small(N, 128, "bf16", causal, B=1, H=1))


def test_forward_tiny_workload():
    parity.check_forward_full(synth.TINY)


def test_forward_many_heads_few_rows():
    parity.check_forward_full(small(64, 64, "fp16", True, B=3, H=5))


def test_forward_empty():
    q = torch.empty(1, 2, 0, 64, dtype=torch.float16, device="cuda")
    o, lse = fa.forward(q, q, q)
    assert o.shape == q.shape and lse.shape == (1, 2, 0)


# --------------------------------------------------------------------- backward, exact over all elements
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_small(d, dtype, causal):
    parity.check_backward_full(small(300, d, dtype, causal))


@pytest.mark.parametrize("N", [1, 64, 65, 127, 129, 200])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_backward_ragged_lengths(N, d):
    # d = 256 streams 64-row tiles in its dK and dQ CTAs and 128-row tiles in its dV
    # CTAs, so 64, 65, 127 and 129 rows put a ragged tail in each
    parity.check_backward_full(small(N, d, "bf16", True, B=1, H=1))


# --------------------------------------------------------------------- the softmax scale argument
@pytest.mark.parametrize("scale", [0.03, 0.3, 1.0])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_softmax_scale_argument(d, scale):
    # Every other case runs at 1/sqrt(d); here the kernels must take the scale they are
    # given, in the exponent of P (forward and backward) and in dQ = scale dS K and
    # dK = scale dS^T Q.  At 1.0 the rows are far from uniform (scores of spread sqrt(d)).
    w = small(200, d, "bf16", True, H=2).with_(softmax_scale=scale, name=f"scale{scale}_d{d}")
    parity.check_backward_full(w)
    for causal in (True, False):
        parity.check_forward_full(w.with_(causal=causal))


# --------------------------------------------------------------------- the five workloads at full size
def test_train_workload_forward_sampled():
    w = synth.TRAIN
    for causal in (False, True):
        wc = w.with_(causal=causal)
        parity.check_forward_sampled(wc, synth.sample_heads(wc), synth.sample_rows(wc.N, 48))


def test_train_workload_backward_sampled():
    for causal in (False, True):
        wc = synth.TRAIN.with_(causal=causal)
        parity.check_backward_sampled(wc, synth.sample_heads(wc, count=3))


def test_long_workload_forward_sampled():
    w = synth.LONG
    parity.check_forward_sampled(w, synth.sample_heads(w), synth.sample_rows(w.N, 64))


def test_long_workload_backward_sampled():
    w = synth.LONG
    parity.check_backward_sampled(w, synth.sample_heads(w, count=2))


def test_d256_workload_forward_sampled():
    for causal in (False, True):
        w = synth.D256.with_(causal=causal)
        parity.check_forward_sampled(w, synth.sample_heads(w), synth.sample_rows(w.N, 48))


def test_d256_workload_backward_sampled():
    for causal in (False, True):
        w = synth.D256.with_(causal=causal)
        parity.check_backward_sampled(w, synth.sample_heads(w, count=2))


def test_ctx32k_workload_forward_sampled():
    w = synth.CTX32K
    parity.check_forward_sampled(w, synth.sample_heads(w), synth.sample_rows(w.N, 64))


def test_ctx32k_backward_one_head():
    # the longest sequence of the workloads (N = 32768), backward included: two heads
    # on the GPU, the second checked in full against the oracle (row chunks)
    w = synth.CTX32K.with_(H=2, backward=True)
    parity.check_backward_sampled(w, [(0, 1)])


def test_ctx128k_causal_forward_and_backward_sampled():
    """N = 131072 (four times the longest workload), causal, two heads: sampled rows
    of O and L, dQ of sampled rows, and dK, dV of the last 512 keys, which under the
    causal mask only the last 512 queries see, so the oracle evaluates those rows
    alone and still gives the exact gradients."""
    N = 131072
    w = synth.CTX32K.with_(name="ctx128k", H=2, N=N, backward=True)
    q, k, v, do = synth.make_inputs(w, with_dout=True)
    o, lse, dq, dk, dv = parity.run_backward(w, q, k, v, do)
    o, lse, dq, dk, dv = (t.float().cpu() for t in (o, lse, dq, dk, dv))
    rows = [0, 1, 4095, 65536, N - 513, N - 512, N - 1]
    tail = np.arange(N - 512, N)
    for h in (0, 1):
        O_ref, L_ref = oracle.forward_rows(q[0, h], k[0, h], v[0, h], w.scale, True, rows)
        parity.compare_o(w, o[0, h, rows].numpy().astype(np.float64), O_ref, f"O[0,{h}]")
        parity.compare_l(lse[0, h, rows].numpy().astype(np.float64), L_ref)
        rdq, _, _, _ = oracle.head_backward_rows(q[0, h], k[0, h], v[0, h], do[0, h], w.scale, True, rows)
        parity.compare_g(dq[0, h, rows].numpy().astype(np.float64), rdq, f"dQ[0,{h}] rows")
        _, rdk, rdv, _ = oracle.head_backward_rows(q[0, h], k[0, h], v[0, h], do[0, h], w.scale, True, tail)
        parity.compare_g(dk[0, h, N - 512:].numpy().astype(np.float64), rdk[N - 512:], f"dK[0,{h}] last keys")
        parity.compare_g(dv[0, h, N - 512:].numpy().astype(np.float64), rdv[N - 512:], f"dV[0,{h}] last keys")


@pytest.mark.parametrize("d,dtype,causal", [(64, "fp16", False), (128, "bf16", True), (256, "bf16", True)])
def test_many_heads_short_sequences(d, dtype, causal):
    """About a thousand heads of a few hundred rows (the ragged tail in every head):
    the CTA order over head groups and the plane indexing at large B*H, checked on
    heads spread over the batch (first, middle, last)."""
    w = Workload(f"many_heads_d{d}", 32, 32, 130, d, dtype, causal, 1.0, (961, 962, 963, 964))
    heads = [(0, 0), (15, 17), (31, 31)]
    parity.check_forward_sampled(w, heads, list(range(0, 130, 7)) + [129])
    parity.check_backward_sampled(w, heads)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_tensors_past_two_to_the_31_elements(d):
    """Every tensor holds more than 2^31 elements (about 4.3 GB each, some 35 GB in all
    with the gradients): the element offset of head h is h N d, which passes 2^31 at
    h* = 2^31 / (N d), so an index computed in 32-bit arithmetic anywhere (a pointer
    offset, a tensor-map plane, a workspace row) would put the heads from h* on in the
    wrong place.  Inputs are N(0, 1) drawn on the device from a seeded generator (a
    host draw of this size takes minutes); the heads on both sides of h* and the last
    one are copied back and checked in full, forward and backward, against the oracle."""
    N = 1024
    h_star = (1 << 31) // (N * d)
    B, H = 2, h_star // 2 + 8  # B*H = h_star + 16 heads
    torch.cuda.empty_cache()
    g = torch.Generator(device="cuda")
    g.manual_seed(20000 + d)
    q, k, v, do = (torch.randn(B, H, N, d, generator=g, device="cuda", dtype=torch.bfloat16) for _ in range(4))
    assert q.numel() > (1 << 31)
    scale = float(np.float32(1.0 / np.sqrt(d)))
    o, lse = fa.forward(q, k, v, scale=scale, causal=True)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, scale=scale, causal=True)
    fa.fa_check_device_status()
    w = Workload("past_2_31", 1, 1, N, d, "bf16", True)
    for i in (0, h_star - 1, h_star, h_star + 1, B * H - 1):
        b, h = divmod(i, H)
        one = lambda t: t[b, h][None, None].cpu()
        q1, k1, v1, do1 = (one(t) for t in (q, k, v, do))
        O_ref, L_ref = oracle.attention_forward(q1, k1, v1, scale, True)
        parity.compare_o(w, parity.to_np(one(o)), O_ref, f"O head {i}")
        parity.compare_l(one(lse).numpy().astype(np.float64), L_ref)
        rdq, rdk, rdv, _ = oracle.attention_backward(q1, k1, v1, do1, scale, True)
        parity.compare_g(parity.to_np(one(dq)), rdq, f"dQ head {i}")
        parity.compare_g(parity.to_np(one(dk)), rdk, f"dK head {i}")
        parity.compare_g(parity.to_np(one(dv)), rdv, f"dV head {i}")
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


def test_forward_allocates_nothing_beyond_its_outputs():
    """O(N) memory: at N = 32768 a single fp32 score matrix of one head would take
    4.3 GB; the forward call's footprint is its two outputs (allocated by torch in
    ``fa.forward``) and nothing else -- the library itself allocates no device memory."""
    w = synth.CTX32K
    q, k, v, _ = synth.make_inputs(w, with_dout=False)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    o, lse = fa.forward(qd, kd, vd, scale=w.scale, causal=w.causal)
    fa.fa_check_device_status()
    free1, _ = torch.cuda.mem_get_info()
    out_bytes = o.numel() * o.element_size() + lse.numel() * lse.element_size()
    assert torch.cuda.max_memory_allocated() - base <= out_bytes + (4 << 20)
    # nothing outside torch's allocator either (the caching allocator may round up its segment)
    assert free0 - free1 <= out_bytes + (64 << 20)
