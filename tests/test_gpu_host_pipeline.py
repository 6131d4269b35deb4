"""The host-buffer entry points (head chunks pipelined over the library's streams)
give the same results as the device entry points on the whole problem, bitwise
(every path is deterministic), whatever the chunk count.  The device scratch is
filled with 0xFF bytes (NaN in both 16-bit formats) before each call, so a copy
to the host that started before the kernel writing its tensor had run (dK and dV
go back while the dQ kernel runs) would show as NaN, not as an earlier call's
identical result.
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


@pytest.mark.parametrize("chunks", [0, 1, 3, 64])
@pytest.mark.parametrize(
    "w",
    [
        Workload("host_d128", 2, 3, 777, 128, "bf16", True, 1.0, (701, 702, 703, 704)),
        Workload("host_d64_odd_n", 1, 5, 513, 64, "fp16", False, 1.0, (705, 706, 707, 708)),
        # 16 heads, N a multiple of 4: the default plan is 2, 4, 4, 4, 2 heads
        Workload("host_d128_16_heads", 2, 8, 256, 128, "bf16", True, 1.0, (709, 710, 711, 712)),
        # 35 heads of odd length: chunk starts must be multiples of 4 heads (L stays
        # 16-byte aligned); the default plan is 8, 12, 4, 11
        Workload("host_d64_35_heads", 5, 7, 33, 64, "fp16", True, 1.0, (713, 714, 715, 716)),
        # kernels long enough that a download racing them would read unwritten scratch
        Workload("host_d128_long", 1, 8, 2048, 128, "bf16", True, 1.0, (717, 718, 719, 720)),
        # one launch writes dQ, dK and dV at d = 256
        Workload("host_d256", 1, 3, 300, 256, "bf16", True, 1.0, (721, 722, 723, 724)),
    ],
    ids=lambda w: w.name,
)
def test_host_pipeline_matches_device_path(w, chunks):
    q, k, v, do = make_inputs(w, with_dout=True)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o_ref, lse_ref = fa.forward(qd, kd, vd, scale=w.scale, causal=w.causal)
    dq_ref, dk_ref, dv_ref = fa.backward(qd, kd, vd, o_ref, lse_ref, dod, scale=w.scale, causal=w.causal)
    B, H, N, d = q.shape
    pin = lambda t: t.contiguous().pin_memory()
    qh, kh, vh, doh = (pin(x) for x in (q, k, v, do))
    oh, dqh, dkh, dvh = (torch.empty_like(x).pin_memory() for x in (q, q, k, v))
    lseh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    scratch = torch.full((fa.fa_host_scratch_size(B, H, N, d, True),), 0xFF, dtype=torch.uint8, device="cuda")
    fa.fa_fwd_bwd_host(qh, kh, vh, doh, oh, lseh, dqh, dkh, dvh, scratch, w.scale, w.causal, chunks)
    torch.cuda.current_stream().synchronize()
    fa.fa_check_device_status()
    for got, ref in ((oh, o_ref), (lseh, lse_ref), (dqh, dq_ref), (dkh, dk_ref), (dvh, dv_ref)):
        assert torch.equal(got, ref.cpu())
    # forward only
    oh2 = torch.empty_like(oh)
    lseh2 = torch.empty_like(lseh)
    scratch_f = torch.full((fa.fa_host_scratch_size(B, H, N, d, False),), 0xFF, dtype=torch.uint8, device="cuda")
    fa.fa_fwd_host(qh, kh, vh, oh2, lseh2, scratch_f, w.scale, w.causal, chunks)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(oh2, o_ref.cpu()) and torch.equal(lseh2, lse_ref.cpu())
