"""The checked build (libfa_attention_debug.so, compiled with -DFA_DEBUG) on the GPU.

It runs the same kernels with device-side checks before every TMA copy, tensor
memory access and tensor-core product, and of every mbarrier's phase count at
CTA exit; a failed check records itself in the device error record and the
kernel runs on.  This is the stand-in for a memory checker on machines where none
can be run.  Two things are shown here:

  - small parity cases (every head dimension, both masks, ragged tails, grouped
    heads with unequal lengths) run clean through the checked build -- no check
    fires -- and still match the fp64 oracle;
  - each kind of check does fire: a self-test hands it a value that breaks its
    rule (nothing is copied or accessed) and the status check reports it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_attention_37_gb300 import _lib
from exact_attention_37_gb300.synth import Workload, make_inputs

from . import parity

pytestmark = pytest.mark.gpu

FA_OK, FA_ERR_DEVICE_CHECK = 0, 7


@pytest.fixture(scope="module")
def dlib():
    from exact_attention_37_gb300 import build

    return _lib.open_library(build.build(debug=True))


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def status(dlib):
    code = dlib.fa_check_device_status(_stream())
    rec = (ctypes.c_uint32 * 4)()
    dlib.fa_last_device_error_detail(rec)
    return code, [int(x) for x in rec]


CASES = [
    Workload("dbg_d64_nc", 1, 2, 300, 64, "fp16", False, 1.0, (701, 702, 703, 704)),
    Workload("dbg_d64_c_ragged", 2, 1, 129, 64, "bf16", True, 1.0, (705, 706, 707, 708)),
    Workload("dbg_d128_c", 1, 2, 300, 128, "bf16", True, 1.0, (709, 710, 711, 712)),
    Workload("dbg_d128_gqa_unequal", 1, 4, 200, 128, "fp16", True, 1.0, (713, 714, 715, 716), True, 2, 333),
    Workload("dbg_d256_nc", 1, 2, 300, 256, "bf16", False, 1.0, (717, 718, 719, 720)),
    Workload("dbg_d256_c_unequal", 1, 4, 333, 256, "bf16", True, 1.0, (721, 722, 723, 724), True, 2, 200),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_checked_build_runs_parity_cases_clean(dlib, w):
    assert status(dlib)[0] == FA_OK  # start from a clear record
    q, k, v, do = make_inputs(w, with_dout=True)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    B, H, Nq, d = qd.shape
    Hkv, Nk = kd.shape[1], kd.shape[2]
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(max(1, dlib.fa_bwd_workspace_size(B, H, Nq, d)), dtype=torch.uint8, device="cuda")
    dt = _lib._dtype_code(qd)
    sc = ctypes.c_float(w.scale)
    assert dlib.fa_fwd_ex(_p(qd), _p(kd), _p(vd), _p(o), _p(lse), B, H, Hkv, Nq, Nk, d, sc, int(w.causal), dt,
                          _stream()) == FA_OK
    assert dlib.fa_bwd_ex(_p(qd), _p(kd), _p(vd), _p(o), _p(dod), _p(lse), _p(dq), _p(dk), _p(dv), _p(ws),
                          ws.numel(), B, H, Hkv, Nq, Nk, d, sc, int(w.causal), dt, _stream()) == FA_OK
    code, rec = status(dlib)
    assert code == FA_OK, f"a device-side check fired: record {rec}"
    O_ref, L_ref = oracle.attention_forward(q, k, v, w.scale, w.causal)
    parity.compare_o(w, parity.to_np(o), O_ref)
    parity.compare_l(lse.cpu().numpy().astype(np.float64), L_ref)
    rdq, rdk, rdv, _ = oracle.attention_backward(q, k, v, do, w.scale, w.causal)
    parity.compare_g(parity.to_np(dq), rdq, "dQ")
    parity.compare_g(parity.to_np(dk), rdk, "dK")
    parity.compare_g(parity.to_np(dv), rdv, "dV")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_checked_build_past_two_to_the_31_elements(dlib, d):
    """The checked build on tensors of more than 2^31 elements (the heads past
    h* = 2^31 / (N d) sit beyond any 32-bit element offset): every tensor-map
    coordinate, tensor-memory column and barrier phase check stays silent."""
    N = 1024
    B, H = 2, (1 << 31) // (N * d) // 2 + 8
    torch.cuda.empty_cache()
    g = torch.Generator(device="cuda")
    g.manual_seed(20000 + d)
    q, k, v, do = (torch.randn(B, H, N, d, generator=g, device="cuda", dtype=torch.bfloat16) for _ in range(4))
    assert q.numel() > (1 << 31)
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(dlib.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    sc = ctypes.c_float(float(np.float32(1.0 / np.sqrt(d))))
    assert status(dlib)[0] == FA_OK
    assert dlib.fa_fwd_ex(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, H, N, N, d, sc, 1, 1, _stream()) == FA_OK
    assert dlib.fa_bwd_ex(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv), _p(ws), ws.numel(),
                          B, H, H, N, N, d, sc, 1, 1, _stream()) == FA_OK
    code, rec = status(dlib)
    assert code == FA_OK, f"a device-side check fired: record {rec}"
    del q, k, v, do, o, lse, dq, dk, dv, ws
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kind", range(1, 8))
def test_each_check_reports_a_planted_violation(dlib, kind):
    assert status(dlib)[0] == FA_OK
    assert dlib.fa_selftest_device_check(kind, _stream()) == FA_OK
    code, rec = status(dlib)
    assert code == FA_ERR_DEVICE_CHECK
    bits, first, cta, _value = rec
    assert first == 0x100 | kind and cta == 0
    assert bits & 64 and not bits & (1 << 31)  # the check bit; checks do not abort the grid
    assert status(dlib)[0] == FA_OK  # the status check cleared the record
