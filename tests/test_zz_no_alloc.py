"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

It runs the same kernels as fa_bwd but keeps its scratch (dQ accumulator and D
rows) in the library's fixed 32 MiB device array instead of a workspace the
caller allocates.  These tests call it through the C ABI twice in a row --
different shapes, masks and types, so a stale accumulator from the first call
would show up in the second -- and check each result against fa_bwd with the
gradient tolerance the parity tests use.  This file is collected last so that a
failure here never hides the other GPU tests.
"""
import ctypes

import pytest
import torch

import exact_attention_37_gb300 as fa
from exact_attention_37_gb300 import _lib, synth
from exact_attention_37_gb300.synth import Workload

pytestmark = pytest.mark.gpu

G_REL = 5e-2  # same bound as the gradient parity tests


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_attention_37_gb300 import build

    build.build()
    fa.load()


def grads_both_ways(w: Workload):
    q, k, v, do = (x.cuda() for x in synth.make_inputs(w, with_dout=True))
    o, lse = fa.forward(q, k, v, scale=w.scale, causal=w.causal)
    ref = fa.backward(q, k, v, o, lse, do, scale=w.scale, causal=w.causal)
    lib = _lib.load()
    got = [torch.empty_like(q) for _ in range(3)]
    B, H, N, d = q.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    code = lib.fa_bwd_noalloc(p(q), p(k), p(v), p(o), p(do), p(lse), p(got[0]), p(got[1]), p(got[2]), B, H, N, d,
                              ctypes.c_float(w.scale), int(w.causal), _lib._dtype_code(q),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, _lib.STATUS.get(code, code)
    fa.fa_check_device_status()
    return ref, got


def check_close(ref, got):
    for name, r, g in zip(("dQ", "dK", "dV"), ref, got):
        r, g = r.float(), g.float()
        err = (g - r).abs().max().item()
        assert err <= G_REL * max(r.abs().max().item(), 1e-3), f"{name}: {err}"


def test_noalloc_matches_workspace_backward_twice_in_a_row():
    first = Workload("noalloc_a", 1, 4, 1000, 128, "bf16", True, 1.0, (201, 202, 203, 204))
    second = Workload("noalloc_b", 2, 3, 777, 64, "fp16", False, 1.0, (301, 302, 303, 304))
    for w in (first, second):
        ref, got = grads_both_ways(w)
        check_close(ref, got)


def test_noalloc_rejects_sizes_over_its_scratch():
    lib = _lib.load()
    z = ctypes.c_void_p(16)
    # d = 256 (fp32 dQ accumulator in the scratch) fits at most 32,513 rows in 32 MiB;
    # one head of 32,514 rows must be refused.
    code = lib.fa_bwd_noalloc(z, z, z, z, z, z, z, z, z, 1, 1, 32514, 256, ctypes.c_float(0.1), 0, 1, None)
    assert code == 4  # FA_ERR_WORKSPACE
