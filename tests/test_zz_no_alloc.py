"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

It runs the same kernels as fa_bwd but keeps its scratch (the fp32 row vectors
L log2 e and D that the pre-pass writes and the main kernels read) in the
library's fixed 32 MiB device array instead of a workspace the caller allocates.
Every call shares that array, so these tests call the entry point through the C
ABI several times in a row, with different shapes, masks, types and head
dimensions whose rows overlap in the array; whatever a previous call left there
must not reach the next result.  Each result is checked element by element
against the fp64 oracle with the gradient tolerance of the parity tests, and
against fa_bwd with a caller workspace.  This file is collected last so that a
failure here never hides the other GPU tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_attention_37_gb300 as fa
import oracle
from exact_attention_37_gb300 import _lib, synth
from exact_attention_37_gb300.synth import Workload

from . import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_attention_37_gb300 import build

    build.build()
    fa.load()


def noalloc_grads(w: Workload):
    """(inputs on the CPU, fa_bwd gradients, fa_bwd_noalloc gradients)."""
    cpu = synth.make_inputs(w, with_dout=True)
    q, k, v, do = (x.cuda() for x in cpu)
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
    return cpu, ref, got


def check_against_oracle_and_workspace_path(w: Workload):
    (q, k, v, do), ref, got = noalloc_grads(w)
    rdq, rdk, rdv, _ = oracle.attention_backward(q, k, v, do, w.scale, w.causal)
    for name, r_or, r_ws, g in zip(("dQ", "dK", "dV"), (rdq, rdk, rdv), ref, got):
        parity.compare_g(parity.to_np(g), r_or, f"{w.name} {name} vs oracle")
        err = (g.float() - r_ws.float()).abs().max().item()
        assert err <= parity.G_REL * max(r_ws.float().abs().max().item(), parity.G_FLOOR), f"{name} vs fa_bwd"


# Calls in this order share the scratch: each later one reads rows an earlier one wrote.
SEQUENCE = [
    Workload("noalloc_d128_bf16_c", 1, 4, 1000, 128, "bf16", True, 1.0, (201, 202, 203, 204)),
    Workload("noalloc_d64_fp16_nc", 2, 3, 777, 64, "fp16", False, 1.0, (301, 302, 303, 304)),
    Workload("noalloc_d256_bf16_c", 1, 2, 1000, 256, "bf16", True, 1.0, (311, 312, 313, 314)),
    Workload("noalloc_d256_fp16_nc", 1, 3, 613, 256, "fp16", False, 1.0, (321, 322, 323, 324)),
    Workload("noalloc_d256_bf16_c_again", 1, 2, 1000, 256, "bf16", True, 1.0, (331, 332, 333, 334)),
]


def test_noalloc_matches_oracle_on_consecutive_calls():
    for w in SEQUENCE:
        check_against_oracle_and_workspace_path(w)


def test_noalloc_rejects_sizes_over_its_scratch():
    lib = _lib.load()
    z = ctypes.c_void_p(16)
    # the scratch holds 32 MiB; one head of 4,194,305 rows needs more at every head dimension
    for d in (64, 128, 256):
        code = lib.fa_bwd_noalloc(z, z, z, z, z, z, z, z, z, 1, 1, 4194305, d, ctypes.c_float(0.1), 0, 1, None)
        assert code == 4  # FA_ERR_WORKSPACE
