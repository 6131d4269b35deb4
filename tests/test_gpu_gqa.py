"""GPU parity for grouped-query / multi-query attention and unequal query and key
lengths (bottom-right causal mask), forward and backward, against the fp64 oracle.
"""
import pytest

import exact_attention_37_gb300 as fa
from exact_attention_37_gb300.synth import Workload

from . import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_attention_37_gb300 import build

    build.build()
    fa.load()


def w_ex(H, H_kv, N, N_k, d, dtype, causal, B=1, seeds=(401, 402, 403, 404)):
    return Workload(f"ex_H{H}_Hkv{H_kv}_Nq{N}_Nk{N_k}_d{d}_{dtype}_{int(causal)}", B, H, N, d, dtype, causal, 1.0,
                    seeds, True, H_kv, N_k)


@pytest.mark.parametrize("H_kv", [1, 2, 4])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_grouped_query_forward_and_backward(H_kv, causal, d):
    w = w_ex(4, H_kv, 300, 300, d, "bf16", causal, B=2)
    parity.check_forward_full(w)
    parity.check_backward_full(w)


@pytest.mark.parametrize("N,N_k", [(100, 300), (300, 100), (1, 257), (257, 1), (129, 640), (640, 129)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_unequal_lengths_forward_and_backward(N, N_k, causal, d):
    w = w_ex(2, 1, N, N_k, d, "fp16", causal)
    parity.check_forward_full(w)
    parity.check_backward_full(w)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_unequal_head_dim_256(causal):
    w = w_ex(4, 2, 200, 330, 256, "bf16", causal)
    parity.check_forward_full(w)
    parity.check_backward_full(w)
