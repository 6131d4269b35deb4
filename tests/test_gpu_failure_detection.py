"""Failure detection on the GPU without a fault: the self-test kernel waits, through
the library's bounded wait, on an mbarrier that nothing arrives on; the wait gives
up after a short limit, the status check reports FA_ERR_DEVICE_TIMEOUT with the
self-test's record, and the context keeps working afterwards.
"""
import pytest
import torch

import exact_attention_37_gb300 as fa
from exact_attention_37_gb300 import _lib
from exact_attention_37_gb300.synth import Workload, make_inputs

from . import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_attention_37_gb300 import build

    build.build()
    fa.load()


def test_timed_out_wait_is_reported_and_the_context_stays_usable():
    fa.fa_check_device_status()  # start from a clear record
    _lib.fa_selftest_wait_timeout(20000)  # 20 ms
    with pytest.raises(_lib.FaError) as exc:
        fa.fa_check_device_status()
    assert exc.value.code == 6  # FA_ERR_DEVICE_TIMEOUT
    bits, code, cta, _bar = exc.value.detail
    assert code == 32 and cta == 0  # the self-test's code, recorded by CTA 0
    assert bits & 32 and bits & (1 << 31)
    # the record was cleared: a normal call runs to completion and matches the oracle
    fa.fa_check_device_status()
    w = Workload("after_selftest", 1, 2, 200, 128, "bf16", True, 1.0, (601, 602, 603, 604))
    parity.check_forward_full(w)
    fa.fa_check_device_status()

