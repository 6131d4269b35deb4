"""Calls from several host threads at once, each on its own stream.

The device-buffer entry points keep no host state between calls (tensor maps are
encoded per call), so concurrent calls must give bitwise the results of the same
calls made one after another; the host-buffer entry points serialize themselves.
ctypes releases the interpreter lock around each foreign call, so the C calls do
overlap.
"""
import threading

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
    Workload("thr_d64", 2, 4, 700, 64, "fp16", False, 1.0, (931, 932, 933, 934)),
    Workload("thr_d128_c", 1, 6, 1000, 128, "bf16", True, 1.0, (935, 936, 937, 938)),
    Workload("thr_d256_gqa", 1, 4, 513, 256, "bf16", True, 1.0, (939, 940, 941, 942), True, 2, 600),
]


def step(w, q, k, v, do):
    o, lse = fa.forward(q, k, v, scale=w.scale, causal=w.causal)
    return (o, lse, *fa.backward(q, k, v, o, lse, do, scale=w.scale, causal=w.causal))


def test_concurrent_device_calls_match_sequential_ones():
    inputs = [tuple(x.cuda() for x in make_inputs(w, with_dout=True)) for w in CASES]
    ref = [step(w, *x) for w, x in zip(CASES, inputs)]
    torch.cuda.synchronize()
    results, errors = {}, []

    def worker(t):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for rep in range(3):
                    i = (t + rep) % len(CASES)
                    results[(t, rep)] = (i, step(CASES[i], *inputs[i]))
            s.synchronize()
        except Exception as e:  # reported below, in the test's thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(6)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    fa.fa_check_device_status()
    assert len(results) == 18
    for (t, rep), (i, got) in results.items():
        for name, a, b in zip(("O", "L", "dQ", "dK", "dV"), got, ref[i]):
            assert torch.equal(a, b), f"thread {t} call {rep} ({CASES[i].name}): {name} differs"


def test_concurrent_host_buffer_calls_match_device_calls():
    w = CASES[1]
    q, k, v, do = make_inputs(w, with_dout=True)
    ref = [t.cpu() for t in step(w, q.cuda(), k.cuda(), v.cuda(), do.cuda())]
    B, H, N, d = q.shape
    pin = lambda t: t.contiguous().pin_memory()
    qh, kh, vh, doh = (pin(x) for x in (q, k, v, do))
    outs, errors = [], []

    def worker():
        try:
            oh, dqh, dkh, dvh = (torch.empty_like(x).pin_memory() for x in (q, q, k, v))
            lseh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
            scratch = torch.empty(fa.fa_host_scratch_size(B, H, N, d, True), dtype=torch.uint8, device="cuda")
            s = torch.cuda.Stream()
            fa.fa_fwd_bwd_host(qh, kh, vh, doh, oh, lseh, dqh, dkh, dvh, scratch, w.scale, w.causal, 0, s)
            s.synchronize()
            outs.append((oh, lseh, dqh, dkh, dvh))
        except Exception as e:
            errors.append(repr(e))

    threads = [threading.Thread(target=worker) for _ in range(3)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    fa.fa_check_device_status()
    assert len(outs) == 3
    for got in outs:
        for name, a, b in zip(("O", "L", "dQ", "dK", "dV"), got, ref):
            assert torch.equal(a, b), f"host-buffer call: {name} differs"
