"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI and
compare it with the fp64 oracle on the same rounded inputs.

Tolerances (written here, used by every GPU test):
  O  : max|g - r| <= 2e-2 (bf16) / 5e-3 (fp16), and max|g - r| / max|r| <= 2e-2
  L  : max|g - r| <= 1e-3
  dQ, dK, dV : max|g - r| / max(max|r|, 1e-3) <= 5e-2
The 1e-3 floor only matters when the reference gradient is (near) zero, e.g. N = 1
where dS = P (dP - D) vanishes identically and what remains is the rounding of O
to 16 bits inside D; it caps the absolute error there at 5e-5.
"""
from __future__ import annotations

import numpy as np
import torch

import exact_attention_37_gb300 as fa
import oracle
from exact_attention_37_gb300.synth import Workload, make_inputs

O_ABS = {"bf16": 2e-2, "fp16": 5e-3}
O_REL = 2e-2
L_ABS = 1e-3
G_REL = 5e-2


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_forward(w: Workload, q, k, v):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.forward(qd, kd, vd, scale=w.scale, causal=w.causal)
    fa.fa_check_device_status()
    return o, lse


def compare_o(w, got, ref, what="O"):
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    mref = float(np.abs(ref).max()) if ref.size else 1.0
    assert err <= O_ABS[w.dtype], f"{what}: max abs err {err:.3e} > {O_ABS[w.dtype]}"
    assert err <= O_REL * mref, f"{what}: max err {err:.3e} > {O_REL} * max|ref| {mref:.3e}"
    return err


def compare_l(got, ref):
    # rows that see no key have L = -inf on both sides
    inf = np.isinf(ref)
    assert np.array_equal(np.isinf(got), inf) and np.all(got[inf] == ref[inf]), "L: infinite rows differ"
    got, ref = got[~inf], ref[~inf]
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    assert err <= L_ABS, f"L: max abs err {err:.3e} > {L_ABS}"
    return err


G_FLOOR = 1e-3


def compare_g(got, ref, what):
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    mref = max(float(np.abs(ref).max()) if ref.size else 1.0, G_FLOOR)
    assert err <= G_REL * mref, f"{what}: max err {err:.3e} > {G_REL} * max|ref| {mref:.3e}"
    return err / max(mref, 1e-30)


def check_forward_full(w: Workload):
    """Every output element of every head against the oracle."""
    q, k, v, _ = make_inputs(w, with_dout=False)
    o, lse = run_forward(w, q, k, v)
    O_ref, L_ref = oracle.attention_forward(q, k, v, w.scale, w.causal)
    compare_o(w, to_np(o), O_ref)
    compare_l(lse.cpu().numpy().astype(np.float64), L_ref)


def check_forward_sampled(w: Workload, heads, rows):
    """Selected rows of selected heads (the oracle evaluates those rows over all keys)."""
    q, k, v, _ = make_inputs(w, with_dout=False)
    o, lse = run_forward(w, q, k, v)
    o_np = o.float().cpu()
    l_np = lse.cpu()
    for b, h in heads:
        O_ref, L_ref = oracle.forward_rows(q[b, h], k[b, h], v[b, h], w.scale, w.causal, rows)
        compare_o(w, o_np[b, h, rows].numpy().astype(np.float64), O_ref, f"O[{b},{h}]")
        compare_l(l_np[b, h, rows].numpy().astype(np.float64), L_ref)


def run_backward(w: Workload, q, k, v, do):
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.forward(qd, kd, vd, scale=w.scale, causal=w.causal)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, scale=w.scale, causal=w.causal)
    fa.fa_check_device_status()
    return o, lse, dq, dk, dv


def check_backward_full(w: Workload):
    q, k, v, do = make_inputs(w, with_dout=True)
    _, _, dq, dk, dv = run_backward(w, q, k, v, do)
    rdq, rdk, rdv, _ = oracle.attention_backward(q, k, v, do, w.scale, w.causal)
    compare_g(to_np(dq), rdq, "dQ")
    compare_g(to_np(dk), rdk, "dK")
    compare_g(to_np(dv), rdv, "dV")


def check_backward_sampled(w: Workload, heads):
    """All rows of selected heads; the oracle walks each head in row chunks."""
    q, k, v, do = make_inputs(w, with_dout=True)
    _, _, dq, dk, dv = run_backward(w, q, k, v, do)
    dq, dk, dv = dq.float().cpu(), dk.float().cpu(), dv.float().cpu()
    for b, h in heads:
        rdq, rdk, rdv, _ = oracle.head_backward_rowwise(q[b, h], k[b, h], v[b, h], do[b, h], w.scale, w.causal)
        compare_g(dq[b, h].numpy().astype(np.float64), rdq, f"dQ[{b},{h}]")
        compare_g(dk[b, h].numpy().astype(np.float64), rdk, f"dK[{b},{h}]")
        compare_g(dv[b, h].numpy().astype(np.float64), rdv, f"dV[{b},{h}]")
