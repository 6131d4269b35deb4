"""Pins for the fp64 oracle: checks against facts fixed by the pages and by mathematics.

None of these re-types the oracle's own formula.  They use invariants of the
softmax, an independently written blockwise online softmax (page
"FlashAttention — فلاش أتنشن", section "Online softmax": a running maximum and a
running sum of exponentials updated block by block give the exact result),
closed forms, hand-derived examples, torch's float64 softmax and autograd, and
central finite differences.  A final test plants plausible mistakes in the
oracle and checks that each one trips at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def one_head(N=37, d=8, seed=0, scale=1.0):
    return (rnd((1, 1, N, d), seed, scale), rnd((1, 1, N, d), seed + 1, scale),
            rnd((1, 1, N, d), seed + 2, scale))


# ----------------------------------------------------------------------------
# pin functions (return the worst error; used by the tests and the mutation test)
# ----------------------------------------------------------------------------

def pin_rows_sum_to_one(causal):
    q, k, _ = one_head(N=41, d=16, seed=3)
    P, _ = oa.probabilities(oa.scores(q[0, 0], k[0, 0], 0.25, causal))
    return float(np.abs(P.sum(axis=1) - 1.0).max())


def online_softmax_attention(q_h, k_h, v_h, scale, causal, block):
    """Independent blockwise pass over keys with a running max m and running sum l per row."""
    N, d = q_h.shape
    O = np.zeros((N, v_h.shape[1]))
    L = np.zeros(N)
    for i in range(N):
        m, l = -math.inf, 0.0
        acc = np.zeros(v_h.shape[1])
        last = i + 1 if causal else k_h.shape[0]
        for j0 in range(0, last, block):
            j1 = min(last, j0 + block)
            s = scale * (k_h[j0:j1] @ q_h[i])
            m_new = max(m, float(s.max()))
            alpha = math.exp(m - m_new) if m != -math.inf else 0.0
            p = np.exp(s - m_new)
            l = alpha * l + float(p.sum())
            acc = alpha * acc + p @ v_h[j0:j1]
            m = m_new
        O[i] = acc / l
        L[i] = m + math.log(l)
    return O, L


def pin_online_equals_full(causal, block):
    q, k, v = one_head(N=70, d=12, seed=5)
    O, L = oracle.attention_forward(q, k, v, 0.3, causal)
    O2, L2 = online_softmax_attention(q[0, 0], k[0, 0], v[0, 0], 0.3, causal, block)
    return max(float(np.abs(O[0, 0] - O2).max()), float(np.abs(L[0, 0] - L2).max()))


def pin_constant_v(causal):
    q, k, _ = one_head(N=33, d=8, seed=7)
    c = rnd((8,), 9)
    v = np.broadcast_to(c, (1, 1, 33, 8)).copy()
    O, _ = oracle.attention_forward(q, k, v, 0.5, causal)
    return float(np.abs(O - c).max())


def pin_causal_row0():
    q, k, v = one_head(N=19, d=8, seed=11)
    O, L = oracle.attention_forward(q, k, v, 0.7, True)
    e1 = float(np.abs(O[0, 0, 0] - v[0, 0, 0]).max())
    s00 = 0.7 * sum(float(a) * float(b) for a, b in zip(q[0, 0, 0], k[0, 0, 0]))
    return max(e1, abs(float(L[0, 0, 0]) - s00))


def pin_uniform(causal):
    N, d = 29, 6
    q = np.zeros((1, 1, N, d))
    k = rnd((1, 1, N, d), 13)
    v = rnd((1, 1, N, d), 14)
    O, L = oracle.attention_forward(q, k, v, 0.9, causal)
    err = 0.0
    for i in range(N):
        n = i + 1 if causal else N
        err = max(err, float(np.abs(O[0, 0, i] - v[0, 0, :n].mean(axis=0)).max()))
        err = max(err, abs(float(L[0, 0, i]) - math.log(n)))
    return err


def pin_single_token():
    q, k, v = one_head(N=1, d=5, seed=17)
    O, L = oracle.attention_forward(q, k, v, 0.4, False)
    s = 0.4 * sum(float(a) * float(b) for a, b in zip(q[0, 0, 0], k[0, 0, 0]))
    return max(float(np.abs(O - v).max()), abs(float(L[0, 0, 0]) - s))


def load_two_token():
    with open(os.path.join(HERE, "golden", "two_token.json")) as f:
        g = json.load(f)
    inp = g["inputs"]
    arr = lambda x: np.array(x, dtype=np.float64)[None, None]
    return g, arr(inp["q"]), arr(inp["k"]), arr(inp["v"]), arr(inp["dout"]), inp["scale"]


def pin_two_token_forward(causal):
    g, q, k, v, _, s = load_two_token()
    exp = g["expected"]["causal" if causal else "noncausal"]
    O, L = oracle.attention_forward(q, k, v, s, causal)
    return max(float(np.abs(O[0, 0] - np.array(exp["O"])).max()),
               float(np.abs(L[0, 0] - np.array(exp["L"])).max()))


def pin_two_token_backward():
    g, q, k, v, do, s = load_two_token()
    exp = g["expected"]["backward_noncausal"]
    dq, dk, dv, _ = oracle.attention_backward(q, k, v, do, s, False)
    return max(float(np.abs(dq[0, 0] - np.array(exp["dQ"])).max()),
               float(np.abs(dk[0, 0] - np.array(exp["dK"])).max()),
               float(np.abs(dv[0, 0] - np.array(exp["dV"])).max()))


def torch_reference(q, k, v, do, scale, causal):
    """torch float64: explicit masked softmax and autograd (a library route, not the oracle's code)."""
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = torch.matmul(tq, tk.transpose(-1, -2)) * scale
    if causal:
        N = q.shape[-2]
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.matmul(torch.softmax(s, dim=-1), tv)
    lse = torch.logsumexp(s, dim=-1)
    (o * torch.tensor(do)).sum().backward()
    return (o.detach().numpy(), lse.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy())


def pin_torch(causal):
    B, H, N, d = 2, 3, 45, 16
    q, k, v, do = (rnd((B, H, N, d), s) for s in (21, 22, 23, 24))
    O, L = oracle.attention_forward(q, k, v, 0.25, causal)
    dq, dk, dv, _ = oracle.attention_backward(q, k, v, do, 0.25, causal)
    rO, rL, rdq, rdk, rdv = torch_reference(q, k, v, do, 0.25, causal)
    return max(float(np.abs(a - b).max()) for a, b in ((O, rO), (L, rL), (dq, rdq), (dk, rdk), (dv, rdv)))


def pin_finite_differences(causal):
    N, d, s, h = 9, 4, 0.6, 1e-6
    q, k, v, do = (rnd((1, 1, N, d), t) for t in (31, 32, 33, 34))
    grads = oracle.attention_backward(q, k, v, do, s, causal)[:3]
    worst = 0.0
    for which, g in enumerate(grads):
        num = np.zeros_like(g)
        base = [q, k, v]
        for idx in np.ndindex(*g.shape):
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            fp = (oracle.attention_forward(*plus, s, causal)[0] * do).sum()
            fm = (oracle.attention_forward(*minus, s, causal)[0] * do).sum()
            num[idx] = (fp - fm) / (2 * h)
        worst = max(worst, float(np.abs(num - g).max() / np.abs(num).max()))
    return worst


def pin_d_identity(causal):
    q, k, v, do = (rnd((1, 1, 23, 8), t) for t in (41, 42, 43, 44))
    _, _, _, D = oracle.attention_backward(q, k, v, do, 0.5, causal)
    P, _ = oa.probabilities(oa.scores(q[0, 0], k[0, 0], 0.5, causal))
    dP = do[0, 0] @ v[0, 0].T
    return float(np.abs(D[0, 0] - (P * dP).sum(axis=1)).max())


# ----------------------------------------------------------------------------
# the tests
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one(causal):
    assert pin_rows_sum_to_one(causal) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 7, 64])
def test_online_softmax_equals_full(causal, block):
    assert pin_online_equals_full(causal, block) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v(causal):
    assert pin_constant_v(causal) < 1e-14


def test_causal_row0():
    assert pin_causal_row0() < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_attention_closed_form(causal):
    assert pin_uniform(causal) < 1e-14


def test_single_token():
    assert pin_single_token() < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_two_token_hand_example(causal):
    assert pin_two_token_forward(causal) < 1e-14


def test_two_token_hand_backward():
    assert pin_two_token_backward() < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_torch_float64_cross_check(causal):
    assert pin_torch(causal) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_backward_finite_differences(causal):
    assert pin_finite_differences(causal) < 1e-6


@pytest.mark.parametrize("causal", [False, True])
def test_d_identity(causal):
    assert pin_d_identity(causal) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_forward_rows_matches_full(causal):
    q, k, v = one_head(N=50, d=8, seed=51)
    O, L = oracle.attention_forward(q, k, v, 0.3, causal)
    rows = [0, 7, 31, 49]
    Or, Lr = oracle.forward_rows(q[0, 0], k[0, 0], v[0, 0], 0.3, causal, rows)
    assert np.abs(Or - O[0, 0, rows]).max() < 1e-14
    assert np.abs(Lr - L[0, 0, rows]).max() < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_rowwise_backward_matches_full(causal):
    q, k, v, do = (rnd((1, 1, 23, 8), t) for t in (61, 62, 63, 64))
    ref = oracle.attention_backward(q, k, v, do, 0.5, causal)
    got = oracle.head_backward_rowwise(q[0, 0], k[0, 0], v[0, 0], do[0, 0], 0.5, causal, chunk=5)
    for a, b in zip(ref, got):
        assert np.abs(a[0, 0] - b).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_row_subset_backward_parts_sum_to_the_full_gradients(causal):
    # an uneven, out-of-order partition of the rows: dQ and D rows match, dK and dV parts add up
    q, k, v, do = (rnd((1, 1, 19, 6), t) for t in (71, 72, 73, 74))
    dQ, dK, dV, D = oracle.attention_backward(q, k, v, do, 0.7, causal)
    parts = [[18, 3, 11], list(range(0, 3)), [4, 5, 6, 7, 8, 9, 10], [12, 13, 14, 15, 16, 17]]
    sk, sv = np.zeros_like(dK[0, 0]), np.zeros_like(dV[0, 0])
    for rows in parts:
        dq, dk, dv, dr = oracle.head_backward_rows(q[0, 0], k[0, 0], v[0, 0], do[0, 0], 0.7, causal, rows)
        assert np.abs(dq - dQ[0, 0, rows]).max() < 1e-12
        assert np.abs(dr - D[0, 0, rows]).max() < 1e-12
        sk += dk
        sv += dv
    assert np.abs(sk - dK[0, 0]).max() < 1e-12
    assert np.abs(sv - dV[0, 0]).max() < 1e-12


def test_accepts_16bit_tensors_exactly():
    x = torch.randn(1, 1, 4, 8).to(torch.bfloat16)
    assert np.array_equal(oa._f64(x), x.float().numpy().astype(np.float64))


# ----------------------------------------------------------------------------
# planted mistakes: each plausible bug in the oracle must trip at least one pin
# ----------------------------------------------------------------------------

def _all_pins():
    out = []
    for c in (False, True):
        out += [pin_rows_sum_to_one(c) < 1e-14, pin_online_equals_full(c, 7) < 1e-12,
                pin_constant_v(c) < 1e-14, pin_uniform(c) < 1e-14, pin_two_token_forward(c) < 1e-14,
                pin_torch(c) < 1e-12, pin_d_identity(c) < 1e-12]
    out += [pin_causal_row0() < 1e-14, pin_single_token() < 1e-14, pin_two_token_backward() < 1e-14]
    return out


def _mutant_scores_no_scale(q_h, k_h, scale, causal, rows=None):
    return ORIG_SCORES(q_h, k_h, 1.0, causal, rows)


def _mutant_scores_mask_flipped(q_h, k_h, scale, causal, rows=None):
    q_h = oa._f64(q_h)
    k_h = oa._f64(k_h)
    idx = np.arange(q_h.shape[0]) if rows is None else np.asarray(rows)
    S = float(scale) * (q_h[idx] @ k_h.T)
    if causal:
        keys = np.arange(k_h.shape[0])
        S = np.where(keys[None, :] < idx[:, None], -np.inf, S)
    return S


def _mutant_probabilities_wrong_axis(S):
    M = S.max(axis=1, keepdims=True)
    E = np.exp(S - M)
    l = E.sum(axis=0, keepdims=True)
    P = E / l
    return P, (M + np.log(E.sum(axis=1, keepdims=True)))[:, 0]


def _mutant_probabilities_log2(S):
    P, L = ORIG_PROBS(S)
    return P, L / math.log(2.0)


def _mutant_backward_sign(q_h, k_h, v_h, do_h, scale, causal):
    dQ, dK, dV, D = ORIG_HEAD_BWD(q_h, k_h, v_h, do_h, scale, causal)
    return -dQ, dK, dV, D


def _mutant_backward_transposed(q_h, k_h, v_h, do_h, scale, causal):
    dQ, dK, dV, D = ORIG_HEAD_BWD(q_h, k_h, v_h, do_h, scale, causal)
    P, _ = oa.probabilities(oa.scores(q_h, k_h, scale, causal))
    return dQ, dK, P @ do_h, D


ORIG_SCORES = oa.scores
ORIG_PROBS = oa.probabilities
ORIG_HEAD_BWD = oa._head_backward


@pytest.mark.parametrize("target,mutant", [
    ("scores", _mutant_scores_no_scale),
    ("scores", _mutant_scores_mask_flipped),
    ("probabilities", _mutant_probabilities_wrong_axis),
    ("probabilities", _mutant_probabilities_log2),
    ("_head_backward", _mutant_backward_sign),
    ("_head_backward", _mutant_backward_transposed),
])
def test_planted_mistakes_are_caught(monkeypatch, target, mutant):
    assert all(_all_pins()), "pins must hold for the unmodified oracle"
    monkeypatch.setattr(oa, target, mutant)
    with np.errstate(all="ignore"):
        try:
            results = _all_pins()
        except Exception:
            results = [False]
    assert not all(results), f"planted mistake in {target} went unnoticed"


# ----------------------------------------------------------------------------
# grouped-query attention and unequal lengths (bottom-right causal mask)
# ----------------------------------------------------------------------------

def gqa_inputs(B=2, H=6, H_kv=2, Nq=19, Nk=23, d=8, seed=71):
    q = rnd((B, H, Nq, d), seed)
    k = rnd((B, H_kv, Nk, d), seed + 1)
    v = rnd((B, H_kv, Nk, d), seed + 2)
    do = rnd((B, H, Nq, d), seed + 3)
    return q, k, v, do


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H_kv", [1, 2, 3, 6])
def test_gqa_equals_repeated_heads(causal, H_kv):
    """A key/value head shared by a group equals giving every query head its own copy."""
    q, k, v, do = gqa_inputs(H=6, H_kv=H_kv)
    G = 6 // H_kv
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    O, L = oracle.attention_forward(q, k, v, 0.4, causal)
    O2, L2 = oracle.attention_forward(q, kr, vr, 0.4, causal)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
    dq, dk, dv, _ = oracle.attention_backward(q, k, v, do, 0.4, causal)
    dq2, dk2, dv2, _ = oracle.attention_backward(q, kr, vr, do, 0.4, causal)
    assert np.abs(dq - dq2).max() < 1e-13
    assert np.abs(dk - dk2.reshape(2, H_kv, G, 23, 8).sum(axis=2)).max() < 1e-12
    assert np.abs(dv - dv2.reshape(2, H_kv, G, 23, 8).sum(axis=2)).max() < 1e-12


def test_unequal_lengths_causal_rows_match_square_causal():
    """N_q < N_k: row i sees keys 0..i+(N_k-N_q), i.e. row i+shift of a square causal problem."""
    Nq, Nk, d = 7, 20, 8
    q = rnd((1, 1, Nq, d), 81)
    k, v = rnd((1, 1, Nk, d), 82), rnd((1, 1, Nk, d), 83)
    O, L = oracle.attention_forward(q, k, v, 0.5, True)
    qs = np.zeros((1, 1, Nk, d))
    qs[0, 0, Nk - Nq:] = q[0, 0]
    Os, Ls = oracle.attention_forward(qs, k, v, 0.5, True)
    assert np.abs(O[0, 0] - Os[0, 0, Nk - Nq:]).max() < 1e-14
    assert np.abs(L[0, 0] - Ls[0, 0, Nk - Nq:]).max() < 1e-14


def test_more_queries_than_keys_leaves_leading_rows_empty():
    """N_q > N_k: the first N_q-N_k rows see no key (O = 0, L = -inf); the rest are square causal."""
    Nq, Nk, d = 12, 5, 4
    q = rnd((1, 1, Nq, d), 91)
    k, v = rnd((1, 1, Nk, d), 92), rnd((1, 1, Nk, d), 93)
    O, L = oracle.attention_forward(q, k, v, 0.5, True)
    assert np.all(O[0, 0, :Nq - Nk] == 0) and np.all(np.isneginf(L[0, 0, :Nq - Nk]))
    Os, Ls = oracle.attention_forward(q[:, :, Nq - Nk:], k, v, 0.5, True)
    assert np.abs(O[0, 0, Nq - Nk:] - Os[0, 0]).max() < 1e-14
    assert np.abs(L[0, 0, Nq - Nk:] - Ls[0, 0]).max() < 1e-14
    dq, dk, dv, _ = oracle.attention_backward(q, k, v, rnd((1, 1, Nq, d), 94), 0.5, True)
    assert np.all(dq[0, 0, :Nq - Nk] == 0)


def test_single_query_row_sees_every_key_under_the_mask():
    q = rnd((1, 1, 1, 8), 101)
    k, v = rnd((1, 1, 30, 8), 102), rnd((1, 1, 30, 8), 103)
    Oc, Lc = oracle.attention_forward(q, k, v, 0.3, True)
    On, Ln = oracle.attention_forward(q, k, v, 0.3, False)
    assert np.array_equal(Oc, On) and np.array_equal(Lc, Ln)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(9, 14), (14, 9)])
def test_gqa_unequal_lengths_against_torch_autograd(causal, Nq, Nk):
    q, k, v, do = gqa_inputs(B=1, H=4, H_kv=2, Nq=Nq, Nk=Nk, d=6, seed=111)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    kr, vr = tk.repeat_interleave(2, dim=1), tv.repeat_interleave(2, dim=1)
    s = torch.matmul(tq, kr.transpose(-1, -2)) * 0.35
    if causal:
        s = s.masked_fill(torch.ones(Nq, Nk, dtype=torch.bool).triu(Nk - Nq + 1), float("-inf"))
    p = torch.softmax(s, dim=-1).nan_to_num(0.0)  # rows with no visible key: P = 0
    o = torch.matmul(p, vr)
    (o * torch.tensor(do)).sum().backward()
    O, _ = oracle.attention_forward(q, k, v, 0.35, causal)
    dq, dk, dv, _ = oracle.attention_backward(q, k, v, do, 0.35, causal)
    assert np.abs(O - o.detach().numpy()).max() < 1e-12
    for a, b in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert np.abs(a - b.numpy()).max() < 1e-12


def test_gqa_unequal_lengths_finite_differences():
    q, k, v, do = gqa_inputs(B=1, H=2, H_kv=1, Nq=5, Nk=7, d=3, seed=121)
    h = 1e-6
    grads = oracle.attention_backward(q, k, v, do, 0.7, True)[:3]
    for which, g in enumerate(grads):
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            plus = [x.copy() for x in (q, k, v)]
            minus = [x.copy() for x in (q, k, v)]
            plus[which][idx] += h
            minus[which][idx] -= h
            fp = (oracle.attention_forward(*plus, 0.7, True)[0] * do).sum()
            fm = (oracle.attention_forward(*minus, 0.7, True)[0] * do).sum()
            num[idx] = (fp - fm) / (2 * h)
        assert np.abs(num - g).max() / np.abs(num).max() < 1e-6
