"""Plain fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` call it.  It shares no code, header, table or helper with the CUDA
kernels; it receives the same rounded 16-bit inputs (as float64) and computes
the textbook definition, materialising the full score matrix S and the
probability matrix P of every head it evaluates.

What it follows
---------------
* Forward, ``O = softmax(Q K^T * scale + mask) V``: the attention formula of the
  page "FlashAttention — فلاش أتنشن", section "The problem of standard
  attention" (the only formula the pages print), with 1/sqrt(d_k) passed in as
  ``scale``.  The mask is the causal one ("masking" is one of the fused steps,
  same page, section "Fusion of the operations into one CUDA kernel"):
  key j is visible to query i iff j <= i, and hidden scores are -inf.
* Logsumexp ``L_i = ln sum_j exp(S_ij)`` of the scaled, masked scores, natural
  log.  The pages keep a running maximum and a running sum of exponentials per
  row (same page, section "Online softmax"); L is the pair folded into one
  number, so the backward pass can rebuild P as exp(S - L).
* Backward with upstream gradient dO: the derivatives of the same formula,
  dV = P^T dO, dP = dO V^T, D_i = sum_c dO_ic O_ic, dS = P o (dP - D),
  dQ = scale dS K, dK = scale dS^T Q.  The pages state only that the method
  speeds up training (page "FlashAttention-2 — فلاش أتنشن-2", section
  "Performance and efficiency"), so a gradient exists; these are the standard
  chain-rule derivatives of softmax, written out.

Extensions (the "next" rows of the build, readings of the pages' MQA support --
page "FlashAttention — فلاش أتنشن", section "FlashAttention-2" -- and of the
causal mask for unequal lengths):
* Grouped / multi-query attention: K and V carry H_kv heads, H_kv divides H, and
  query head h attends to key/value head h // (H / H_kv).  H_kv = 1 is multi-query
  attention, H_kv = H plain multi-head attention.
* Unequal lengths: Q has N_q rows, K and V have N_k rows.  Under the causal mask
  key j is visible to query i iff j <= i + (N_k - N_q) (the last query row sees
  every key).  A row that sees no key has O = 0 and L = -inf.

Pins (tests/test_oracle.py): rows of P sum to 1; a blockwise online softmax
written independently in the tests equals this two-pass softmax; constant V
rows reproduce the constant; causal row 0 attends to key 0 only; Q = 0 gives
uniform attention with L = ln(#visible keys); N = 1; hand-derived two-token
examples; torch float64 softmax + autograd as a library cross-check; central
finite differences for the backward pass; and the identity
sum_c dO o O = sum_j P o dP.  Every function below is pinned by at least one.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "scores",
    "probabilities",
    "attention_forward",
    "attention_backward",
    "forward_rows",
    "head_backward_rows",
    "head_backward_rowwise",
]


def _f64(x) -> np.ndarray:
    """Exact widening of the stored values (fp16/bf16/fp32 tensors or arrays) to float64."""
    if hasattr(x, "detach"):  # a torch tensor: widen through float32, which is exact for 16-bit types
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float64)


def scores(q_h, k_h, scale: float, causal: bool, rows=None) -> np.ndarray:
    """S = scale * q k^T for one head, with -inf where the causal mask hides key j from query i.

    ``rows`` selects query rows (their absolute indices decide the mask).  With N_q
    query rows and N_k keys the mask is aligned at the bottom right: key j is
    visible to query i iff j <= i + N_k - N_q.
    """
    q_h = _f64(q_h)
    k_h = _f64(k_h)
    idx = np.arange(q_h.shape[0]) if rows is None else np.asarray(rows)
    S = float(scale) * (q_h[idx] @ k_h.T)
    if causal:
        shift = k_h.shape[0] - q_h.shape[0]
        keys = np.arange(k_h.shape[0])
        S = np.where(keys[None, :] > idx[:, None] + shift, -np.inf, S)
    return S


def probabilities(S: np.ndarray):
    """Row softmax of S by the two-pass textbook form; returns (P, L) with L the natural logsumexp.

    A row whose scores are all -inf (no visible key) gets P = 0 and L = -inf.
    """
    M = S.max(axis=1, keepdims=True)
    empty = ~np.isfinite(M)
    Msafe = np.where(empty, 0.0, M)
    E = np.exp(S - Msafe)
    l = E.sum(axis=1, keepdims=True)
    P = np.where(empty, 0.0, E / np.where(empty, 1.0, l))
    with np.errstate(divide="ignore"):
        L = np.where(empty, -np.inf, Msafe + np.log(l))[:, 0]
    return P, L


def kv_head(h: int, H: int, H_kv: int) -> int:
    """Key/value head that query head h reads under grouped-query attention."""
    return h // (H // H_kv)


def attention_forward(q, k, v, scale: float, causal: bool):
    """O [B,H,N_q,d] and L [B,H,N_q] in float64, one head at a time, S and P materialised.

    k and v are [B,H_kv,N_k,d]; H_kv divides H (grouped-query attention).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    O = np.empty((B, H, N, v.shape[3]))
    L = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            g = kv_head(h, H, H_kv)
            P, Lh = probabilities(scores(q[b, h], k[b, g], scale, causal))
            O[b, h] = P @ v[b, g]
            L[b, h] = Lh
    return O, L


def _head_backward(q_h, k_h, v_h, do_h, scale, causal):
    P, _ = probabilities(scores(q_h, k_h, scale, causal))
    O = P @ v_h
    dV = P.T @ do_h
    dP = do_h @ v_h.T
    D = (do_h * O).sum(axis=1)
    dS = P * (dP - D[:, None])
    dQ = scale * (dS @ k_h)
    dK = scale * (dS.T @ q_h)
    return dQ, dK, dV, D


def attention_backward(q, k, v, dout, scale: float, causal: bool):
    """dQ [B,H,N_q,d], dK and dV [B,H_kv,N_k,d], D [B,H,N_q] in float64 for the loss sum(O o dout).

    Under grouped-query attention a key/value head's gradient is the sum of the
    gradients it receives from every query head of its group.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    dQ = np.empty_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    D = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            g = kv_head(h, H, H_kv)
            dq, dk, dv, D[b, h] = _head_backward(q[b, h], k[b, g], v[b, g], dout[b, h], float(scale), causal)
            dQ[b, h] = dq
            dK[b, g] += dk
            dV[b, g] += dv
    return dQ, dK, dV, D


def forward_rows(q_h, k_h, v_h, scale: float, causal: bool, rows):
    """O and L of selected query rows of one head: the definition applied row by row.

    Each row's softmax depends on that row's scores only, so evaluating a subset
    of rows is the same computation as the full forward pass restricted to them.
    """
    v_h = _f64(v_h)
    P, L = probabilities(scores(q_h, k_h, scale, causal, rows=rows))
    return P @ v_h, L


def head_backward_rows(q_h, k_h, v_h, do_h, scale: float, causal: bool, rows):
    """One head's backward pass restricted to the query rows ``rows``.

    Returns (dQ[rows], dK part, dV part, D[rows]): the rows' own dQ and D, and
    their contributions to dK and dV (the full dK, dV are the sums of these parts
    over any partition of the rows).  Every quantity comes from the definition
    for those rows alone: P, then O = P V, dP = dO V^T, D, dS = P o (dP - D).
    """
    q_h, k_h, v_h, do_h = _f64(q_h), _f64(k_h), _f64(v_h), _f64(do_h)
    rows = np.asarray(rows)
    P, _ = probabilities(scores(q_h, k_h, scale, causal, rows=rows))
    O = P @ v_h
    dP = do_h[rows] @ v_h.T
    Dr = (do_h[rows] * O).sum(axis=1)
    dS = P * (dP - Dr[:, None])
    return scale * (dS @ k_h), scale * (dS.T @ q_h[rows]), P.T @ do_h[rows], Dr


def head_backward_rowwise(q_h, k_h, v_h, do_h, scale: float, causal: bool, chunk: int = 1024):
    """dQ, dK, dV, D of one head, evaluating the definition over chunks of query rows.

    For long sequences the N x N matrices of one head do not fit comfortably in
    host memory, so rows are taken ``chunk`` at a time (``head_backward_rows``):
    dQ rows are written directly and the dK, dV sums over rows are accumulated
    chunk after chunk.
    """
    q_h, k_h, v_h, do_h = _f64(q_h), _f64(k_h), _f64(v_h), _f64(do_h)
    N, d = q_h.shape
    dQ = np.empty_like(q_h)
    dK = np.zeros_like(k_h)
    dV = np.zeros_like(v_h)
    D = np.empty(N)
    for r0 in range(0, N, chunk):
        rows = np.arange(r0, min(N, r0 + chunk))
        dQ[rows], dk, dv, D[rows] = head_backward_rows(q_h, k_h, v_h, do_h, scale, causal, rows)
        dK += dk
        dV += dv
    return dQ, dK, dV, D
