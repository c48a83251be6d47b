"""FP64 reference attention, forward and backward -- TEST INFRASTRUCTURE ONLY.

This module is the oracle that the CUDA library is checked against.  It is
plain, slow and written to be read against the pages it follows; it shares
no code with the CUDA path and must never be imported by the product path
(only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg call it).

Sources (page title, section):
  * "FlashAttention 训练时为什么会梯度爆炸？一次拆透反向传播的坑" (cnnetsun.cn),
    §3.1 Attention(Q,K,V) = softmax(QK^T/sqrt(d_k)) V and §3.2 the safe
    softmax e^{x_i - max} / sum_j e^{x_j - max}; §2 the backward recomputes
    the forward from Q, K, V.
  * ijyty.com/news/896914 (BF16 FlashAttention stability), §2.1 the online
    softmax and final O = diag(l)^-1 O; §3.1 delta = rowsum(dO o O);
    §4.1 the stabilised shift rule (repeated row maximum -> m = beta*rm for
    a positive maximum, m = 0 for a negative maximum), beta in [1.1, 1.5].
  * "為什么BF16的FlashAttention會把訓練「炸掉」？" (web578.cn), "mechanism 2":
    detect whether the row maximum of S occurs more than once and move the
    shift so that the exponent at the maximum is strictly below 1.

Readings where the pages are garbled or silent:
  * Shift rule (the comparison operators are stripped in §4.1): with
    rm = max_j S_raw[i, j] over visible j and rs = #{j : S_raw[i, j] == rm},
    m = beta*rm if rm > 0 and rs > 1; m = 0 if rm < 0 and rs > 1; else m = rm.
    A row with rm == 0 and rs > 1 matches neither branch and keeps m = 0.
  * Ties are decided on the raw (unscaled) dot products S_raw = Q K^T.
  * The gradient formulas are not printed on the pages; the backward is the
    calculus of the forward with loss L = sum(dO o O):
        P = exp(scale*S_raw - LSE), dV = P^T dO, dP = dO V^T,
        delta = rowsum(dO o O), dS = P o (dP - delta),
        dQ = scale * dS K, dK = scale * dS^T Q.
  * Causal masking is top-left aligned: query i sees keys j <= i.
  * LSE is the natural-log logsumexp of the scaled logits.

Parity status: pinned by closed forms and invariants in
``tests/test_oracle_pins.py`` (row sums, k tied maxima -> 1/k, uniform and
single-key cases, shift invariance, translation invariance, finite
differences of the gradients, the delta identity, sum_j dK_j = 0).
"""
from __future__ import annotations

import numpy as np

BRANCH_RM = 0      # m = rm
BRANCH_BETA = 1    # m = beta * rm   (repeated positive maximum)
BRANCH_ZERO = 2    # m = 0           (repeated negative maximum)


def _f64(x) -> np.ndarray:
    """Widen a tensor/array (bf16 torch tensors included) to a float64 numpy array."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float64)


def visible(rows: np.ndarray, n_keys: int, causal: bool) -> np.ndarray:
    """Boolean [len(rows), n_keys]: which keys each query row may attend to."""
    cols = np.arange(n_keys)
    if causal:
        return cols[None, :] <= rows[:, None]
    return np.ones((len(rows), n_keys), dtype=bool)


def shift_rule(rm, rs, beta: float, stable: int):
    """Stabilised shift (ijyty.com/news/896914 §4.1), applied to a whole row.

    Returns (m, branch).  In plain mode (stable == 0) m = rm and branch = 0.
    """
    rm = np.asarray(rm, dtype=np.float64)
    rs = np.asarray(rs)
    if not stable:
        return rm.copy(), np.zeros(rm.shape, dtype=np.int8)
    repeated = rs > 1
    pos = repeated & (rm > 0)
    neg = repeated & (rm < 0)
    m = np.where(pos, beta * rm, np.where(neg, 0.0, rm))
    branch = np.where(pos, BRANCH_BETA, np.where(neg, BRANCH_ZERO, BRANCH_RM)).astype(np.int8)
    return m, branch


def row_max_and_ties(s_raw: np.ndarray, vis: np.ndarray):
    """rm = max over visible entries, rs = how many visible entries equal rm."""
    masked = np.where(vis, s_raw, -np.inf)
    rm = masked.max(axis=1)
    rs = ((masked == rm[:, None]) & vis).sum(axis=1)
    return rm, rs


def forward(q, k, v, scale: float, causal: bool, stable: int = 0, beta: float = 1.25,
            row_block: int = 512):
    """One-shot softmax attention in FP64.

    q, k, v: [B, H, N, d].  Returns a dict with
      o   [B, H, N, d]  softmax(scale * q k^T) v
      lse [B, H, N]     logsumexp_j(scale * S_raw[i, j]) over visible j
      rm  [B, H, N]     raw row maximum;  rs: how often it occurs
      rmin [B, H, N]    raw row minimum over visible keys (the monitor's softmax-input min)
      branch [B, H, N]  which shift the stabilised rule picks (0, 1, 2)
      m   [B, H, N]     the shift used (raw units)
    The outputs are computed with the shift the rule picks; o and lse do not
    depend on it (a softmax is invariant to a constant shift of its row).
    Rows are processed in blocks of ``row_block`` only to bound memory; each
    row is still the plain one-shot definition.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    out = {
        "o": np.zeros((B, H, N, v.shape[-1])),
        "lse": np.zeros((B, H, N)),
        "rm": np.zeros((B, H, N)),
        "rmin": np.zeros((B, H, N)),
        "rs": np.zeros((B, H, N), dtype=np.int64),
        "branch": np.zeros((B, H, N), dtype=np.int8),
        "m": np.zeros((B, H, N)),
    }
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, row_block):
                rows = np.arange(r0, min(N, r0 + row_block))
                s_raw = q[b, h, rows] @ k[b, h].T
                vis = visible(rows, N, causal)
                rm, rs = row_max_and_ties(s_raw, vis)
                m, br = shift_rule(rm, rs, beta, stable)
                shift = scale * m
                e = np.where(vis, np.exp(scale * s_raw - shift[:, None]), 0.0)
                l = e.sum(axis=1)
                out["o"][b, h, rows] = (e / l[:, None]) @ v[b, h]
                out["lse"][b, h, rows] = shift + np.log(l)
                out["rm"][b, h, rows] = rm
                out["rmin"][b, h, rows] = np.where(vis, s_raw, np.inf).min(axis=1)
                out["rs"][b, h, rows] = rs
                out["branch"][b, h, rows] = br
                out["m"][b, h, rows] = m
    return out


def probabilities(q, k, scale: float, causal: bool, b: int = 0, h: int = 0):
    """The normalised attention matrix P of one head (for the row-sum pin)."""
    q, k = _f64(q), _f64(k)
    N = q.shape[2]
    rows = np.arange(N)
    s_raw = q[b, h] @ k[b, h].T
    vis = visible(rows, N, causal)
    rm, _ = row_max_and_ties(s_raw, vis)
    e = np.where(vis, np.exp(scale * (s_raw - rm[:, None])), 0.0)
    return e / e.sum(axis=1, keepdims=True)


def backward(q, k, v, o, lse, do, scale: float, causal: bool, row_block: int = 512):
    """FP64 gradients of L = sum(dO o O) by recomputing P from Q, K and LSE.

    Returns dict(dq, dk, dv, delta) with delta = rowsum(dO o O)
    (ijyty.com/news/896914 §3.1).
    """
    q, k, v, o, lse, do = _f64(q), _f64(k), _f64(v), _f64(o), _f64(lse), _f64(do)
    B, H, N, d = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    delta = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, row_block):
                rows = np.arange(r0, min(N, r0 + row_block))
                s_raw = q[b, h, rows] @ k[b, h].T
                vis = visible(rows, N, causal)
                p = np.where(vis, np.exp(scale * s_raw - lse[b, h, rows][:, None]), 0.0)
                dov = do[b, h, rows]
                dv[b, h] += p.T @ dov
                dp = dov @ v[b, h].T
                dl = (dov * o[b, h, rows]).sum(axis=1)
                ds = p * (dp - dl[:, None])
                dq[b, h, rows] = scale * (ds @ k[b, h])
                dk[b, h] += scale * (ds.T @ q[b, h, rows])
                delta[b, h, rows] = dl
    return {"dq": dq, "dk": dk, "dv": dv, "delta": delta}


def fp32_dot_error_bound(q_row: np.ndarray, k_rows: np.ndarray) -> np.ndarray:
    """gamma_d * sum_c |q_c k_c|: the classic bound on an FP32 dot product's error.

    gamma_d = d u / (1 - d u) with u = 2^-24 (Higham, "Accuracy and Stability of
    Numerical Algorithms", Thm 3.1), for each key row against one query row.
    """
    d = q_row.shape[-1]
    u = 2.0 ** -24
    gamma = d * u / (1.0 - d * u)
    return gamma * (np.abs(k_rows) @ np.abs(q_row))


def _fp32_exact(q_row: np.ndarray, k_row: np.ndarray) -> bool:
    """True when every FP32 summation order of q.k gives the exact value.

    bf16 x bf16 products are exact in FP32 (<= 16 significant bits).  If all
    products are multiples of a common quantum g and sum_c |p_c| < 2^24 g,
    every partial sum is an exactly representable multiple of g.
    """
    p = q_row * k_row
    nz = p[p != 0]
    if nz.size == 0:
        return True
    _, e = np.frexp(nz)
    g = np.ldexp(1.0, int(e.min()) - 16)
    return float(np.abs(nz).sum()) < g * 2.0 ** 24


def decidable_rows(q, k, causal: bool, b: int = 0, h: int = 0, safety: float = 2.0, row_block: int = 256):
    """Which rows' (rm, rs, branch) an FP32 computation must reproduce exactly.

    A row is decidable when (a) the gap between its maximum and the next
    distinct visible value exceeds ``safety`` x the sum of the two entries'
    FP32 error bounds, and (b) every tied maximum comes from a bit-identical
    key row or is exact in FP32 whatever the summation order.  Returns
    (decidable [N] bool, bound [N] error bound of the maximum entry).
    Rows are taken ``row_block`` at a time only to bound memory and time; each
    row's decision uses that row alone.
    """
    q, k = _f64(q), _f64(k)
    N, d = q.shape[2], q.shape[3]
    qb, kb = q[b, h], k[b, h]
    u = 2.0 ** -24
    gamma = d * u / (1.0 - d * u)
    dec = np.zeros(N, dtype=bool)
    bound = np.zeros(N)
    abs_k = np.abs(kb)
    for r0 in range(0, N, row_block):
        rows = np.arange(r0, min(N, r0 + row_block))
        vis = visible(rows, N, causal)
        s = np.where(vis, qb[rows] @ kb.T, -np.inf)
        err = gamma * (np.abs(qb[rows]) @ abs_k.T)           # fp32_dot_error_bound per entry
        rm = s.max(axis=1)
        at_max = vis & (s == rm[:, None])
        bound[rows] = np.where(at_max, err, -np.inf).max(axis=1)
        below = vis & (s < rm[:, None])
        nxt = np.where(below, s, -np.inf).max(axis=1)
        has_below = below.any(axis=1)
        e_next = np.where(below & (s == nxt[:, None]), err, -np.inf).max(axis=1)
        ok = ~has_below | ((rm - nxt) > safety * (bound[rows] + e_next))
        for t in np.nonzero(ok & (at_max.sum(axis=1) > 1))[0]:
            i = rows[t]
            js = np.nonzero(at_max[t])[0]
            ref = kb[js[0]]
            for j in js[1:]:
                if not np.array_equal(kb[j], ref) and not (_fp32_exact(qb[i], kb[j]) and _fp32_exact(qb[i], ref)):
                    ok[t] = False
                    break
        dec[rows] = ok
    return dec, bound
