"""CPU fp64 oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
baseline leg of the benchmark may import this module; the library never
does, and shares no code with it.

It computes the plain definition that FlashAttention-2 reproduces "with no
approximation" (FlashAttention-2 paper abstract): the full score matrix is
materialised, in float64, from the bf16-rounded inputs.

Notation follows "FlashAttention V2 in depth" (infra-guide, section 6.1):
Q, K, V are N x d per head, S = Q K^T * scale, the causal mask lets query
row i see key columns j <= i (section 5.1), O = softmax(S) V and
L = m + log(l) is the row logsumexp kept for the backward pass (sections
6.1 and 7.1).  The backward pass is the derivative of that definition, with
D_i = rowsum(dO_i * O_i) (section 7.3).

Every function takes float64 arrays; the caller upcasts bf16 inputs.
Arrays are [B, H, N, d] (or one head, [N, d]).

Queries and keys may differ in length (Nq query rows, Nk key rows per head;
the pages only treat Nq = Nk).  The causal mask then needs an alignment,
which the pages do not fix: ``offset`` shifts it so that query row i sees key
j iff j <= i + offset.  Top-left alignment is offset 0 (the pages' mask when
Nq = Nk); bottom-right alignment, where the last query row sees every key,
is offset Nk - Nq (``causal_offset``).  A query row that sees no key (only
possible with a negative offset) has no softmax weights: its output row is 0,
its logsumexp is -inf (the log of an empty sum) and its gradients are 0.
"""

from __future__ import annotations

import numpy as np

# Rows of S materialised at once in the forward pass (bounds memory only;
# each output row depends on its own score row alone, so blocking the rows
# changes no arithmetic).
_ROW_ELEMS = 1 << 24


def _scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * Q K^T  (section 6.1, "local attention scores")."""
    return scale * (q @ k.T)


def causal_offset(n_q: int, n_k: int, align: str) -> int:
    """Mask offset of an alignment: "top_left" (query row i sees keys j <= i)
    or "bottom_right" (query row i sees keys j <= i + n_k - n_q)."""
    if align == "top_left":
        return 0
    if align == "bottom_right":
        return n_k - n_q
    raise ValueError(f"unknown causal alignment {align!r}")


def _visible(rows: np.ndarray, n_k: int, offset: int = 0) -> np.ndarray:
    """Causal visibility: query row i may attend to key j iff j <= i + offset
    (section 5.1, where offset = 0: a position sees itself and the ones
    before it)."""
    cols = np.arange(n_k)
    return cols[None, :] <= rows[:, None] + offset


def _masked_scores(q, k, scale, causal, rows, offset=0):
    s = _scores(q, k, scale)
    if causal:
        s = np.where(_visible(rows, k.shape[0], offset), s, -np.inf)
    return s


def _softmax_stats(s: np.ndarray):
    """Row max m, unnormalised weights exp(S - m), row sum l.  A row whose
    scores are all -inf (no visible key) gets m = -inf, weights 0, l = 0."""
    m = np.max(s, axis=1)
    ref = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - ref[:, None])
    l = np.sum(p, axis=1)
    return m, p, l


def _normalise(p: np.ndarray, l: np.ndarray) -> np.ndarray:
    """P / l row by row; a row with l = 0 (no visible key) stays 0."""
    return np.divide(p, l[:, None], out=np.zeros_like(p), where=l[:, None] > 0)


def _lse(m: np.ndarray, l: np.ndarray) -> np.ndarray:
    """L = m + log(l), natural log (section 6.1, last line); -inf for a row
    that sees no key."""
    with np.errstate(divide="ignore"):
        return m + np.log(l)


def probabilities_head(q, k, scale, causal, rows=None, offset=0):
    """P = softmax(S) for one head, rows selected by ``rows`` (all if None)."""
    if rows is None:
        rows = np.arange(q.shape[0])
    rows = np.asarray(rows)
    s = _masked_scores(q[rows], k, scale, causal, rows, offset)
    m, p, l = _softmax_stats(s)
    return _normalise(p, l)


def forward_head(q, k, v, scale, causal, rows=None, offset=0):
    """O and L of one head for the query rows ``rows`` (all rows if None).

    q: [Nq, d], k: [Nk, d], v: [Nk, d], float64.  Returns (O [r, d], L [r]).
    """
    n = q.shape[0]
    if rows is None:
        rows = np.arange(n)
    rows = np.asarray(rows)
    blk = max(1, _ROW_ELEMS // max(1, k.shape[0]))
    o = np.empty((rows.shape[0], v.shape[1]), dtype=np.float64)
    L = np.empty(rows.shape[0], dtype=np.float64)
    for r0 in range(0, rows.shape[0], blk):
        rr = rows[r0:r0 + blk]
        s = _masked_scores(q[rr], k, scale, causal, rr, offset)
        m, p, l = _softmax_stats(s)
        o[r0:r0 + blk] = _normalise(p, l) @ v
        L[r0:r0 + blk] = _lse(m, l)
    return o, L


def forward(q, k, v, scale, causal, offset=0):
    """O [B,H,Nq,d] and L [B,H,Nq] for the whole problem (k, v: [B,H,Nk,d])."""
    B, H, N, d = q.shape
    o = np.empty_like(q)
    L = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], L[b, h] = forward_head(q[b, h], k[b, h], v[b, h], scale, causal, offset=offset)
    return o, L


def forward_rows(q, k, v, scale, causal, rows_per_head, offset=0):
    """O and L on a subset of query rows per head.

    rows_per_head: int array [B, H, r] (or [r], shared by every head).
    Returns O [B, H, r, d] and L [B, H, r].
    """
    B, H, N, d = q.shape
    rows_per_head = np.asarray(rows_per_head)
    if rows_per_head.ndim == 1:
        rows_per_head = np.broadcast_to(rows_per_head, (B, H, rows_per_head.shape[0]))
    r = rows_per_head.shape[-1]
    o = np.empty((B, H, r, d), dtype=np.float64)
    L = np.empty((B, H, r), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], L[b, h] = forward_head(q[b, h], k[b, h], v[b, h], scale, causal,
                                            rows_per_head[b, h], offset)
    return o, L


def _d_vector(do: np.ndarray, o: np.ndarray) -> np.ndarray:
    """D_i = rowsum(dO_i * O_i)  (section 7.3)."""
    return np.sum(do * o, axis=1)


def backward_head(q, k, v, do, scale, causal, offset=0):
    """dQ, dK, dV of one head, the derivative of O = softmax(scale Q K^T) V.

    With P = softmax(S) and dP = dO V^T:
      dV = P^T dO,  dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q,
    where D_i = rowsum(dO_i * O_i) equals rowsum(P_i * dP_i)
    (section 7.3).  O is the oracle's own fp64 output.
    """
    n = q.shape[0]
    rows = np.arange(n)
    s = _masked_scores(q, k, scale, causal, rows, offset)
    m, e, l = _softmax_stats(s)
    p = _normalise(e, l)
    o = p @ v
    dv = p.T @ do
    dp = do @ v.T
    D = _d_vector(do, o)
    ds = p * (dp - D[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


def backward(q, k, v, do, scale, causal, heads=None, offset=0):
    """dQ [B,H,Nq,d], dK, dV [B,H,Nk,d]; ``heads`` restricts to a list of (b, h)."""
    B, H = q.shape[:2]
    dq = np.full_like(q, np.nan)
    dk = np.full_like(k, np.nan)
    dv = np.full_like(v, np.nan)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads:
        dq[b, h], dk[b, h], dv[b, h] = backward_head(q[b, h], k[b, h], v[b, h], do[b, h],
                                                     scale, causal, offset)
    return dq, dk, dv


def backward_dq_rows_head(q, k, v, do, scale, causal, rows, offset=0):
    """dQ on selected query rows of one head (each dQ row needs only its own
    score row, its own O row and D_i)."""
    rows = np.asarray(rows)
    s = _masked_scores(q[rows], k, scale, causal, rows, offset)
    m, e, l = _softmax_stats(s)
    p = _normalise(e, l)
    o = p @ v
    dp = do[rows] @ v.T
    D = _d_vector(do[rows], o)
    ds = p * (dp - D[:, None])
    return scale * (ds @ k)


def backward_dkdv_rows_head(q, k, v, do, scale, causal, key_rows, offset=0):
    """dK and dV on selected key rows of one head.

    dV_j = sum_i P_ij dO_i and dK_j = scale sum_i dS_ij Q_i take column j of P
    and of dS over every query row i.  P_ij = exp(S_ij - L_i) with the row's
    logsumexp L_i (section 7.1), and D_i = rowsum(dO_i * O_i) needs the row's
    output (section 7.3), so the whole forward pass (forward_head) runs first;
    then only the selected columns of S, P, dP and dS are formed.  A row that
    sees no key (L_i = -inf) has no weights.
    """
    key_rows = np.asarray(key_rows)
    n = q.shape[0]
    o, L = forward_head(q, k, v, scale, causal, offset=offset)
    s = scale * (q @ k[key_rows].T)
    if causal:
        s = np.where(_visible(np.arange(n), k.shape[0], offset)[:, key_rows], s, -np.inf)
    seen = np.isfinite(L)
    p = np.zeros_like(s)
    p[seen] = np.exp(s[seen] - L[seen][:, None])
    dp = do @ v[key_rows].T
    D = _d_vector(do, o)
    ds = p * (dp - D[:, None])
    dv = p.T @ do
    dk = scale * (ds.T @ q)
    return dk, dv


def merge_partials(o_parts, L_parts):
    """Merge attention results computed over disjoint key subsets.

    Softmax over a union of key sets, written with each part's normalised
    output O_s and logsumexp L_s: L = log(sum_s exp(L_s)) and
    O = sum_s exp(L_s - L) O_s.  Parts with L_s = -inf (no visible key)
    weigh zero.  o_parts: [S, r, d], L_parts: [S, r].
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    L_parts = np.asarray(L_parts, dtype=np.float64)
    mx = np.max(L_parts, axis=0)
    w = np.exp(L_parts - mx[None, :])
    tot = np.sum(w, axis=0)
    L = mx + np.log(tot)
    o = np.sum((w / tot[None, :])[:, :, None] * o_parts, axis=0)
    return o, L


def forward_head_keys(q, k, v, scale, causal, key_lo, key_hi):
    """O and L of one head when only keys [key_lo, key_hi) exist (causal
    visibility still uses absolute positions).  Rows that see no key get
    O = 0 and L = -inf."""
    n = q.shape[0]
    rows = np.arange(n)
    s = _masked_scores(q, k, scale, causal, rows)
    cols = np.arange(k.shape[0])
    inside = (cols >= key_lo) & (cols < key_hi)
    s = np.where(inside[None, :], s, -np.inf)
    o = np.zeros((n, v.shape[1]))
    L = np.full(n, -np.inf)
    ok = np.isfinite(np.max(s, axis=1))
    if np.any(ok):
        m, e, l = _softmax_stats(s[ok])
        o[ok] = (e @ v) / l[:, None]
        L[ok] = _lse(m, l)
    return o, L


# ------------------------------------------------- grouped-query attention
# Grouped-query attention is listed on the pages as not evaluated; it is the
# same computation per query head with K and V shared: the H query heads of
# a batch read Hkv key/value heads, query head h reading key/value head
# h // (H // Hkv).  The oracle writes that definition out by repeating each
# key/value head over its group and reusing the functions above; dK and dV of
# a shared head are the sums over the query heads that read it (the
# derivative of a sum of per-query-head terms).

def expand_kv(x, H):
    """[B, Hkv, N, d] -> [B, H, N, d]: head h of the result is head
    h // (H // Hkv) of x."""
    Hkv = x.shape[1]
    assert H % Hkv == 0
    return np.repeat(x, H // Hkv, axis=1)


def reduce_kv(g, Hkv):
    """[B, H, N, d] gradient w.r.t. the expanded K or V -> [B, Hkv, N, d],
    summed over each group of H // Hkv query heads."""
    B, H, N, d = g.shape
    assert H % Hkv == 0
    return g.reshape(B, Hkv, H // Hkv, N, d).sum(axis=2)


def forward_gqa(q, k, v, scale, causal, offset=0):
    """O [B,H,Nq,d] and L [B,H,Nq] with k, v of Hkv heads."""
    H = q.shape[1]
    return forward(q, expand_kv(k, H), expand_kv(v, H), scale, causal, offset)


def backward_gqa(q, k, v, do, scale, causal, offset=0):
    """dQ [B,H,Nq,d] and dK, dV [B,Hkv,Nk,d] with k, v of Hkv heads."""
    H, Hkv = q.shape[1], k.shape[1]
    dq, dk, dv = backward(q, expand_kv(k, H), expand_kv(v, H), do, scale, causal, offset=offset)
    return dq, reduce_kv(dk, Hkv), reduce_kv(dv, Hkv)
