"""fp64 emulation of the tiled forward algorithm of FlashAttention-2.

TEST INFRASTRUCTURE ONLY (see oracle/attention.py).  This is not the
oracle: it is a CPU restatement of the algorithm the GPU kernels implement,
used by the tests to confirm, without a GPU, that the algorithm equals the
plain definition ("derive correctness of delayed normalize" and "the three
block-skip cases" in the self-check list of "FlashAttention V2 in depth").

The steps follow "FlashAttention V2 in depth", section 6.1 (full forward
algorithm), with the block classification of section 5.3:

* the outer loop walks query blocks Q_i of B_r rows; each is independent;
* a running row max m (starting at -inf), a running row sum l (starting at 0)
  and an unnormalised accumulator O~ (starting at 0) are kept per block;
* the inner loop walks key/value blocks of B_c rows; with the causal mask it
  stops after the block holding the last row of Q_i;
* a key block wholly above the diagonal is skipped, one wholly below is used
  as is, one that crosses it gets the element mask col > row -> -inf;
* per block: m_new = max(m, rowmax S); P = exp(S - m_new);
  l = exp(m - m_new) l + rowsum P; O~ = exp(m - m_new) O~ + P V;
* after the inner loop: O = O~ / l (the single normalisation) and
  L = m + log l.
"""

from __future__ import annotations

import numpy as np


def classify_block(q_first: int, q_last: int, k_first: int, k_last: int) -> str:
    """Causal class of the tile rows [q_first, q_last] x cols [k_first, k_last]
    (section 5.3): 'skip' if every col > every row, 'full' if every col <=
    every row, else 'diagonal'."""
    if q_last < k_first:
        return "skip"
    if q_first >= k_last:
        return "full"
    return "diagonal"


def forward_head(q, k, v, scale, causal, B_r, B_c, counts=None):
    """Tiled forward of one head in fp64.  Returns (O [N, d], L [N]).

    ``counts`` (a dict, optional) receives: q_blocks, kv_steps (inner
    iterations run), skipped (causal blocks never visited), diagonal, full,
    final_divides (rows normalised after the inner loop) and step_rescales
    (rows whose accumulator was multiplied by exp(m - m_new) in a step).
    """
    N, d = q.shape
    O = np.zeros((N, d))
    L = np.zeros(N)
    c = dict(q_blocks=0, kv_steps=0, skipped=0, diagonal=0, full=0,
             final_divides=0, step_rescales=0)
    n_kv_blocks = -(-N // B_c)
    for i in range(0, N, B_r):
        rows = np.arange(i, min(N, i + B_r))
        Qi = q[rows]
        m = np.full(rows.size, -np.inf)
        l = np.zeros(rows.size)
        acc = np.zeros((rows.size, d))
        c["q_blocks"] += 1
        # With the causal mask no key past the block's last row is visible.
        kv_end = min(N, i + B_r) if causal else N
        visited = 0
        for j in range(0, kv_end, B_c):
            cols = np.arange(j, min(N, j + B_c))
            kind = classify_block(rows[0], rows[-1], cols[0], cols[-1]) if causal else "full"
            if kind == "skip":
                c["skipped"] += 1
                continue
            visited += 1
            S = scale * (Qi @ k[cols].T)
            if kind == "diagonal":
                S = np.where(cols[None, :] <= rows[:, None], S, -np.inf)
                c["diagonal"] += 1
            else:
                c["full"] += 1
            m_new = np.maximum(m, np.max(S, axis=1))
            P = np.exp(S - m_new[:, None])
            alpha = np.exp(m - m_new)
            c["step_rescales"] += int(np.count_nonzero(alpha != 1.0)) if visited > 1 else 0
            l = alpha * l + np.sum(P, axis=1)
            acc = alpha[:, None] * acc + P @ v[cols]
            m = m_new
            c["kv_steps"] += 1
        if causal:
            c["skipped"] += n_kv_blocks - -(-kv_end // B_c)
        O[rows] = acc / l[:, None]
        c["final_divides"] += rows.size
        L[rows] = m + np.log(l)
    if counts is not None:
        counts.update(c)
    return O, L
