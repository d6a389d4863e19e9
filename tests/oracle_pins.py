"""Checks that pin the fp64 oracle to facts other than itself.

Each ``pin_*`` function raises AssertionError when the oracle module given
to it disagrees with a closed form, an invariant, brute force on tiny inputs
or a finite-difference derivative.  ``tests/test_oracle.py`` runs them on the
oracle as it stands; ``tests/test_oracle_mutants.py`` runs them on copies of
the oracle with a planted mistake and requires that at least one fails.
"""

from __future__ import annotations

import math

import numpy as np

from exact_attention_92_gb300 import inputs


def _rng_f64(seed, shape, std=1.0):
    return inputs.bits_to_f64(inputs.normal_bits(np.random.default_rng(seed), shape, std))


# --------------------------------------------------------------------------
# Brute force: scalar loops, math.exp / math.log / math.fsum, written as
# O_i = sum_j exp(S_ij - L_i) V_j with L_i = log sum_j exp(S_ij) and no max
# subtraction (tiny inputs keep exp in range).  No NumPy arithmetic.
# --------------------------------------------------------------------------

def brute_force_head(q, k, v, scale, causal):
    N, d = len(q), len(q[0])
    O, L = [], []
    for i in range(N):
        js = [j for j in range(N) if (not causal) or j <= i]
        s = {j: scale * math.fsum(float(q[i][c]) * float(k[j][c]) for c in range(d)) for j in js}
        Li = math.log(math.fsum(math.exp(s[j]) for j in js))
        O.append([math.fsum(math.exp(s[j] - Li) * float(v[j][c]) for j in js) for c in range(d)])
        L.append(Li)
    return np.array(O), np.array(L)


def pin_brute_force(att):
    for N in (1, 2, 3, 5, 8):
        for d in (1, 2, 4):
            for causal in (False, True):
                seed = 17 * N + d + (100 if causal else 0)
                q = _rng_f64(seed, (N, d))
                k = _rng_f64(seed + 1, (N, d))
                v = _rng_f64(seed + 2, (N, d))
                scale = 1.0 / math.sqrt(d)
                O, L = att.forward_head(q, k, v, scale, causal)
                Ob, Lb = brute_force_head(q.tolist(), k.tolist(), v.tolist(), scale, causal)
                assert np.allclose(O, Ob, rtol=0, atol=1e-12), (N, d, causal)
                assert np.allclose(L, Lb, rtol=0, atol=1e-12), (N, d, causal)


# --------------------------------------------------------------------------
# Invariants and closed forms
# --------------------------------------------------------------------------

def pin_rows_sum_to_one(att):
    for causal in (False, True):
        q = _rng_f64(3, (37, 16), 2.0)
        k = _rng_f64(4, (37, 16), 2.0)
        P = att.probabilities_head(q, k, 0.25, causal)
        assert np.all(P >= 0)
        assert np.max(np.abs(P.sum(axis=1) - 1.0)) < 1e-12
        if causal:
            assert np.all(P[np.triu_indices(37, 1)] == 0.0)


def pin_identical_keys(att):
    """All keys equal k: every visible key has the same score, so O_i is the
    mean of the visible V rows and L_i = scale q_i.k + ln(n_visible)."""
    N, d = 23, 8
    q = _rng_f64(5, (N, d))
    k = np.broadcast_to(_rng_f64(6, (1, d)), (N, d)).copy()
    v = _rng_f64(7, (N, d))
    scale = 0.3
    for causal in (False, True):
        O, L = att.forward_head(q, k, v, scale, causal)
        for i in range(N):
            n_vis = i + 1 if causal else N
            assert np.allclose(O[i], v[:n_vis].mean(axis=0), rtol=0, atol=1e-12)
            assert abs(L[i] - (scale * float(q[i] @ k[0]) + math.log(n_vis))) < 1e-12


def pin_causal_first_row(att):
    """Causal row 0 sees only key 0: O_0 = V_0 and L_0 = scale q_0.k_0."""
    q = _rng_f64(8, (19, 4))
    k = _rng_f64(9, (19, 4))
    v = _rng_f64(10, (19, 4))
    O, L = att.forward_head(q, k, v, 0.5, True)
    assert np.array_equal(O[0], v[0])
    assert abs(L[0] - 0.5 * float(q[0] @ k[0])) < 1e-14


def pin_dominant_key(att):
    """A key whose score beats every other by >= 40 takes all the weight."""
    N, d = 16, 4
    q = np.abs(_rng_f64(11, (N, d))) + 0.5
    k = _rng_f64(12, (N, d)) * 0.01
    jstar = 3
    k[jstar] = 60.0
    v = _rng_f64(13, (N, d))
    O, L = att.forward_head(q, k, v, 1.0, False)
    for i in range(N):
        assert np.allclose(O[i], v[jstar], rtol=0, atol=1e-12)
        assert abs(L[i] - float(q[i] @ k[jstar])) < 1e-12
    Oc, _ = att.forward_head(q, k, v, 1.0, True)
    for i in range(jstar, N):
        assert np.allclose(Oc[i], v[jstar], rtol=0, atol=1e-12)


def pin_convexity(att):
    """O_i is a convex combination of the visible V rows; L_i lies in
    [max_j S_ij, max_j S_ij + ln n_i]."""
    N, d = 29, 6
    q = _rng_f64(14, (N, d), 2.0)
    k = _rng_f64(15, (N, d), 2.0)
    v = _rng_f64(16, (N, d))
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        O, L = att.forward_head(q, k, v, scale, causal)
        for i in range(N):
            n = i + 1 if causal else N
            vis = v[:n]
            assert np.all(O[i] >= vis.min(axis=0) - 1e-12)
            assert np.all(O[i] <= vis.max(axis=0) + 1e-12)
            smax = max(scale * float(q[i] @ k[j]) for j in range(n))
            assert smax - 1e-12 <= L[i] <= smax + math.log(n) + 1e-12


def pin_key_permutation(att):
    """Without the mask, permuting keys and values together changes nothing;
    permuting queries permutes the outputs."""
    N, d = 21, 8
    rng = np.random.default_rng(19)
    q = _rng_f64(17, (N, d))
    k = _rng_f64(18, (N, d))
    v = _rng_f64(20, (N, d))
    O, L = att.forward_head(q, k, v, 0.4, False)
    p = rng.permutation(N)
    O2, L2 = att.forward_head(q, k[p], v[p], 0.4, False)
    assert np.allclose(O, O2, rtol=0, atol=1e-12) and np.allclose(L, L2, rtol=0, atol=1e-12)
    O3, L3 = att.forward_head(q[p], k, v, 0.4, False)
    assert np.allclose(O[p], O3, rtol=0, atol=1e-12) and np.allclose(L[p], L3, rtol=0, atol=1e-12)


def pin_full_problem_and_rows(att):
    """forward / forward_rows on [B,H,N,d] agree with the per-head brute force."""
    B, H, N, d = 2, 3, 7, 4
    q = _rng_f64(21, (B, H, N, d))
    k = _rng_f64(22, (B, H, N, d))
    v = _rng_f64(23, (B, H, N, d))
    for causal in (False, True):
        O, L = att.forward(q, k, v, 0.5, causal)
        rows = np.array([0, 3, 6])
        Or, Lr = att.forward_rows(q, k, v, 0.5, causal, rows)
        for b in range(B):
            for h in range(H):
                Ob, Lb = brute_force_head(q[b, h].tolist(), k[b, h].tolist(), v[b, h].tolist(), 0.5, causal)
                assert np.allclose(O[b, h], Ob, atol=1e-12) and np.allclose(L[b, h], Lb, atol=1e-12)
                assert np.allclose(Or[b, h], Ob[rows], atol=1e-12) and np.allclose(Lr[b, h], Lb[rows], atol=1e-12)


# --------------------------------------------------------------------------
# Backward: central finite differences of the scalar sum(dO * O)
# --------------------------------------------------------------------------

def _fd_grad(f, x, h=1e-5):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        xp = x.copy(); xp[idx] += h
        xm = x.copy(); xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


def pin_backward_finite_differences(att):
    for causal in (False, True):
        for (N, d) in ((5, 3), (9, 4)):
            seed = 31 * N + d + (7 if causal else 0)
            q = _rng_f64(seed, (N, d))
            k = _rng_f64(seed + 1, (N, d))
            v = _rng_f64(seed + 2, (N, d))
            do = _rng_f64(seed + 3, (N, d))
            scale = 0.7

            def loss(qq, kk, vv):
                O, _ = brute_force_head(qq.tolist(), kk.tolist(), vv.tolist(), scale, causal)
                return float(np.sum(do * O))

            gq = _fd_grad(lambda x: loss(x, k, v), q)
            gk = _fd_grad(lambda x: loss(q, x, v), k)
            gv = _fd_grad(lambda x: loss(q, k, x), v)
            dq, dk, dv = att.backward_head(q, k, v, do, scale, causal)
            for g, a in ((gq, dq), (gk, dk), (gv, dv)):
                assert np.max(np.abs(g - a)) <= 1e-7 * max(1.0, np.max(np.abs(g))), (causal, N, d)
            rows = np.array([0, N // 2, N - 1])
            dqr = att.backward_dq_rows_head(q, k, v, do, scale, causal, rows)
            assert np.max(np.abs(dqr - gq[rows])) <= 1e-7 * max(1.0, np.max(np.abs(gq)))
            dkr, dvr = att.backward_dkdv_rows_head(q, k, v, do, scale, causal, rows)
            assert np.max(np.abs(dkr - gk[rows])) <= 1e-7 * max(1.0, np.max(np.abs(gk)))
            assert np.max(np.abs(dvr - gv[rows])) <= 1e-7 * max(1.0, np.max(np.abs(gv)))


def pin_d_identity(att):
    """D_i = rowsum(dO_i * O_i) equals rowsum(P_i * dP_i) with dP = dO V^T."""
    N, d = 33, 8
    q = _rng_f64(40, (N, d))
    k = _rng_f64(41, (N, d))
    v = _rng_f64(42, (N, d))
    do = _rng_f64(43, (N, d))
    for causal in (False, True):
        P = att.probabilities_head(q, k, 0.35, causal)
        O, _ = att.forward_head(q, k, v, 0.35, causal)
        dP = do @ v.T
        lhs = np.sum(P * dP, axis=1)
        rhs = att._d_vector(do, O)
        assert np.max(np.abs(lhs - rhs)) < 1e-12


def pin_merge(att):
    """Merging results over a partition of the keys equals the whole."""
    N, d = 40, 8
    q = _rng_f64(50, (N, d))
    k = _rng_f64(51, (N, d))
    v = _rng_f64(52, (N, d))
    for causal in (False, True):
        O, L = att.forward_head(q, k, v, 0.3, causal)
        cuts = [0, 7, 16, 31, 40]
        parts = [att.forward_head_keys(q, k, v, 0.3, causal, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
        Om, Lm = att.merge_partials([p[0] for p in parts], [p[1] for p in parts])
        assert np.allclose(O, Om, rtol=0, atol=1e-12) and np.allclose(L, Lm, rtol=0, atol=1e-12)
        # a part that covers every key is the plain result
        Of, Lf = att.forward_head_keys(q, k, v, 0.3, causal, 0, N)
        assert np.allclose(O, Of, atol=1e-14) and np.allclose(L, Lf, atol=1e-14)


def pin_gqa_routing(att):
    """Grouped-query attention, closed form: with V = 0 on key/value head 0
    and V = 1 on head 1, every softmax row sums to one, so O is exactly 0 for
    the query heads of the first group and exactly 1 for those of the second
    (H = 6, Hkv = 2)."""
    rng = np.random.default_rng(7)
    B, H, Hkv, N, d = 1, 6, 2, 9, 4
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = np.zeros((B, Hkv, N, d))
    v[:, 1] = 1.0
    for causal in (False, True):
        o, _ = att.forward_gqa(q, k, v, 0.5, causal)
        assert np.array_equal(o[:, :3], np.zeros((B, 3, N, d)))
        assert np.allclose(o[:, 3:], 1.0, rtol=0, atol=1e-15)


def pin_gqa_finite_differences(att):
    """Grouped-query attention: dQ, dK, dV against central differences of the
    forward loss sum(O * dO); a dropped group member or a wrong head in the
    sum of a shared head's gradient moves it by a whole term."""
    rng = np.random.default_rng(11)
    B, H, Hkv, N, d = 1, 4, 2, 5, 3
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    do = rng.standard_normal((B, H, N, d))
    scale = 0.7
    for causal in (False, True):
        dq, dk, dv = att.backward_gqa(q, k, v, do, scale, causal)
        assert dk.shape == k.shape and dv.shape == v.shape and dq.shape == q.shape

        def loss(q_, k_, v_):
            return float(np.sum(att.forward_gqa(q_, k_, v_, scale, causal)[0] * do))

        eps = 1e-6
        for name, x, g in (("k", k, dk), ("v", v, dv), ("q", q, dq)):
            for ix in [(0, 0, 1, 2), (0, 1, 4, 0), (0, x.shape[1] - 1, 2, 1)]:
                xp, xm = x.copy(), x.copy()
                xp[ix] += eps
                xm[ix] -= eps
                args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
                args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
                fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
                assert abs(fd - g[ix]) <= 1e-6 * max(1.0, abs(fd)), (name, causal, ix, fd, g[ix])


def pin_gqa_one_group_per_head(att):
    """Hkv = H: the grouped functions give the multi-head results."""
    rng = np.random.default_rng(3)
    q, k, v, do = (rng.standard_normal((2, 3, 7, 4)) for _ in range(4))
    o1, l1 = att.forward_gqa(q, k, v, 0.5, True)
    o2, l2 = att.forward(q, k, v, 0.5, True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    for a, b in zip(att.backward_gqa(q, k, v, do, 0.5, True), att.backward(q, k, v, do, 0.5, True)):
        assert np.array_equal(a, b)


# --------------------------------------------------------------------------
# Queries and keys of different lengths.  Each alignment is pinned through
# the square causal case (Nq = Nk, pinned by brute force above) and closed
# forms, not by restating its mask:
#  * bottom-right: the Nq rows are the last Nq rows of a causal self-attention
#    over all Nk positions (what a decoder computes for the newest Nq tokens);
#    rows that no position of that self-attention corresponds to (Nq > Nk)
#    see no key: O = 0, L = -inf;
#  * top-left: the Nq rows are the first rows of a causal self-attention over
#    the keys, and rows past the last key see every key (no mask);
#  * one query row: bottom-right sees every key (the unmasked result),
#    top-left sees key 0 alone (O = V_0, L = scale q . k_0).
# --------------------------------------------------------------------------

def _square_causal_rows(att, q_rows, k, v, scale, rows):
    """Rows ``rows`` of causal self-attention over len(k) positions whose
    queries at those rows are q_rows (other queries do not matter)."""
    nk, d = k.shape
    qq = np.zeros((nk, d))
    qq[rows] = q_rows
    O, L = att.forward_head(qq, k, v, scale, True)
    return O[rows], L[rows]


def pin_unequal_lengths_alignments(att):
    d, scale = 4, 0.5
    for nq, nk in ((1, 9), (3, 9), (9, 9), (5, 2), (12, 7), (1, 1), (4, 1)):
        seed = 100 * nq + nk
        q = _rng_f64(seed, (nq, d))
        k = _rng_f64(seed + 1, (nk, d))
        v = _rng_f64(seed + 2, (nk, d))
        # bottom-right
        off = att.causal_offset(nq, nk, "bottom_right")
        O, L = att.forward_head(q, k, v, scale, True, offset=off)
        empty = max(0, nq - nk)
        assert np.all(O[:empty] == 0.0) and np.all(L[:empty] == -np.inf), (nq, nk)
        rows = np.arange(nk - (nq - empty), nk)
        Ow, Lw = _square_causal_rows(att, q[empty:], k, v, scale, rows)
        assert np.allclose(O[empty:], Ow, atol=1e-12) and np.allclose(L[empty:], Lw, atol=1e-12), (nq, nk)
        # top-left
        off = att.causal_offset(nq, nk, "top_left")
        O, L = att.forward_head(q, k, v, scale, True, offset=off)
        m = min(nq, nk)
        Ow, Lw = _square_causal_rows(att, q[:m], k, v, scale, np.arange(m))
        assert np.allclose(O[:m], Ow, atol=1e-12) and np.allclose(L[:m], Lw, atol=1e-12), (nq, nk)
        if nq > nk:
            Of, Lf = att.forward_head(q[nk:], k, v, scale, False)
            assert np.allclose(O[nk:], Of, atol=1e-12) and np.allclose(L[nk:], Lf, atol=1e-12), (nq, nk)
        if nq == 1:
            Ob, Lb = att.forward_head(q, k, v, scale, True, offset=att.causal_offset(1, nk, "bottom_right"))
            Of, Lf = brute_force_head(q.tolist() + [[0.0] * d] * (nk - 1), k.tolist(), v.tolist(), scale, False)
            assert np.allclose(Ob, Of[:1], atol=1e-12) and np.allclose(Lb, Lf[:1], atol=1e-12)
            assert np.allclose(O[0], v[0], atol=1e-14) and abs(L[0] - scale * float(q[0] @ k[0])) < 1e-12


def pin_unequal_lengths_finite_differences(att):
    """Gradients with Nq != Nk, both alignments (rows that see no key
    included), against central differences of the forward pass."""
    d, scale = 3, 0.6
    for nq, nk, align in ((3, 7, "bottom_right"), (6, 4, "bottom_right"), (6, 4, "top_left"),
                          (2, 5, "top_left")):
        seed = 7 * nq + nk
        q = _rng_f64(seed, (nq, d))
        k = _rng_f64(seed + 1, (nk, d))
        v = _rng_f64(seed + 2, (nk, d))
        do = _rng_f64(seed + 3, (nq, d))
        off = att.causal_offset(nq, nk, align)

        def loss(qq, kk, vv):
            O, _ = att.forward_head(qq, kk, vv, scale, True, offset=off)
            return float(np.sum(do * O))

        gq = _fd_grad(lambda x: loss(x, k, v), q)
        gk = _fd_grad(lambda x: loss(q, x, v), k)
        gv = _fd_grad(lambda x: loss(q, k, x), v)
        dq, dk, dv = att.backward_head(q, k, v, do, scale, True, offset=off)
        for g, a in ((gq, dq), (gk, dk), (gv, dv)):
            assert np.max(np.abs(g - a)) <= 1e-7 * max(1.0, np.max(np.abs(g))), (nq, nk, align)
        rows = np.arange(nq)
        dqr = att.backward_dq_rows_head(q, k, v, do, scale, True, rows, offset=off)
        assert np.max(np.abs(dqr - gq)) <= 1e-7 * max(1.0, np.max(np.abs(gq)))
        keys = np.arange(nk)
        dkr, dvr = att.backward_dkdv_rows_head(q, k, v, do, scale, True, keys, offset=off)
        assert np.max(np.abs(dkr - gk)) <= 1e-7 * max(1.0, np.max(np.abs(gk)))
        assert np.max(np.abs(dvr - gv)) <= 1e-7 * max(1.0, np.max(np.abs(gv)))


ALL_PINS = [
    pin_brute_force,
    pin_rows_sum_to_one,
    pin_identical_keys,
    pin_causal_first_row,
    pin_dominant_key,
    pin_convexity,
    pin_key_permutation,
    pin_full_problem_and_rows,
    pin_backward_finite_differences,
    pin_d_identity,
    pin_merge,
    pin_gqa_routing,
    pin_gqa_finite_differences,
    pin_gqa_one_group_per_head,
    pin_unequal_lengths_alignments,
    pin_unequal_lengths_finite_differences,
]
