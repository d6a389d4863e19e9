"""Comparison of CUDA results with the fp64 oracle, at the stated tolerances.

Tolerances (attention forward / backward on bf16 inputs):
  O    : max |O_gpu - O_ref| <= 1e-2, element by element relaxed to one bf16
         ulp of O_ref where |O_ref| >= 2 (a correctly rounded bf16 output can
         sit half an ulp away from the fp64 value, more than 1e-2 once
         |O| > 5); and mean |O_gpu - bf16(O_ref)| <= 1e-3.
         An element above that flat bound must still lie within the bound
         that follows from the precisions the method is read to use (P
         rounded to bf16 for the P V product, O the weighted mean under those
         weights): each weight has relative error <= u = 2^-8, so the rounded
         weights renormalised differ from P_ij by at most 2u P_ij and
           |dO_ic| <= 0.5 ulp(O_ic) + 2u * sum_j P_ij |V_jc - O_ic| + 1e-4,
         computed from the oracle's weights for that row.  Such elements may
         be at most 1 in 10^6 of the elements checked (none in a check of
         fewer than 10^6 elements); how many there were is
         recorded per case (O_EXCEPTIONS) and printed at the end of the run.
  LSE  : |L_gpu - L_ref| <= 1e-4 * max(1, |L_ref|) (relative error, with an
         absolute floor where L is near 0, e.g. causal row 0).
  grads: max |g_gpu - g_ref| <= 5e-2 * max |g_ref|, per tensor.
The oracle works in fp64 on the same bf16-rounded inputs.
"""

import numpy as np

from exact_attention_92_gb300 import inputs

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_REL = 1e-4
GRAD_REL = 5e-2


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (2^(e-7) for |x| in [2^e, 2^(e+1)))."""
    a = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    e = np.floor(np.log2(a))
    return np.exp2(e - 7)


def round_bf16(x):
    return inputs.bits_to_f64(inputs.bf16_bits(np.asarray(x, dtype=np.float32)))


U_BF16 = 2.0 ** -8
O_EXCEPTION_BUDGET = 10 ** -6

# (what, elements checked, elements above the flat bound) of every check_o
# call of the session; the test session prints it as a summary.
O_EXCEPTIONS = []


def check_o(o_gpu, o_ref, what="", row_weights=None):
    """row_weights(index_without_column) -> (P_row [n_keys], V [n_keys, d]):
    the oracle's softmax weights and values of one output row, used to bound
    elements above the flat bound."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    err = np.abs(o_gpu - o_ref)
    allowed = np.maximum(O_MAX_ABS, bf16_ulp(o_ref))
    bad = err > allowed
    assert not np.isnan(o_gpu).any(), f"{what}: NaN in O"
    O_EXCEPTIONS.append((what, int(err.size), int(bad.sum())))
    if bad.any():
        idx = np.argwhere(bad)
        msg = (f"{what}: O max-abs error {err.max():.3e} over the flat bound at {idx[:5].tolist()} "
               f"(ref {o_ref[bad][:5]}, gpu {o_gpu[bad][:5]})")
        assert row_weights is not None and len(idx) <= int(err.size * O_EXCEPTION_BUDGET), msg
        for ix in idx:
            P, V = row_weights(tuple(ix[:-1]))
            c = ix[-1]
            ref = o_ref[tuple(ix)]
            derived = 0.5 * bf16_ulp(ref) + 2 * U_BF16 * float(np.sum(P * np.abs(V[:, c] - ref))) + 1e-4
            assert err[tuple(ix)] <= derived, f"{msg}; derived bound {derived:.3e} at {ix.tolist()}"
    mean = float(np.mean(np.abs(o_gpu - round_bf16(o_ref))))
    assert mean <= O_MEAN_ABS, f"{what}: O mean-abs error {mean:.3e} > {O_MEAN_ABS}"
    return float(err.max()), mean


def check_lse(l_gpu, l_ref, what=""):
    """A row that sees no key has L = -inf in the oracle; the GPU must give
    exactly -inf there and finite values elsewhere."""
    l_gpu = np.asarray(l_gpu, dtype=np.float64)
    l_ref = np.asarray(l_ref, dtype=np.float64)
    assert not np.isnan(l_gpu).any(), f"{what}: NaN in LSE"
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(l_gpu), empty), (
        f"{what}: LSE -inf at {np.argwhere(np.isneginf(l_gpu) != empty)[:5].tolist()} disagrees with the oracle")
    l_gpu = np.where(empty, 0.0, l_gpu)
    l_ref = np.where(empty, 0.0, l_ref)
    err = np.abs(l_gpu - l_ref)
    bound = LSE_REL * np.maximum(1.0, np.abs(l_ref))
    bad = err > bound
    assert not bad.any(), (f"{what}: LSE error {err.max():.3e} at {np.argwhere(bad)[:5].tolist()} "
                           f"(ref {l_ref[bad][:5]}, gpu {l_gpu[bad][:5]})")
    return float(np.max(err / np.maximum(1.0, np.abs(l_ref))))


def check_grad(g_gpu, g_ref, name, what=""):
    g_gpu = np.asarray(g_gpu, dtype=np.float64)
    assert not np.isnan(g_gpu).any(), f"{what}: NaN in {name}"
    scale = float(np.max(np.abs(g_ref)))
    err = float(np.max(np.abs(g_gpu - g_ref)))
    if scale == 0.0:
        # e.g. a single key: dQ = dK = 0 exactly; allow rounding noise only
        assert err <= 1e-6, f"{what}: {name} should be 0, max-abs {err:.3e}"
        return err
    assert err <= GRAD_REL * scale, f"{what}: {name} max-abs error {err:.3e} > {GRAD_REL} x {scale:.3e}"
    return err / scale
