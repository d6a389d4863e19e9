"""Plant plausible mistakes in the oracle (CPU only) and require that at least
one pin catches each.  Each mutant replaces one step of ``oracle.attention``
through monkeypatch, so the oracle's own code is what runs, with one error."""

import numpy as np
import pytest

from oracle import attention as att

from oracle_pins import ALL_PINS


def _fails_some_pin():
    failed = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(att)
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            failed.append(pin.__name__)
    return failed


MUTANTS = {
    # forward
    "scale_dropped": ("_scores", lambda q, k, scale: q @ k.T),
    "operands_transposed": ("_scores", lambda q, k, scale: scale * (k @ q.T)),
    "mask_flipped": ("_visible", lambda rows, n_k, off=0: np.arange(n_k)[None, :] >= rows[:, None] + off),
    "mask_strict": ("_visible", lambda rows, n_k, off=0: np.arange(n_k)[None, :] < rows[:, None] + off),
    "mask_off_by_one": ("_visible", lambda rows, n_k, off=0: np.arange(n_k)[None, :] <= rows[:, None] + off + 1),
    # queries and keys of different lengths
    "offset_ignored": ("_visible", lambda rows, n_k, off=0: np.arange(n_k)[None, :] <= rows[:, None]),
    "offset_negated": ("_visible", lambda rows, n_k, off=0: np.arange(n_k)[None, :] <= rows[:, None] - off),
    "bottom_right_as_top_left": ("causal_offset", lambda n_q, n_k, align: 0),
    "bottom_right_reversed": ("causal_offset", lambda n_q, n_k, align: 0 if align == "top_left" else n_q - n_k),
    "empty_rows_uniform": ("_normalise", lambda p, l: p / np.where(l > 0, l, 1.0)[:, None]
                           + (l == 0)[:, None] / p.shape[1]),
    "max_sign": ("_softmax_stats", lambda s: (lambda m: (m, np.exp(s + m[:, None]), np.sum(np.exp(s + m[:, None]), axis=1)))(np.max(s, axis=1))),
    "lse_without_max": ("_lse", lambda m, l: np.log(l)),
    "lse_log2": ("_lse", lambda m, l: m + np.log2(l)),
    # backward
    "d_dropped": ("_d_vector", lambda do, o: np.zeros(do.shape[0])),
    "d_wrong_axis": ("_d_vector", lambda do, o: np.sum(do * o, axis=1)[::-1].copy()),
    # grouped-query attention
    "gqa_heads_interleaved": ("expand_kv", lambda x, H: np.tile(x, (1, H // x.shape[1], 1, 1))),
    "gqa_sum_interleaved": ("reduce_kv", lambda g, Hkv: g.reshape(g.shape[0], g.shape[1] // Hkv, Hkv,
                                                                  *g.shape[2:]).sum(axis=1)),
    "gqa_mean_not_sum": ("reduce_kv", lambda g, Hkv: g.reshape(g.shape[0], Hkv, g.shape[1] // Hkv,
                                                               *g.shape[2:]).mean(axis=2)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(att, attr, fn)
    failed = _fails_some_pin()
    assert failed, f"no pin caught the planted mistake {name!r}"
