"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""

import json
import math
import os

import numpy as np
import pytest

from exact_attention_92_gb300 import inputs
from oracle import attention as att
from oracle import blockwise

from oracle_pins import ALL_PINS, _rng_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(att)


# --------------------------------------------------------------------------
# The tiled algorithm ("FlashAttention V2 in depth", section 6.1) equals the
# definition: delayed normalisation and the causal block skip are exact.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,B_r,B_c", [(64, 16, 16), (100, 32, 16), (100, 16, 32), (129, 64, 64), (7, 4, 3), (1, 64, 64)])
def test_blockwise_equals_definition(causal, N, B_r, B_c):
    d = 8
    q = _rng_f64(60 + N, (N, d), 2.0)
    k = _rng_f64(61 + N, (N, d), 2.0)
    v = _rng_f64(62 + N, (N, d))
    scale = 1 / math.sqrt(d)
    O, L = att.forward_head(q, k, v, scale, causal)
    Ob, Lb = blockwise.forward_head(q, k, v, scale, causal, B_r, B_c)
    assert np.max(np.abs(O - Ob)) < 1e-12
    assert np.max(np.abs(L - Lb)) < 1e-12


def test_blockwise_counts_page1_worked_example():
    """Page "FlashAttention-2 Improvements", section "Reduced Non-Matrix-Multiply
    FLOPs": at n=4096 and 64-row blocks one query block walks 64 key/value
    blocks; per-block rescaling would touch 64 x 64 = 4096 rows, the single
    final normalisation 64."""
    g = json.load(open(os.path.join(GOLDEN, "page1_counts.json")))
    n, B_r, B_c = g["n"], g["B_r"], g["B_c"]
    d = 2
    q = _rng_f64(70, (n, d))
    k = _rng_f64(71, (n, d))
    v = _rng_f64(72, (n, d))
    c = {}
    blockwise.forward_head(q, k, v, 0.5, False, B_r, B_c, counts=c)
    steps_per_block = c["kv_steps"] // c["q_blocks"]
    assert steps_per_block == g["kv_blocks"]
    assert steps_per_block * B_r == g["fa1_rescales"]
    assert c["final_divides"] // c["q_blocks"] == g["fa2_rescales"]
    assert g["fa1_rescales"] // g["fa2_rescales"] == g["reduction"]


@pytest.mark.parametrize("N,B_r,B_c", [(256, 64, 64), (512, 128, 64), (512, 64, 128), (1024, 128, 128)])
def test_blockwise_causal_block_classes(N, B_r, B_c):
    """Section 5.3: tiles above the diagonal are skipped, tiles below it run
    unmasked, tiles crossing it are masked element by element.  The expected
    counts come from the two inequalities alone (first row >= last column:
    visible; last row < first column: skipped), and the skipped fraction is
    (T-1)/(2T) for T blocks per side, close to the half of section 5.4."""
    d = 4
    q = _rng_f64(80, (N, d))
    k = _rng_f64(81, (N, d))
    v = _rng_f64(82, (N, d))
    c = {}
    blockwise.forward_head(q, k, v, 0.5, True, B_r, B_c, counts=c)
    full = diag = skip = 0
    nk = N // B_c
    for i in range(N // B_r):
        r0, r1 = i * B_r, (i + 1) * B_r - 1
        f = sum(1 for j in range(nk) if r0 >= (j + 1) * B_c - 1)
        s = sum(1 for j in range(nk) if r1 < j * B_c)
        full += f
        skip += s
        diag += nk - f - s
    assert (c["full"], c["diagonal"], c["skipped"]) == (full, diag, skip)
    total = (N // B_r) * nk
    # about half of the tiles are skipped
    assert abs(skip / total - 0.5) <= 0.5 * max(B_r, B_c) / N + 1e-9


def test_inputs_bf16_rounding_is_rne():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e-3], dtype=np.float32)
    bits = inputs.bf16_bits(x)
    back = inputs.bits_to_f64(bits)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert back[0] == 1.0 and back[1] == 1.0
    # 1 + 1.5 * 2^-8 rounds up to 1 + 2^-7
    assert back[2] == 1.0078125
    assert back[3] == -2.5
    assert abs(back[4] - 3.0e-3) <= 2.0 ** -8 * 3.0e-3  # half an ulp: 2^-8 relative


def test_inputs_seeded_and_degenerate():
    c1 = inputs.make_case(1, 2, 64, 16, False, 123)
    c2 = inputs.make_case(1, 2, 64, 16, False, 123)
    assert np.array_equal(c1.q, c2.q) and np.array_equal(c1.v, c2.v)
    ci = inputs.make_case(1, 2, 64, 16, False, 5, degenerate="identical_keys")
    assert np.all(ci.k == ci.k[:, :, :1, :])
    cd = inputs.make_case(1, 2, 64, 16, True, 5, degenerate="dominant_key")
    assert 0 <= cd.dominant_key < 16
    base = inputs.make_case(1, 2, 64, 16, True, 5)
    ratio = cd.f64("k")[:, :, cd.dominant_key] / base.f64("k")[:, :, cd.dominant_key]
    assert np.all(np.abs(ratio - 50) <= 50 * 2.0 ** -8)
    rows = inputs.sample_rows(9, 4096)
    assert rows.size == 1024 and np.unique(rows).size == 1024


def test_flop_counts():
    assert inputs.fwd_flops(8, 32, 4096, 128, True) == 4 * 8 * 32 * 4096 ** 2 * 128 / 2
    assert inputs.bwd_flops(2, 16, 4096, 128, True) == 2.5 * inputs.fwd_flops(2, 16, 4096, 128, True)

