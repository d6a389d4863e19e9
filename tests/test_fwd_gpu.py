"""Forward pass on the GPU against the fp64 oracle (through the C ABI)."""

import numpy as np
import pytest

from exact_attention_92_gb300 import inputs
from oracle import attention as att

from gpu_util import case_tensors, ensure_built, host, torch_cuda
from parity import check_lse, check_o, round_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    torch_cuda()
    return ensure_built()


def run_fwd(fa, case, num_splits=0):
    q, k, v, _ = case_tensors(case)
    o, lse = fa.forward(q, k, v, causal=case.causal, num_splits=num_splits)
    st = fa.fa_poll_status()
    assert st == 0, fa.fa_strerror(st)
    return host(o), lse.cpu().numpy().astype(np.float64)


def weights_of(case, rows=None):
    """Oracle softmax weights and values of one output row (for the derived
    O bound of elements above the flat bound)."""
    q, k, v = case.f64("q"), case.f64("k"), case.f64("v")

    def fn(ix):
        b, h, r = ix
        row = int(rows[b, h, r]) if rows is not None else int(r)
        P = att.probabilities_head(q[b, h], k[b, h], case.scale, case.causal, rows=np.array([row]))[0]
        return P, v[b, h]

    return fn


def check_full(fa, case, num_splits=0, what=""):
    o, lse = run_fwd(fa, case, num_splits)
    O, L = att.forward(case.f64("q"), case.f64("k"), case.f64("v"), case.scale, case.causal)
    check_o(o, O, what, weights_of(case))
    check_lse(lse, L, what)
    return o, lse, O, L


def check_sampled(fa, case, num_splits=0, what=""):
    o, lse = run_fwd(fa, case, num_splits)
    rows = inputs.sample_rows_per_head(case.seed, case.B, case.H, case.N)
    O, L = att.forward_rows(case.f64("q"), case.f64("k"), case.f64("v"), case.scale, case.causal, rows)
    og = np.take_along_axis(o, rows[..., None], axis=2)
    lg = np.take_along_axis(lse, rows, axis=2)
    check_o(og, O, what, weights_of(case, rows))
    check_lse(lg, L, what)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    return o, lse


# Small shapes: several tiles, ragged tails, a single row, both head dims.
SMALL = [
    (1, 1, 128, 64), (1, 1, 128, 128), (2, 3, 257, 64), (1, 2, 1, 64), (1, 1, 63, 128),
    (1, 2, 129, 128), (2, 2, 200, 64), (1, 1, 384, 128), (1, 1, 1000, 128), (3, 1, 640, 64),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(fa, shape, causal):
    B, H, N, d = shape
    case = inputs.make_case(B, H, N, d, causal, seed=100 + N + d + (1 if causal else 0))
    check_full(fa, case, 1, f"{shape} causal={causal}")


@pytest.mark.parametrize("splits", [2, 3, 5, 64])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1000, 128), (2, 1, 640, 64), (1, 2, 1, 128)],
                         ids=lambda s: "x".join(map(str, s)))
def test_split_kv_small(fa, shape, causal, splits):
    B, H, N, d = shape
    case = inputs.make_case(B, H, N, d, causal, seed=200 + N + d)
    check_full(fa, case, splits, f"{shape} causal={causal} splits={splits}")


@pytest.mark.parametrize("c", inputs.workload_cases()[1], ids=lambda c: f"causal{int(c['causal'])}")
def test_single_head_n128_d64(fa, c):
    case = inputs.make_case(**c)
    o, lse, O, L = check_full(fa, case, what=str(c))
    if case.causal:
        # causal row 0 sees only key 0: O_0 = V_0 and L_0 = scale q_0 . k_0
        assert np.array_equal(o[0, 0, 0], case.f64("v")[0, 0, 0])
        l0 = case.scale * float(case.f64("q")[0, 0, 0] @ case.f64("k")[0, 0, 0])
        assert abs(lse[0, 0, 0] - l0) <= 1e-4 * max(1.0, abs(l0))


@pytest.mark.parametrize("c", inputs.workload_cases()[2],
                         ids=lambda c: f"causal{int(c['causal'])}-{c.get('degenerate', 'iid')}")
def test_b4_h16_n1024_d64(fa, c):
    case = inputs.make_case(**c)
    o, lse, O, L = check_full(fa, case, what=str(c))
    if c.get("degenerate") == "identical_keys":
        v = case.f64("v")
        n_vis = np.arange(1, case.N + 1)[:, None] if case.causal else case.N
        mean = np.cumsum(v, axis=2) / n_vis if case.causal else np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
        check_o(o, mean, "identical keys: O = mean of visible V")
    if c.get("degenerate") == "dominant_key":
        j = case.dominant_key
        q, k, v = case.f64("q"), case.f64("k"), case.f64("v")
        checked = 0
        for b in range(case.B):
            for h in range(case.H):
                s = case.scale * (q[b, h] @ k[b, h].T)
                if case.causal:
                    s = np.where(np.tril(np.ones((case.N, case.N), bool)), s, -np.inf)
                other = np.max(np.delete(s, j, axis=1), axis=1)
                dom = (s[:, j] - other >= 20.0) & (np.arange(case.N) >= (j if case.causal else 0))
                if dom.any():
                    checked += int(dom.sum())
                    assert np.all(np.abs(o[b, h][dom] - round_bf16(v[b, h, j])[None, :]) <= 1e-2)
                    assert np.all(np.abs(lse[b, h][dom] - s[dom, j]) <= 1e-4 * np.maximum(1, np.abs(s[dom, j])))
        assert checked > 0


@pytest.mark.parametrize("d", [64, 96, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_rising_keys_rescale_every_tile(fa, d, causal):
    """Logits that climb by some 46 log2 units per 128-key tile: every row's
    running maximum moves past the correction threshold at every key tile,
    so the O~ correction (and, at d=64, its wait for the tile's previous
    P V product) runs at every step ("FlashAttention V2 in depth" 6.1)."""
    case = inputs.make_case(2, 3, 1000, d, causal, seed=70 + d + int(causal), degenerate="rising_keys")
    q, k = case.f64("q"), case.f64("k")
    s = case.scale * np.einsum("bhc,bhmc->bhm", q[:, :, -1], k)  # logits of the last query row
    tile_max = s[..., :896].reshape(2, 3, 7, 128).max(-1)
    assert np.all(np.diff(tile_max, axis=-1) * np.log2(np.e) > 24.0)
    check_full(fa, case, what=f"rising keys d{d} causal{int(causal)}")


SWEEP = inputs.workload_cases()[3]


@pytest.mark.parametrize("c", SWEEP, ids=lambda c: f"N{c['N']}-d{c['d']}-causal{int(c['causal'])}")
def test_sweep_16k_tokens(fa, c):
    case = inputs.make_case(**c)
    check_sampled(fa, case, what=str(c))


@pytest.mark.parametrize("c", inputs.workload_cases()[4], ids=lambda c: f"B{c['B']}H{c['H']}N{c['N']}causal{int(c['causal'])}")
def test_gpt_layer_and_long_single_head(fa, c):
    case = inputs.make_case(**c)
    check_sampled(fa, case, what=str(c))


@pytest.mark.parametrize("splits", [1, 4])
def test_long_single_head_forced_splits(fa, splits):
    c = inputs.workload_cases()[4][1]
    case = inputs.make_case(**c)
    check_sampled(fa, case, num_splits=splits, what=f"N=65536 splits={splits}")


def test_repeatable(fa):
    """The forward pass has no atomics: two runs give identical bits."""
    torch = torch_cuda()
    case = inputs.make_case(2, 4, 777, 128, True, seed=31)
    q, k, v, _ = case_tensors(case)
    o1, l1 = fa.forward(q, k, v, causal=True)
    o2, l2 = fa.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_grid_larger_than_units_and_many_units(fa):
    """Persistent CTAs that get no unit, and CTAs that walk many units."""
    for (B, H, N) in [(1, 1, 256), (64, 8, 384)]:
        case = inputs.make_case(B, H, N, 64, True, seed=40 + B)
        q, k, v, _ = case_tensors(case)
        o, lse = fa.forward(q, k, v, causal=True)
        rows = inputs.sample_rows_per_head(case.seed, B, H, N, n=64)
        O, L = att.forward_rows(case.f64("q"), case.f64("k"), case.f64("v"), case.scale, True, rows)
        check_o(np.take_along_axis(host(o), rows[..., None], axis=2), O, f"B{B}H{H}N{N}")
        check_lse(np.take_along_axis(lse.cpu().numpy().astype(np.float64), rows, axis=2), L, f"B{B}H{H}N{N}")
