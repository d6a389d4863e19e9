"""Launch plans of the forward and backward calls, checked on the host.

fa_fwd_plan / fa_bwd_plan return what fa_fwd_general / fa_bwd_general do
for given sizes (the calls fill in the same plan with the current device's
SM count and L2 size): head packing, the key splits and the decoding dual
mode, the CTA grid, the unit order's head window, the kernels launched and
the workspace taken.  These tests run without a GPU.  They check the plans
against what must hold for any sizes (no empty split, every key tile in one
split, the workspace of the partial results that are merged), against brute
force (which query and key tiles some row sees under each causal
alignment), and pin the decisions measured fastest on GB300 for the
workloads named in the tests.
"""

import math
import random

import pytest

import exact_attention_92_gb300 as fa
from exact_attention_92_gb300 import build

SM = 152  # GB300
L2 = 126 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    fa.load()


def fwd_plan(B, H, Hkv, Nq, Nk, d, causal=0, splits=0, sm=SM, l2=L2):
    return fa.fa_fwd_plan(B, H, Hkv, Nq, Nk, d, causal, splits, sm, l2)


def bwd_plan(B, H, Hkv, Nq, Nk, d, causal=0, sm=SM):
    return fa.fa_bwd_plan(B, H, Hkv, Nq, Nk, d, causal, sm)


def sees(i, j, Nq, Nk, causal):
    """Query row i sees key j under the causal code (the mask the header
    defines: top-left j <= i, bottom-right j <= i + Nk - Nq)."""
    if causal == fa.FA_CAUSAL_NONE:
        return True
    if causal == fa.FA_CAUSAL_TOP_LEFT:
        return j <= i
    return j <= i + Nk - Nq


def random_sizes(rng):
    Hkv = rng.randint(1, 8)
    H = Hkv * rng.choice([1, 1, 2, 4, 8])
    B = rng.randint(1, 16)
    kind = rng.randrange(4)
    if kind == 0:  # decoding
        Nq, Nk = rng.randint(1, 8), rng.randint(1, 70000)
    elif kind == 1:  # short chunks over long keys
        Nq, Nk = rng.randint(1, 400), rng.randint(1, 30000)
    elif kind == 2:  # self-attention
        Nq = Nk = rng.randint(1, 40000)
    else:
        Nq, Nk = rng.randint(1, 20000), rng.randint(1, 20000)
    return B, H, Hkv, Nq, Nk, rng.choice([64, 96, 128, 256]), rng.randrange(3)


def test_plan_argument_errors():
    def fwd_status(*a):
        try:
            fwd_plan(*a)
            return fa.FA_OK
        except fa.FaError as e:
            return e.status

    assert fwd_status(1, 4, 2, 100, 300, 48) == fa.FA_ERR_UNSUPPORTED
    assert fwd_status(1, 4, 3, 100, 300, 64) == fa.FA_ERR_INVALID_ARG
    assert fwd_status(1, 4, 2, 0, 300, 64) == fa.FA_ERR_INVALID_ARG
    assert fwd_status(1, 4, 2, 100, 300, 64, 3) == fa.FA_ERR_INVALID_ARG
    assert fwd_status(1, 4, 2, 100, 300, 64, 0, -1) == fa.FA_ERR_INVALID_ARG
    assert fwd_status(1, 4, 2, 100, 300, 64, 0, 0, 0) == fa.FA_ERR_INVALID_ARG
    # A forced split count whose units (65536 query blocks x 131072 splits of
    # one 2^24-token head) overflow a 32-bit unit index; the same head with
    # the automatic count is fine.
    assert fwd_status(1, 1, 1, 1 << 24, 1 << 24, 64, 0, 1 << 20) == fa.FA_ERR_INVALID_ARG
    assert fwd_status(1, 1, 1, 1 << 24, 1 << 24, 64, 0, 0) == fa.FA_OK
    lib = fa.load()
    assert lib.fa_fwd_plan(1, 1, 1, 128, 128, 64, 0, 0, SM, L2, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_plan(1, 1, 1, 128, 128, 64, 0, SM, None) == fa.FA_ERR_INVALID_ARG
    with pytest.raises(fa.FaError):
        bwd_plan(1, 4, 2, 100, 300, 80)
    with pytest.raises(fa.FaError):
        bwd_plan(1, 4, 2, 100, 300, 64, 0, 0)


def test_fwd_plan_invariants():
    rng = random.Random(20261203)
    seen = {"dual": 0, "split": 0, "packed": 0, "window": 0, "forced": 0}
    for _ in range(3000):
        B, H, Hkv, Nq, Nk, d, causal = random_sizes(rng)
        forced = rng.choice([0, 0, 0, rng.randint(1, 20)])
        sm = rng.choice([SM, rng.randint(1, 200)])
        l2 = rng.choice([L2, rng.randint(1, 256) << 20])
        p = fwd_plan(B, H, Hkv, Nq, Nk, d, causal, forced, sm, l2)
        G = H // Hkv
        wide = d == 256
        what = (B, H, Hkv, Nq, Nk, d, causal, forced, sm, l2, p)
        # Head packing: grouped heads with short query blocks share a tile.
        assert p["packed_heads"] == int(G > 1 and Nq < 128), what
        assert p["unit_heads"] * p["unit_rows"] == B * H * Nq, what
        assert p["unit_heads"] == B * (Hkv if p["packed_heads"] else H), what
        assert (p["query_block"], p["key_tile"]) == ((128, 64) if wide else (256, 128)), what
        nkv = math.ceil(Nk / p["key_tile"])
        assert p["key_tiles"] == nkv, what
        # Splits: S >= 1, every key tile in exactly one split, none empty.
        S, per = p["num_splits"], p["key_tiles_per_split"]
        assert 1 <= S <= nkv and per * S >= nkv and per * (S - 1) < nkv, what
        if forced:
            f = min(forced, nkv)
            assert per == math.ceil(nkv / f) and S == math.ceil(nkv / per), what
            assert p["dual"] == 0, what
        elif S > 1:
            assert nkv // S >= (8 if wide else 4), what  # no split shorter than the minimum
        if p["dual"]:
            assert not forced and not wide and p["unit_rows"] <= 128 and per >= 8, what
        # Units, grid, the merge and its workspace.
        qblocks = math.ceil(p["unit_rows"] / p["query_block"])
        assert p["num_units"] == p["unit_heads"] * qblocks * S, what
        assert p["grid"] == min(p["num_units"], sm), what
        parts = 2 * S if p["dual"] else S
        assert p["partials"] == (parts if parts > 1 else 0), what
        assert p["launches"] == (2 if p["partials"] else 1), what
        assert p["workspace_bytes"] == p["partials"] * B * H * Nq * (d + 1) * 4, what
        # Head windows: only without the mask, one split, K and V beyond
        # half the L2; the fewest heads whose query blocks fill the grid.
        w = p["head_window"]
        if w:
            assert causal == 0 and S == 1 and 4 * B * Hkv * Nk * d > l2 / 2, what
            assert w < p["unit_heads"] and w * qblocks >= p["grid"] and (w - 1) * qblocks < p["grid"], what
        seen["dual"] += p["dual"]
        seen["split"] += S > 1
        seen["packed"] += p["packed_heads"]
        seen["window"] += w > 0
        seen["forced"] += forced > 0
    assert all(v > 50 for v in seen.values()), seen


def test_fwd_plan_automatic_split_only_when_units_are_few():
    """Without a forced count, prefill with enough (head, query block) units
    for every SM twice over is never split and takes no workspace."""
    rng = random.Random(7)
    for _ in range(500):
        B, H, Hkv, Nq, Nk, d, causal = random_sizes(rng)
        p = fwd_plan(B, H, Hkv, Nq, Nk, d, causal)
        units = p["unit_heads"] * math.ceil(p["unit_rows"] / p["query_block"])
        if units >= 2 * SM and p["unit_rows"] > 128:
            assert p["num_splits"] == 1 and p["partials"] == 0 and p["workspace_bytes"] == 0


def test_fwd_plan_decisions_on_gb300():
    """The plans of the measured workloads (152 SMs, 126 MiB of L2)."""
    # fwd+bwd step, B=2 H=16 N=4096 d=128 causal: one launch, no workspace.
    p = fwd_plan(2, 16, 16, 4096, 4096, 128, fa.FA_CAUSAL_TOP_LEFT)
    assert (p["num_splits"], p["partials"], p["grid"], p["head_window"]) == (1, 0, SM, 0)
    # Non-causal B=4 H=16 N=4096 d=128: K, V (134 MB) exceed half the L2, so
    # units go by windows of ten heads (16 query blocks a head fill 152 CTAs).
    p = fwd_plan(4, 16, 16, 4096, 4096, 128)
    assert p["head_window"] == 10 and p["num_splits"] == 1
    # The same with K, V within half the L2 (B=1 H=4): no window.
    assert fwd_plan(1, 4, 4, 4096, 4096, 128)["head_window"] == 0
    # One long causal head, N=65536: split along the keys, merged.
    p = fwd_plan(1, 1, 1, 65536, 65536, 128, fa.FA_CAUSAL_TOP_LEFT)
    assert p["num_splits"] > 1 and p["partials"] == p["num_splits"] and p["launches"] == 2
    # GQA decoding, B=8 H=32 Hkv=8, one query over 8192 keys: the four query
    # heads of a group share a tile, both tiles of a CTA take its key tiles.
    p = fwd_plan(8, 32, 8, 1, 8192, 128, fa.FA_CAUSAL_BOTTOM_RIGHT)
    assert p["packed_heads"] == 1 and p["unit_rows"] == 4 and p["dual"] == 1
    assert p["partials"] == 2 * p["num_splits"]
    # Head dim 256 never runs dual (one query tile per CTA).
    assert fwd_plan(8, 32, 8, 1, 8192, 256, fa.FA_CAUSAL_BOTTOM_RIGHT)["dual"] == 0
    # A forced split count is kept (clamped to the key tiles, no empty split).
    p = fwd_plan(1, 2, 2, 1000, 1000, 64, 0, 5)  # 8 key tiles: 5 -> 2 a split -> 4 splits
    assert (p["num_splits"], p["key_tiles_per_split"], p["partials"]) == (4, 2, 4)
    assert fwd_plan(1, 2, 2, 1000, 1000, 64, 0, 100)["num_splits"] == 8


@pytest.mark.parametrize("d", [64, 96, 128, 256])
def test_bwd_plan_against_brute_force(d):
    """Query tiles with no visible key and key tiles no row sees, by
    enumeration of the mask, for every causal alignment and ragged sizes."""
    rng = random.Random(d)
    cases = [(300, 100), (100, 300), (128, 128), (129, 1), (1, 129), (640, 333), (257, 256), (1000, 1000)]
    cases += [(rng.randint(1, 700), rng.randint(1, 700)) for _ in range(12)]
    for Nq, Nk in cases:
        for causal in range(3):
            B, Hkv, G = 2, 3, 2
            H = Hkv * G
            p = bwd_plan(B, H, Hkv, Nq, Nk, d, causal)
            qt, kt = math.ceil(Nq / 128), math.ceil(Nk / 128)
            q_live = [any(sees(i, j, Nq, Nk, causal) for i in range(t * 128, min(Nq, t * 128 + 128))
                          for j in range(Nk)) for t in range(qt)]
            k_live = [any(sees(i, j, Nq, Nk, causal) for j in range(t * 128, min(Nk, t * 128 + 128))
                          for i in range(Nq)) for t in range(kt)]
            what = (Nq, Nk, causal, p)
            assert (p["q_tiles"], p["k_tiles"]) == (qt, kt), what
            # Visibility is monotone: dead query tiles lead, dead key tiles trail.
            first = q_live.index(True) if any(q_live) else qt
            used = kt - k_live[::-1].index(True) if any(k_live) else 0
            assert p["q_tile_first"] == first and all(q_live[first:]), what
            assert p["kv_tiles_used"] == used and all(k_live[:used]), what
            assert p["dq_units"] == B * H * (qt - first), what
            assert p["dq_grid"] == min(p["dq_units"], SM), what
            assert p["kv_units"] == B * Hkv * (math.ceil(used / 2) if d == 128 else used), what
            assert p["zeroed_dq_bytes"] == B * H * min(Nq, first * 128) * d * 2, what
            assert p["zeroed_dkdv_bytes"] == 2 * B * Hkv * (Nk - min(Nk, used * 128)) * d * 2, what
            assert p["workspace_bytes"] == B * H * Nq * 4, what
            assert (p["kv_cta_pair"], p["kv_passes"]) == (int(d == 128), 2 if d == 256 else 1), what
            assert p["launches"] == 2 + p["kv_passes"], what


def test_bwd_plan_rows_that_see_no_key_are_exactly_the_zeroed_ones():
    """Bottom-right with Nq > Nk: rows i < Nq - Nk see nothing.  The zeroed
    dQ rows are whole leading tiles of such rows; the rest of them (in the
    first live tile) are left to the kernel, which writes zeros there."""
    for Nq, Nk in [(300, 100), (1000, 1), (129, 1), (256, 128), (257, 128)]:
        p = bwd_plan(1, 1, 1, Nq, Nk, 64, fa.FA_CAUSAL_BOTTOM_RIGHT)
        dead_rows = Nq - Nk
        assert p["q_tile_first"] == dead_rows // 128
        assert p["zeroed_dq_bytes"] == min(Nq, p["q_tile_first"] * 128) * 64 * 2
        assert p["kv_tiles_used"] == math.ceil(Nk / 128)
