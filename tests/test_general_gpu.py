"""Queries and keys of different lengths (both causal alignments), head dim
96, and their combinations with grouped-query attention and key splits, on
the GPU against the fp64 oracle (through the C ABI: fa_fwd_general,
fa_bwd_general)."""

import numpy as np
import pytest

from exact_attention_92_gb300 import inputs
from oracle import attention as att

from gpu_util import dev, ensure_built, host, torch_cuda
from parity import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu

CAUSAL = {"none": (False, None), "top_left": (True, "top_left"), "bottom_right": (True, "bottom_right")}


@pytest.fixture(scope="module")
def fa():
    torch_cuda()
    return ensure_built()


def make(B, H, Hkv, Nq, Nk, d, seed, with_do=False):
    """Seeded bf16 Q, dO [B,H,Nq,d] and K, V [B,Hkv,Nk,d] (bit patterns)."""
    rng = np.random.default_rng(seed)
    q = inputs.normal_bits(rng, (B, H, Nq, d))
    k = inputs.normal_bits(rng, (B, Hkv, Nk, d))
    v = inputs.normal_bits(rng, (B, Hkv, Nk, d))
    do = inputs.normal_bits(rng, (B, H, Nq, d)) if with_do else None
    return q, k, v, do


def f64(bits):
    return inputs.bits_to_f64(bits)


def offset_of(mode, Nq, Nk):
    causal, align = CAUSAL[mode]
    return causal, (att.causal_offset(Nq, Nk, align) if causal else 0)


def run_fwd(fa, q, k, v, mode, num_splits=0):
    torch = torch_cuda()
    tq, tk, tv = dev(q), dev(k), dev(v)
    B, H, Nq, d = q.shape
    o = torch.empty_like(tq)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    fa.fa_fwd_general(tq, tk, tv, o, lse, mode, None, num_splits)
    st = fa.fa_poll_status()
    assert st == 0, fa.fa_strerror(st)
    return host(o), lse.cpu().numpy().astype(np.float64), (tq, tk, tv, o, lse)


def oracle_fwd(q, k, v, mode, rows=None):
    B, H, Nq, d = q.shape
    causal, off = offset_of(mode, Nq, k.shape[2])
    Q, K, V = f64(q), att.expand_kv(f64(k), H), att.expand_kv(f64(v), H)
    scale = 1 / np.sqrt(d)
    if rows is None:
        O, L = att.forward(Q, K, V, scale, causal, off)
    else:
        O, L = att.forward_rows(Q, K, V, scale, causal, rows, off)

    def weights(ix):
        b, h, r = ix
        row = int(rows[r]) if rows is not None else int(r)
        P = att.probabilities_head(Q[b, h], K[b, h], scale, causal, rows=np.array([row]), offset=off)[0]
        return P, V[b, h]

    return O, L, weights


FWD_SHAPES = [
    # (B, H, Hkv, Nq, Nk, d)
    (1, 2, 2, 1, 8192, 128), (1, 2, 2, 128, 8192, 128), (1, 2, 2, 1000, 8192, 128),
    (1, 2, 2, 1000, 8192, 64), (1, 2, 2, 1000, 8192, 96), (2, 2, 2, 1, 8192, 96),
    (1, 1, 1, 300, 100, 128), (1, 2, 2, 257, 130, 64), (2, 3, 3, 200, 200, 96),
    (1, 1, 1, 1000, 1000, 96), (1, 4, 2, 200, 700, 96), (1, 4, 1, 129, 383, 64),
    # head dim 256 (its own kernel: one query tile per CTA, 64-key tiles)
    (1, 2, 2, 1, 8192, 256), (1, 2, 2, 128, 8192, 256), (1, 2, 2, 1000, 8192, 256),
    (1, 1, 1, 300, 100, 256), (2, 3, 3, 200, 200, 256), (1, 4, 2, 200, 700, 256), (1, 1, 1, 63, 63, 256),
    # grouped query heads with fewer than 128 query rows: the heads of a group share a tile
    (2, 8, 2, 1, 4096, 128), (1, 8, 2, 37, 1000, 64), (1, 32, 1, 3, 5000, 96), (1, 4, 1, 5, 3000, 256),
    (1, 6, 2, 100, 60, 128), (2, 4, 2, 127, 129, 128),
    # a few rows per key/value head (decoding steps), grouped and not: 2 x 4, 5, 3, 8 x 1, 8 rows
    (1, 8, 2, 2, 3000, 64), (1, 1, 1, 5, 700, 128), (3, 4, 4, 3, 1000, 64), (1, 16, 2, 1, 257, 128),
    (2, 2, 2, 8, 33, 128),
    # single-tile units over long keys: both query tiles of a CTA take a unit's rows and split its
    # key tiles (even / odd), with an odd count per split, a ragged last key tile, 100 and 64 rows
    (4, 32, 8, 1, 8192, 64), (2, 16, 16, 100, 4000, 128), (8, 8, 8, 64, 6000, 96),
]


@pytest.mark.parametrize("mode", ["none", "top_left", "bottom_right"])
@pytest.mark.parametrize("shape", FWD_SHAPES, ids=lambda s: "B{}H{}Hkv{}Nq{}Nk{}d{}".format(*s))
def test_forward(fa, shape, mode):
    B, H, Hkv, Nq, Nk, d = shape
    q, k, v, _ = make(B, H, Hkv, Nq, Nk, d, seed=7000 + Nq + 3 * Nk + d)
    o, lse, _ = run_fwd(fa, q, k, v, mode)
    O, L, weights = oracle_fwd(q, k, v, mode)
    what = f"{shape} {mode}"
    check_o(o, O, what, weights)
    check_lse(lse, L, what)
    causal, off = offset_of(mode, Nq, Nk)
    if causal and off < 0:
        # rows that see no key: O = 0 exactly
        assert np.all(o[:, :, :-off] == 0.0), what


@pytest.mark.parametrize("d", [64, 128])
def test_decoding_runs_dual_tiles(fa, d):
    """GQA decoding at scale (B=8, 32 query heads over 8 key/value heads, one
    query row, 8192 keys): the automatic plan puts both query tiles of a CTA
    on a unit's rows (each tile writes a partial, so the merge kernel runs)
    and the result matches the oracle."""
    before = fa.fa_launch_count(fa.FA_KERNEL_COMBINE)
    q, k, v, _ = make(8, 32, 8, 1, 8192, d, seed=7300 + d)
    o, lse, _ = run_fwd(fa, q, k, v, "bottom_right")
    assert fa.fa_launch_count(fa.FA_KERNEL_COMBINE) == before + 1
    O, L, weights = oracle_fwd(q, k, v, "bottom_right")
    check_o(o, O, f"decode d={d}", weights)
    check_lse(lse, L, f"decode d={d}")


@pytest.mark.parametrize("shape", [(1, 2, 2, 300, 4000, 96, "top_left"), (8, 32, 8, 1, 8192, 128, "bottom_right"),
                                   (2, 4, 4, 1000, 1000, 256, "none"), (1, 4, 2, 300, 100, 128, "bottom_right"),
                                   (1, 1, 1, 65536, 65536, 128, "top_left")],
                         ids=lambda s: "B{}H{}Hkv{}Nq{}Nk{}d{}-{}".format(*s))
def test_calls_follow_their_plans(fa, shape):
    """fa_fwd_general and fa_bwd_general launch what fa_fwd_plan and
    fa_bwd_plan report for this device: the merge exactly when partial
    results are planned, two key/value passes at head dim 256."""
    torch = torch_cuda()
    B, H, Hkv, Nq, Nk, d, mode = shape
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    sm, l2 = props.multi_processor_count, getattr(props, "L2_cache_size", 126 << 20)
    fplan = fa.fa_fwd_plan(B, H, Hkv, Nq, Nk, d, mode, 0, sm, l2)
    bplan = fa.fa_bwd_plan(B, H, Hkv, Nq, Nk, d, mode, sm)
    q, k, v, do = make(B, H, Hkv, Nq, Nk, d, seed=7400 + Nq + d, with_do=True)
    kernels = (fa.FA_KERNEL_FWD, fa.FA_KERNEL_COMBINE, fa.FA_KERNEL_BWD_PRE, fa.FA_KERNEL_BWD, fa.FA_KERNEL_BWD_DQ)
    before = [fa.fa_launch_count(kid) for kid in kernels]
    _, _, (tq, tk, tv, o, lse) = run_fwd(fa, q, k, v, mode)
    tdo = dev(do)
    dq, dk, dv = torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv)
    fa.fa_bwd_general(tq, tk, tv, o, lse, tdo, dq, dk, dv, mode)
    assert fa.fa_poll_status() == fa.FA_OK
    got = [fa.fa_launch_count(kid) - b for kid, b in zip(kernels, before)]
    assert got == [1, 1 if fplan["partials"] else 0, 1, bplan["kv_passes"], 1], (got, fplan, bplan)
    assert fplan["launches"] == got[0] + got[1] and bplan["launches"] == sum(got[2:])


@pytest.mark.parametrize("d", [96, 256])
@pytest.mark.parametrize("splits", [1, 3, 16])
@pytest.mark.parametrize("mode", ["top_left", "bottom_right"])
def test_forward_forced_splits(fa, mode, splits, d):
    q, k, v, _ = make(1, 2, 2, 300, 4000, d, seed=7100 + splits + d)
    o, lse, _ = run_fwd(fa, q, k, v, mode, splits)
    O, L, weights = oracle_fwd(q, k, v, mode)
    check_o(o, O, f"splits={splits} {mode}", weights)
    check_lse(lse, L, f"splits={splits} {mode}")


@pytest.mark.parametrize("mode", ["none", "top_left", "bottom_right"])
@pytest.mark.parametrize("c", [dict(B=16384 // N, H=2048 // d, N=N, d=d) for d in (96, 256) for N in (1024, 4096)],
                         ids=lambda c: f"B{c['B']}H{c['H']}N{c['N']}d{c['d']}")
def test_forward_16k_tokens_other_head_dims(fa, c, mode):
    """Head dims 96 and 256 at the 16K-token sweep's sizes (hidden 2016 = 21
    heads of 96, 2048 = 8 heads of 256), checked on 1024 seeded rows per
    head."""
    B, H, N, d = c["B"], c["H"], c["N"], c["d"]
    q, k, v, _ = make(B, H, H, N, N, d, seed=7200 + N + d)
    o, lse, _ = run_fwd(fa, q, k, v, mode)
    rows = inputs.sample_rows(7200 + N, N)
    O, L, weights = oracle_fwd(q, k, v, mode, rows)
    check_o(o[:, :, rows], O, f"{c} {mode}", weights)
    check_lse(lse[:, :, rows], L, f"{c} {mode}")


BWD_SHAPES = [
    (1, 2, 2, 1, 8192, 128), (1, 2, 2, 128, 8192, 64), (1, 1, 1, 1000, 8192, 96),
    (1, 2, 2, 1000, 8192, 128), (1, 1, 1, 300, 100, 128), (1, 2, 2, 257, 130, 96),
    (2, 3, 3, 200, 200, 96), (1, 1, 1, 640, 640, 96), (1, 4, 2, 200, 700, 96), (1, 4, 1, 129, 383, 64),
    # head dim 256 (its own kernels: dV and dK passes over 64-row query steps, dQ over 64-key steps)
    (1, 1, 1, 1, 4096, 256), (1, 2, 2, 1000, 4096, 256), (1, 1, 1, 300, 100, 256), (2, 3, 3, 200, 200, 256),
    (1, 4, 2, 200, 700, 256), (1, 1, 1, 63, 63, 256), (1, 2, 2, 640, 640, 256),
    (1, 8, 2, 37, 1000, 64), (1, 6, 2, 100, 60, 128), (1, 8, 2, 300, 1000, 256), (2, 4, 1, 70, 50, 256),
    # head dim 128, whose dK/dV run on CTA pairs (two neighbouring key tiles a unit): an odd number of key
    # tiles (the last pair's second tile past Nk), grouped heads, more query rows than keys
    (1, 2, 2, 640, 640, 128), (1, 4, 2, 200, 700, 128), (1, 2, 2, 700, 389, 128), (2, 3, 3, 257, 513, 128),
]


@pytest.mark.parametrize("mode", ["none", "top_left", "bottom_right"])
@pytest.mark.parametrize("shape", BWD_SHAPES, ids=lambda s: "B{}H{}Hkv{}Nq{}Nk{}d{}".format(*s))
def test_backward(fa, shape, mode):
    torch = torch_cuda()
    B, H, Hkv, Nq, Nk, d = shape
    q, k, v, do = make(B, H, Hkv, Nq, Nk, d, seed=7300 + Nq + 3 * Nk + d, with_do=True)
    _, _, (tq, tk, tv, o, lse) = run_fwd(fa, q, k, v, mode)
    tdo = dev(do)
    dq, dk, dv = torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv)
    # Every gradient element is written, including the rows no key / query
    # reaches: start from NaN so that a missed row shows.
    for t in (dq, dk, dv):
        t.fill_(float("nan"))
    fa.fa_bwd_general(tq, tk, tv, o, lse, tdo, dq, dk, dv, mode)
    st = fa.fa_poll_status()
    assert st == 0, fa.fa_strerror(st)
    causal, off = offset_of(mode, Nq, Nk)
    rq, rk, rv = att.backward_gqa(f64(q), f64(k), f64(v), f64(do), 1 / np.sqrt(d), causal, off)
    what = f"{shape} {mode}"
    check_grad(host(dq), rq, "dQ", what)
    check_grad(host(dk), rk, "dK", what)
    check_grad(host(dv), rv, "dV", what)
    if causal and off < 0:
        assert np.all(host(dq)[:, :, :-off] == 0.0), what
    if causal and Nq - 1 + off < Nk - 1:
        # keys past the last one the last query row sees: zero gradients
        assert np.all(host(dk)[:, :, Nq + off:] == 0.0) and np.all(host(dv)[:, :, Nq + off:] == 0.0), what


@pytest.mark.parametrize("causal", [False, True])
def test_backward_d96_b8_h21_n2048(fa, causal):
    """Head dim 96 backward at N = 2048 (B=8, H=21): dK, dV in full on 3
    seeded heads, dQ on 1024 seeded rows of every head."""
    torch = torch_cuda()
    B, H, N, d = 8, 21, 2048, 96
    case = inputs.make_case(B, H, N, d, causal, seed=7400 + int(causal), with_do=True)
    tq, tk, tv, tdo = dev(case.q), dev(case.k), dev(case.v), dev(case.do)
    o, lse = fa.forward(tq, tk, tv, causal=causal)
    dq, dk, dv = fa.backward(tq, tk, tv, o, lse, tdo, causal=causal)
    assert fa.fa_poll_status() == 0
    dq, dk, dv = host(dq), host(dk), host(dv)
    Q, K, V, DO = (case.f64(n) for n in ("q", "k", "v", "do"))
    rng = np.random.default_rng(case.seed + 11)
    for i in rng.choice(B * H, 3, replace=False):
        b, h = int(i) // H, int(i) % H
        rq, rk, rv = att.backward_head(Q[b, h], K[b, h], V[b, h], DO[b, h], case.scale, causal)
        check_grad(dk[b, h], rk, "dK", f"head {(b, h)}")
        check_grad(dv[b, h], rv, "dV", f"head {(b, h)}")
    rows = inputs.sample_rows_per_head(case.seed, B, H, N)
    for b in range(B):
        for h in range(H):
            ref = att.backward_dq_rows_head(Q[b, h], K[b, h], V[b, h], DO[b, h], case.scale, causal, rows[b, h])
            check_grad(dq[b, h, rows[b, h]], ref, "dQ", f"head {(b, h)}")


@pytest.mark.parametrize("causal", [False, True])
def test_backward_d256_b2_h8_n2048(fa, causal):
    """Head dim 256 backward at N = 2048 (B=2, H=8, hidden 2048): dK, dV in
    full on 3 seeded heads, dQ on 1024 seeded rows of every head."""
    B, H, N, d = 2, 8, 2048, 256
    case = inputs.make_case(B, H, N, d, causal, seed=7600 + int(causal), with_do=True)
    tq, tk, tv, tdo = dev(case.q), dev(case.k), dev(case.v), dev(case.do)
    o, lse = fa.forward(tq, tk, tv, causal=causal)
    dq, dk, dv = fa.backward(tq, tk, tv, o, lse, tdo, causal=causal)
    assert fa.fa_poll_status() == 0
    dq, dk, dv = host(dq), host(dk), host(dv)
    Q, K, V, DO = (case.f64(n) for n in ("q", "k", "v", "do"))
    rng = np.random.default_rng(case.seed + 11)
    for i in rng.choice(B * H, 3, replace=False):
        b, h = int(i) // H, int(i) % H
        rq, rk, rv = att.backward_head(Q[b, h], K[b, h], V[b, h], DO[b, h], case.scale, causal)
        check_grad(dk[b, h], rk, "dK", f"head {(b, h)}")
        check_grad(dv[b, h], rv, "dV", f"head {(b, h)}")
    rows = inputs.sample_rows_per_head(case.seed, B, H, N)
    for b in range(B):
        for h in range(H):
            ref = att.backward_dq_rows_head(Q[b, h], K[b, h], V[b, h], DO[b, h], case.scale, causal, rows[b, h])
            check_grad(dq[b, h, rows[b, h]], ref, "dQ", f"head {(b, h)}")


@pytest.mark.parametrize("d", [96, 256])
def test_general_repeatable(fa, d):
    """No atomics with unequal lengths either: identical bits run to run."""
    torch = torch_cuda()
    q, k, v, do = make(1, 4, 2, 333, 1111, d, seed=7500, with_do=True)
    outs = []
    for _ in range(2):
        _, _, (tq, tk, tv, o, lse) = run_fwd(fa, q, k, v, "bottom_right")
        grads = fa.backward(tq, tk, tv, o, lse, dev(do), causal="bottom_right")
        torch.cuda.synchronize()
        outs.append([o, lse, *grads])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
