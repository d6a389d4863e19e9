"""Backward pass on the GPU against the fp64 oracle (through the C ABI)."""

import numpy as np
import pytest

from exact_attention_92_gb300 import inputs
from oracle import attention as att

from gpu_util import case_tensors, dev, ensure_built, host, torch_cuda
from parity import check_grad

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    torch_cuda()
    return ensure_built()


def run(fa, case):
    q, k, v, do = case_tensors(case)
    o, lse = fa.forward(q, k, v, causal=case.causal)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=case.causal)
    st = fa.fa_poll_status()
    assert st == 0, fa.fa_strerror(st)
    return host(dq), host(dk), host(dv)


SMALL = [(1, 1, 128, 64), (1, 2, 128, 128), (1, 1, 200, 128), (2, 2, 257, 64), (1, 1, 1, 64),
         (1, 1, 63, 128), (2, 1, 384, 128), (1, 3, 640, 64)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(fa, shape, causal):
    B, H, N, d = shape
    case = inputs.make_case(B, H, N, d, causal, seed=500 + N + d, with_do=True)
    dq, dk, dv = run(fa, case)
    rq, rk, rv = att.backward(case.f64("q"), case.f64("k"), case.f64("v"), case.f64("do"), case.scale, causal)
    what = f"{shape} causal={causal}"
    check_grad(dq, rq, "dQ", what)
    check_grad(dk, rk, "dK", what)
    check_grad(dv, rv, "dV", what)


def test_fwd_bwd_b2_h16_n4096_d128_causal(fa):
    """dK, dV in full on 8 seeded heads; dQ on 1024 seeded rows of every head."""
    c = inputs.workload_cases()[5][0]
    case = inputs.make_case(**c)
    dq, dk, dv = run(fa, case)
    q, k, v, do = case.f64("q"), case.f64("k"), case.f64("v"), case.f64("do")
    rng = np.random.default_rng(case.seed + 11)
    heads = [(int(i) // case.H, int(i) % case.H) for i in rng.choice(case.B * case.H, 8, replace=False)]
    rq, rk, rv = att.backward(q, k, v, do, case.scale, True, heads=heads)
    for b, h in heads:
        check_grad(dk[b, h], rk[b, h], "dK", f"head {(b, h)}")
        check_grad(dv[b, h], rv[b, h], "dV", f"head {(b, h)}")
    rows = inputs.sample_rows_per_head(case.seed, case.B, case.H, case.N)
    for b in range(case.B):
        for h in range(case.H):
            ref = att.backward_dq_rows_head(q[b, h], k[b, h], v[b, h], do[b, h], case.scale, True, rows[b, h])
            check_grad(dq[b, h, rows[b, h]], ref, "dQ", f"head {(b, h)}")
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()


@pytest.mark.parametrize("d", [64, 128])
def test_gradients_bitwise_repeatable(fa, d):
    """No atomics anywhere in the backward pass: two runs give identical bits."""
    case = inputs.make_case(2, 3, 777, d, True, seed=77, with_do=True)
    a = run(fa, case)
    b = run(fa, case)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_back_to_back_calls_on_shared_buffers(fa, d):
    """Forward and backward calls of two problems queued on one stream with no
    synchronisation, writing the same O and L: each call's gradients equal,
    bit for bit, those of the same problem run alone.  The backward's kernels
    may start before the kernel ahead of them in the stream has ended, so
    this checks that each waits for what it reads (the new O, the new D)."""
    torch = torch_cuda()
    cases = [inputs.make_case(2, 4, 1000, d, True, seed=300 + d + i, with_do=True) for i in range(2)]
    tens = [case_tensors(c) for c in cases]
    alone = []
    for q, k, v, do in tens:
        o, lse = fa.forward(q, k, v, causal=True)
        alone.append(fa.backward(q, k, v, o, lse, do, causal=True))
    torch.cuda.synchronize()
    q0 = tens[0][0]
    o = torch.empty_like(q0)
    lse = torch.empty(q0.shape[:3], dtype=torch.float32, device="cuda")
    outs = [tuple(torch.empty_like(q0) for _ in range(3)) for _ in range(6)]
    side = torch.cuda.Stream()  # the last three calls on a stream of their own
    side.wait_stream(torch.cuda.current_stream())
    for i, (dq, dk, dv) in enumerate(outs):
        q, k, v, do = tens[i % 2]
        st = side if i >= 3 else None
        if i == 3:
            side.wait_stream(torch.cuda.current_stream())
        fa.fa_fwd(q, k, v, o, lse, True, stream=st)
        fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, True, stream=st)
    torch.cuda.synchronize()
    assert fa.fa_poll_status() == fa.FA_OK
    for i, got in enumerate(outs):
        for name, x, y in zip(("dQ", "dK", "dV"), got, alone[i % 2]):
            assert torch.equal(x, y), f"call {i}: {name} differs from the problem run alone"


@pytest.mark.parametrize("d", [64, 128])
def test_outputs_only_16_byte_aligned(fa, d):
    """Gradient buffers that are 16- but not 32-byte aligned take the 16-byte
    store path; the results are the same bits as with aligned buffers."""
    torch = torch_cuda()
    case = inputs.make_case(1, 2, 300, d, True, seed=91, with_do=True)
    q, k, v, do = case_tensors(case)
    o, lse = fa.forward(q, k, v, causal=True)
    ref = fa.backward(q, k, v, o, lse, do, causal=True)
    n = q.numel()
    outs = []
    for _ in range(3):
        buf = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
        t = buf[8:].view(q.shape)  # 16 bytes past a 256-byte-aligned allocation
        assert t.data_ptr() % 32 == 16
        outs.append(t)
    fa.fa_bwd(q, k, v, o, lse, do, outs[0], outs[1], outs[2], True)
    torch.cuda.synchronize()
    assert fa.fa_poll_status() == fa.FA_OK
    for got, want in zip(outs, ref):
        assert torch.equal(got, want)


def test_many_heads_many_units_per_cta(fa):
    """272 heads at N=1024, d=64 causal: every persistent CTA walks many
    units of both backward kernels and of the forward kernel, across the last
    partial round.  O, L and the gradients of heads spread over the unit order
    match the oracle."""
    from parity import check_lse, check_o

    case = inputs.make_case(17, 16, 1024, 64, True, seed=601, with_do=True)
    q, k, v, do = case_tensors(case)
    o, lse = fa.forward(q, k, v, causal=True)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True)
    st = fa.fa_poll_status()
    assert st == 0, fa.fa_strerror(st)
    o, lse = host(o), lse.cpu().numpy().astype(np.float64)
    dq, dk, dv = host(dq), host(dk), host(dv)
    Q, K, V, DO = case.f64("q"), case.f64("k"), case.f64("v"), case.f64("do")
    for b, h in [(0, 0), (7, 9), (15, 15), (16, 0), (16, 7), (16, 15)]:
        what = f"head {(b, h)}"
        O, L = att.forward_head(Q[b, h], K[b, h], V[b, h], case.scale, True)

        def row_weights(ix, b=b, h=h):
            P = att.probabilities_head(Q[b, h], K[b, h], case.scale, True, rows=[ix[-1]])[0]
            return P, V[b, h]

        check_o(o[b, h][None, None], O[None, None], what, row_weights)
        check_lse(lse[b, h], L, what)
        rq, rk, rv = att.backward_head(Q[b, h], K[b, h], V[b, h], DO[b, h], case.scale, True)
        check_grad(dq[b, h], rq, "dQ", what)
        check_grad(dk[b, h], rk, "dK", what)
        check_grad(dv[b, h], rv, "dV", what)


def _sweep_case(N, d, causal):
    """The 16K-token sweep case with these sizes (its seed), with dO."""
    c = next(c for c in inputs.workload_cases()[3] if (c["N"], c["d"], c["causal"]) == (N, d, causal))
    return inputs.make_case(**c, with_do=True)


def _check_dq_rows(case, dq):
    q, k, v, do = case.f64("q"), case.f64("k"), case.f64("v"), case.f64("do")
    rows = inputs.sample_rows_per_head(case.seed, case.B, case.H, case.N)
    for b in range(case.B):
        for h in range(case.H):
            ref = att.backward_dq_rows_head(q[b, h], k[b, h], v[b, h], do[b, h], case.scale, case.causal, rows[b, h])
            check_grad(dq[b, h, rows[b, h]], ref, "dQ", f"head {(b, h)} sampled rows")


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_b4_h16_n4096_d128(fa, causal):
    """The backward the bench times at N = 4096: dK, dV in full on 4 seeded
    heads, dQ on 1024 seeded rows of every head."""
    case = _sweep_case(4096, 128, causal)
    dq, dk, dv = run(fa, case)
    q, k, v, do = case.f64("q"), case.f64("k"), case.f64("v"), case.f64("do")
    rng = np.random.default_rng(case.seed + 11)
    heads = [(int(i) // case.H, int(i) % case.H) for i in rng.choice(case.B * case.H, 4, replace=False)]
    rq, rk, rv = att.backward(q, k, v, do, case.scale, causal, heads=heads)
    for b, h in heads:
        check_grad(dk[b, h], rk[b, h], "dK", f"head {(b, h)}")
        check_grad(dv[b, h], rv[b, h], "dV", f"head {(b, h)}")
    _check_dq_rows(case, dq)
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_b1_h16_n16384_d128(fa, causal):
    """The backward the bench times at N = 16384: dK, dV on 1024 seeded key
    rows of 4 seeded heads, dQ on 1024 seeded rows of every head."""
    case = _sweep_case(16384, 128, causal)
    dq, dk, dv = run(fa, case)
    q, k, v, do = case.f64("q"), case.f64("k"), case.f64("v"), case.f64("do")
    rng = np.random.default_rng(case.seed + 11)
    for i in rng.choice(case.B * case.H, 4, replace=False):
        b, h = int(i) // case.H, int(i) % case.H
        keys = np.sort(rng.choice(case.N, inputs.SAMPLE_ROWS, replace=False))
        rk, rv = att.backward_dkdv_rows_head(q[b, h], k[b, h], v[b, h], do[b, h], case.scale, causal, keys)
        check_grad(dk[b, h, keys], rk, "dK", f"head {(b, h)} sampled key rows")
        check_grad(dv[b, h, keys], rv, "dV", f"head {(b, h)} sampled key rows")
    _check_dq_rows(case, dq)
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_b4_h16_n1024_d64(fa, causal):
    """Backward at the B=4 H=16 N=1024 d=64 shape, every head in full."""
    c = next(c for c in inputs.workload_cases()[2] if c["causal"] == causal and "degenerate" not in c)
    case = inputs.make_case(**c, with_do=True)
    dq, dk, dv = run(fa, case)
    rq, rk, rv = att.backward(case.f64("q"), case.f64("k"), case.f64("v"), case.f64("do"), case.scale, causal)
    for b in range(case.B):
        for h in range(case.H):
            what = f"head {(b, h)} causal={causal}"
            check_grad(dq[b, h], rq[b, h], "dQ", what)
            check_grad(dk[b, h], rk[b, h], "dK", what)
            check_grad(dv[b, h], rv[b, h], "dV", what)
