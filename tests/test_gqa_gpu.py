"""Grouped-query attention on the GPU (fa_fwd_gqa and fa_bwd_gqa through the
C ABI) against the fp64 oracle: H query heads share Hkv key/value heads,
dK and dV of a shared head sum over its query heads."""

import numpy as np
import pytest

from exact_attention_92_gb300 import inputs
from oracle import attention as att

from gpu_util import dev, ensure_built, host, torch_cuda
from parity import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    torch_cuda()
    return ensure_built()


def make_gqa(B, H, Hkv, N, d, seed):
    """Seeded N(0,1) bf16 inputs: q, dO of H heads, k, v of Hkv heads (bits
    and their fp64 values)."""
    rng = np.random.default_rng(seed)
    q = inputs.normal_bits(rng, (B, H, N, d))
    k = inputs.normal_bits(rng, (B, Hkv, N, d))
    v = inputs.normal_bits(rng, (B, Hkv, N, d))
    do = inputs.normal_bits(rng, (B, H, N, d))
    return (q, k, v, do), tuple(inputs.bits_to_f64(x) for x in (q, k, v, do))


SHAPES = [(2, 8, 2, 300, 64), (1, 4, 1, 257, 128), (2, 6, 3, 128, 128), (1, 8, 4, 640, 64), (1, 2, 1, 1, 128)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gqa_forward_and_backward(fa, shape, causal):
    torch = torch_cuda()
    B, H, Hkv, N, d = shape
    bits, (Q, K, V, DO) = make_gqa(B, H, Hkv, N, d, seed=700 + N + d + H + Hkv)
    q, k, v, do = (dev(x) for x in bits)
    scale = 1.0 / np.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa.fa_fwd_gqa(q, k, v, o, lse, causal)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.fa_bwd_gqa(q, k, v, o, lse, do, dq, dk, dv, causal)
    st = fa.fa_poll_status()
    assert st == 0, fa.fa_strerror(st)
    what = f"{shape} causal={causal}"
    O, L = att.forward_gqa(Q, K, V, scale, causal)
    Vx = att.expand_kv(V, H)
    Kx = att.expand_kv(K, H)

    def row_weights(ix):
        b, h, r = ix
        P = att.probabilities_head(Q[b, h], Kx[b, h], scale, causal, rows=[r])[0]
        return P, Vx[b, h]

    check_o(host(o), O, what, row_weights)
    check_lse(lse.cpu().numpy().astype(np.float64), L, what)
    rq, rk, rv = att.backward_gqa(Q, K, V, DO, scale, causal)
    check_grad(host(dq), rq, "dQ", what)
    check_grad(host(dk), rk, "dK", what)
    check_grad(host(dv), rv, "dV", what)


def test_gqa_with_hkv_equal_h_is_fa_fwd_fa_bwd(fa):
    """Hkv = H through the grouped entry points gives the same bits as fa_fwd
    and fa_bwd."""
    torch = torch_cuda()
    bits, _ = make_gqa(2, 3, 3, 333, 128, seed=77)
    q, k, v, do = (dev(x) for x in bits)
    outs = []
    for grouped in (False, True):
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        if grouped:
            fa.fa_fwd_gqa(q, k, v, o, lse, True)
            fa.fa_bwd_gqa(q, k, v, o, lse, do, dq, dk, dv, True)
        else:
            fa.fa_fwd(q, k, v, o, lse, True)
            fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, True)
        outs.append([t.clone() for t in (o, lse, dq, dk, dv)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_mqa_long_sequence_sampled(fa):
    """MQA (Hkv = 1) at N = 4096, d = 128, causal: 8 query heads, one
    key/value head; O and L on seeded rows of every head, dK and dV of the
    shared head in full."""
    torch = torch_cuda()
    B, H, Hkv, N, d = 1, 8, 1, 4096, 128
    bits, (Q, K, V, DO) = make_gqa(B, H, Hkv, N, d, seed=4096)
    q, k, v, do = (dev(x) for x in bits)
    scale = 1.0 / np.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa.fa_fwd_gqa(q, k, v, o, lse, True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.fa_bwd_gqa(q, k, v, o, lse, do, dq, dk, dv, True)
    st = fa.fa_poll_status()
    assert st == 0, fa.fa_strerror(st)
    rows = inputs.sample_rows_per_head(4096, B, H, N)
    Kx, Vx = att.expand_kv(K, H), att.expand_kv(V, H)
    O, L = att.forward_rows(Q, Kx, Vx, scale, True, rows)
    og = np.take_along_axis(host(o), rows[..., None], axis=2)
    lg = np.take_along_axis(lse.cpu().numpy().astype(np.float64), rows, axis=2)
    def row_weights(ix):
        b, h, i = ix
        P = att.probabilities_head(Q[b, h], Kx[b, h], scale, True, rows=[rows[b, h, i]])[0]
        return P, Vx[b, h]

    check_o(og, O, "MQA sampled rows", row_weights)
    check_lse(lg, L, "MQA sampled rows")
    _, rk, rv = att.backward_gqa(Q, K, V, DO, scale, True)
    check_grad(host(dk), rk, "dK", "MQA")
    check_grad(host(dv), rv, "dV", "MQA")
