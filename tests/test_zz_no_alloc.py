"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory during the call.

fa_bwd takes its fp32 workspace from cudaMallocAsync on every call.  A
caller that has given almost all device memory to its own pool beforehand,
or whose memory budget is fixed when it starts, cannot let the library do
that; fa_bwd_noalloc uses a static device array instead.

These tests call it through the C ABI (ctypes, raw device pointers) and check
that two calls in a row give the same bits as fa_bwd (both run the same
deterministic kernels, so a stale or wrongly addressed workspace would show
as a difference), that such a call leaves the device's free memory
unchanged, and that a problem larger than the static array is refused before
any device work.  This file is collected last (its name), so a run that
stops at the first failure has run every other test before it.
"""

import ctypes

import numpy as np
import pytest

import exact_attention_92_gb300 as fa_mod
from exact_attention_92_gb300 import inputs

from gpu_util import case_tensors, ensure_built, host, torch_cuda

P = ctypes.c_void_p


def _call_noalloc(lib, q, k, v, o, lse, do, dq, dk, dv, causal, scale, stream):
    B, H, N, d = q.shape
    return lib.fa_bwd_noalloc(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), P(o.data_ptr()),
                              P(lse.data_ptr()), P(do.data_ptr()), P(dq.data_ptr()), P(dk.data_ptr()),
                              P(dv.data_ptr()), B, H, N, d, 1 if causal else 0, scale, P(stream))


@pytest.mark.gpu
@pytest.mark.parametrize("shape,causal", [((2, 4, 1000, 128), True), ((1, 2, 640, 128), False), ((1, 8, 640, 64), False),
                                          ((1, 3, 333, 96), True)])
def test_noalloc_matches_fa_bwd_on_two_calls(shape, causal):
    torch = torch_cuda()
    fa = ensure_built()
    lib = fa.load()
    B, H, N, d = shape
    case = inputs.make_case(B, H, N, d, causal, seed=900 + N, with_do=True)
    q, k, v, do = case_tensors(case)
    o, lse = fa.forward(q, k, v, causal=causal)
    ref = [host(t) for t in fa.backward(q, k, v, o, lse, do, causal=causal)]
    assert fa.fa_poll_status() == fa.FA_OK
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        st = _call_noalloc(lib, q, k, v, o, lse, do, dq, dk, dv, causal, case.scale, stream)
        # Read before the stream is synchronised: a stream-ordered allocation
        # would still hold its memory here.  The first call may load the
        # library's module (and with it the static array), so only the second
        # call is held to an unchanged figure.
        free_after = torch.cuda.mem_get_info()[0]
        assert st == fa.FA_OK, fa.fa_strerror(st)
        assert fa.fa_poll_status() == fa.FA_OK
        if call == 1:
            assert free_after == free_before, (free_before, free_after)
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert np.array_equal(host(got), want), f"fa_bwd_noalloc call {call + 1} vs fa_bwd, {shape}: {name}"


def test_noalloc_refuses_problems_beyond_the_scratch():
    fa = ensure_built()
    lib = fa.load()
    # The scratch holds D, one fp32 per row: 2 x 33 x 262144 rows x 4 bytes =
    # 69.2 MB > 64 MiB; refused on the host before any pointer is touched, so
    # placeholder addresses suffice.
    ptrs = [P(0x10000 * (i + 1)) for i in range(9)]
    need = 2 * 33 * 262144 * 4
    assert need > fa_mod.FA_BWD_NOALLOC_SCRATCH_BYTES
    st = lib.fa_bwd_noalloc(*ptrs, 2, 33, 262144, 128, 1, 0.088, None)
    assert st == fa.FA_ERR_SCRATCH_TOO_SMALL
    assert "scratch" in fa.fa_strerror(st)
