"""Failure detection on the GPU without a fault: a bounded device wait that
runs out records FA_ERR_TIMEOUT, the kernel returns, and the context stays
usable."""

import numpy as np
import pytest

from exact_attention_92_gb300 import inputs
from oracle import attention as att

from gpu_util import case_tensors, ensure_built, host, torch_cuda
from parity import check_grad, check_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    torch_cuda()
    return ensure_built()


def test_wait_gives_up_and_reports(fa):
    assert fa.fa_poll_status() == fa.FA_OK
    fa.fa_selftest_wait_timeout(50_000_000)  # 50 ms on a barrier nothing arrives on
    assert fa.fa_poll_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_poll_status() == fa.FA_OK  # read clears the word


def test_context_usable_after_timeout(fa):
    fa.fa_selftest_wait_timeout(10_000_000)
    assert fa.fa_poll_status() == fa.FA_ERR_TIMEOUT
    case = inputs.make_case(1, 2, 300, 64, True, seed=9)
    q, k, v, _ = case_tensors(case)
    o, lse = fa.forward(q, k, v, causal=True)
    assert fa.fa_poll_status() == fa.FA_OK
    O, _ = att.forward(case.f64("q"), case.f64("k"), case.f64("v"), case.scale, True)
    check_o(host(o), O, "after timeout")


def test_bad_arguments_raise_before_launch(fa):
    torch = torch_cuda()
    q = torch.zeros(1, 1, 64, 80, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.forward(q, q, q)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    q = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.forward(q, q, q, scale=float("nan"))
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    assert fa.fa_poll_status() == fa.FA_OK


def test_timing_counts_launches(fa):
    torch = torch_cuda()
    case = inputs.make_case(1, 2, 1024, 128, True, seed=3, with_do=True)
    q, k, v, do = case_tensors(case)
    fa.fa_timing_enable(True)
    o, lse = fa.forward(q, k, v, causal=True, num_splits=1)
    fa.backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    counts = {kid: fa.fa_timing_read(kid) for kid in range(5)}
    fa.fa_timing_enable(False)
    assert counts[fa.FA_KERNEL_FWD][0] == 1 and counts[fa.FA_KERNEL_FWD][1] > 0
    assert counts[fa.FA_KERNEL_COMBINE][0] == 0
    assert counts[fa.FA_KERNEL_BWD][0] == 1 and counts[fa.FA_KERNEL_BWD_PRE][0] == 1
    assert counts[fa.FA_KERNEL_BWD_DQ][0] == 1


def test_launch_counter_without_events(fa):
    """fa_launch_count advances by exactly the kernels a call launches, with
    per-launch timing off."""
    torch = torch_cuda()
    case = inputs.make_case(1, 2, 1024, 128, True, seed=4, with_do=True)
    q, k, v, do = case_tensors(case)
    before = [fa.fa_launch_count(kid) for kid in range(5)]
    o, lse = fa.forward(q, k, v, causal=True, num_splits=1)
    fa.backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    after = [fa.fa_launch_count(kid) for kid in range(5)]
    delta = [a - b for a, b in zip(after, before)]
    assert delta[fa.FA_KERNEL_FWD] == 1 and delta[fa.FA_KERNEL_COMBINE] == 0
    assert delta[fa.FA_KERNEL_BWD_PRE] == 1 and delta[fa.FA_KERNEL_BWD] == 1 and delta[fa.FA_KERNEL_BWD_DQ] == 1


def test_workspace_allocation_failure_is_reported(fa, monkeypatch):
    """A workspace allocation that fails (injected on the host with
    FA_TEST_FAIL_ALLOC) is reported as FA_ERR_NO_MEMORY before any launch;
    the stream and the device stay usable and the next call is correct."""
    torch = torch_cuda()
    case = inputs.make_case(1, 2, 512, 64, True, seed=5, with_do=True)
    q, k, v, do = case_tensors(case)
    o, lse = fa.forward(q, k, v, causal=True)
    monkeypatch.setenv("FA_TEST_FAIL_ALLOC", "1")
    with pytest.raises(fa.FaError) as e:
        fa.backward(q, k, v, o, lse, do, causal=True)
    assert e.value.status == fa.FA_ERR_NO_MEMORY
    with pytest.raises(fa.FaError) as e:
        fa.forward(q, k, v, causal=True, num_splits=2)  # split partials need workspace
    assert e.value.status == fa.FA_ERR_NO_MEMORY
    monkeypatch.delenv("FA_TEST_FAIL_ALLOC")
    assert fa.fa_poll_status() == fa.FA_OK
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True)
    assert fa.fa_poll_status() == fa.FA_OK
    rq, rk, rv = att.backward(case.f64("q"), case.f64("k"), case.f64("v"), case.f64("do"), case.scale, True)
    for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        check_grad(host(g), r, name, "after an allocation failure")


def test_workspace_pool_keeps_memory_until_trimmed(fa):
    """The split partials of one 65536-token causal head come from the
    library's pool, which keeps them reserved across synchronisations (a
    second call maps nothing new) until fa_trim_workspace gives them back;
    a call after the trim takes memory again and gives the same bits."""
    torch = torch_cuda()
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    plan = fa.fa_fwd_plan(1, 1, 1, 65536, 65536, 128, fa.FA_CAUSAL_TOP_LEFT, 0, props.multi_processor_count,
                          getattr(props, "L2_cache_size", 126 << 20))
    assert plan["workspace_bytes"] > 0
    g = torch.Generator(device="cuda").manual_seed(77)
    q, k, v = (torch.randn((1, 1, 65536, 128), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    o1, lse1 = fa.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    o2, lse2 = fa.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    free2 = torch.cuda.mem_get_info()[0]
    fa.fa_trim_workspace()
    free3 = torch.cuda.mem_get_info()[0]
    o3, lse3 = fa.forward(q, k, v, causal=True)
    assert fa.fa_poll_status() == fa.FA_OK
    # The second call's outputs are new tensors from torch's cache (not the
    # device); the workspace came back from the library's pool.
    assert free1 - free2 <= o2.numel() * 2 + lse2.numel() * 4 + (8 << 20), (free1, free2)
    assert free3 - free2 >= plan["workspace_bytes"], (free2, free3, plan["workspace_bytes"])
    for a, b in ((o1, o2), (o1, o3), (lse1, lse2), (lse1, lse3)):
        assert torch.equal(a, b)
