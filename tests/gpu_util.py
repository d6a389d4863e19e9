"""Helpers of the GPU tests: moving seeded bf16 inputs to the device and
results back, and running the oracle on the same inputs."""

import numpy as np
import pytest

from exact_attention_92_gb300 import inputs


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def ensure_built():
    from exact_attention_92_gb300 import build

    build.build()
    import exact_attention_92_gb300 as fa

    fa.load()
    return fa


def dev(bits):
    torch = torch_cuda()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def case_tensors(case):
    q, k, v = dev(case.q), dev(case.k), dev(case.v)
    do = dev(case.do) if case.do is not None else None
    return q, k, v, do
