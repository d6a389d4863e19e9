"""The C ABI library without a GPU: it loads, exports every entry point
include/fa.h declares, and rejects bad arguments on the host before any
device work (no compute call is made here)."""

import ctypes
import os
import subprocess

import pytest

import exact_attention_92_gb300 as fa
from exact_attention_92_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa.load()


def test_exports_every_declared_symbol(lib):
    declared = fa.declared_symbols()
    assert {"fa_fwd", "fa_fwd_ex", "fa_bwd", "fa_poll_status", "fa_strerror", "fa_abi_version"} <= set(declared)
    out = subprocess.run(["nm", "-D", "--defined-only", _binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [s for s in declared if s not in exported]
    assert not missing, missing
    for s in declared:
        assert hasattr(lib, s)


def test_no_driver_dependency():
    out = subprocess.run(["ldd", _binding.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart" not in out


def test_version_and_strerror(lib):
    assert fa.fa_abi_version() == 5
    for code in range(6):
        assert fa.fa_strerror(code).startswith("FA_")
    assert "unknown" in fa.fa_strerror(99)


P = ctypes.c_void_p


def _fwd(lib, q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=1, N=128, d=64, causal=0,
         scale=0.125, splits=0):
    return lib.fa_fwd_ex(P(q), P(k), P(v), P(o), P(lse), B, H, N, d, causal, scale, splits, None)


def test_fwd_argument_errors(lib):
    assert _fwd(lib, q=0) == fa.FA_ERR_INVALID_ARG          # null
    assert _fwd(lib, k=0x2008) == fa.FA_ERR_INVALID_ARG     # not 16-byte aligned
    assert _fwd(lib, lse=0x5004) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, B=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, N=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, H=-3) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("inf")) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, splits=-1) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, d=32) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, d=80) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, d=512) == fa.FA_ERR_UNSUPPORTED


def test_general_argument_errors(lib):
    """fa_fwd_general / fa_bwd_general: lengths, causal codes and head counts
    are checked on the host before anything touches a device."""
    ptrs = [P(0x1000 * (i + 1)) for i in range(9)]

    def fwd(B=1, H=4, Hkv=2, Nq=100, Nk=300, d=96, causal=2, scale=0.1, splits=0):
        return lib.fa_fwd_general(*ptrs[:5], B, H, Hkv, Nq, Nk, d, causal, scale, splits, None)

    def bwd(B=1, H=4, Hkv=2, Nq=100, Nk=300, d=96, causal=2, scale=0.1):
        return lib.fa_bwd_general(*ptrs, B, H, Hkv, Nq, Nk, d, causal, scale, None)

    for call in (fwd, bwd):
        assert call(Nq=0) == fa.FA_ERR_INVALID_ARG
        assert call(Nk=0) == fa.FA_ERR_INVALID_ARG
        assert call(causal=3) == fa.FA_ERR_INVALID_ARG
        assert call(causal=-1) == fa.FA_ERR_INVALID_ARG
        assert call(Hkv=3) == fa.FA_ERR_INVALID_ARG
        assert call(d=48) == fa.FA_ERR_UNSUPPORTED
        assert call(scale=0.0) == fa.FA_ERR_INVALID_ARG
        assert call(B=1 << 16, H=1 << 10, Nq=1 << 10) == fa.FA_ERR_INVALID_ARG  # 2^36 query rows
    assert fwd(splits=-2) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_noalloc(*ptrs, 1, 1, 128, 256, 1, 0.06, None) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_general(*ptrs[:4], P(0x5004), 1, 4, 2, 100, 300, 96, 2, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert fa.FA_CAUSAL_NONE == 0 and fa.FA_CAUSAL_TOP_LEFT == 1 and fa.FA_CAUSAL_BOTTOM_RIGHT == 2


def test_gqa_argument_errors(lib):
    """Key/value head counts that do not divide the query heads are refused
    before anything touches a device."""
    ptrs = [P(0x1000 * (i + 1)) for i in range(9)]
    for hkv in (0, -1, 3, 5):
        assert lib.fa_fwd_gqa(*ptrs[:5], 2, 8, hkv, 256, 64, 1, 0.125, 0, None) == fa.FA_ERR_INVALID_ARG
        assert lib.fa_bwd_gqa(*ptrs, 2, 8, hkv, 256, 64, 1, 0.125, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_gqa(P(0), *ptrs[1:5], 2, 8, 2, 256, 64, 1, 0.125, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_gqa(*ptrs[:8], P(0x9008), 2, 8, 2, 256, 64, 1, 0.125, None) == fa.FA_ERR_INVALID_ARG


def test_bwd_argument_errors(lib):
    ptrs = [P(0x1000 * (i + 1)) for i in range(9)]

    def call(ptrs=ptrs, B=1, H=1, N=64, d=64, scale=0.125):
        return lib.fa_bwd(*ptrs, B, H, N, d, 1, scale, None)

    for i in range(9):
        bad = list(ptrs)
        bad[i] = P(0)
        assert call(bad) == fa.FA_ERR_INVALID_ARG
        bad[i] = P(0x1000 * (i + 1) + 2)
        assert call(bad) == fa.FA_ERR_INVALID_ARG
    assert call(N=0) == fa.FA_ERR_INVALID_ARG
    assert call(d=32) == fa.FA_ERR_UNSUPPORTED
    assert call(scale=0.0) == fa.FA_ERR_INVALID_ARG


def test_timing_read_argument_errors(lib):
    n = ctypes.c_int()
    ms = ctypes.c_double()
    assert lib.fa_timing_read(7, ctypes.byref(n), ctypes.byref(ms)) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_timing_read(0, None, ctypes.byref(ms)) == fa.FA_ERR_INVALID_ARG


def test_launch_count_arguments(lib):
    """The launch counter is host-side: it answers without a GPU and rejects
    bad ids and null pointers."""
    n = ctypes.c_uint64(123)
    assert lib.fa_launch_count(0, ctypes.byref(n)) == fa.FA_OK
    assert n.value >= 0
    assert lib.fa_launch_count(5, ctypes.byref(n)) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_launch_count(-1, ctypes.byref(n)) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_launch_count(0, None) == fa.FA_ERR_INVALID_ARG


def test_python_binding_rejects_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.forward(q, q, q)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "libfa.so"))
    with pytest.raises(fa.FaError):
        _binding.load()


def test_build_refuses_spills_in_tmem_kernels():
    """A spill between tcgen05.ld and its wait would store garbage: the build
    rejects any spill in the kernels that read tensor memory."""
    bad = ("ptxas info    : Compiling entry function '_ZN2fa18fa_bwd_dkdv_kernelILi128EEEv' for 'sm_103a'\n"
           "    64 bytes stack frame, 32 bytes spill stores, 36 bytes spill loads\n")
    with pytest.raises(RuntimeError):
        build.check_spills(bad)
    ok = ("ptxas info    : Compiling entry function '_ZN2fa13fa_fwd_kernelILi64EEEv' for 'sm_103a'\n"
          "    24 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads\n"
          "ptxas info    : Compiling entry function '_ZN2fa17fa_bwd_preprocessILi64EEEv' for 'sm_103a'\n"
          "    8 bytes stack frame, 8 bytes spill stores, 8 bytes spill loads\n")
    build.check_spills(ok)


def _prototypes():
    """(name, return type, parameter list) of every function include/fa.h declares."""
    import re

    text = open(_binding.HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    protos = {}
    for m in re.finditer(r"(int|uint64_t|const char\s*\*)\s+(fa_\w+)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(3).split(",") if p.strip() and p.strip() != "void"]
        protos[m.group(2)] = (m.group(1).replace(" ", ""), params)
    return protos


def test_binding_signatures_match_the_header():
    """Every ctypes signature of the binding has the header's parameter count
    and types (pointers as pointers, 64-bit integers as 64-bit), so a drift
    between fa.h and _binding.py cannot pass arguments in the wrong slots."""
    protos = _prototypes()
    assert set(protos) == set(fa.declared_symbols())
    assert set(protos) == set(_binding._SIGNATURES), set(protos) ^ set(_binding._SIGNATURES)
    ret = {"int": ctypes.c_int, "uint64_t": ctypes.c_uint64, "constchar*": ctypes.c_char_p}
    for name, (rtype, params) in protos.items():
        args, res = _binding._SIGNATURES[name]
        assert res is ret[rtype], name
        assert len(args) == len(params), (name, len(args), params)
        for a, p in zip(args, params):
            if "*" in p:
                assert a is ctypes.c_void_p or issubclass(a, ctypes._Pointer), (name, p, a)
            elif p.startswith("uint64_t"):
                assert a is ctypes.c_uint64, (name, p, a)
            elif p.startswith("float"):
                assert a is ctypes.c_float, (name, p, a)
            else:
                assert p.startswith("int") and a is ctypes.c_int, (name, p, a)


C_CLIENT = r"""
#include <stdio.h>
#include "fa.h"

int main(void) {
  fa_fwd_plan_t f;
  fa_bwd_plan_t b;
  if (fa_abi_version() != FA_ABI_VERSION) return 10;
  /* GQA decoding, 8 x 32 query heads over 8 key/value heads, 8192 keys. */
  if (fa_fwd_plan(8, 32, 8, 1, 8192, 128, FA_CAUSAL_BOTTOM_RIGHT, 0, 152, 132120576ull, &f) != FA_OK) return 11;
  if (fa_bwd_plan(1, 4, 2, 300, 100, 128, FA_CAUSAL_BOTTOM_RIGHT, 152, &b) != FA_OK) return 12;
  if (fa_fwd_plan(1, 1, 1, 128, 128, 48, 0, 0, 152, 0, &f) != FA_ERR_UNSUPPORTED) return 13;
  if (fa_fwd(0, 0, 0, 0, 0, 1, 1, 128, 64, 0, 0.125f, 0) != FA_ERR_INVALID_ARG) return 14;
  printf("%d %d %d %llu %d %d\n", f.packed_heads, f.dual, f.partials, (unsigned long long)f.workspace_bytes,
         b.q_tile_first, b.launches);
  printf("%s\n", fa_strerror(FA_ERR_NO_MEMORY));
  return 0;
}
"""


def test_header_is_plain_c(tmp_path, lib):
    """include/fa.h is a C header: a C99 program that includes it compiles
    with warnings as errors, links against libfa.so and calls the host-only
    entry points (plans, version, strerror, an argument check)."""
    import shutil

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(_binding.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), "-L", libdir, "-lfa", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stderr)
    first, second = out.stdout.splitlines()
    plan = fa.fa_fwd_plan(8, 32, 8, 1, 8192, 128, fa.FA_CAUSAL_BOTTOM_RIGHT, 0, 152, 132120576)
    bplan = fa.fa_bwd_plan(1, 4, 2, 300, 100, 128, fa.FA_CAUSAL_BOTTOM_RIGHT, 152)
    assert first.split() == [str(plan["packed_heads"]), str(plan["dual"]), str(plan["partials"]),
                             str(plan["workspace_bytes"]), str(bplan["q_tile_first"]), str(bplan["launches"])]
    assert second.startswith("FA_ERR_NO_MEMORY")


def test_build_checks_the_register_split_budget():
    """Kernels that move registers between warpgroups with setmaxnreg are
    launched with the per-thread count their split is sized for; an entry
    that ptxas gave any other count is refused (a warpgroup asking for more
    than the launch holds would wait forever)."""
    log = ("ptxas info    : Compiling entry function '_ZN2fa13fa_fwd_kernelILi128ELb0EEEv' for 'sm_103a'\n"
           "ptxas info    : Used {} registers, used 1 barriers, 0 bytes cmem[0]\n"
           "    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads\n")
    build.check_spills(log.format(build.REG_SPLIT_KERNELS["fa_fwd_kernel"]))
    for regs in (160, 176):
        with pytest.raises(RuntimeError):
            build.check_spills(log.format(regs))
    # A kernel without a register split may use any count.
    build.check_spills(log.replace("fa_fwd_kernel", "fa_combine_kernel").format(40))
