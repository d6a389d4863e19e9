"""Host logic of bench.py (no GPU): the source hash that ties a recorded
ncu traffic figure to the kernel sources it was taken on, the FLOP counts
behind the throughput figures, and the summary of the clock record."""

import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_code_only_drops_comments_and_keeps_literals():
    b = _bench()
    src = ('int a = 1;  // trailing\n'
           '/* block\n   comment */\n'
           '\n'
           'asm("x // not a comment /* nor this */");\n'
           "char c = '/';  /* after */ int d;\n")
    out = b._code_only(src)
    assert "trailing" not in out and "block" not in out and "after" not in out
    assert 'asm("x // not a comment /* nor this */");' in out
    assert "char c = '/';" in out and "int d;" in out
    assert "\n\n" not in out


def test_hash_ignores_comments_but_not_code():
    b = _bench()
    base = "int f(int x) {\n  return x + 1;  // one\n}\n"
    same = "// header\nint f(int x) {\n\n  return x + 1;  /* two */\n}\n"
    other = "int f(int x) {\n  return x + 2;\n}\n"
    asm_changed = 'asm("add %0, 1;");\n', 'asm("add %0, 2;");\n'
    assert b._code_only(base) == b._code_only(same)
    assert b._code_only(base) != b._code_only(other)
    assert b._code_only(asm_changed[0]) != b._code_only(asm_changed[1])


def test_every_timed_kernel_has_a_source_hash():
    b = _bench()
    for name in b.KERNEL_NAMES:
        h = b.kernel_source_hash(name)
        assert len(h) == 16 and int(h, 16) >= 0


def test_visible_pairs_by_enumeration():
    """The (query, key) pairs each causal alignment lets through, which the
    FLOP counts of the Nq != Nk cases use, against enumerating the mask."""
    b = _bench()
    for Nq, Nk in [(1, 1), (1, 9), (9, 1), (7, 7), (5, 12), (12, 5), (130, 64), (64, 300)]:
        assert b.visible_pairs(Nq, Nk, False, "top_left") == Nq * Nk
        for align, off in (("top_left", 0), ("bottom_right", Nk - Nq)):
            want = sum(1 for i in range(Nq) for j in range(Nk) if j <= i + off)
            assert b.visible_pairs(Nq, Nk, True, align) == want, (Nq, Nk, align)


def test_flop_convention():
    """Throughput counts the forward as 4 B H N^2 d FLOPs (two N x N x d
    products of 2 FLOPs a multiply-add), halved with the causal mask, and
    the backward as 2.5 times that (five such products instead of two)."""
    b = _bench()
    f, g = b.workload_flops(2, 16, 4096, 128, True)
    assert f == 4 * 2 * 16 * 4096 ** 2 * 128 / 2 and g == 2.5 * f
    assert round(f / 1e9, 1) == 137.4 and round(g / 1e9, 1) == 343.6
    f_nc, g_nc = b.workload_flops(1, 1, 1000, 64, False)
    assert f_nc == 4 * 1000 ** 2 * 64 and g_nc == 2.5 * f_nc


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_sampler_summary(tmp_path):
    """The clock record of a timed region: median SM clock over the samples
    under load (utilisation >= 50%), the highest max clock seen, and every
    throttle reason active under load."""
    b = _bench()
    rows = ["0, 2070, 2070, 900.0, 100, Not Active, Not Active, Not Active, Not Active",
            "0, 1980, 2070, 1400.0, 100, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 950.0, 98, Not Active, Not Active, Not Active, Not Active",
            "0, 600, 2070, 90.0, 0, Active, Not Active, Not Active, Not Active",  # idle: ignored
            "garbage line",
            ""]
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")
    s = b.ClockSampler(0)
    s.proc, s.path = _DoneProc(), str(path)
    out = s.stop()
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert not path.exists()
    s = b.ClockSampler(0)  # nvidia-smi missing: an empty record, not an error
    assert s.stop() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
