"""Host logic of bench.py (no GPU): the source hash that ties a recorded
ncu traffic figure to the kernel sources it was taken on."""

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
