"""CPU checks of bench.py's host logic: the kernel-source hash that decides whether
the recorded ncu traffic still applies ignores comments and layout but not code."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_comments_and_layout_do_not_count():
    b = _bench()
    code = 'int f(int x) {\n  return x + 1;  // add one\n}\n/* block\n comment */\n'
    same = '// header\nint f(int x) { return x + 1; }\n'
    assert b._strip_comments(code) == b._strip_comments(same)


def test_code_and_string_literals_count():
    b = _bench()
    assert b._strip_comments("int f() { return 1; }") != b._strip_comments("int f() { return 2; }")
    # a "//" inside a string literal is code, not a comment
    assert b._strip_comments('const char* s = "a // b";') != b._strip_comments('const char* s = "a ";')


def test_recorded_traffic_is_for_a_hash_of_the_right_form():
    b = _bench()
    sha = b._src_sha()
    assert len(sha) == 16 and int(sha, 16) >= 0
    assert set(b.NCU_TRAFFIC) == {"src_sha", "bytes_per_launch"}
    assert b.NCU_TRAFFIC["bytes_per_launch"] > 140_000_000     # at least the algorithmic 140.7 MB
