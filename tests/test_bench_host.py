"""Host-side helpers of bench.py: the code hash that ties a committed ncu summary to
the sources it was taken on (comments do not count, code does)."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_comments_and_blank_lines_go_literals_stay():
    b = load_bench()
    src = ('int a = 1;  // note\n\n/* block\n   comment */ const char* s = "x // y /* z */";\n'
           "char q = '\"'; char e = '\\\\'; const char* t = \"a\\\"// b\";  /**/ int y;\n")
    out = b.strip_c_comments(src)
    assert out == ('int a = 1;\n const char* s = "x // y /* z */";\n'
                   "char q = '\"'; char e = '\\\\'; const char* t = \"a\\\"// b\";   int y;")


def test_a_comment_edit_keeps_the_hash_and_a_code_edit_changes_it():
    b = load_bench()
    base = "int f(int x) {\n  return x + 1;  // one\n}\n"
    assert b.strip_c_comments(base) == b.strip_c_comments(base.replace("// one", "// the successor"))
    assert b.strip_c_comments(base) != b.strip_c_comments(base.replace("x + 1", "x + 2"))
