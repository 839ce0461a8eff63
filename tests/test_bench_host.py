"""Host-side helpers of bench.py: the code hash that ties a committed ncu summary to
the sources it was taken on (comments do not count, code does), the lookup of a
summary's traffic, the algorithmic bytes the roofline fractions divide, and the
selection-overlap statistic."""
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


def test_algorithmic_bytes_of_a_loop32_layer_match_the_profiled_figures():
    """The bench's algorithmic bytes for one loop32 layer are the figures the committed
    ncu summaries quote: 1,270,087,680 B of K/V for the verify call, and per draft step
    8 sequences x (2048 + s + 1) token pages of 4096 B (67.14-67.31 MB for s = 0..5)."""
    import synth
    b = load_bench()
    w = synth.scaled(synth.WORKLOADS["loop32"], layers=1)
    lengths = w.lengths(0)
    assert min(lengths) >= w.k  # every sequence selects k entries
    got = b.algorithmic_bytes(w, lengths)
    assert got["per_token"] == 4096
    assert got["verify"] == 1270087680
    steps = [8 * (2048 + s + 1) * 4096 for s in range(w.gamma)]
    assert steps[0] == 67141632 and steps[-1] == 67305472
    assert got["draft"] == sum(steps)


def test_short_sequences_select_everything_in_the_draft_bytes():
    import synth
    b = load_bench()
    w = synth.Workload("t", B=2, Hq=4, Hkv=2, d=64, gamma=2, k=100, n=None, ragged=(1, 2))
    got = b.algorithmic_bytes(w, [40, 300])
    per = 2 * 64 * 2 * 2
    assert got["verify"] == 340 * per
    # sequence 0 selects its 40 entries, sequence 1 its top 100; step s adds s + 1 draft tokens
    assert got["draft"] == ((40 + 1) + (40 + 2) + (100 + 1) + (100 + 2)) * per


def test_profiled_traffic_is_read_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    b = load_bench()
    csrc = tmp_path / "self_speculative_sparse_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = "__global__ void k(int* x) {\n  x[0] = 1;  // one\n}\n"
    (csrc / "k.cu").write_text(src)
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    sha = b.source_sha(("k.cu",))
    (tmp_path / "profiles" / "kern_wl.md").write_text(
        f"# summary\n\n- source_sha256: `{sha}`\n- dram_bytes_per_launch: 123456\n")
    assert b.profiled_traffic("kern", "wl", ("k.cu",)) == 123456
    (csrc / "k.cu").write_text(src.replace("// one", "// the first element"))  # a comment: same code
    assert b.profiled_traffic("kern", "wl", ("k.cu",)) == 123456
    (csrc / "k.cu").write_text(src.replace("x[0] = 1", "x[0] = 2"))  # the code changed
    assert b.profiled_traffic("kern", "wl", ("k.cu",)) is None
    assert b.profiled_traffic("other", "wl", ("k.cu",)) is None  # no summary at all


def test_the_committed_summaries_name_their_figures_in_the_form_the_bench_reads():
    """Each committed kernel summary carries a 64-hex source hash and an integer byte
    count under the keys profiled_traffic looks for (whether the hash is current is the
    bench's business: it reports null traffic for an old summary)."""
    import re
    for name in ("verify_attn_loop32.md", "draft_attn_loop32.md"):
        text = open(os.path.join(ROOT, "profiles", name)).read()
        assert re.search(r"^- source_sha256: `[0-9a-f]{64}`$", text, re.M), name
        assert re.search(r"^- dram_bytes_per_launch: [0-9]+$", text, re.M), name


def test_overlap_fraction():
    b = load_bench()
    assert b.overlap_fraction([1, 2, 3, 4], [3, 4, 5, 6], 4) == 0.5
    assert b.overlap_fraction([1, 2], [1, 2], 2) == 1.0
    assert b.overlap_fraction([], [], 0) == 1.0
