"""The DRAM-traffic records under profiles/ and the source hash that keeps
them honest: bench.py reports a kernel's recorded traffic only while the code
of its sources (comments removed) is the code that was captured."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_only_drops_comments_and_blank_lines_only():
    src = ("int a = 1;  // one\n"
           "/* block\n   comment */\n"
           "\n"
           "int b = a / 2;   \n"
           "float c = 1.f;  /* inline */ int d = 3;\n")
    assert bench._code_only(src) == "int a = 1;\nint b = a / 2;\nfloat c = 1.f;   int d = 3;"
    # a code change is visible, a comment change is not
    assert bench._code_only(src.replace("// one", "// two")) == bench._code_only(src)
    assert bench._code_only(src.replace("a / 2", "a / 3")) != bench._code_only(src)


def test_read_traffic_keeps_only_records_of_the_current_code():
    """Every kernel the bench reports has a record; a record counts only while
    its sources hash to the stored value, so the bench reports traffic null
    for a kernel changed since its capture."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        rec = json.load(fh)["kernels"]
    assert set(rec) == set(bench.KERNEL_SOURCES)
    fresh = bench.read_traffic()
    for k, v in rec.items():
        assert (k in fresh) == (v["sources_sha256"] == bench.kernel_source_hash(k)), k
        assert all(isinstance(x, int) and x > 0 for key, x in v.items() if key != "sources_sha256")
