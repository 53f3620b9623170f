"""Host-side pieces of bench.py that need no GPU."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_profile_key_ignores_comments_but_not_code():
    a = "int f(int x) {\n    return x + 1;  // add one\n}\n"
    b = "/* a note */\nint f(int x) {\n\n    return x + 1;  // add one, said differently\n}\n"
    c = "int f(int x) {\n    return x + 2;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_kernel_source_sha_is_stable():
    for k in ("k_topk16", "k_verify", "k_gate_tc", "k_pair_score_walk"):
        h = bench.kernel_source_sha(k)
        assert len(h) == 16 and h == bench.kernel_source_sha(k)
