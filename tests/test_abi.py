"""The C ABI: the library builds, loads and exports every entry point the
header declares; host-side argument checks reject bad arguments before any
GPU work (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(dflash2_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from dflash_draft_selection_gb300 import build
    build.build()
    import dflash_draft_selection_gb300 as d2
    return d2.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, text in [(0, b"ok"), (1, b"invalid argument"), (2, b"unsupported"), (3, b"CUDA error"),
                       (4, b"workspace too small")]:
        assert lib.dflash2_status_string(code) == text


def test_workspace_sizes(lib):
    assert lib.dflash2_verify_workspace_bytes(64, 7) >= 64 * 8 * 520
    assert lib.dflash2_verify_workspace_bytes(1, 0) == 0
    assert lib.dflash2_verify_workspace_bytes(1, 16) == 0
    assert lib.dflash2_topk16_workspace_bytes(448) >= 448 * 4
    assert lib.dflash2_topk16_workspace_bytes(-1) == 0


def test_argument_checks_fail_before_any_launch(lib):
    bad = 1  # DFLASH2_ERR_INVALID_ARG
    p = ctypes.c_void_p(16)  # never dereferenced: the checks fail first
    # V < 16
    assert lib.dflash2_topk16(p, 1, 4, 8, 8, None, 1, p, p, p, p, 1 << 22, None) == bad
    # ld * 2 bytes not a multiple of 16
    assert lib.dflash2_topk16(p, 1, 4, 100, 100, None, 1, p, p, p, p, 1 << 22, None) == bad
    # rows_per_param < 1
    assert lib.dflash2_topk16(p, 1, 4, 128, 128, None, 0, p, p, p, p, 1 << 22, None) == bad
    # no workspace
    assert lib.dflash2_topk16(p, 1, 4, 128, 128, None, 1, p, p, p, None, 1 << 22, None) == bad
    # K outside 1..15
    assert lib.dflash2_verify(p, 1, 2, 16, 128, 128, p, p, p, p, None, None, None, 0, p, p, p, p, 1 << 20,
                              None) == bad
    assert lib.dflash2_pair_score_walk(2, 0, p, p, p, p, p, 1, 128, 256, p, None, None, p, p, p, p, None) == bad
    # D not a power of two
    assert lib.dflash2_pair_score_walk(2, 3, p, p, p, p, p, 1, 128, 100, p, None, None, p, p, p, p, None) == bad
    assert lib.dflash2_ctx_gate(p, 1, 4, 128, p, 48, p, None) == bad
    # bf16 hidden not a multiple of 64
    assert lib.dflash2_ctx_gate(p, 1, 4, 100, p, 256, p, None) == bad
    # conv group size must divide H
    assert lib.dflash2_conv2tap(p, p, p, p, 1, 2, 3, 10, 3, p, None) == bad
    # workspace too small
    assert lib.dflash2_verify(p, 1, 2, 3, 128, 128, p, p, p, p, None, None, None, 0, p, p, p, p, 16, None) == 4
    assert lib.dflash2_topk16(p, 1, 4, 128, 128, None, 1, p, p, p, p, 16, None) == 4
