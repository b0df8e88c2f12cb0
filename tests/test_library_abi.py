"""The C-ABI library builds, loads and exports every entry point include/ddt.h declares;
host-side argument checks fail fast (no GPU needed: no kernel is launched)."""
import ctypes
import os
import re
import shutil

import pytest

from tree_speculative_decoding_02_gb300 import build_ext, ddt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ddt.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ddt_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return ddt.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert {"ddt_build_tree", "ddt_tree_attn", "ddt_tree_gdn", "ddt_walk_accept", "ddt_commit"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ddt.EXPORTS)


def test_library_is_in_tree_and_versioned(lib):
    assert os.path.dirname(build_ext.LIB).startswith(ROOT)
    assert lib.ddt_version().decode().endswith("sm_103a")
    assert lib.ddt_launch_count() >= 0
    for code, text in [(0, "ok"), (3, "cache capacity exceeded"), (6, "non-finite logits"), (7, "malformed tree")]:
        assert lib.ddt_status_string(code).decode() == text


def test_status_codes_match_header():
    text = open(HEADER).read()
    codes = dict((m.group(1), int(m.group(2))) for m in re.finditer(r"(DDT_[A-Z0-9_]+)\s*=\s*(\d+)", text))
    assert codes["DDT_OK"] == 0 and codes["DDT_ERR_CAPACITY"] == 3 and codes["DDT_ERR_NONFINITE"] == 6
    assert codes["DDT_ERR_TREE"] == 7 and codes["DDT_F32"] == 0 and codes["DDT_BF16"] == 1


def test_host_checks_fail_fast(lib):
    """Bad sizes / null pointers are refused on the host before any launch."""
    p = ctypes.c_void_p(16)
    nul = None
    launched = lib.ddt_launch_count()
    # build: B = 0, top_k > 32, null workspace
    assert lib.ddt_build_tree(0, 1, 10, 1, 1, 1, *([p] * 11), p, 1 << 20, nul) == 1
    assert lib.ddt_build_tree(1, 1, 100, 33, 1, 1, *([p] * 11), p, 1 << 20, nul) == 2
    assert lib.ddt_build_tree(1, 1, 100, 4, 1, 1, *([p] * 11), nul, 1 << 20, nul) == 1
    assert lib.ddt_build_tree(1, 1, 100, 4, 2000, 1, *([p] * 11), p, 1 << 20, nul) == 2
    # attention: head size not compiled, Hq not a multiple of Hkv
    assert lib.ddt_tree_attn(1, 1, 5, 4, 1, 96, 10, 1, 1, *([p] * 8), 1.0, p, p, p, 256, nul) == 2
    assert lib.ddt_tree_attn(1, 1, 5, 5, 2, 64, 10, 1, 1, *([p] * 8), 1.0, p, p, p, 256, nul) == 1
    # GDN: unsupported head dims
    assert lib.ddt_tree_gdn(1, 1, 5, 1, 1, 48, 48, 4, 1, 1, *([p] * 11), p, 256, nul) == 2
    # walk / commit: bad sizes
    assert lib.ddt_walk_accept(0, 5, 10, 4, 1, *([p] * 11), p, 256, nul) == 1
    assert lib.ddt_commit(1, 5, 0, 0, 1, 64, 10, 1, p, p, p, p, 0, 1, 1, 32, 32, 4, 1, *([p] * 12), nul) == 1
    assert lib.ddt_launch_count() == launched   # refused before any launch


def test_workspace_queries(lib):
    assert lib.ddt_build_tree_workspace(32, 15, 151936, 8) > 0
    assert lib.ddt_walk_accept_workspace(32, 65, 151936) > 0
    assert lib.ddt_build_tree_workspace(0, 15, 151936, 8) == 0
