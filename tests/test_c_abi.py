"""include/ddt.h is a plain C header: a C99 program (and a C++ one) that includes it
compiles with warnings as errors, links against the in-tree libddt.so, and gets the
documented answers from the calls that need no GPU (version, status text, launch
counter, and argument refusals that return before anything is launched)."""
import os
import shutil
import subprocess

import pytest

from tree_speculative_decoding_02_gb300 import build_ext, ddt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

pytestmark = pytest.mark.skipif(
    shutil.which("gcc") is None or (shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc")),
    reason="needs gcc and nvcc (to build libddt.so)")

C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "ddt.h"

#define EXPECT(cond) do { if (!(cond)) { printf("FAILED line %d: %s\n", __LINE__, #cond); return 1; } } while (0)

int main(void) {
    ddt_stream_t stream = NULL;
    int32_t word = 0;
    int32_t* p = &word;             /* never dereferenced: every call below is refused first */
    uint64_t before;
    EXPECT(strstr(ddt_version(), "sm_103a") != NULL);
    EXPECT(strcmp(ddt_status_string(DDT_OK), "ok") == 0);
    EXPECT(strcmp(ddt_status_string(DDT_ERR_TIMEOUT), "bounded device wait gave up") == 0);
    before = ddt_launch_count();
    EXPECT(ddt_wait_selftest(NULL, stream) == DDT_ERR_INVALID_ARG);
    EXPECT(ddt_build_tree_workspace(0, 15, 151936, 8) == 0);
    EXPECT(ddt_build_tree(0, 15, 151936, 8, 64, DDT_BF16, p, p, p, p, p, p, p, p, (uint32_t*)p, NULL, p, p,
                          1 << 20, stream) == DDT_ERR_INVALID_ARG);
    EXPECT(ddt_build_tree(1, 15, 151936, 33, 64, DDT_BF16, p, p, p, p, p, p, p, p, (uint32_t*)p, NULL, p, p,
                          1 << 20, stream) == DDT_ERR_UNSUPPORTED);
    EXPECT(ddt_build_tree_noalloc(1, 15, 151936, 8, 64, DDT_BF16, NULL, p, p, p, p, p, p, p, (uint32_t*)p,
                                  NULL, p, stream) == DDT_ERR_INVALID_ARG);
    EXPECT(ddt_tree_attn(1, 1, 5, 4, 1, 96, 10, DDT_BF16, DDT_BF16, p, p, p, p, p, p, p, (uint32_t*)p, 0.125f,
                         p, p, p, 256, stream) == DDT_ERR_UNSUPPORTED);
    EXPECT(ddt_tree_gdn(1, 1, 5, 1, 1, 48, 48, 4, DDT_BF16, DDT_BF16, p, p, p, (float*)p, (float*)p, (float*)p,
                        p, p, p, NULL, p, p, 256, stream) == DDT_ERR_UNSUPPORTED);
    EXPECT(ddt_walk_accept(0, 5, 10, 4, DDT_BF16, p, p, p, p, p, p, p, p, p, p, p, p, 256, stream)
           == DDT_ERR_INVALID_ARG);
    EXPECT(ddt_walk_accept_sample_workspace(0, 65, 151936) == 0);
    EXPECT(ddt_walk_accept_sample_workspace(32, 65, 151936) == 1248000);  /* 32*65*75 partials of 8 B */
    EXPECT(ddt_walk_accept_sample(1, 5, 10, 4, 2, 0.0f, DDT_BF16, p, (const float*)p, p, p, p, p, p, p, p, p, p,
                                  p, 1 << 20, stream) == DDT_ERR_INVALID_ARG);
    EXPECT(ddt_walk_accept_sample(1, 5, 10, 4, 2, 1e-40f, DDT_BF16, p, (const float*)p, p, p, p, p, p, p, p, p,
                                  p, p, 1 << 20, stream) == DDT_ERR_INVALID_ARG);
    EXPECT(ddt_walk_accept_sample(1, 5, 10, 4, 33, 1.0f, DDT_BF16, p, (const float*)p, p, p, p, p, p, p, p, p,
                                  p, p, 1 << 20, stream) == DDT_ERR_UNSUPPORTED);
    EXPECT(ddt_walk_accept_sample(1, 5, 10, 4, 2, 1.0f, DDT_BF16, p, NULL, p, p, p, p, p, p, p, p, p, p,
                                  1 << 20, stream) == DDT_ERR_INVALID_ARG);
    EXPECT(ddt_commit(1, 5, 0, 0, 1, 64, 10, DDT_BF16, p, p, p, p, 0, 1, 1, 32, 32, 4, DDT_BF16, p, p,
                      (float*)p, (float*)p, (float*)p, p, p, p, p, p, p, p, stream) == DDT_ERR_INVALID_ARG);
    /* more accepted rows than any tree can have: refused before the KV part runs */
    EXPECT(ddt_commit(1, 5, 1000, 1, 1, 64, 10, DDT_BF16, p, p, p, p, 0, 1, 1, 32, 32, 4, DDT_BF16, p, p,
                      (float*)p, (float*)p, (float*)p, p, p, p, p, p, p, p, stream) == DDT_ERR_UNSUPPORTED);
    EXPECT(ddt_launch_count() == before);
    printf("ok\n");
    return 0;
}
"""


@pytest.fixture(scope="module")
def libdir():
    ddt.load()
    return os.path.dirname(build_ext.LIB)


@pytest.mark.parametrize("lang", ["c99", "c++11"])
def test_header_compiles_links_and_refuses(tmp_path, libdir, lang):
    ext, cc = (".c", "gcc") if lang == "c99" else (".cpp", "g++")
    src = tmp_path / ("caller" + ext)
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    cmd = [cc, "-std=" + lang, "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, str(src), "-o", str(exe),
           "-L", libdir, "-lddt", "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip() == "ok", run.stdout + run.stderr
