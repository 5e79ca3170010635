"""The headers are plain C: a C99 program that includes all of them compiles with warnings as
errors, links against libeagle3.so and gets the documented host-side answers (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

from tests._util import ROOT, built_lib

C_SOURCE = r"""
#include "eagle3.h"
#include "eagle3_linear.h"
#include "eagle3_f32.h"
#include "eagle3_chain.h"
#include "eagle3_testing.h"
#include "eagle3_ttt.h"

#include <stdio.h>
#include <string.h>

int main(void) {
    eagle3_accept_args_t a;
    eagle3_draft_tree_args_t d;
    memset(&a, 0, sizeof a);
    a.mode = EAGLE3_ACCEPT_GREEDY;
    a.n_nodes = 5;
    a.vocab = 100;
    a.max_path = 7;
    if (eagle3_accept(&a, NULL, 0, NULL) != EAGLE3_OK) return 1;            /* batch 0: nothing to do */
    a.batch = 2;
    a.vocab = 0;
    if (eagle3_accept(&a, NULL, 0, NULL) != EAGLE3_ERR_INVALID_ARGUMENT) return 2;
    memset(&d, 0, sizeof d);
    d.hidden = 256;
    d.n_heads = 4;
    d.n_kv_heads = 2;
    d.head_dim = 128;
    d.ffn = 512;
    d.vocab = 1000;
    d.depth = 4;
    d.top_k = 4;
    d.n_nodes = 12;
    d.tc_max = 2;
    d.s_max = 64;
    d.draft_vocab = 300;                                                     /* reduced, without d2t */
    if (eagle3_draft_tree(NULL, &d, NULL, 0, NULL) != EAGLE3_ERR_INVALID_ARGUMENT) return 3;
    {
        eagle3_chain_verify_args_t c;
        eagle3_spec_decode_metadata_args_t m;
        memset(&c, 0, sizeof c);
        c.vocab = 10;
        c.temperature = 1.0f;
        if (eagle3_chain_verify(&c, NULL) != EAGLE3_OK) return 6;                 /* no requests */
        c.n_requests = 3;
        c.max_drafts = 256;                                                      /* above 255 */
        if (eagle3_chain_verify(&c, NULL) != EAGLE3_ERR_INVALID_ARGUMENT) return 7;
        memset(&m, 0, sizeof m);
        m.n_requests = -1;
        if (eagle3_spec_decode_metadata(&m, NULL) != EAGLE3_ERR_INVALID_ARGUMENT) return 8;
        if (eagle3_test_verify_attn_timeout(NULL, NULL, 0, -1, 1000, NULL) != EAGLE3_ERR_INVALID_ARGUMENT) return 9;
    }
    {
        eagle3_ttt_attn_args_t t;
        memset(&t, 0, sizeof t);
        t.seq_len = 96;                                                          /* not a multiple of 64 */
        t.n_heads = 32;
        t.n_kv_heads = 8;
        t.head_dim = 128;
        t.n_steps = 2;
        t.batch = 1;
        if (eagle3_ttt_attn(&t, NULL, 0, NULL) != EAGLE3_ERR_UNSUPPORTED) return 10;
    }
    if (strlen(eagle3_status_string(EAGLE3_ERR_CAPACITY)) == 0) return 4;
    if (eagle3_version() < 100) return 5;
    printf("ok %d\n", eagle3_version());
    return 0;
}
"""


def test_headers_compile_as_c99_and_link(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = built_lib()
    libdir = os.path.dirname(lib._name)
    src = tmp_path / "abi.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "abi"
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", libdir, "-leagle3", "-Wl,-rpath," + libdir]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    assert run.stdout.startswith("ok ")
