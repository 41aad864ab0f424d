"""The header is a plain C ABI: a C99 client compiles against include/kvc.h
with -pedantic, links against libkvc, and sees the same struct layouts as
the Python binding (no GPU needed: only host-side calls)."""
import ctypes
import os
import shutil
import subprocess

import pytest

from kv_cache_eviction_kvc_gb300 import _build, kvc as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CLIENT = r"""
#include <stddef.h>
#include <stdio.h>
#include "kvc.h"
int main(void)
{
    kvc_params p;
    p.U = 2; p.G = 4; p.d = 128; p.cap = 100; p.L = 10; p.rule = KVC_RULE_EMA;
    p.alpha = 0.9f; p.refresh_period = 1; p.correction = KVC_CORR_FIRST_ORDER;
    p.merge = 0; p.merge_recent = 0; p.budget = NULL; p.chain_layers = 0; p.chain_heads = 0;
    printf("%zu %zu %zu %zu %zu %zu %d %zu\n", sizeof(kvc_params), sizeof(kvc_cache),
           sizeof(kvc_moments), offsetof(kvc_params, alpha), offsetof(kvc_params, merge_recent),
           kvc_decode_workspace_size(&p), kvc_version(), offsetof(kvc_params, budget));
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c99_client_sees_the_binding_layouts(tmp_path):
    lib = K.load() and _build.LIB
    src = tmp_path / "client.c"
    src.write_text(CLIENT)
    exe = tmp_path / "client"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), lib,
                    "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    sp, sc, sm, off_alpha, off_mr, ws, ver, off_b = map(int, out)
    assert sp == ctypes.sizeof(K.kvc_params)
    assert sc == ctypes.sizeof(K.kvc_cache)
    assert sm == ctypes.sizeof(K.kvc_moments)
    assert off_alpha == K.kvc_params.alpha.offset
    assert off_mr == K.kvc_params.merge_recent.offset
    assert ws == K.kvc_decode_workspace_size(K.make_params(U=2, G=4, cap=100, L=10))
    assert ver == K.kvc_version()
    assert off_b == K.kvc_params.budget.offset
