"""The boundary is a C ABI: a plain C program includes include/rdkv.h, links the built library and
calls its host-side entry points (no GPU, no Python binding); its results equal the binding's."""
import ctypes
import os
import shutil
import subprocess

import pytest

from mixed_bit_kv_gb300 import rdkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_links_and_calls_the_library(tmp_path):
    import __graft_entry__
    __graft_entry__.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(rdkv.LIB_PATH)
    exe = str(tmp_path / "c_abi_check")
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_check.c"), "-L", libdir, "-lrdkv",
                    "-Wl,-rpath," + libdir, "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    got = dict(line.split() for line in out.stdout.splitlines())
    L = rdkv.lib()
    s = rdkv.make_shape(1, 32768, 24, 8, 128, 128, "f16")
    assert int(got["ws_score"]) == L.rdkv_score_workspace_bytes(ctypes.byref(s))
    assert int(got["plan_bytes"]) == L.rdkv_plan_bytes(ctypes.byref(s))
    b = rdkv.Sizes()
    assert L.rdkv_zone_bounds(ctypes.byref(s), ctypes.c_float(2.5), ctypes.c_float(2.5), ctypes.byref(b)) == 0
    assert int(got["bound_zone_a"]) == b.zone_a_bytes
    assert int(got["bad_head_dim_status"]) == rdkv.RDKV_ERR_UNSUPPORTED
    assert int(got["ws_allocate_pack"]) == L.rdkv_allocate_pack_workspace_bytes(ctypes.byref(s), 0)
