"""The C-ABI library builds for sm_103a, loads, and exports every entry point declared in include/hs.h. Only
host-side calls that touch no device are made here (descriptor arithmetic, error strings)."""
import ctypes
import os
import re

import pytest

import hierarchical_sparse_attention_hs_gb300 as hs
from hierarchical_sparse_attention_hs_gb300 import build as hs_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "hs.h")


@pytest.fixture(scope="module")
def lib():
    hs_build.build()
    return hs.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hs_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["hs_pool_create", "hs_resolve", "hs_prefetch", "hs_step_begin", "hs_pool_destroy",
                 "hs_meta_bytes", "hs_get_error", "hs_get_counters"]:
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_has_the_same_names():
    for n in declared_functions():
        assert callable(getattr(hs, n)), n


def test_descriptor_struct_matches_c_layout():
    assert ctypes.sizeof(hs.hs_pool_desc) == 6 * 4 + 8 + 8 + 8 + 8 + 8 + 8
    assert hs.hs_pool_desc.host_pool.offset == 24


def _desc(**kw):
    d = dict(layers=2, max_batch=3, ctx=1000, slots=64, topk_max=32, row_bytes=48)
    d.update(kw)
    return hs.hs_pool_desc(d["layers"], d["max_batch"], d["ctx"], d["slots"], d["topk_max"], d["row_bytes"],
                           None, 0, 0, None, None, None)


def test_meta_layout_arithmetic(lib):
    lay = hs.hs_get_meta_layout(_desc())
    assert lay["step"] == 0 and lay["error"] == 4 and lay["counters"] == 256
    assert lay["tok2slot"] % 256 == 0 and lay["tok2slot"] >= 256 + 2 * 4 * 8
    assert lay["slot_tok"] >= lay["tok2slot"] + 2 * 3 * 1000 * 4
    assert lay["slot_stamp"] >= lay["slot_tok"] + 2 * 3 * 64 * 4
    assert lay["total"] == hs.hs_meta_bytes(_desc()) >= lay["slot_stamp"] + 2 * 3 * 64 * 4


@pytest.mark.parametrize("bad", [dict(row_bytes=40), dict(topk_max=65), dict(slots=70000, topk_max=8),
                                 dict(layers=0), dict(ctx=0), dict(max_batch=-1)])
def test_invalid_geometry_is_rejected(lib, bad):
    assert hs.hs_meta_bytes(_desc(**bad)) == 0
    with pytest.raises(hs.HsError) as e:
        hs.hs_get_meta_layout(_desc(**bad))
    assert e.value.code == hs.HS_ERR_INVALID_ARG


def test_error_strings(lib):
    assert hs.hs_error_string(0) == "ok"
    assert "argument" in hs.hs_error_string(-1)
    assert hs.hs_error_string(-99) == "unknown error"


def test_plain_c_caller(lib, tmp_path):
    """include/hs.h is plain C: a C99 program compiles against it with warnings as errors, links libhs.so, and
    gets the same metadata layout as the binding."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c_caller.c")
    exe = str(tmp_path / "c_caller")
    libdir = os.path.dirname(hs.LIB_PATH)
    subprocess.check_call([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.dirname(HEADER), src, "-L", libdir, "-lhs", f"-Wl,-rpath,{libdir}",
                           "-o", exe])
    out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    d = hs.hs_pool_desc(2, 3, 1000, 64, 32, 656, None, 0, 0, None, None, None)
    lay = hs.hs_get_meta_layout(d)
    assert out[0].split() == [str(hs.hs_meta_bytes(d)), str(lay["tok2slot"]), str(lay["slot_stamp"]),
                              str(lay["total"])]
    assert out[1] == hs.hs_error_string(hs.HS_ERR_INVALID_ARG)
    assert out[2].split() == [str(hs.HS_ERR_INVALID_ARG), "0"]


def test_host_side_argument_errors_need_no_device(lib):
    """Calls whose arguments are refused return before any CUDA call, so they can be checked without a GPU."""
    for call in (lambda: hs.hs_host_alloc(0), lambda: hs.hs_host_free(0),
                 lambda: hs.hs_probe_launch(0, 0, 1, 1, 1, 0), lambda: hs.hs_pool_destroy(0),
                 lambda: hs.hs_step_begin_fused(0)):
        with pytest.raises(hs.HsError) as e:
            call()
        assert e.value.code == hs.HS_ERR_INVALID_ARG
