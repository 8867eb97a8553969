"""The C-ABI library builds, loads, and exports every function include/*.h declares (CPU only)."""
import ctypes
import glob
import os
import re

import pytest

import mxfp4_moe_expert_gb300 as pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(moe_mxfp4_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib_path():
    if not os.path.exists(pkg.LIB_PATH):
        from mxfp4_moe_expert_gb300 import build
        build.build()
    return pkg.LIB_PATH


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert {"moe_mxfp4_create", "moe_mxfp4_forward", "moe_mxfp4_destroy"} <= names
    assert names == set(pkg.EXPORTED), names ^ set(pkg.EXPORTED)


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_host_side_validation(lib_path):
    pkg.load_library(lib_path)
    assert pkg.moe_mxfp4_status_string(pkg.MOE_OK) == "ok"
    assert "workspace" in pkg.moe_mxfp4_status_string(pkg.MOE_ERR_WORKSPACE)
    # argument checks that return before touching a device
    st, h = pkg.moe_mxfp4_create(pkg.moe_mxfp4_config(0, 256, 128, 8, 2, 8, 1e-6, 0, 0, 0, 0), [pkg.moe_mxfp4_layer()])
    assert st == pkg.MOE_ERR_INVALID_ARG and not h
    st, h = pkg.moe_mxfp4_create(pkg.moe_mxfp4_config(1, 200, 128, 8, 2, 8, 1e-6, 0, 0, 0, 0), [pkg.moe_mxfp4_layer()])
    assert st == pkg.MOE_ERR_INVALID_ARG
    st, h = pkg.moe_mxfp4_create(pkg.moe_mxfp4_config(1, 256, 128, 8, 9, 8, 1e-6, 0, 0, 0, 0), [pkg.moe_mxfp4_layer()])
    assert st == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_quantize(None, 1, 32, None, None, None) == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_forward(None, None, 8, None, None, 0, None) == pkg.MOE_ERR_INVALID_ARG
    pkg.moe_mxfp4_destroy(None)


def test_every_entry_point_rejects_a_null_handle_or_bad_sizes_without_a_device(lib_path):
    """Host-side argument checks of the entry points, all before any CUDA call."""
    pkg.load_library(lib_path)
    assert pkg.moe_mxfp4_workspace_bytes(None, 8)[0] == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_forward_host(None, None, 8, None, None, 0, None) == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_check(None, None, None) == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_forward_static(None, None, 8, None, None) == pkg.MOE_ERR_INVALID_ARG
    # acceptance: sizes are checked first; zero streams is a no-op; null buffers are refused
    assert pkg.moe_mxfp4_accept(None, None, -1, 8, 100, None, None, None, None) == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_accept(None, None, 1, 0, 100, None, None, None, None) == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_accept(None, None, 1, 8, 0, None, None, None, None) == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_accept(None, None, 1, 8, 1 << 31, None, None, None, None) == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_accept(None, None, 0, 8, 100, None, None, None, None) == pkg.MOE_OK
    assert pkg.moe_mxfp4_accept(None, None, 1, 8, 100, None, None, None, None) == pkg.MOE_ERR_INVALID_ARG
    # the activation split: sizes and pointers are checked before any launch; nothing to do is OK
    assert pkg.moe_mxfp4_split_terms(None, -1, None, None, None) == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_split_terms(None, 4, None, None, None) == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_split_terms(None, 0, None, None, None) == pkg.MOE_OK


def _up256(v):
    return (v + 255) // 256 * 256


@pytest.mark.parametrize("H,I,E", [(512, 512, 1), (1024, 512, 16), (4096, 1536, 64), (7168, 2048, 384)])
def test_packed_layout_size_is_the_sum_of_its_sections(lib_path, H, I, E):
    """moe_mxfp4_packed_bytes (host arithmetic only) against the layout the header states:
    the codes of gate, up and down (E * 3 * H * I / 2 bytes), the gate/up scales (E * 2 * H * I
    / 32) and the down scales (E * H * I / 32), each section starting on a 256-byte
    boundary, nothing else."""
    pkg.load_library(lib_path)
    st, n = pkg.moe_mxfp4_packed_bytes(H, I, E)
    assert st == pkg.MOE_OK
    codes = E * 3 * H * I // 2
    scales_gu = E * 2 * H * I // 32
    scales_d = E * H * I // 32
    assert n == _up256(_up256(_up256(codes) + scales_gu) + scales_d)
    assert n - (codes + scales_gu + scales_d) < 3 * 256


def test_packed_layout_refuses_shapes_outside_the_tensor_core_path(lib_path):
    pkg.load_library(lib_path)
    assert pkg.moe_mxfp4_packed_bytes(768, 512, 4)[0] == pkg.MOE_ERR_UNSUPPORTED   # H not a multiple of 512
    assert pkg.moe_mxfp4_packed_bytes(1024, 384, 4)[0] == pkg.MOE_ERR_UNSUPPORTED  # I not a multiple of 512
    assert pkg.moe_mxfp4_packed_bytes(1024, 512, 0)[0] == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_packed_bytes(-512, 512, 4)[0] == pkg.MOE_ERR_INVALID_ARG
