"""Host-side checks of the C ABI (no GPU needed): the library builds for sm_103a, loads, and
exports every entry point that include/moe.h declares; size helpers follow the documented rules."""
import os
import re

import pytest

from bit_expert_ffn_moe_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    return B.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.EXPORTED) == names


def test_status_strings_and_version(lib):
    assert B.moe_abi_version() == 13
    header = open(os.path.join(ROOT, "include", "moe.h")).read()
    assert int(re.search(r"#define MOE_ABI_VERSION (\d+)", header).group(1)) == B.moe_abi_version()
    assert B.status_string(0) == "MOE_OK"
    assert B.status_string(5) == "MOE_ERR_TIMEOUT"


def test_size_helpers():
    # tensor-core scale layout: one 512-byte atom per 128 rows x 128 columns
    assert B.moe_mxfp4_mma_scale_bytes(128, 128) == 512
    assert B.moe_mxfp4_mma_scale_bytes(256, 8192) == 2 * 64 * 512
    assert B.moe_mxfp4_mma_scale_bytes(100, 128) == 0
    # padded rows: every touched expert may waste up to 127 rows
    assert B.moe_padded_rows(4096, 8, 128) == 32768 + 128 * 127 + 0 or B.moe_padded_rows(4096, 8, 128) % 128 == 0
    assert B.moe_padded_rows(1, 8, 128) == 1024
    assert B.moe_workspace_size(16, 256, 8, 2, 512, B.MOE_ACT_BF16) > 0
    assert B.moe_workspace_size(16, 256, 8, 2, 512, B.MOE_ACT_MXFP4) > B.moe_workspace_size(16, 256, 8, 2, 512, 0)
    # shape rules
    assert B.moe_workspace_size(16, 200, 8, 2, 512, 0) == 0      # d % 128
    assert B.moe_workspace_size(16, 256, 8, 9, 512, 0) == 0      # k > E
    assert B.moe_workspace_size(16, 256, 2048, 2, 512, 0) == 0   # E > 1024
    assert B.moe_workspace_size(16, 256, 8, 2, 96, B.MOE_ACT_MXFP4) == 0  # I % 256 on the MXFP4 path
    assert B.moe_workspace_size(16, 256, 8, 2, 384, B.MOE_ACT_MXFP4) == 0
    assert B.moe_workspace_size(16, 384, 8, 2, 512, B.MOE_ACT_MXFP4) == 0  # d % 256 on the MXFP4 path
    assert B.moe_workspace_size(16, 384, 8, 2, 384, B.MOE_ACT_BF16) > 0
    # MXFP8: the MXFP4 shape rules, one byte per value in the operand buffers
    assert B.moe_workspace_size(16, 256, 8, 2, 512, B.MOE_ACT_MXFP8) > B.moe_workspace_size(16, 256, 8, 2, 512, 1)
    assert B.moe_workspace_size(16, 384, 8, 2, 512, B.MOE_ACT_MXFP8) == 0
    assert B.moe_workspace_size(16, 256, 8, 2, 384, B.MOE_ACT_MXFP8) == 0
    assert B.moe_workspace_size(16, 256, 8, 2, 512, 3) == 0      # unknown format
    # decode pieces: up to 16 tokens, d % 256
    assert B.moe_decode_pieces_bytes(16, 8192, 0) == 128 * 8192 // 2
    assert B.moe_decode_pieces_bytes(16, 8192, 1) == 64 * 512
    assert B.moe_decode_pieces_bytes(17, 8192, 0) == 0
    assert B.moe_decode_pieces_bytes(4, 384, 0) == 0


def test_library_is_built_for_sm103a_only():
    from bit_expert_ffn_moe_gb300 import _build
    assert "arch=compute_103a,code=sm_103a" in _build.NVCC_FLAGS
    assert os.path.exists(_build.LIB)


def test_decode_pieces_arguments_are_checked_on_the_host(lib):
    # format and shape rules are checked before anything is launched
    assert lib.moe_decode_pieces(256, 4, 8192, B.MOE_ACT_MXFP4, 256, 256, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_decode_pieces(256, 17, 8192, B.MOE_ACT_BF16, 256, 256, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_decode_pieces(256, 4, 384, B.MOE_ACT_MXFP8, 256, 256, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_decode_pieces(256, 0, 8192, B.MOE_ACT_MXFP8, None, None, None) == B.MOE_OK
    assert lib.moe_decode_pieces(None, 4, 8192, B.MOE_ACT_MXFP8, 256, 256, None) == B.MOE_ERR_INVALID_ARG
    W = B.moe_expert_weights()
    assert lib.moe_expert_ffn_decode(256, 256, B.MOE_ACT_MXFP4, 256, 256, 256, 256, 4, 8192, 128, 8, 2048, W, 256, None,
                                     256, 1 << 30, None) == B.MOE_ERR_INVALID_ARG


def test_selftest_arguments_are_checked_on_the_host(lib):
    # rejected before anything is launched (no GPU needed)
    assert lib.moe_selftest_wait_timeout(None, 0, 10, None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_selftest_wait_timeout(256, 1 << 20, 0, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_wait_timeout(256, 1 << 20, 2000000, None) == B.MOE_ERR_INVALID_ARG


def test_expert_norm_arguments_are_checked_on_the_host(lib):
    # eps must lie in (0, 1]; shapes follow moe_combine; both are rejected before any launch
    for eps in (0.0, -1e-6, 2.0, float("nan")):
        assert lib.moe_combine_norm(256, 256, 256, 4, 2, 256, eps, 256, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_combine_norm(256, 256, 256, 4, 33, 256, 1e-6, 256, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_combine_norm(256, 256, 256, 4, 2, 100, 1e-6, 256, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_combine_norm(256, 256, 256, 0, 2, 256, 1e-6, 256, None) == B.MOE_OK
    W = B.moe_expert_weights()
    assert lib.moe_layer_forward_norm(256, 256, None, 4, 256, 8, 2, 512, W, B.MOE_ACT_BF16, 0.0, 256, None, None,
                                      256, 1 << 30, None) == B.MOE_ERR_INVALID_ARG


def test_host_buffer_layer_arguments_are_checked_on_the_host(lib):
    # null host or staging pointers, misaligned or shared staging buffers, and the layer's own shape
    # rules are refused before any copy or launch; T = 0 is a no-op
    W = B.moe_expert_weights()
    args = lambda xh, yh, xd, yd, T=4, d=256: (xh, 256, None, T, d, 8, 2, 512, W, B.MOE_ACT_BF16, yh, None, None,
                                               xd, yd, 256, 1 << 30, None, None, None)
    assert lib.moe_layer_forward_host(*args(None, 4096, 8192, 16384)) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_host(*args(4096, None, 8192, 16384)) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_host(*args(4096, 4096, None, 16384)) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_host(*args(4096, 4096, 8192, 8192)) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_host(*args(4096, 4096, 8200, 16384)) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_host(*args(4096, 4096, 8192, 16384, d=200)) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_layer_forward_host(*args(None, None, None, None, T=0)) == B.MOE_OK


def test_dense_linear_shapes_and_arguments_are_checked_on_the_host(lib):
    assert B.moe_dense_workspace_size(4, 8192, 4096, B.MOE_ACT_MXFP4) > B.moe_dense_workspace_size(4, 8192, 4096, 0)
    assert B.moe_dense_workspace_size(4, 384, 256, B.MOE_ACT_MXFP4) == 0    # K % 256 on the MXFP4 path
    assert B.moe_dense_workspace_size(4, 8192, 4096, B.MOE_ACT_MXFP8) > B.moe_dense_workspace_size(4, 8192, 4096, 1)
    assert B.moe_dense_workspace_size(4, 384, 256, B.MOE_ACT_MXFP8) == 0
    assert B.moe_dense_workspace_size(4, 384, 256, B.MOE_ACT_BF16) > 0
    assert B.moe_dense_workspace_size(4, 200, 256, B.MOE_ACT_BF16) == 0     # K % 128
    assert B.moe_dense_workspace_size(4, 16384, 256, B.MOE_ACT_BF16) == 0   # K <= 8192 on the GEMV path
    W = B.moe_mxfp4_matrix()
    assert lib.moe_dense_linear(256, 4, 256, 256, W, B.MOE_ACT_BF16, 256, 256, 1 << 20, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_dense_linear(256, 4, 200, 256, W, B.MOE_ACT_BF16, 256, 256, 1 << 20, None) == \
        B.MOE_ERR_UNSUPPORTED_SHAPE


def test_nvfp4_arguments_are_checked_on_the_host(lib):
    # pack / unpack: K % 32, at most 65535 matrices, pointers and alignment; n_mats == 0 is a no-op
    assert lib.moe_nvfp4_pack(256, 1, 4, 48, 256, 256, 256, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_nvfp4_pack(256, 70000, 4, 64, 256, 256, 256, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_nvfp4_pack(256, 1, 4, 64, 256, 256, None, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_nvfp4_pack(256, 1, 4, 64, 256, 257, 256, None) == B.MOE_ERR_INVALID_ARG  # s 2-byte aligned
    assert lib.moe_nvfp4_pack(None, 0, 4, 64, None, None, None, None) == B.MOE_OK
    assert lib.moe_nvfp4_unpack(256, 256, 256, 1, 4, 40, 256, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    # NVFP4 expert weights: the bf16-activation GEMVs, or MXFP4 activations on the tensor cores
    # with the weights' tensor-core copies; not MXFP8; global scales required; known formats
    W = B.nvfp4_expert_weights_struct(256, 256, 256, 256, 256, 256, 256, 256, 256)
    args = (256, 256, None, 4, 256, 8, 2, 512)
    tail = (256, None, None, 256, 1 << 30, None)
    assert lib.moe_layer_forward(*args, W, B.MOE_ACT_MXFP8, *tail) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_layer_forward(*args, W, B.MOE_ACT_MXFP4, *tail) == B.MOE_ERR_INVALID_ARG  # no copies
    W.down_gs = None
    assert lib.moe_layer_forward(*args, W, B.MOE_ACT_BF16, *tail) == B.MOE_ERR_INVALID_ARG
    W.down_gs = 256
    W.up_s = 257
    assert lib.moe_layer_forward(*args, W, B.MOE_ACT_BF16, *tail) == B.MOE_ERR_INVALID_ARG
    W.wfmt = 7
    assert lib.moe_layer_forward(*args, W, B.MOE_ACT_BF16, *tail) == B.MOE_ERR_INVALID_ARG


def _c_struct_fields(name):
    """(field, C type) pairs of `typedef struct ... { ... } name;` in include/moe.h."""
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    m = re.search(r"typedef struct\s*\w*\s*\{([^}]*)\}\s*" + name + r"\s*;", src)
    assert m, name
    out = []
    for decl in m.group(1).split(";"):
        decl = " ".join(decl.split())
        if not decl:
            continue
        typ, _, rest = decl.rpartition(" ")
        for field in rest.split(","):
            out.append((field.strip().lstrip("*"), typ + ("*" if field.strip().startswith("*") else "")))
    return out


@pytest.mark.parametrize("name", ["moe_expert_weights", "moe_mxfp4_matrix"])
def test_ctypes_structs_mirror_the_header(name):
    import ctypes
    fields = _c_struct_fields(name)
    cls = getattr(B, name)
    assert [f for f, _ in fields] == [f for f, _ in cls._fields_]
    for (f, ctype), (_, pytype) in zip(fields, cls._fields_):
        if ctype.endswith("*"):
            assert pytype is ctypes.c_void_p, f
        else:
            assert ctype == "int32_t" and pytype is ctypes.c_int32, f
    # the C layout of these fields on an LP64 ABI: pointers 8-byte aligned
    assert ctypes.sizeof(cls) % 8 == 0


@pytest.mark.parametrize("name", ["moe_expert_weights", "moe_mxfp4_matrix"])
def test_ctypes_struct_offsets_equal_the_c_compilers(name, tmp_path):
    import ctypes
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    cls = getattr(B, name)
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe.h"', "int main(void) {",
             '  printf("%%zu\\n", sizeof(%s));' % name]
    lines += ['  printf("%%zu\\n", offsetof(%s, %s));' % (name, f) for f, _ in cls._fields_]
    lines += ["  return 0;", "}"]
    c = tmp_path / "layout.c"
    c.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(c), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(cls)
    assert got[1:] == [getattr(cls, f).offset for f, _ in cls._fields_]
