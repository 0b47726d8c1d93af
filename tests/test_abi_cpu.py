"""Host-side checks of the C-ABI library that need no GPU: it loads, exports
every entry point the header declares, sizes its workspace, and rejects bad
arguments before launching anything."""

import ctypes
import os
import re

import pytest

from dropless_mixture_experts_gb300 import abi

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(abi.LIB_PATH):
        from dropless_mixture_experts_gb300 import build
        build.build()
    return abi.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+(moe_\w+)\s*\(", text, re.M)))


def declared_parameter_counts():
    """Name -> number of parameters of every prototype in the header
    (comments stripped; `void` alone counts as none)."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    out = {}
    for m in re.finditer(r"(moe_\w+)\s*\(([^;{]*?)\)\s*;", text, re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header():
    # the Python binding passes exactly as many arguments as each prototype
    # declares (an ABI change that misses the binding fails here, not on a GPU)
    counts = declared_parameter_counts()
    assert set(counts) == set(abi.EXPORTS)
    for name, (argtypes, _) in abi._SIGS.items():
        assert len(argtypes) == counts[name], (name, len(argtypes), counts[name])


def test_header_declarations_are_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    assert sorted(abi.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(7):
        assert abi.status_string(s)
    assert abi.status_string(0) == "ok"


def test_workspace_and_padded_rows(lib):
    d = abi.make_dims(32768, 512, 1024, 8, 2, 0, abi.MOE_BF16)
    fwd = abi.moe_workspace_bytes(d, abi.MOE_FWD_ONLY)
    train = abi.moe_workspace_bytes(d, abi.MOE_SAVE_FOR_BWD)
    assert 0 < fwd < train
    # h = 1024, d = 512: the down and input-gradient GEMMs run as CTA pairs
    # over 256-row units, so each expert's rows are padded to 256
    assert abi.moe_padded_rows(d) == ((32768 * 2 + 8 * 255 + 255) // 256) * 256
    # fine-grained experts (h = 128, HBM-bound: single CTAs) and float32: 128
    d1 = abi.make_dims(16384, 512, 128, 64, 8, 1024, abi.MOE_BF16)
    assert abi.moe_padded_rows(d1) == ((16384 * 8 + 64 * 127 + 127) // 128) * 128
    d2 = abi.make_dims(32768, 512, 1024, 8, 2, 0, abi.MOE_F32)
    assert abi.moe_padded_rows(d2) == ((32768 * 2 + 8 * 127 + 127) // 128) * 128
    d0 = abi.make_dims(0, 512, 1024, 8, 2, 0, abi.MOE_BF16)
    assert abi.moe_workspace_bytes(d0, abi.MOE_FWD_ONLY) > 0


@pytest.mark.parametrize("field,value", [("tokens", -1), ("experts", 0), ("experts", 257),
                                          ("top_k", 0), ("top_k", 9), ("d_model", 0),
                                          ("dtype", 7), ("shared_hidden", -64),
                                          ("capacity", -1)])
def test_invalid_dims_rejected(lib, field, value):
    d = abi.make_dims(64, 128, 128, 8, 2, 0, abi.MOE_F32)
    setattr(d, field, value)
    out = ctypes.c_size_t(0)
    assert lib.moe_workspace_bytes(ctypes.byref(d), 0, ctypes.byref(out)) == abi.MOE_ERR_INVALID_ARG
    s = abi.moe_route(d, 256, 256, None, None, 256, 256, 256, 1 << 30, None, check=False)
    assert s == abi.MOE_ERR_INVALID_ARG


def test_unsupported_shape(lib):
    d = abi.make_dims(64, 96, 128, 8, 2, 0, abi.MOE_F32)
    s = abi.moe_route(d, 256, 256, None, None, 256, 256, 256, 1 << 30, None, check=False)
    assert s == abi.MOE_ERR_UNSUPPORTED


def test_workspace_errors(lib):
    d = abi.make_dims(64, 128, 128, 8, 2, 0, abi.MOE_F32)
    need = abi.moe_workspace_bytes(d, abi.MOE_FWD_ONLY)
    # missing, misaligned, too small: all rejected before any launch
    assert abi.moe_permute(d, 256, 256, 256, 256, 256, None, need, None, check=False) == abi.MOE_ERR_WORKSPACE
    assert abi.moe_permute(d, 256, 256, 256, 256, 256, 0x1010, need, None, check=False) == abi.MOE_ERR_WORKSPACE
    assert abi.moe_permute(d, 256, 256, 256, 256, 256, 0x1000, need - 1, None, check=False) == abi.MOE_ERR_WORKSPACE
    need_t = abi.moe_workspace_bytes(d, abi.MOE_SAVE_FOR_BWD)
    ptrs = [256] * 25
    s = abi.moe_backward(d, *ptrs, 0x1000, need_t - 1, None, check=False)
    assert s == abi.MOE_ERR_WORKSPACE


def test_null_pointers_rejected(lib):
    d = abi.make_dims(64, 128, 128, 8, 2, 0, abi.MOE_F32)
    need = abi.moe_workspace_bytes(d, abi.MOE_FWD_ONLY)
    assert abi.moe_route(d, None, None, None, None, 256, 256, 0x1000, need, None, check=False) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_route(d, 256, 256, None, None, None, 256, 0x1000, need, None, check=False) == abi.MOE_ERR_INVALID_ARG
    # train mode without the saved pre-activation buffers
    assert abi.moe_grouped_ffn_fwd(d, 1, 256, 256, 256, 256, 256, 256, None, None, 0x1000, need, None,
                                   check=False) == abi.MOE_ERR_INVALID_ARG
    # unknown mode
    assert abi.moe_grouped_ffn_fwd(d, 5, 256, 256, 256, 256, 256, 256, 256, 256, 0x1000, need, None,
                                   check=False) == abi.MOE_ERR_INVALID_ARG
    # no output buffer
    assert abi.moe_combine(d, 0, None, None, None, None, None, None, None, None, None, None, 0x1000,
                           need, None, check=False) == abi.MOE_ERR_INVALID_ARG
    # a value without a place to put it
    assert abi.moe_combine(d, 0, None, None, None, None, 256, None, None, None, 256, None, 0x1000,
                           need, None, check=False) == abi.MOE_ERR_INVALID_ARG
    # a backward without the forward's saved H (routed; and shared, hs > 0)
    need_t = abi.moe_workspace_bytes(d, abi.MOE_SAVE_FOR_BWD)
    ptrs = [256] * 25
    ptrs[13] = None
    assert abi.moe_backward(d, *ptrs, 0x1000, need_t, None, check=False) == abi.MOE_ERR_INVALID_ARG
    ds = abi.make_dims(64, 128, 128, 8, 2, 64, abi.MOE_F32)
    need_s = abi.moe_workspace_bytes(ds, abi.MOE_SAVE_FOR_BWD)
    ptrs = [256] * 25
    ptrs[16] = None
    assert abi.moe_backward(ds, *ptrs, 0x1000, need_s, None, check=False) == abi.MOE_ERR_INVALID_ARG


def test_misaligned_row_data_rejected(lib):
    # row data moves in 16-byte vectors and bulk copies: an array that does
    # not start on a 16-byte boundary is refused before anything launches
    d = abi.make_dims(64, 128, 128, 8, 2, 0, abi.MOE_BF16)
    need = abi.moe_workspace_bytes(d, abi.MOE_FWD_ONLY)
    need_t = abi.moe_workspace_bytes(d, abi.MOE_SAVE_FOR_BWD)
    assert abi.moe_route(d, 0x108, 256, None, None, 256, 256, 0x1000, need, None,
                         check=False) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_grouped_ffn_fwd(d, 0, 256, 256, 256, 256, 0x2008, 256, None, None, 0x1000,
                                   need, None, check=False) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_combine(d, 0, None, None, None, None, 0x2004, None, None, None, None, None,
                           0x1000, need, None, check=False) == abi.MOE_ERR_INVALID_ARG
    for pos in (13, 17):  # the saved H, dx
        ptrs = [256] * 25
        ptrs[pos] = 0x3002
        assert abi.moe_backward(d, *ptrs, 0x1000, need_t, None,
                                check=False) == abi.MOE_ERR_INVALID_ARG


def test_capacity_routing_is_refused_by_the_allocation_free_sort(lib):
    d = abi.make_dims(64, 128, 128, 8, 2, 0, abi.MOE_BF16, capacity=8)
    assert abi.moe_permute_noalloc(d, 256, 256, 256, 256, 256, None,
                                   check=False) == abi.MOE_ERR_UNSUPPORTED
