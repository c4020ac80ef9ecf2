"""The C-ABI library builds, loads and exports every symbol include/*.h
declares; host-side validation rejects bad arguments before touching a GPU.
(No compute call runs here: these tests need no GPU.)"""

import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def libdcp():
    from context_decode_attention_gb300 import build
    build.build()
    import context_decode_attention_gb300 as dcp
    return dcp.lib()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(dcp_\w+)\s*\(", text, re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["dcp_slot_mapping", "dcp_partial_attention", "dcp_lse_merge", "dcp_decode_attention",
              "dcp_workspace_size", "dcp_get_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(libdcp):
    from context_decode_attention_gb300._lib import EXPORTS
    declared = _declared()
    assert declared == set(EXPORTS)
    for n in declared:
        assert hasattr(libdcp, n), n
    assert libdcp.dcp_version() == 1
    assert libdcp.dcp_error_string(1) == b"invalid argument"


def test_params_struct_layout():
    from context_decode_attention_gb300 import DcpParams
    assert ctypes.sizeof(DcpParams) == 14 * 4
    assert DcpParams.kv_scale.offset == 12 * 4


def _good():
    from context_decode_attention_gb300 import params_from_config
    from dcp_workloads import config
    return params_from_config(config("gqa_llama8b"))


@pytest.mark.parametrize("field,value", [
    ("N", 0), ("I", 0), ("block_size", 0), ("layout", 7), ("Hq", 0), ("Hkv", 3), ("Dk", 0),
    ("Tq", 0), ("q_dtype", 2), ("kv_dtype", 9), ("out_dtype", 2), ("kv_scale", 2.0),
    ("softmax_scale", float("nan")),
])
def test_host_validation_rejects_bad_params(libdcp, field, value):
    p = _good()
    setattr(p, field, value)
    n = ctypes.c_size_t(0)
    assert libdcp.dcp_workspace_size(ctypes.byref(p), 4, 100, ctypes.byref(n)) == 1
    dummy = ctypes.c_void_p(256)
    rc = libdcp.dcp_decode_attention(ctypes.byref(p), 4, dummy, dummy, dummy, 10, dummy, 4, dummy, dummy,
                                     dummy, None, dummy, 1 << 20, None)
    assert rc == 1


def test_mla_params_need_one_kv_head_and_no_value_pool(libdcp):
    from context_decode_attention_gb300 import params_from_config
    from dcp_workloads import config
    p = params_from_config(config("mla_bf16_32k"))
    p.Hkv = 2
    n = ctypes.c_size_t(0)
    assert libdcp.dcp_workspace_size(ctypes.byref(p), 4, 100, ctypes.byref(n)) == 1
    p = params_from_config(config("mla_bf16_32k"))
    dummy = ctypes.c_void_p(256)
    rc = libdcp.dcp_decode_attention(ctypes.byref(p), 4, dummy, dummy, dummy, 10, dummy, 4, dummy, dummy,
                                     dummy, None, dummy, 1 << 20, None)
    assert rc == 1  # v_pool must be NULL for MLA


def test_null_pointers_and_workspace_rejected(libdcp):
    p = _good()
    dummy = ctypes.c_void_p(256)
    rc = libdcp.dcp_decode_attention(ctypes.byref(p), 4, None, dummy, dummy, 10, dummy, 4, dummy, dummy,
                                     dummy, None, dummy, 1 << 20, None)
    assert rc == 1
    rc = libdcp.dcp_decode_attention(ctypes.byref(p), 4, dummy, dummy, dummy, 10, dummy, 4, dummy, dummy,
                                     dummy, None, None, 0, None)
    assert rc == 4
    assert libdcp.dcp_lse_merge(0, 5, 8, dummy, dummy, dummy, 0, None, None) == 1
    assert libdcp.dcp_lse_merge(2, 5, 8, dummy, dummy, dummy, 2, None, None) == 1
    # misaligned pool pointer
    rc = libdcp.dcp_decode_attention(ctypes.byref(p), 4, dummy, ctypes.c_void_p(258), dummy, 10, dummy, 4,
                                     dummy, dummy, dummy, None, dummy, 1 << 20, None)
    assert rc == 1


def test_slot_mapping_argument_rules(libdcp):
    p = _good()
    dummy = ctypes.c_void_p(256)
    # slots requested without block tables
    rc = libdcp.dcp_slot_mapping(ctypes.byref(p), 2, dummy, 5, dummy, dummy, None, 0, 0, None, dummy, None,
                                 None, None, None, None, None, None, dummy, 1024, None)
    assert rc == 1
    # GQA scatter without values
    rc = libdcp.dcp_slot_mapping(ctypes.byref(p), 2, dummy, 5, dummy, dummy, dummy, 4, 10, None, None, None,
                                 None, None, dummy, None, dummy, None, dummy, 1024, None)
    assert rc == 1
    # workspace too small for the error word
    rc = libdcp.dcp_slot_mapping(ctypes.byref(p), 2, dummy, 0, None, None, None, 0, 0, None, None, dummy,
                                 None, None, None, None, None, None, dummy, 16, None)
    assert rc == 4


@pytest.mark.parametrize("name,kernel", [
    ("gqa_toy", "generic"), ("gqa_llama8b", "gqa_mma"), ("mla_bf16_32k", "mla_tcgen05"),
    ("mla_fp8_mixed", "mla_tcgen05"), ("mla_fp8_1m", "mla_tcgen05"),
])
def test_each_workload_selects_its_kernel(libdcp, name, kernel):
    from context_decode_attention_gb300 import dcp_attention_kernel, params_from_config
    from dcp_workloads import config
    assert dcp_attention_kernel(params_from_config(config(name), kv_scale=0.01 if "fp8" in name else 1.0)) == kernel
