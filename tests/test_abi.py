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


def test_plan_ahead_entry_points_validate_before_launching(libdcp):
    """dcp_decode_plan and dcp_decode_attention_planned refuse bad arguments on
    the host, before any device query or launch (codes: 1 invalid argument, 4
    workspace), and an empty batch is a no-op."""
    p = _good()
    dummy = ctypes.c_void_p(256)
    # the plan: lengths and a block-table width are all it needs
    assert libdcp.dcp_decode_plan(ctypes.byref(p), 0, None, None, 4, None, 0, None) == 0
    assert libdcp.dcp_decode_plan(ctypes.byref(p), -1, dummy, dummy, 4, dummy, 1 << 20, None) == 1
    assert libdcp.dcp_decode_plan(ctypes.byref(p), 4, None, dummy, 4, dummy, 1 << 20, None) == 1
    assert libdcp.dcp_decode_plan(ctypes.byref(p), 4, dummy, None, 4, dummy, 1 << 20, None) == 1
    assert libdcp.dcp_decode_plan(ctypes.byref(p), 4, dummy, dummy, 0, dummy, 1 << 20, None) == 1
    assert libdcp.dcp_decode_plan(ctypes.byref(p), 4, dummy, dummy, 4, None, 1 << 20, None) == 4
    bad = _good()
    bad.N = 0
    assert libdcp.dcp_decode_plan(ctypes.byref(bad), 4, dummy, dummy, 4, dummy, 1 << 20, None) == 1
    # the planned attention: the fused call's argument rules
    f = libdcp.dcp_decode_attention_planned
    assert f(ctypes.byref(p), 0, None, None, None, 0, None, 4, None, None, None, None, None, 0, None) == 0
    assert f(ctypes.byref(p), 4, None, dummy, dummy, 10, dummy, 4, dummy, dummy, dummy, None, dummy, 1 << 20,
             None) == 1
    assert f(ctypes.byref(p), 4, dummy, dummy, None, 10, dummy, 4, dummy, dummy, dummy, None, dummy, 1 << 20,
             None) == 1  # a GQA call needs the value pool
    assert f(ctypes.byref(p), 4, dummy, dummy, dummy, 10, dummy, 4, dummy, dummy, None, None, dummy, 1 << 20,
             None) == 1  # no output
    assert f(ctypes.byref(p), 4, dummy, dummy, dummy, 10, dummy, 4, dummy, dummy, dummy, None, None, 0,
             None) == 4  # no workspace
    assert f(ctypes.byref(p), 4, dummy, ctypes.c_void_p(258), dummy, 10, dummy, 4, dummy, dummy, dummy, None,
             dummy, 1 << 20, None) == 1  # misaligned pool


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
    # owner ranks are stored as int8: more than 127 ranks with an owner output is refused
    # (the same call without owner passes these checks; 127 ranks with owner too)
    for N, owner, want in [(128, dummy, 1), (300, dummy, 1)]:
        p.N = N
        rc = libdcp.dcp_slot_mapping(ctypes.byref(p), 2, dummy, 5, dummy, dummy, None, 0, 0, owner, None, None,
                                     None, None, None, None, None, None, dummy, 1024, None)
        assert rc == want, (N, rc)


@pytest.mark.parametrize("name,kernel", [
    ("gqa_toy", "generic"), ("gqa_llama8b", "gqa_mma"), ("mla_bf16_32k", "mla_tcgen05"),
    ("mla_fp8_mixed", "mla_tcgen05"), ("mla_fp8_1m", "mla_tcgen05"),
])
def test_each_workload_selects_its_kernel(libdcp, name, kernel):
    from context_decode_attention_gb300 import dcp_attention_kernel, params_from_config
    from dcp_workloads import config
    assert dcp_attention_kernel(params_from_config(config(name), kv_scale=0.01 if "fp8" in name else 1.0)) == kernel


# ----- host validation of the entry points beyond decode (no GPU is touched:
# every call below returns before its first CUDA call)

def _mla(name="mla_fp8_mixed", **kw):
    from context_decode_attention_gb300 import params_from_config
    from dcp_workloads import config
    return params_from_config(config(name, **kw))


def test_sparse_workspace_size_rules(libdcp):
    """Argument rules of the size query (the size itself needs the device's SM
    count: tests/test_gpu_sparse.py checks it)."""
    p = _mla()
    n = ctypes.c_size_t(0)
    assert libdcp.dcp_sparse_workspace_size(ctypes.byref(p), 4, 0, ctypes.byref(n)) == 1
    assert libdcp.dcp_sparse_workspace_size(ctypes.byref(p), -1, 64, ctypes.byref(n)) == 1
    g = _good()  # GQA: the sparse path is MLA only
    assert libdcp.dcp_sparse_workspace_size(ctypes.byref(g), 4, 64, ctypes.byref(n)) == 2
    wide = _mla(N=33)
    assert libdcp.dcp_sparse_workspace_size(ctypes.byref(wide), 4, 64, ctypes.byref(n)) == 2


def test_sparse_entry_points_validate_before_launching(libdcp):
    p = _mla()
    dummy = ctypes.c_void_p(256)
    # empty batch: nothing to do
    assert libdcp.dcp_sparse_decode_attention(ctypes.byref(p), 0, 64, dummy, dummy, dummy, 10, dummy, 4, dummy,
                                              dummy, None, dummy, 1 << 20, None) == 0
    # missing query / candidates / output
    for i in (3, 4, 10):
        args = [ctypes.byref(p), 2, 64, dummy, dummy, dummy, 10, dummy, 4, dummy, dummy, None, dummy, 1 << 30, None]
        args[i] = None
        assert libdcp.dcp_sparse_decode_attention(*args) == 1, i
    # no workspace
    assert libdcp.dcp_sparse_decode_attention(ctypes.byref(p), 2, 64, dummy, dummy, dummy, 10, dummy, 4, dummy,
                                              dummy, None, None, 0, None) == 4
    assert libdcp.dcp_sparse_localize(ctypes.byref(p), 2, 0, dummy, dummy, dummy, dummy, dummy, 1 << 20,
                                      None) == 1


def test_pcp_partition_and_prefill_rules(libdcp):
    dummy = ctypes.c_void_p(256)
    # K >= 1, B >= 0, max_q >= 0; a workspace for the error word; empty batch is a no-op
    assert libdcp.dcp_pcp_partition(0, 2, dummy, dummy, 8, dummy, dummy, dummy, 256, None) == 1
    assert libdcp.dcp_pcp_partition(2, -1, dummy, dummy, 8, dummy, dummy, dummy, 256, None) == 1
    assert libdcp.dcp_pcp_partition(2, 2, dummy, dummy, 8, dummy, dummy, None, 0, None) == 4
    assert libdcp.dcp_pcp_partition(2, 0, None, None, 8, None, None, dummy, 256, None) == 0
    assert libdcp.dcp_pcp_partition(2, 2, dummy, None, 8, dummy, dummy, dummy, 256, None) == 1
    g = _good()
    args = [ctypes.byref(g), 0, 16, dummy, dummy, dummy, dummy, 10, dummy, 4, dummy, dummy, dummy, dummy,
            None, None, dummy, 256, None]
    assert libdcp.dcp_prefill_attention(*args) == 0  # empty batch
    args[1] = -1
    assert libdcp.dcp_prefill_attention(*args) == 1
    args[1] = 2
    args[3] = None  # no query
    assert libdcp.dcp_prefill_attention(*args) == 1
    args[3] = dummy
    args[16], args[17] = None, 0
    assert libdcp.dcp_prefill_attention(*args) == 4
    m = _mla()  # MLA prefill is not built
    args = [ctypes.byref(m), 2, 16, dummy, dummy, dummy, dummy, 10, dummy, 4, dummy, dummy, dummy, dummy,
            None, None, dummy, 256, None]
    assert libdcp.dcp_prefill_attention(*args) == 2


def test_transfer_blocks_rules(libdcp):
    p = _good()
    dummy = ctypes.c_void_p(256)
    # B < 0; no workspace; empty batch with no totals is a no-op; missing inputs
    assert libdcp.dcp_transfer_blocks(ctypes.byref(p), -1, dummy, dummy, 4, 10, dummy, dummy, dummy, None,
                                      dummy, 256, None) == 1
    assert libdcp.dcp_transfer_blocks(ctypes.byref(p), 2, dummy, dummy, 4, 10, dummy, dummy, dummy, None,
                                      None, 0, None) == 4
    assert libdcp.dcp_transfer_blocks(ctypes.byref(p), 0, None, None, 4, 10, None, None, None, None,
                                      dummy, 256, None) == 0
    assert libdcp.dcp_transfer_blocks(ctypes.byref(p), 2, None, dummy, 4, 10, dummy, dummy, dummy, None,
                                      dummy, 256, None) == 1


def test_binding_refuses_host_tensors(libdcp):
    """The Python binding passes plain pointers, so it refuses a host tensor
    before calling into the library (no GPU is touched)."""
    import torch
    import context_decode_attention_gb300 as dcp
    o = torch.zeros((2, 3, 8))
    l = torch.zeros((2, 3))
    with pytest.raises(ValueError, match="device tensors"):
        dcp.dcp_lse_merge(2, 3, 8, o, l, torch.zeros((3, 8)), dcp.DCP_F32, torch.zeros(3))
    with pytest.raises(ValueError, match="device tensors"):
        dcp.dcp_pcp_partition(2, torch.zeros(2, dtype=torch.int32), torch.zeros(2, dtype=torch.int32), 8,
                              torch.zeros((2, 8), dtype=torch.int32), torch.zeros(2, dtype=torch.int32),
                              workspace=torch.zeros(256, dtype=torch.uint8))


def test_binding_refuses_buffers_too_small_for_the_params(libdcp):
    """The library reads through plain pointers, so a short buffer or one of
    the wrong element size would be read past its end on the device.  The
    binding compares every buffer with the params and sizes before calling in
    (checked here on host tensors: the size check comes first)."""
    import torch
    import context_decode_attention_gb300 as dcp
    from dcp_workloads import config

    cfg = config("gqa_llama8b", B=2)
    p = dcp.params_from_config(cfg)
    B, Tq, Hq, Hkv, D, N, bs, nb, mb = 2, 1, 32, 8, 128, 4, 16, 10, 3
    ok = dict(
        q=torch.zeros((B, Tq, Hq, D), dtype=torch.bfloat16),
        k_pool=torch.zeros((nb, Hkv, bs, D), dtype=torch.bfloat16),
        v_pool=torch.zeros((nb, Hkv, bs, D), dtype=torch.bfloat16),
        block_tables=torch.zeros((N, B, mb), dtype=torch.int32),
        seq_lens=torch.zeros(B, dtype=torch.int32), local_lens=torch.zeros((N, B), dtype=torch.int32),
        out=torch.zeros((B, Tq, Hq, D), dtype=torch.bfloat16), lse=torch.zeros((B, Tq, Hq)),
    )

    def decode(**over):
        a = dict(ok, **over)
        dcp.dcp_decode_attention(p, a["q"], a["k_pool"], a["v_pool"], nb, a["block_tables"], a["seq_lens"],
                                 a["local_lens"], a["out"], a["lse"], torch.zeros(256, dtype=torch.uint8))

    # right sizes: the checks pass and the host-tensor refusal follows
    with pytest.raises(ValueError, match="device tensors"):
        decode()
    bad = {
        "q": ok["q"][:1],                                             # one request short
        "k_pool": ok["k_pool"][:-1],                                  # one block short
        "v_pool": ok["v_pool"].to(torch.float32),                     # 4-byte elements for a bf16 cache
        "block_tables": ok["block_tables"].to(torch.int64),
        "local_lens": ok["local_lens"][:1],
        "out": ok["out"].to(torch.float32)[..., :64],                 # f32 where the params say bf16
        "lse": ok["lse"][:1],
    }
    for name, t in bad.items():
        with pytest.raises(ValueError, match=name):
            decode(**{name: t.contiguous()})

    # the merge: N partials of rows x Dv
    o, l = torch.zeros((2, 3, 8)), torch.zeros((2, 3))
    with pytest.raises(ValueError, match="out_partial"):
        dcp.dcp_lse_merge(2, 3, 8, o[:1].contiguous(), l, torch.zeros((3, 8)), dcp.DCP_F32, torch.zeros(3))
    with pytest.raises(ValueError, match="out"):
        dcp.dcp_lse_merge(2, 3, 8, o, l, torch.zeros((3, 8), dtype=torch.bfloat16), dcp.DCP_F32, torch.zeros(3))

    # slot mapping: slots are int64 [N][T]
    T = 5
    with pytest.raises(ValueError, match="slots"):
        dcp.dcp_slot_mapping(p, ok["seq_lens"], torch.zeros(T, dtype=torch.int32), torch.zeros(T, dtype=torch.int64),
                             ok["block_tables"], nb, slots=torch.zeros((N, T), dtype=torch.int32))
    with pytest.raises(ValueError, match="new_k"):
        dcp.dcp_slot_mapping(p, ok["seq_lens"], torch.zeros(T, dtype=torch.int32), torch.zeros(T, dtype=torch.int64),
                             ok["block_tables"], nb, new_k=torch.zeros((T - 1, Hkv, D), dtype=torch.bfloat16),
                             k_pool=ok["k_pool"], v_pool=ok["v_pool"])


def test_binding_size_checks_cover_the_other_entry_points(libdcp):
    """Transfer listing, PCP partition, prefill and sparse calls refuse short
    buffers on the host too (host tensors: the size check comes first)."""
    import torch
    import context_decode_attention_gb300 as dcp
    from dcp_workloads import config

    i32 = dict(dtype=torch.int32)
    p = dcp.params_from_config(config("gqa_llama8b", B=2))
    N, B, M = 4, 2, 3
    seq, bt = torch.zeros(B, **i32), torch.zeros((N, B, M), **i32)
    with pytest.raises(ValueError, match="fills"):
        dcp.dcp_transfer_blocks(p, seq, bt, 10, torch.zeros((N, B), **i32), torch.zeros((N, B, M), **i32),
                                torch.zeros((N, B, M - 1), **i32), torch.zeros(2, dtype=torch.int64))
    with pytest.raises(ValueError, match="totals"):
        dcp.dcp_transfer_blocks(p, seq, bt, 10, torch.zeros((N, B), **i32), totals=torch.zeros(2, **i32))
    with pytest.raises(ValueError, match="pos"):
        dcp.dcp_pcp_partition(2, seq, seq, 8, torch.zeros((B, 7), **i32), torch.zeros(B, **i32))
    with pytest.raises(ValueError, match="device tensors"):  # right sizes: only the host refusal remains
        dcp.dcp_pcp_partition(2, seq, seq, 8, torch.zeros((B, 8), **i32), torch.zeros(B, **i32))

    Tq, Hq, D = 4, 32, 128
    pool = torch.zeros((10, 8, 16, D), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out_partial"):
        dcp.dcp_prefill_attention(p, torch.zeros((B, Tq, Hq, D), dtype=torch.bfloat16), torch.zeros((B, Tq), **i32),
                                  pool, pool, 10, bt, seq, torch.zeros((N, B), **i32),
                                  torch.zeros((N, B, Tq, Hq, D - 1)), torch.zeros((N, B, Tq, Hq)))

    m = dcp.params_from_config(config("mla_fp8_mixed", B=2))
    k = 64
    q = torch.zeros((B, 1, 128, 576), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="local"):
        dcp.dcp_sparse_localize(m, torch.zeros((B, k), **i32), seq, torch.zeros((8, B, k - 1), **i32),
                                torch.zeros((8, B), **i32))
    with pytest.raises(ValueError, match="k_pool"):
        dcp.dcp_sparse_decode_attention(m, q, torch.zeros((B, k), **i32), torch.zeros((10, 64, 575), dtype=torch.uint8),
                                        10, torch.zeros((8, B, M), **i32), seq,
                                        torch.zeros((B, 1, 128, 512), dtype=torch.bfloat16))


def test_a_plain_c_program_compiles_links_and_calls_the_library(libdcp, tmp_path):
    """The boundary is a C ABI: a C99 program that includes include/dcp.h,
    links libdcp.so and calls the entry points that need no device (version,
    error strings, host validation) works without any C++ or torch."""
    import shutil
    import subprocess
    from context_decode_attention_gb300 import build
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "caller.c"
    src.write_text(
        '#include <stdio.h>\n#include "dcp.h"\n'
        "int main(void) {\n"
        "    dcp_params p = {0};  /* N = 0: rejected by host validation, no device touched */\n"
        "    size_t n = 0;\n"
        "    int rc = dcp_workspace_size(&p, 1, 1, &n);\n"
        '    printf("%d %d %s\\n", dcp_version(), rc, dcp_error_string(rc));\n'
        "    return 0;\n"
        "}\n")
    exe = tmp_path / "caller"
    libdir = os.path.dirname(build.LIB)
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src),
                        "-L", libdir, "-ldcp", f"-Wl,-rpath,{libdir}", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "1 1 invalid argument"
