"""The no-allocation decode entry point, through the C ABI, against the
workspace-taking dcp_decode_attention.

dcp_decode_attention_noalloc serves callers that may not allocate device
memory while they run attention: a plugin inside an engine that owns all
device memory and hands none out, or a path where an allocation's latency or
possible failure is not acceptable.  Its scratch is a static device buffer
inside the library.  It runs the same plan and kernels as the workspace path,
so it must give the same results bit for bit, call after call, since every
call reuses (and so inherits) the same buffer; and it must not allocate.
Collected last (file name) so a failure here cannot hide another test's
result.
"""

import pytest
import torch

from dcp_workloads import config, make_workload

pytestmark = pytest.mark.gpu


def _static_scratch_bytes():
    """DCP_STATIC_SCRATCH_BYTES as include/dcp.h defines it."""
    import os
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dcp.h")
    m = re.search(r"#define DCP_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)", open(hdr).read())
    assert m, "DCP_STATIC_SCRATCH_BYTES not found in include/dcp.h"
    return int(m.group(1)) << int(m.group(2))


@pytest.mark.parametrize("cfg", [
    config("gqa_llama8b", B=3, lengths=("list", [900, 41, 300])),
    config("mla_fp8_mixed", B=2, lengths=("list", [1500, 260])),
])
def test_noalloc_decode_matches_workspace_decode_twice(cfg):
    import context_decode_attention_gb300 as dcp
    from context_decode_attention_gb300.harness import DeviceWorkload
    wl = make_workload(cfg, seed=21)
    dw = DeviceWorkload(wl)
    ref_out, ref_lse = dw.decode()
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    out = torch.empty_like(dw.out)
    lse = torch.empty_like(dw.lse)

    def call():
        dcp.dcp_decode_attention_noalloc(dw.params, dw.q, dw.k_pool, dw.v_pool, dw.num_blocks, dw.block_tables,
                                         dw.seq_lens, dw.local_lens, out, lse)

    call()  # the first call on a device looks up the buffer (and loads the kernels)
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    for _ in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        call()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), "noalloc differs from the workspace path"
        assert dcp.dcp_noalloc_get_error() == 0
    # no allocation by the calls: torch's pool and the device's free memory are unchanged
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_reports_device_errors():
    """A block id outside the pool is caught on the device (the access is
    skipped) and its bit is read back from the static buffer; the next clean
    call reports nothing."""
    import context_decode_attention_gb300 as dcp
    from context_decode_attention_gb300.harness import DeviceWorkload
    wl = make_workload(config("gqa_llama8b", B=2, lengths=("list", [300, 77])), seed=5)
    dw = DeviceWorkload(wl)
    bad = dw.block_tables.clone()
    bad[0, 0, 0] = dw.num_blocks + 9
    out, lse = torch.empty_like(dw.out), torch.empty_like(dw.lse)
    for tables, want in [(bad, 0x1), (dw.block_tables, 0)]:
        dcp.dcp_decode_attention_noalloc(dw.params, dw.q, dw.k_pool, dw.v_pool, dw.num_blocks, tables,
                                         dw.seq_lens, dw.local_lens, out, lse)
        bits = dcp.dcp_noalloc_get_error()
        assert (bits & 0x1) == want, hex(bits)
    assert dcp.dcp_noalloc_get_error() == 0  # read and cleared


def test_noalloc_rejects_problems_beyond_its_scratch():
    """The C entry point itself turns down a problem whose scratch would not
    fit in the static buffer (DCP_ERR_WORKSPACE), before it reads any of the
    argument buffers.  Called through the C ABI directly: the Python binding
    would already refuse these deliberately tiny stand-in buffers.  The
    problem's scratch is checked first, on the host, so that a smaller one
    could never reach the kernels with these buffers."""
    import ctypes
    import context_decode_attention_gb300 as dcp
    from context_decode_attention_gb300 import params_from_config
    p = params_from_config(config("mla_bf16_32k"))
    B = 4096  # needs far more partial slots than the static buffer holds
    need = dcp.dcp_workspace_size(p, B, 1)
    scratch = _static_scratch_bytes()
    if not need > scratch:
        pytest.fail(f"the rejection case needs {need} B, not more than the {scratch} B scratch: not calling")
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    seq = torch.ones(B, dtype=torch.int32, device="cuda")
    d, s = dummy.data_ptr(), seq.data_ptr()
    stream = torch.cuda.current_stream().cuda_stream
    rc = dcp.lib().dcp_decode_attention_noalloc(ctypes.byref(p), B, d, d, None, 1, d, 16, s, d, d, None, stream)
    assert rc == 4  # DCP_ERR_WORKSPACE
