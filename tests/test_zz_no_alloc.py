"""The no-allocation decode entry point, through the C ABI, against the
workspace-taking dcp_decode_attention.

dcp_decode_attention_noalloc serves callers that may not allocate device
memory while they run attention: a plugin inside an engine that owns all
device memory and hands none out, or a path where an allocation's latency or
possible failure is not acceptable.  Its scratch is a static device buffer
inside the library.  It must give the workspace path's results, call after call,
since every call reuses (and so inherits) the same buffer.  Collected last
(file name) so a failure here cannot hide another test's result.
"""

import pytest
import torch

from dcp_workloads import config, make_workload

from gpu_common import assert_close_rows, f64, tol_for

pytestmark = pytest.mark.gpu


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
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(dw.out, float("nan"))
        lse = torch.full_like(dw.lse, float("nan"))
        dcp.dcp_decode_attention_noalloc(dw.params, dw.q, dw.k_pool, dw.v_pool, dw.num_blocks, dw.block_tables,
                                         dw.seq_lens, dw.local_lens, out, lse)
        torch.cuda.synchronize()
        assert_close_rows(f64(out).reshape(-1, dw.Dv), f64(lse).reshape(-1), f64(ref_out).reshape(-1, dw.Dv),
                          f64(ref_lse).reshape(-1), tol_for(cfg), "noalloc vs workspace")


def test_noalloc_rejects_problems_beyond_its_scratch():
    """The C entry point itself turns down a problem whose scratch would not
    fit in the static buffer (DCP_ERR_WORKSPACE), before it reads any of the
    argument buffers.  Called through the C ABI directly: the Python binding
    would already refuse these deliberately tiny stand-in buffers."""
    import ctypes
    import context_decode_attention_gb300 as dcp
    from context_decode_attention_gb300 import params_from_config
    p = params_from_config(config("mla_bf16_32k"))
    B = 4096  # needs far more partial slots than the static buffer holds
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    seq = torch.ones(B, dtype=torch.int32, device="cuda")
    d, s = dummy.data_ptr(), seq.data_ptr()
    stream = torch.cuda.current_stream().cuda_stream
    rc = dcp.lib().dcp_decode_attention_noalloc(ctypes.byref(p), B, d, d, None, 1, d, 16, s, d, d, None, stream)
    assert rc == 4  # DCP_ERR_WORKSPACE
