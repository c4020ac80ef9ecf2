"""Parity of the DCP-localised sparse (top-k) attention path through the C ABI
with the fp64 oracle: the localisation bit-exact, the merged attention over
each query row's candidates within the cache dtype's tolerance."""

import numpy as np
import pytest
import torch

import oracle
from dcp_workloads import config, make_workload, sparse_candidates

from gpu_common import assert_close_rows, f64, tol_for

pytestmark = pytest.mark.gpu

CASES = {
    # name: (config, k)
    "fp8_mixed_k256": (config("mla_fp8_mixed", B=3, lengths=("list", [700, 3000, 90])), 256),
    "bf16_tq2_k128_I64": (config("mla_bf16_32k", B=2, Tq=2, lengths=("list", [1500, 50])), 128),
    "fp8_n3_i5_k512": (config("mla_fp8_mixed", B=2, N=3, I=5, lengths=("list", [4000, 600])), 512),
    # k not a multiple of the 64-token staging page; an empty row, a short
    # list, an unsorted list (see _edit)
    "fp8_n2_k100_ragged": (config("mla_fp8_mixed", B=3, Tq=2, N=2, lengths=("list", [900, 40, 3000])), 100),
    # one rank: the sparse result without any merge
    "bf16_n1_k64": (config("mla_bf16_32k", B=2, N=1, I=1, lengths=("list", [64, 500])), 64),
}


def _edit(name, cand):
    """Candidate lists the synthetic indexer does not produce by itself."""
    if name == "fp8_n2_k100_ragged":
        cand = cand.copy()
        cand[1] = -1             # no candidate at all: zeros and -inf
        cand[3, 10:] = -1        # ten candidates
        cand[4] = cand[4][::-1]  # descending order (the result does not depend on it)
    return cand

_cache = {}


def _setup(name):
    if name not in _cache:
        import context_decode_attention_gb300 as dcp
        from context_decode_attention_gb300.harness import DeviceWorkload
        cfg, k = CASES[name]
        wl = make_workload(cfg, seed=8)
        params = dcp.params_from_config(cfg, wl.kv_scale)
        ws = dcp.dcp_sparse_workspace_size(params, int(cfg["B"]), k)
        dw = DeviceWorkload(wl, workspace_bytes=ws)
        cand = _edit(name, sparse_candidates(wl, k, seed=1))
        _cache.clear()
        _cache[name] = (wl, dw, cand, k)
    return _cache[name]


@pytest.mark.parametrize("name", list(CASES))
def test_sparse_localize_bit_exact(name):
    import context_decode_attention_gb300 as dcp
    wl, dw, cand, k = _setup(name)
    c = wl.cfg
    N, Tq = int(c["N"]), int(c["Tq"])
    rows = wl.B * Tq
    local = torch.full((N, rows, k), -7, dtype=torch.int32, device="cuda")
    counts = torch.full((N, rows), -7, dtype=torch.int32, device="cuda")
    dcp.dcp_sparse_localize(dw.params, torch.from_numpy(cand).cuda(), dw.seq_lens, local, counts,
                            workspace=dw.workspace)
    ref_local, ref_counts = oracle.sparse_localize(cand, N, int(c["I"]), wl.seq_lens, Tq)
    assert np.array_equal(counts.cpu().numpy(), ref_counts)
    assert np.array_equal(local.cpu().numpy(), ref_local)
    assert dw.error_bits() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_sparse_decode_matches_oracle(name):
    import context_decode_attention_gb300 as dcp
    wl, dw, cand, k = _setup(name)
    c = wl.cfg
    out = torch.empty_like(dw.out)
    lse = torch.empty_like(dw.lse)
    dcp.dcp_sparse_decode_attention(dw.params, dw.q, torch.from_numpy(cand).cuda(), dw.k_pool, dw.num_blocks,
                                    dw.block_tables, dw.seq_lens, out, lse, workspace=dw.workspace)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ref_o, ref_l = oracle.sparse_attention(wl, cand)
    assert_close_rows(f64(out).reshape(ref_o.shape), f64(lse).reshape(-1), ref_o, ref_l, tol_for(c), name)
    # a second call on the same workspace gives the same bits
    out2 = torch.empty_like(out)
    dcp.dcp_sparse_decode_attention(dw.params, dw.q, torch.from_numpy(cand).cuda(), dw.k_pool, dw.num_blocks,
                                    dw.block_tables, dw.seq_lens, out2, None, workspace=dw.workspace)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_sparse_candidate_past_position_is_reported():
    import context_decode_attention_gb300 as dcp
    wl, dw, cand, k = _setup("fp8_mixed_k256")
    bad = cand.copy()
    bad[0, 0] = int(wl.seq_lens[0])  # past the query's own position
    out = torch.empty_like(dw.out)
    dcp.dcp_sparse_decode_attention(dw.params, dw.q, torch.from_numpy(bad).cuda(), dw.k_pool, dw.num_blocks,
                                    dw.block_tables, dw.seq_lens, out, None, workspace=dw.workspace)
    torch.cuda.synchronize()
    assert dw.error_bits() & 0x2
    # the dropped candidate: the row equals the oracle over the remaining ones
    ref_o, _ = oracle.sparse_attention(wl, np.where(bad >= int(wl.seq_lens[0]), -1, bad))
    Hq = int(wl.cfg["Hq"])
    assert np.abs(f64(out).reshape(ref_o.shape)[:Hq] - ref_o[:Hq]).max() <= tol_for(wl.cfg)[0]


def test_sparse_workspace_size_grows_with_batch_and_k():
    """The size query on the device: the staging area alone holds every rank's
    copy of every row's k candidates (k rounded up to 64 tokens); a smaller
    workspace is refused before any work is enqueued."""
    import ctypes
    import context_decode_attention_gb300 as dcp
    lib = dcp.lib()
    p = dcp.params_from_config(config("mla_fp8_mixed"))
    sizes = {}
    for B, k in [(0, 64), (1, 64), (4, 64), (4, 100), (4, 2048), (16, 2048)]:
        sizes[(B, k)] = dcp.dcp_sparse_workspace_size(p, B, k)
    assert sizes[(1, 64)] < sizes[(4, 64)] < sizes[(16, 2048)]
    assert sizes[(4, 64)] < sizes[(4, 100)] <= sizes[(4, 2048)]
    assert sizes[(16, 2048)] >= p.N * 16 * p.Tq * 2048 * 576
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    dummy = ctypes.c_void_p(small.data_ptr())
    rc = lib.dcp_sparse_decode_attention(ctypes.byref(p), 2, 64, dummy, dummy, dummy, 10, dummy, 4, dummy, dummy,
                                         None, dummy, 1024, None)
    assert rc == 4
