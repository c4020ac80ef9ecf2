"""Parity at the full workload sizes, in the launch configuration the bench
times: metadata and slots bit-exact against the oracle, and every element of
the decode step's attention output (all query rows of all requests) against
the threaded fp64 oracle; the prefill and sparse workloads on sampled rows."""

import numpy as np
import pytest
import torch

import oracle
from dcp_workloads import CONFIG_ORDER, config, make_workload

from gpu_common import assert_close_rows, f64, tol_for

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_full_size(name):
    from context_decode_attention_gb300.harness import DeviceWorkload
    wl = make_workload(config(name))
    dw = DeviceWorkload(wl)
    c = wl.cfg
    N, I, bs = int(c["N"]), int(c["I"]), int(c["block_size"])
    # metadata, bit-exact
    meta = oracle.slot_mapping(N, I, bs, wl.seq_lens, np.zeros(0, np.int32), np.zeros(0, np.int64))
    assert np.array_equal(dw.local_lens.cpu().numpy(), meta["local_lens"])
    assert np.array_equal(dw.virt_blocks.cpu().numpy(), meta["virt_blocks"])
    assert np.array_equal(dw.rank_blocks.cpu().numpy(), meta["rank_blocks"])
    # slots of the decode step's tokens and of a random token sample, bit-exact
    nr, npos = wl.new_token_lists()
    rng = np.random.default_rng(1)
    sr = rng.integers(0, int(c["B"]), size=4096).astype(np.int32)
    sp = (rng.random(4096) * wl.seq_lens[sr]).astype(np.int64)
    tok_req, tok_pos = np.concatenate([nr, sr]), np.concatenate([npos, sp])
    ref = oracle.slot_mapping(N, I, bs, wl.seq_lens, tok_req, tok_pos, dw.block_tables_host)
    owner, slots = dw.slot_mapping(tok_req, tok_pos)
    assert np.array_equal(owner.cpu().numpy(), ref["owner"])
    assert np.array_equal(slots.cpu().numpy(), ref["slots"])
    # one decode step exactly as the bench runs it
    out, lse = dw.step()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    lse_h = f64(lse).reshape(-1)
    out_h = f64(out).reshape(lse_h.size, -1)
    assert np.all(np.isfinite(lse_h)) and np.all(np.isfinite(out_h))
    # a convex combination of values: |out| <= max |v|
    assert np.abs(out_h).max() <= np.abs(oracle.decode(wl.k[:4096], c["kv_dtype"], wl.kv_scale)).max() * 2 + 10
    # every row, every element (fp64 oracle over all host cores)
    ref_o, ref_l = oracle.attention(wl)
    assert_close_rows(out_h, lse_h, ref_o, ref_l, tol_for(c), f"{name} all rows")


def test_full_size_prefill():
    """The PCP prefill workload (2 x a 2K chunk on a 64K context, PCP 4 x DCP 4,
    64-token pages) exactly as the bench runs it: partition bit-exact, merged
    rows sampled across the chunk (both ends, the head-tail split points, random
    tokens) against the oracle's causal attention of those rows."""
    from context_decode_attention_gb300.harness import DeviceWorkload
    cfg = config("gqa_prefill_64k")
    wl = make_workload(cfg, seed=int(cfg["index"]))
    dw = DeviceWorkload(wl, workspace_bytes=256)
    K = int(cfg["pcp"])
    dw.prefill_setup(K)
    B, Tq, Hq = int(cfg["B"]), int(cfg["Tq"]), int(cfg["Hq"])
    for _ in range(2):
        dw.write_new_tokens()
        out, lse = dw.prefill()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ref = oracle.pcp_partition(K, wl.seq_lens - Tq, np.full(B, Tq), dw.max_q)
    assert np.array_equal(dw.q_pos.cpu().numpy(), ref["pos"])
    pos = ref["pos"].astype(np.int64)
    ctx = wl.seq_lens.astype(np.int64) - Tq
    rng = np.random.default_rng(11)
    piece = Tq // (2 * K)
    toks = sorted(set([0, Tq - 1] + [p * piece for p in range(2 * K)] + [p * piece - 1 for p in range(1, 2 * K)]
                      + rng.integers(0, Tq, size=16).tolist()))
    picks = []  # (b, gathered index, natural token, head)
    for b in range(B):
        where = {int(p - ctx[b]): j for j, p in enumerate(pos[b]) if p >= 0}
        assert sorted(where) == list(range(Tq))
        for t in toks:
            for h in sorted({int(rng.integers(0, Hq)), (7 * t + b) % Hq}):
                picks.append((b, where[t], t, h))
    rows = np.array([(b * Tq + t) * Hq + h for b, _, t, h in picks], dtype=np.int64)
    ref_o, ref_l = oracle.attention(wl, rows=rows)
    got_o, got_l = f64(out), f64(lse)
    bi = np.array([p[0] for p in picks])
    ji = np.array([p[1] for p in picks])
    hi = np.array([p[3] for p in picks])
    assert_close_rows(got_o[bi, ji, hi], got_l[bi, ji, hi], ref_o, ref_l, tol_for(cfg), "prefill sampled rows")


def test_full_size_sparse():
    """The sparse workload (the 16 mixed-context MLA requests, 4 query tokens per request,
    2,048 candidates per token) exactly as the bench runs it: localisation
    bit-exact for every row, merged output of sampled query tokens (all heads)
    against the oracle's attention over their candidates."""
    import context_decode_attention_gb300 as dcp
    from context_decode_attention_gb300.harness import DeviceWorkload
    from dcp_workloads import sparse_candidates
    cfg = config("mla_fp8_sparse_2k")
    wl = make_workload(cfg, seed=int(cfg["index"]))
    k = int(cfg["topk"])
    params = dcp.params_from_config(cfg, wl.kv_scale)
    B, Tq, N = int(cfg["B"]), int(cfg["Tq"]), int(cfg["N"])
    dw = DeviceWorkload(wl, workspace_bytes=dcp.dcp_sparse_workspace_size(params, B, k))
    cand_h = sparse_candidates(wl, k, seed=1)
    cand = torch.from_numpy(cand_h).cuda()
    out = torch.empty_like(dw.out)
    lse = torch.empty_like(dw.lse)
    for _ in range(2):
        dcp.dcp_sparse_decode_attention(dw.params, dw.q, cand, dw.k_pool, dw.num_blocks, dw.block_tables,
                                        dw.seq_lens, out, lse, workspace=dw.workspace)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    rows = B * Tq
    local = torch.full((N, rows, k), -7, dtype=torch.int32, device="cuda")
    counts = torch.full((N, rows), -7, dtype=torch.int32, device="cuda")
    dcp.dcp_sparse_localize(dw.params, cand, dw.seq_lens, local, counts, workspace=dw.workspace)
    ref_local, ref_counts = oracle.sparse_localize(cand_h, N, int(cfg["I"]), wl.seq_lens, Tq)
    assert np.array_equal(counts.cpu().numpy(), ref_counts)
    assert np.array_equal(local.cpu().numpy(), ref_local)
    # sampled query tokens: the longest and the shortest request, random others
    rng = np.random.default_rng(5)
    b_long, b_short = int(np.argmax(wl.seq_lens)), int(np.argmin(wl.seq_lens))
    pick = sorted({b_long * Tq + Tq - 1, b_short * Tq, *rng.integers(0, rows, size=4).tolist()})
    sub = np.full_like(cand_h, -1)
    sub[pick] = cand_h[pick]
    ref_o, ref_l = oracle.sparse_attention(wl, sub)
    Hq = int(cfg["Hq"])
    sel = np.concatenate([np.arange(i * Hq, (i + 1) * Hq) for i in pick])
    got_o = f64(out).reshape(ref_o.shape)
    got_l = f64(lse).reshape(-1)
    assert_close_rows(got_o[sel], got_l[sel], ref_o[sel], ref_l[sel], tol_for(cfg), "sparse sampled tokens")
