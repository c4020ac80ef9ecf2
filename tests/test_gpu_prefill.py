"""Parity of the PCP prefill path through the C ABI with the fp64 CPU oracle:
the head-tail partition bit-exact, and causal prefill attention of the
gathered query rows (per-rank partials and their merge) element by element.

The chunk is each request's newest Tq tokens, already in the cache; the
oracle computes attention in position order (query t at position L - Tq + t),
and the GPU rows, gathered in head-tail order, are mapped back by position."""

import numpy as np
import pytest
import torch

import oracle
from dcp_workloads import config, make_workload

from gpu_common import assert_close_rows, f64, tol_for

pytestmark = pytest.mark.gpu

CASES = {
    # name: (config, PCP ranks K)
    "llama8b_chunk256_k4": (config("gqa_llama8b", B=2, Tq=256, lengths=("list", [1200, 3000])), 4),
    "llama8b_chunk250_k4_pad": (config("gqa_llama8b", B=2, Tq=250, lengths=("list", [700, 2100])), 4),
    "llama8b_chunk96_k1": (config("gqa_llama8b", B=1, Tq=96, lengths=("list", [1500])), 1),
    "llama8b_chunk64_k8_I16": (config("gqa_llama8b", B=2, Tq=64, N=4, I=16, lengths=("list", [64, 900])), 8),
    "d64_g2_n3_i5": (config("gqa_llama8b", B=2, Tq=40, Hq=8, Hkv=4, Dk=64, Dv=64, N=3, I=5,
                            lengths=("list", [333, 77])), 2),
    "whole_prompt_k3": (config("gqa_llama8b", B=1, Tq=300, lengths=("list", [300])), 3),
    # block sizes that are multiples of 64: K/V come in through TMA boxes
    "bs64_chunk192_k4": (config("gqa_llama8b", B=2, Tq=192, block_size=64, lengths=("list", [1000, 2600])), 4),
    "bs128_chunk100_k2_N3": (config("gqa_llama8b", B=2, Tq=100, block_size=128, N=3, I=2,
                                    lengths=("list", [100, 777])), 2),
    # 64-token pages and the CTA's 128-row tiles: one row tile, an odd number of
    # row tiles with G = 8, a last row tile that is mostly padding
    "bs64_chunk24_k1_one_tile": (config("gqa_llama8b", B=2, Tq=24, block_size=64, lengths=("list", [500, 90])), 1),
    "bs64_chunk72_k2_g8_odd_tiles": (config("gqa_llama8b", B=2, Tq=72, Hq=16, Hkv=2, block_size=64,
                                            lengths=("list", [800, 300])), 2),
    "bs64_chunk40_k3_part_pair": (config("gqa_llama8b", B=2, Tq=40, block_size=64, N=2, I=3,
                                         lengths=("list", [1000, 77])), 3),
}

_cache = {}


def _setup(name):
    if name not in _cache:
        from context_decode_attention_gb300.harness import DeviceWorkload
        cfg, K = CASES[name]
        wl = make_workload(cfg, seed=3)
        dw = DeviceWorkload(wl, workspace_bytes=256)
        dw.prefill_setup(K)
        _cache.clear()
        _cache[name] = (wl, dw, K)
    return _cache[name]


@pytest.mark.parametrize("name", list(CASES))
def test_pcp_partition_bit_exact(name):
    wl, dw, K = _setup(name)
    Tq = int(wl.cfg["Tq"])
    ctx = wl.seq_lens.astype(np.int64) - Tq
    ref = oracle.pcp_partition(K, ctx, np.full(len(ctx), Tq), dw.max_q)
    assert ref["status"] == 0
    assert np.array_equal(dw.q_pos.cpu().numpy(), ref["pos"])
    assert np.array_equal(dw.padded_lens.cpu().numpy(), ref["padded_len"])
    assert dw.error_bits() == 0


def _natural_rows(wl, dw):
    """For every gathered row (b, j): the oracle's row block (b, t) or -1."""
    Tq = int(wl.cfg["Tq"])
    pos = dw.q_pos.cpu().numpy().astype(np.int64)
    ctx = wl.seq_lens.astype(np.int64)[:, None] - Tq
    t = np.where(pos >= 0, pos - ctx, -1)
    return t


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_merged_matches_oracle(name):
    wl, dw, K = _setup(name)
    c = wl.cfg
    B, Tq, Hq, Dv = (int(c[k]) for k in ("B", "Tq", "Hq", "Dv"))
    out, lse = dw.prefill()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ref_o, ref_l = oracle.attention(wl)
    ref_o = ref_o.reshape(B, Tq, Hq, Dv)
    ref_l = ref_l.reshape(B, Tq, Hq)
    t = _natural_rows(wl, dw)
    got_o, got_l = f64(out), f64(lse)
    live = t >= 0
    bi, ji = np.nonzero(live)
    assert len(bi) == B * Tq  # every new token appears exactly once
    assert sorted(zip(bi.tolist(), t[live].tolist())) == [(b, x) for b in range(B) for x in range(Tq)]
    assert_close_rows(got_o[bi, ji], got_l[bi, ji], ref_o[bi, t[live]], ref_l[bi, t[live]], tol_for(c), name)
    # padding rows: zeros and -inf
    pb, pj = np.nonzero(~live)
    if len(pb):
        assert np.all(got_o[pb, pj] == 0.0) and np.all(np.isneginf(got_l[pb, pj]))


@pytest.mark.parametrize("name", ["llama8b_chunk256_k4", "llama8b_chunk64_k8_I16", "d64_g2_n3_i5", "bs64_chunk192_k4"])
def test_prefill_rank_partials_match_oracle(name):
    wl, dw, K = _setup(name)
    c = wl.cfg
    B, Tq, Hq, Dv, N = (int(c[k]) for k in ("B", "Tq", "Hq", "Dv", "N"))
    dw.prefill(merged=False)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    t = _natural_rows(wl, dw)
    live = t >= 0
    bi, ji = np.nonzero(live)
    po, pl = f64(dw.p_out), f64(dw.p_lse)
    for r in range(N):
        ro, rl = oracle.attention(wl, rank=r)
        ro = ro.reshape(B, Tq, Hq, Dv)
        rl = rl.reshape(B, Tq, Hq)
        # fp32 partials: the bf16 inputs are exact, so only the accumulation order differs
        assert_close_rows(po[r][bi, ji], pl[r][bi, ji], ro[bi, t[live]], rl[bi, t[live]], (1e-2, 1e-3),
                          f"{name} rank {r}")


def test_prefill_position_past_context_is_reported():
    import context_decode_attention_gb300 as dcp
    wl, dw, K = _setup("llama8b_chunk96_k1")
    bad = dw.q_pos.clone()
    bad[0, 5] = int(wl.seq_lens[0]) + 3          # past the cached tokens
    dcp.dcp_prefill_attention(dw.params, dw.q_gathered, bad, dw.k_pool, dw.v_pool, dw.num_blocks, dw.block_tables,
                              dw.seq_lens, dw.local_lens, dw.p_out, dw.p_lse, dw.g_out, dw.g_lse,
                              workspace=dw.workspace)
    torch.cuda.synchronize()
    assert dw.error_bits() & 0x2
    assert np.isneginf(f64(dw.g_lse)[0, 5]).all() and (f64(dw.g_out)[0, 5] == 0).all()


def test_pcp_partition_row_overflow_is_reported():
    import context_decode_attention_gb300 as dcp
    wl, dw, K = _setup("llama8b_chunk96_k1")
    pos = torch.empty((1, 64), dtype=torch.int32, device="cuda")
    plen = torch.empty(1, dtype=torch.int32, device="cuda")
    dcp.dcp_pcp_partition(4, dw.ctx_lens, dw.q_lens, 64, pos, plen, workspace=dw.workspace)  # 96 rows > 64
    torch.cuda.synchronize()
    assert dw.error_bits() == 0x20
    assert (pos == -1).all() and plen.item() == 96
