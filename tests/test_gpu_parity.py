"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle, element
by element, at sizes the oracle finishes in seconds that still span several
chunks, splits and a ragged tail; plus the degenerate cases of the method."""

import numpy as np
import pytest
import torch

import oracle
from dcp_workloads import allocate_blocks, config, make_workload

from gpu_common import assert_close_rows, f64, tol_for

pytestmark = pytest.mark.gpu

CASES = {
    "gqa_toy_fp32": config("gqa_toy"),
    "gqa_bf16_ragged": config("gqa_llama8b", B=3, lengths=("list", [1000, 37, 513])),
    "gqa_bf16_tq2": config("gqa_llama8b", B=2, Tq=2, lengths=("list", [301, 77])),
    "gqa_bf16_tq3_rows24": config("gqa_llama8b", B=2, Tq=3, Hq=16, Hkv=2, lengths=("list", [100, 260])),
    "gqa_bf16_bs8": config("gqa_llama8b", B=2, block_size=8, lengths=("list", [333, 64])),
    "gqa_bf16_I64_short": config("gqa_llama8b", B=3, N=4, I=64, lengths=("list", [100, 700, 3])),
    "gqa_bf16_N1": config("gqa_llama8b", B=2, N=1, lengths=("list", [257, 16])),
    "gqa_bf16_single_token": config("gqa_llama8b", B=3, lengths=("list", [1, 1, 2])),
    "gqa_bf16_d64": config("gqa_llama8b", B=2, Hq=8, Hkv=2, Dk=64, Dv=64, N=3, I=5, lengths=("list", [600, 91])),
    "gqa_fp8": config("gqa_llama8b", B=2, kv_dtype="fp8", lengths=("list", [400, 129])),
    # more units (B x Hkv x N = 5120) than the planner keeps in shared memory
    "gqa_bf16_many_units": config("gqa_llama8b", B=160, lengths=("lognormal", 40, 0.8, 1, 300)),
    "mla_bf16": config("mla_bf16_32k", B=2, lengths=("list", [700, 1531])),
    "mla_bf16_I64_short": config("mla_bf16_32k", B=2, lengths=("list", [100, 64])),
    "mla_fp8_mixed": config("mla_fp8_mixed", B=3, lengths=("list", [300, 1100, 77])),
    "mla_fp8_tq4": config("mla_fp8_1m", lengths=("list", [2000])),
}

_cache = {}


def _setup(name, seed=1):
    key = (name, seed)
    if key not in _cache:
        from context_decode_attention_gb300.harness import DeviceWorkload
        wl = make_workload(CASES[name], seed=seed)
        dw = DeviceWorkload(wl)
        _cache.clear()
        _cache[key] = (wl, dw)
    return _cache[key]


@pytest.mark.parametrize("name", list(CASES))
def test_slot_mapping_and_cache_write_bit_exact(name):
    wl, dw = _setup(name)
    c = wl.cfg
    N, I, bs = int(c["N"]), int(c["I"]), int(c["block_size"])
    tok_req, tok_pos = wl.token_lists()
    ref = oracle.slot_mapping(N, I, bs, wl.seq_lens, tok_req, tok_pos, dw.block_tables_host)
    assert ref["status"] == 0
    owner, slots = dw.slot_mapping(tok_req, tok_pos)
    assert np.array_equal(owner.cpu().numpy(), ref["owner"])
    assert np.array_equal(slots.cpu().numpy(), ref["slots"])
    assert np.array_equal(dw.local_lens.cpu().numpy(), ref["local_lens"])
    assert np.array_equal(dw.virt_blocks.cpu().numpy(), ref["virt_blocks"])
    assert np.array_equal(dw.rank_blocks.cpu().numpy(), ref["rank_blocks"])
    # every token's row sits, bit for bit, in its owner's slot
    own_slot = ref["slots"][ref["owner"].astype(np.int64), np.arange(tok_req.size)]
    blk, off = own_slot // bs, own_slot % bs
    kp = dw.k_pool.view(torch.uint8).cpu().numpy() if dw.k_pool.dtype != torch.uint8 else dw.k_pool.cpu().numpy()
    kraw = wl.k.view(np.uint8).reshape(wl.k.shape[0], wl.k.shape[1], -1)
    if dw.mla:
        got = kp.reshape(dw.num_blocks, bs, -1)[blk, off]
        assert np.array_equal(got, kraw[:, 0])
    else:
        got = kp.reshape(dw.num_blocks, dw.Hkv, bs, -1)[blk, :, off]
        assert np.array_equal(got, kraw)
        vp = dw.v_pool.view(torch.uint8).cpu().numpy() if dw.v_pool.dtype != torch.uint8 else dw.v_pool.cpu().numpy()
        vraw = wl.v.view(np.uint8).reshape(wl.v.shape[0], wl.v.shape[1], -1)
        assert np.array_equal(vp.reshape(dw.num_blocks, dw.Hkv, bs, -1)[blk, :, off], vraw)
    assert dw.error_bits() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_decode_attention_matches_oracle(name):
    wl, dw = _setup(name)
    out, lse = dw.decode()
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attention(wl)
    assert_close_rows(f64(out).reshape(ref_o.shape), f64(lse).reshape(-1), ref_o, ref_l, tol_for(wl.cfg), name)
    assert dw.error_bits() == 0


@pytest.mark.parametrize("name", list(CASES))
def test_partial_attention_per_rank_matches_oracle(name):
    wl, dw = _setup(name)
    op, lp = dw.partial()
    torch.cuda.synchronize()
    N = int(wl.cfg["N"])
    for r in range(N):
        ref_o, ref_l = oracle.attention(wl, rank=r)
        assert_close_rows(f64(op[r]).reshape(ref_o.shape), f64(lp[r]).reshape(-1), ref_o, ref_l,
                          tol_for(wl.cfg), f"{name} rank {r}")
    assert dw.error_bits() == 0


@pytest.mark.parametrize("name", ["gqa_bf16_ragged", "gqa_bf16_I64_short", "mla_fp8_tq4", "gqa_toy_fp32"])
def test_lse_merge_of_partials_matches_unsharded_oracle(name):
    wl, dw = _setup(name)
    dw.partial()
    out = torch.empty_like(dw.out)
    lse = torch.empty_like(dw.lse)
    dw.merge(out, lse)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attention(wl)
    assert_close_rows(f64(out).reshape(ref_o.shape), f64(lse).reshape(-1), ref_o, ref_l, tol_for(wl.cfg), name)


def test_lse_merge_standalone_random_partials():
    import context_decode_attention_gb300 as dcp
    rng = np.random.default_rng(9)
    N, rows, Dv = 5, 77, 96
    o = rng.standard_normal((N, rows, Dv))
    l = rng.standard_normal((N, rows)) * 3
    l[1, :10] = -np.inf
    l[:, 20] = -np.inf  # a row with no tokens at all
    o[1, :10] = 0
    o[:, 20] = 0
    ref_o, ref_l = oracle.merge(o, l)
    od = torch.from_numpy(o.astype(np.float32)).cuda()
    ld = torch.from_numpy(l.astype(np.float32)).cuda()
    # the oracle merges the same fp32-rounded partials
    ref_o, ref_l = oracle.merge(o.astype(np.float32).astype(np.float64), l.astype(np.float32).astype(np.float64))
    for dt, torch_dt in [(dcp.DCP_F32, torch.float32), (dcp.DCP_BF16, torch.bfloat16)]:
        out = torch.empty((rows, Dv), dtype=torch_dt, device="cuda")
        lse = torch.empty(rows, dtype=torch.float32, device="cuda")
        dcp.dcp_lse_merge(N, rows, Dv, od, ld, out, dt, lse)
        torch.cuda.synchronize()
        got_o, got_l = f64(out), f64(lse)
        assert np.array_equal(np.isneginf(got_l), np.isneginf(ref_l))
        fin = ~np.isneginf(ref_l)
        assert np.abs(got_l[fin] - ref_l[fin]).max() <= 1e-5
        assert np.all(got_o[~fin] == 0.0)
        # These partials are unnormalised N(0, 1) draws, so the merged outputs
        # reach |out| ~ 4, where a fixed bf16 bar means little.  The bound is
        # relative: the fp32 merge is good to ~1e-6 of |out|, and the final
        # rounding to nearest costs at most half a unit in the last place,
        # 2^-8 |out| for bf16 (8 significant bits) and 2^-24 |out| for fp32.
        unit = 2.0 ** -8 if dt == dcp.DCP_BF16 else 2.0 ** -24
        err = np.abs(got_o[fin] - ref_o[fin])
        bound = (unit + 2e-6) * np.abs(ref_o[fin]) + 1e-6
        assert np.all(err <= bound), f"standalone merge: worst err/bound {(err / bound).max():.3g}"


@pytest.mark.parametrize("name", ["gqa_bf16_ragged", "mla_fp8_tq4"])
def test_decode_step_with_cache_write(name):
    wl, dw = _setup(name)
    out, lse = dw.step()
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attention(wl)
    assert_close_rows(f64(out).reshape(ref_o.shape), f64(lse).reshape(-1), ref_o, ref_l, tol_for(wl.cfg), name)


@pytest.mark.parametrize("seed", [2, 3])
def test_decode_is_deterministic_and_seed_independent_of_layout(seed):
    wl, dw = _setup("gqa_bf16_ragged", seed=seed)
    a, la = dw.decode()
    a = a.clone(); la = la.clone()
    b, lb = dw.decode()
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(la, lb)


# ---------------------------------------------------------------- device errors

def test_out_of_range_block_id_sets_error_bit():
    import context_decode_attention_gb300 as dcp
    wl, dw = _setup("gqa_bf16_ragged")
    bt = dw.block_tables.clone()
    bt[0, 0, 0] = dw.num_blocks + 5  # outside the pool: the kernels check before reading
    dcp.dcp_decode_attention(dw.params, dw.q, dw.k_pool, dw.v_pool, dw.num_blocks, bt, dw.seq_lens,
                             dw.local_lens, dw.out, dw.lse, dw.workspace)
    assert dw.error_bits() & 0x1
    assert dw.error_bits() == 0  # cleared by the read
    owner = torch.empty(4, dtype=torch.int8, device="cuda")
    slots = torch.empty((int(wl.cfg["N"]), 4), dtype=torch.int64, device="cuda")
    req = torch.zeros(4, dtype=torch.int32, device="cuda")
    pos = torch.arange(4, dtype=torch.int64, device="cuda")
    dcp.dcp_slot_mapping(dw.params, dw.seq_lens, req, pos, bt, dw.num_blocks, owner=owner, slots=slots,
                         workspace=dw.workspace)
    assert dw.error_bits() & 0x1
    assert (slots[:, 0] == -1).all()


def test_stale_local_lengths_detected():
    import context_decode_attention_gb300 as dcp
    wl, dw = _setup("gqa_bf16_ragged")
    stale = dw.local_lens.clone()
    stale[1, 0] -= 1
    dcp.dcp_decode_attention(dw.params, dw.q, dw.k_pool, dw.v_pool, dw.num_blocks, dw.block_tables, dw.seq_lens,
                             stale, dw.out, dw.lse, dw.workspace)
    assert dw.error_bits() & 0x8


def test_token_outside_request_detected():
    import context_decode_attention_gb300 as dcp
    wl, dw = _setup("gqa_bf16_ragged")
    owner = torch.empty(2, dtype=torch.int8, device="cuda")
    slots = torch.empty((int(wl.cfg["N"]), 2), dtype=torch.int64, device="cuda")
    req = torch.tensor([1, 7], dtype=torch.int32, device="cuda")      # request 7 does not exist
    pos = torch.tensor([37, 0], dtype=torch.int64, device="cuda")     # request 1 has 37 tokens
    dcp.dcp_slot_mapping(dw.params, dw.seq_lens, req, pos, dw.block_tables, dw.num_blocks, owner=owner,
                         slots=slots, workspace=dw.workspace)
    assert dw.error_bits() & 0x2
    assert (slots == -1).all() and (owner == -1).all()


# ------------------------------------------------------- PD block transfer

def _transfer(dw, bt=None, num_blocks=None):
    import context_decode_attention_gb300 as dcp
    bt = dw.block_tables if bt is None else bt
    N, B, M = bt.shape
    counts = torch.full((N, B), -7, dtype=torch.int32, device="cuda")
    blocks = torch.full((N, B, M), -7, dtype=torch.int32, device="cuda")
    fills = torch.full((N, B, M), -7, dtype=torch.int32, device="cuda")
    totals = torch.full((2,), -7, dtype=torch.int64, device="cuda")
    dcp.dcp_transfer_blocks(dw.params, dw.seq_lens, bt, dw.num_blocks if num_blocks is None else num_blocks,
                            counts, blocks, fills, totals, workspace=dw.workspace)
    return [t.cpu().numpy() for t in (counts, blocks, fills, totals)]


@pytest.mark.parametrize("name", list(CASES))
def test_transfer_blocks_bit_exact(name):
    wl, dw = _setup(name)
    c = wl.cfg
    ref = oracle.transfer_blocks(int(c["N"]), int(c["I"]), int(c["block_size"]), wl.seq_lens,
                                 dw.block_tables_host, dw.num_blocks)
    assert ref["status"] == 0
    counts, blocks, fills, totals = _transfer(dw)
    assert np.array_equal(counts, ref["counts"])
    assert np.array_equal(blocks, ref["blocks"])
    assert np.array_equal(fills, ref["fills"])
    assert np.array_equal(totals, ref["totals"])
    assert dw.error_bits() == 0


def test_transfer_blocks_errors_match_oracle():
    wl, dw = _setup("gqa_bf16_ragged")
    c = wl.cfg
    N, I, bs = int(c["N"]), int(c["I"]), int(c["block_size"])
    host = dw.block_tables_host.copy()
    host[1, 0, 0] = dw.num_blocks + 3            # a listed entry outside the pool
    ref = oracle.transfer_blocks(N, I, bs, wl.seq_lens, host, dw.num_blocks)
    assert ref["status"] == -1
    counts, blocks, fills, totals = _transfer(dw, torch.from_numpy(host).cuda())
    assert dw.error_bits() == 0x1
    for got, key in zip((counts, blocks, fills, totals), ("counts", "blocks", "fills", "totals")):
        assert np.array_equal(got, ref[key]), key
    short = np.ascontiguousarray(dw.block_tables_host[:, :, :2])   # request 0 needs more than two blocks
    ref = oracle.transfer_blocks(N, I, bs, wl.seq_lens, short, dw.num_blocks)
    assert ref["status"] == -1
    counts, blocks, fills, totals = _transfer(dw, torch.from_numpy(short).cuda())
    assert dw.error_bits() == 0x4
    for got, key in zip((counts, blocks, fills, totals), ("counts", "blocks", "fills", "totals")):
        assert np.array_equal(got, ref[key]), key


def test_transfer_blocks_empty_batch():
    import context_decode_attention_gb300 as dcp
    wl, dw = _setup("gqa_bf16_ragged")
    totals = torch.full((2,), 9, dtype=torch.int64, device="cuda")
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    dcp.dcp_transfer_blocks(dw.params, e, dw.block_tables[:, :0], dw.num_blocks, e, totals=totals,
                            workspace=dw.workspace)
    assert totals.tolist() == [0, 0] and dw.error_bits() == 0


@pytest.mark.parametrize("N,I,bs,B", [(8, 16, 16, 3000), (3, 5, 8, 700), (1, 1, 64, 40)])
def test_transfer_blocks_many_requests_and_repeated_calls(N, I, bs, B):
    """More (rank, request) pairs than the grid holds warps (the grid-stride
    path and the cross-block totals), and back-to-back calls on one workspace
    (the totals' accumulators must come back to zero after every call)."""
    import context_decode_attention_gb300 as dcp
    rng = np.random.default_rng(B)
    seq_lens = rng.integers(0, 600, size=B).astype(np.int32)
    seq_lens[::7] = 0
    cfg = config("gqa_llama8b", N=N, I=I, block_size=bs, B=B)
    params = dcp.params_from_config(cfg)
    sm = oracle.slot_mapping(N, I, bs, seq_lens, np.zeros(0, np.int32), np.zeros(0, np.int64))
    tables, nblk = allocate_blocks(sm["rank_blocks"], seed=B, spare=5)
    ref = oracle.transfer_blocks(N, I, bs, seq_lens, tables, nblk)
    assert ref["status"] == 0
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    dcp.dcp_workspace_init(ws)
    sl, bt = torch.from_numpy(seq_lens).cuda(), torch.from_numpy(tables).cuda()
    M = tables.shape[-1]
    for rep in range(3):
        counts = torch.full((N, B), -7, dtype=torch.int32, device="cuda")
        blocks = torch.full((N, B, M), -7, dtype=torch.int32, device="cuda")
        fills = torch.full((N, B, M), -7, dtype=torch.int32, device="cuda")
        totals = torch.full((2,), -7, dtype=torch.int64, device="cuda")
        if rep == 1:   # no totals requested: the accumulators are left alone
            dcp.dcp_transfer_blocks(params, sl, bt, nblk, counts, blocks, fills, None, workspace=ws)
            totals = torch.from_numpy(ref["totals"]).cuda()
        else:
            dcp.dcp_transfer_blocks(params, sl, bt, nblk, counts, blocks, fills, totals, workspace=ws)
        got = [t.cpu().numpy() for t in (counts, blocks, fills, totals)]
        for g, key in zip(got, ("counts", "blocks", "fills", "totals")):
            assert np.array_equal(g, ref[key]), (rep, key)
    assert dcp.dcp_get_error(ws) == 0
    assert not ws.cpu().numpy().any()  # the header's accumulators are back to zero


# ------------------------------------------------- peaked long contexts

@pytest.mark.parametrize("kv_dtype", ["fp8", "bf16"])
def test_long_flat_tail_below_a_sink(kv_dtype):
    """One 256K-token request on 8 ranks (32K tokens per rank) whose keys are
    a flat tail of identical rows (values with mean ~0.5) except two sinks
    (token 3 and token 100,000: ranks 3 and 0), which the 128 query heads
    score 6 to 20 nats above the tail.  Each tail token then weighs e^-6 to
    e^-20 of a sink, yet together the tail carries up to half of its rank's
    softmax mass, so an output that loses small probabilities (a two-term
    e4m3 split that underflows) misses that share.  Merged output and the
    sink ranks' partials, every element, against the oracle; the bf16 cache
    runs the same case as a control."""
    from context_decode_attention_gb300.harness import DeviceWorkload
    from dcp_workloads import sink_tail_workload
    cfg = config("mla_fp8_mixed" if kv_dtype == "fp8" else "mla_bf16_32k", B=1, I=1,
                 lengths=("list", [262144]))
    wl = sink_tail_workload(cfg, [3, 100000], np.linspace(6.0, 20.0, int(cfg["Hq"])), seed=4)
    dw = DeviceWorkload(wl)
    out, lse = dw.decode()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ref_o, ref_l = oracle.attention(wl)
    assert_close_rows(f64(out).reshape(ref_o.shape), f64(lse).reshape(-1), ref_o, ref_l, tol_for(cfg),
                      f"{kv_dtype} sink + flat tail")
    op, lp = dw.partial()
    torch.cuda.synchronize()
    for r in (3, 0):
        ref_o, ref_l = oracle.attention(wl, rank=r)
        assert_close_rows(f64(op[r]).reshape(ref_o.shape), f64(lp[r]).reshape(-1), ref_o, ref_l, tol_for(cfg),
                          f"{kv_dtype} sink + flat tail, rank {r}")


@pytest.mark.parametrize("name", ["mla_fp8_tq4", "mla_bf16"])
def test_mla_output_off_a_16_byte_boundary(name):
    """An MLA output that starts 2 bytes past a 16-byte boundary: the merge
    then takes its element-by-element path instead of 16-byte pieces (a
    different order of the same arithmetic), and must still match the oracle
    at the stated tolerance."""
    import context_decode_attention_gb300 as dcp
    wl, dw = _setup(name)
    flat = torch.zeros(dw.out.numel() + 1, dtype=dw.out.dtype, device="cuda")
    out = flat[1:].view(dw.out.shape)
    assert out.data_ptr() % 16 == 2
    lse = torch.empty_like(dw.lse)
    dcp.dcp_decode_attention(dw.params, dw.q, dw.k_pool, dw.v_pool, dw.num_blocks, dw.block_tables, dw.seq_lens,
                             dw.local_lens, out, lse, dw.workspace)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attention(wl)
    assert_close_rows(f64(out).reshape(ref_o.shape), f64(lse).reshape(-1), ref_o, ref_l, tol_for(wl.cfg),
                      f"{name} unaligned output")
    assert dw.error_bits() == 0
