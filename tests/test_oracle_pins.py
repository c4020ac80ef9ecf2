"""Pins for the CPU oracle: values the pages print, closed forms, invariants,
and special cases that reduce to a library routine (torch SDPA in fp64).

Each check is chosen so that a plausible slip in the oracle (a wrong index,
a dropped max shift, a transposed operand, a wrong head mapping or causal
bound, a wrong merge weight) fails at least one of them.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from dcp_workloads import allocate_blocks, config, make_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    lines = []
    for ln in open(os.path.join(GOLDEN, name)):
        ln = ln.split("#")[0].strip()
        if ln:
            lines.append(ln)
    return lines


# ---------------------------------------------------------------- ownership

def test_worked_interleave_table():
    lines = _read("interleave_I4_N4.txt")
    N = int(lines[0].split()[1])
    I = int(lines[1].split()[1])
    for ln in lines[2:]:
        a, b, r = map(int, ln.split())
        for t in range(a, b + 1):
            assert oracle.rank_of(t, N, I) == r, (t, r)


def test_contiguous_ranges_are_interleave_with_large_I():
    lines = _read("contiguous_ranges.txt")
    L = int(lines[0].split()[1])
    N = int(lines[1].split()[1])
    I = int(lines[2].split()[1])
    rank, _ = oracle.local_layout(L, N, I)
    for ln in lines[3:]:
        a, b, r = map(int, ln.split())
        assert np.all(rank[a:b + 1] == r)
    for r in range(N):
        assert oracle.local_len(L, r, N, I) == L // N


@pytest.mark.parametrize("N,I", [(1, 1), (2, 1), (3, 2), (4, 4), (8, 1), (8, 64), (5, 3)])
def test_ownership_period(N, I):
    # ownership repeats every N x I tokens ("vLLM DCP and PCP", TL;DR)
    for t in range(0, 3 * N * I + 7):
        assert oracle.rank_of(t + N * I, N, I) == oracle.rank_of(t, N, I)
    # and within one period every rank owns exactly I consecutive tokens
    rank, _ = oracle.local_layout(N * I, N, I)
    assert np.all(np.bincount(rank, minlength=N) == I)


# ------------------------------------------------------------ local lengths

def test_even_split_8k_on_4():
    for ln in _read("even_split.txt"):
        L, N, I, each = map(int, ln.split())
        assert [oracle.local_len(L, r, N, I) for r in range(N)] == [each] * N


@pytest.mark.parametrize("N,I", [(2, 1), (4, 2), (4, 4), (3, 5), (8, 1), (8, 64), (4, 16)])
def test_local_lengths_partition_and_spread(N, I):
    rng = np.random.default_rng(7)
    for L in list(range(0, 3 * N * I + 3)) + list(rng.integers(1, 5000, size=20)):
        lens = [oracle.local_len(int(L), r, N, I) for r in range(N)]
        assert sum(lens) == L
        # "local sequence lengths can differ by at most one interleave group"
        assert max(lens) - min(lens) <= I
        # lower ranks never hold fewer tokens than higher ranks
        assert all(lens[r] >= lens[r + 1] for r in range(N - 1))


@pytest.mark.parametrize("N,I", [(2, 1), (4, 2), (3, 5), (8, 64)])
def test_local_positions_form_a_prefix(N, I):
    # each rank's tokens among the first L occupy local positions 0..len-1 in order
    L = 4 * N * I + 3
    rank, lpos = oracle.local_layout(L, N, I)
    for Lp in range(L + 1):
        for r in range(N):
            mine = lpos[:Lp][rank[:Lp] == r]
            assert np.array_equal(mine, np.arange(oracle.local_len(Lp, r, N, I)))


def test_pd_block_fill_example():
    lines = _read("pd_block_fill.txt")
    L = int(lines[0].split()[1])
    bs = int(lines[1].split()[1])
    N = int(lines[2].split()[1])
    for ln in lines[3:]:
        head, blocks, virt = ln.split("|")
        head = list(map(int, head.split()))
        I, lens = head[0], head[1:]
        sm = oracle.slot_mapping(N, I, bs, np.array([L]), np.zeros(L, np.int32), np.arange(L))
        assert sm["local_lens"][:, 0].tolist() == lens
        assert sm["rank_blocks"][:, 0].tolist() == list(map(int, blocks.split()))
        assert sm["virt_blocks"].tolist() == [int(virt)]
        # fill ratio of each non-empty block: 25% at I=1, 100% at I=bs
        fill = [n / (math.ceil(n / bs) * bs) for n in lens if n]
        assert fill == ([0.25] * 4 if I == 1 else [1.0])


@pytest.mark.parametrize("N,I,bs", [(4, 1, 16), (4, 4, 16), (8, 64, 64), (2, 8, 16), (8, 1, 64)])
def test_rank_blocks_fit_in_virtual_blocks_when_I_divides_bs(N, I, bs):
    assert bs % I == 0
    for L in [1, 5, bs, bs * N, bs * N + 1, 3 * bs * N - 1, 1000, 4097]:
        sm = oracle.slot_mapping(N, I, bs, np.array([L]), np.zeros(0, np.int32), np.zeros(0, np.int64))
        v = int(sm["virt_blocks"][0])
        assert v == math.ceil(L / (bs * N))
        assert np.all(sm["rank_blocks"][:, 0] <= v)


# ------------------------------------------------------------------- slots

def _random_tables(N, I, bs, seq_lens, seed):
    sm = oracle.slot_mapping(N, I, bs, seq_lens, np.zeros(0, np.int32), np.zeros(0, np.int64))
    tables, nblk = allocate_blocks(sm["rank_blocks"], seed=seed, spare=3)
    return tables, nblk


@pytest.mark.parametrize("N,I,bs", [(1, 1, 4), (2, 1, 16), (4, 4, 16), (3, 2, 8), (4, 3, 8), (8, 64, 64)])
def test_slots_are_a_bijection(N, I, bs):
    seq_lens = np.array([1, 7, 64, 130, 257], dtype=np.int32)
    tables, nblk = _random_tables(N, I, bs, seq_lens, seed=N * 100 + I)
    tok_req = np.repeat(np.arange(len(seq_lens), dtype=np.int32), seq_lens)
    tok_pos = np.concatenate([np.arange(n) for n in seq_lens]).astype(np.int64)
    perm = np.random.default_rng(3).permutation(tok_req.size)  # token order must not matter
    tok_req, tok_pos = tok_req[perm], tok_pos[perm]
    sm = oracle.slot_mapping(N, I, bs, seq_lens, tok_req, tok_pos, tables)
    assert sm["status"] == 0
    slots, owner = sm["slots"], sm["owner"]
    # exactly one rank stores each token: its owner; everybody else skips (-1)
    assert np.all((slots >= 0).sum(axis=0) == 1)
    assert np.all(np.argmax(slots >= 0, axis=0) == owner)
    assert np.all(owner == (tok_pos // I) % N)
    flat = slots[slots >= 0]
    assert flat.size == tok_req.size and np.unique(flat).size == flat.size
    assert flat.min() >= 0 and flat.max() < nblk * bs
    # the slot's block is in the owner's table for that request, at lpos // bs
    for i in range(tok_req.size):
        r, b = owner[i], tok_req[i]
        blk, off = divmod(int(slots[r, i]), bs)
        k = list(tables[r, b]).index(blk)
        lp = k * bs + off
        assert lp < sm["local_lens"][r, b]


def test_slot_mapping_brute_force_tiny():
    # brute force: build each rank's token list by appending tokens in order
    for N in range(1, 5):
        for I in range(1, 9):
            for bs in (1, 2, 3, 8):
                L = 37
                lists = [[] for _ in range(N)]
                for t in range(L):
                    lists[(t // I) % N].append(t)
                counts = np.array([[len(x)] for x in lists])
                tables, _ = allocate_blocks(np.ceil(counts / bs).astype(np.int64), seed=N * 31 + I)
                sm = oracle.slot_mapping(N, I, bs, np.array([L]), np.zeros(L, np.int32), np.arange(L), tables)
                assert sm["status"] == 0
                assert sm["local_lens"][:, 0].tolist() == [len(x) for x in lists]
                for r in range(N):
                    for idx, t in enumerate(lists[r]):
                        assert sm["slots"][r, t] == tables[r, 0, idx // bs] * bs + idx % bs


def test_slot_mapping_reports_bad_tokens():
    seq_lens = np.array([10], dtype=np.int32)
    tables, _ = _random_tables(2, 1, 4, seq_lens, seed=1)
    sm = oracle.slot_mapping(2, 1, 4, seq_lens, np.array([0, 0, 1], np.int32), np.array([3, 10, 0]), tables)
    assert sm["status"] == -1
    assert sm["owner"][1] == -1 and sm["owner"][2] == -1
    assert np.all(sm["slots"][:, 1:] == -1) and (sm["slots"][:, 0] >= 0).sum() == 1


# ------------------------------------------------------------ storage types

def test_fp8_e4m3_decode_all_codes_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.decode(codes, "fp8", 1.0)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan) and nan.sum() == 2
    assert np.array_equal(mine[~nan], ref[~nan])
    assert oracle.decode(np.array([0x7E], np.uint8), "fp8", 0.5)[0] == 224.0


def test_bf16_decode_all_codes_against_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.decode(codes, "bf16")
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


# --------------------------------------------------------------- attention

def _dense(wl):
    c = wl.cfg
    q = oracle.decode(wl.q, c["q_dtype"])
    k = oracle.decode(wl.k, c["kv_dtype"], wl.kv_scale)
    v = None if wl.v is None else oracle.decode(wl.v, c["kv_dtype"], wl.kv_scale)
    return q, k, v


def _sdpa_reference(wl):
    """torch SDPA in fp64 (library routine) with an explicit causal mask."""
    c = wl.cfg
    B, Tq, Hq, Hkv, Dk, Dv = (int(c[x]) for x in ("B", "Tq", "Hq", "Hkv", "Dk", "Dv"))
    q, k, v = _dense(wl)
    outs, lses = [], []
    for b in range(B):
        L = int(wl.seq_lens[b])
        s, e = int(wl.req_start[b]), int(wl.req_start[b + 1])
        qb = torch.from_numpy(q[b]).permute(1, 0, 2)            # [Hq, Tq, Dk]
        kb = torch.from_numpy(k[s:e]).permute(1, 0, 2)          # [Hkv, L, Dk]
        if c["layout"] == "mla":
            vb = kb[..., :Dv]
        else:
            vb = torch.from_numpy(v[s:e]).permute(1, 0, 2)
        G = Hq // Hkv
        kb = kb.repeat_interleave(G, dim=0)
        vb = vb.repeat_interleave(G, dim=0)
        pos = torch.arange(L)
        qpos = torch.arange(L - Tq, L)
        mask = pos[None, :] <= qpos[:, None]                    # [Tq, L]
        o = torch.nn.functional.scaled_dot_product_attention(
            qb, kb, vb, attn_mask=mask, scale=float(c["softmax_scale"]))
        scores = (qb @ kb.transpose(-1, -2)) * float(c["softmax_scale"])
        scores = scores.masked_fill(~mask, float("-inf"))
        lse = torch.logsumexp(scores, dim=-1)                   # [Hq, Tq]
        outs.append(o.permute(1, 0, 2).numpy())                 # [Tq, Hq, Dv]
        lses.append(lse.permute(1, 0).numpy())
    return np.stack(outs).reshape(-1, Dv), np.stack(lses).reshape(-1)


@pytest.mark.parametrize("name,kw", [
    ("gqa_toy", dict(L=100)),
    ("gqa_llama8b", dict(B=2, Hq=8, Hkv=2, Dk=32, Dv=32, L=77)),
    ("gqa_llama8b", dict(B=2, Hq=6, Hkv=3, Dk=16, Dv=24, L=40, Tq=3)),
    ("mla_bf16_32k", dict(B=2, Hq=4, Dk=40, Dv=32, L=70)),
    ("mla_fp8_1m", dict(Hq=4, Dk=48, Dv=32, L=90)),
])
def test_attention_matches_torch_sdpa(name, kw):
    wl = make_workload(config(name, **kw), seed=5)
    out, lse = oracle.attention(wl)
    ref_o, ref_l = _sdpa_reference(wl)
    assert np.abs(out - ref_o).max() < 1e-12
    assert np.abs(lse - ref_l).max() < 1e-12


def test_single_key_closed_form():
    wl = make_workload(config("gqa_llama8b", B=1, Hq=4, Hkv=2, Dk=16, Dv=16, L=1), seed=2)
    out, lse = oracle.attention(wl)
    q, k, v = _dense(wl)
    for h in range(4):
        kv = h // 2
        assert np.array_equal(out[h], v[0, kv])
        assert lse[h] == pytest.approx(wl.cfg["softmax_scale"] * float(q[0, 0, h] @ k[0, kv]), abs=1e-13)


def test_zero_query_gives_mean_and_log_count():
    wl = make_workload(config("gqa_toy", L=50, Tq=3), seed=3, zero_q=True)
    out, lse = oracle.attention(wl)
    _, _, v = _dense(wl)
    for t in range(3):
        g = 50 - 3 + t + 1
        for h in range(4):
            row = t * 4 + h
            assert lse[row] == pytest.approx(math.log(g), abs=1e-13)
            assert np.abs(out[row] - v[:g, 0].mean(axis=0)).max() < 1e-13


def test_identical_keys_give_mean():
    wl = make_workload(config("mla_bf16_32k", B=1, Hq=3, Dk=24, Dv=16, L=33), seed=4)
    wl.k[:] = wl.k[0]  # every token carries the same latent row
    out, lse = oracle.attention(wl)
    q, k, _ = _dense(wl)
    for h in range(3):
        s = wl.cfg["softmax_scale"] * float(q[0, 0, h] @ k[0, 0])
        assert lse[h] == pytest.approx(s + math.log(33), abs=1e-12)
        assert np.abs(out[h] - k[0, 0, :16]).max() < 1e-14


# ------------------------------------------------------------------- merge

@pytest.mark.parametrize("N,I", [(1, 1), (2, 1), (3, 2), (4, 1), (4, 5), (8, 1), (8, 64)])
def test_merge_of_rank_partials_equals_unsharded(N, I):
    cfg = config("gqa_llama8b", B=3, Hq=4, Hkv=2, Dk=16, Dv=16, Tq=2, N=N, I=I,
                 lengths=("list", [3, 150, 600]))
    wl = make_workload(cfg, seed=N * 10 + I)
    full_o, full_l = oracle.attention(wl)
    parts = [oracle.attention(wl, rank=r) for r in range(N)]
    o_parts = np.stack([p[0] for p in parts])
    l_parts = np.stack([p[1] for p in parts])
    m_o, m_l = oracle.merge(o_parts, l_parts)
    assert np.abs(m_o - full_o).max() < 1e-12
    assert np.abs(m_l - full_l).max() < 1e-12
    # rank order does not matter
    perm = np.random.default_rng(N).permutation(N)
    p_o, p_l = oracle.merge(o_parts[perm], l_parts[perm])
    assert np.abs(p_o - m_o).max() < 1e-13 and np.abs(p_l - m_l).max() < 1e-13
    # ranks that own none of a short request carry weight zero (-inf LSE)
    if N * I > 3:
        short_rows = slice(0, 2 * 4)  # request 0 (3 tokens), both query tokens
        empty = [r for r in range(N) if oracle.local_len(3, r, N, I) == 0]
        for r in empty:
            assert np.all(np.isneginf(l_parts[r, short_rows]))
            assert np.all(o_parts[r, short_rows] == 0)


def test_merge_single_part_is_identity():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((1, 5, 7))
    l = rng.standard_normal((1, 5))
    mo, ml = oracle.merge(o, l)
    assert np.abs(mo - o[0]).max() < 1e-15 and np.abs(ml - l[0]).max() < 1e-15


def test_merge_weights_by_lse():
    # two parts with LSEs log(1) and log(3): weights 1/4 and 3/4, merged LSE log(4)
    o = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    l = np.log(np.array([[1.0], [3.0]]))
    mo, ml = oracle.merge(o, l)
    assert np.allclose(mo, [[0.25, 0.75]], atol=1e-15)
    assert ml[0] == pytest.approx(math.log(4.0), abs=1e-15)


# ------------------------------------------------------- PD block transfer

def test_transfer_blocks_pd_example():
    """Section 2 example of the PD-disaggregation page: 16 tokens, block size
    16, four ranks.  Interleave 1 moves four blocks a quarter full; interleave
    16 moves one full block and nothing from the other ranks."""
    lines = _read("pd_block_fill.txt")
    L, bs, N = (int(lines[i].split()[1]) for i in range(3))
    tables = np.arange(N * 2, dtype=np.int32).reshape(N, 1, 2) + 100
    for ln in lines[3:]:
        head, nblocks, _ = ln.split("|")
        I, *lens = map(int, head.split())
        tb = oracle.transfer_blocks(N, I, bs, np.array([L]), tables, num_blocks=200)
        assert tb["status"] == 0
        assert tb["counts"][:, 0].tolist() == list(map(int, nblocks.split()))
        for r in range(N):
            c = int(tb["counts"][r, 0])
            assert tb["fills"][r, 0, :c].tolist() == ([lens[r]] if c else [])
            assert tb["blocks"][r, 0, :c].tolist() == tables[r, 0, :c].tolist()
            assert tb["blocks"][r, 0, c:].tolist() == [-1] * (2 - c)
        # slots moved and tokens moved: fill 25% at I=1, 100% at I=bs
        assert tb["totals"].tolist() == ([64, 16] if I == 1 else [16, 16])


@pytest.mark.parametrize("N,I,bs", [(1, 1, 16), (4, 1, 16), (4, 16, 16), (3, 5, 8), (8, 64, 64), (2, 100, 16)])
def test_transfer_blocks_invariants(N, I, bs):
    """Fills add up to the request's length; every listed block is full but
    the rank's last; the list is the table's first ceil(local_len / bs)
    entries; totals are the sums.  Checked against the closed-form local
    length, not the enumeration the oracle uses."""
    seq_lens = np.array([0, 1, 15, 16, 17, 100, 1000, 4097], dtype=np.int32)
    sm = oracle.slot_mapping(N, I, bs, seq_lens, np.zeros(0, np.int32), np.zeros(0, np.int64))
    tables, nblk = allocate_blocks(sm["rank_blocks"], seed=3, spare=2)
    tb = oracle.transfer_blocks(N, I, bs, seq_lens, tables, nblk)
    assert tb["status"] == 0
    slots = toks = 0
    for b, L in enumerate(seq_lens.tolist()):
        assert int(tb["fills"][:, b].sum()) == L
        for r in range(N):
            ln = oracle.local_len(L, r, N, I)
            c = int(tb["counts"][r, b])
            assert c == -(-ln // bs)
            f = tb["fills"][r, b, :c]
            assert np.all(f[:-1] == bs) and (c == 0 or 0 < f[-1] <= bs)
            assert np.array_equal(tb["blocks"][r, b, :c], tables[r, b, :c])
            assert np.all(tb["blocks"][r, b, c:] == -1) and np.all(tb["fills"][r, b, c:] == 0)
            slots += c * bs
            toks += ln
    assert tb["totals"].tolist() == [slots, toks]


def test_transfer_blocks_brute_force_tiny():
    """Tiny case listed by hand: N=2, I=3, bs=4, L=14.  Tokens 0-2, 6-8, 12-13
    go to rank 0 (8 tokens), 3-5, 9-11 to rank 1 (6 tokens)."""
    tables = np.array([[[7, 3, 9]], [[2, 5, 0]]], dtype=np.int32)
    tb = oracle.transfer_blocks(2, 3, 4, np.array([14]), tables, num_blocks=10)
    assert tb["status"] == 0
    assert tb["counts"][:, 0].tolist() == [2, 2]
    assert tb["blocks"][:, 0].tolist() == [[7, 3, -1], [2, 5, -1]]
    assert tb["fills"][:, 0].tolist() == [[4, 4, 0], [4, 2, 0]]
    assert tb["totals"].tolist() == [16, 14]


def test_transfer_blocks_reports_bad_tables():
    tables = np.array([[[7, 30]], [[2, 5]]], dtype=np.int32)   # 30 is outside a 10-block pool
    tb = oracle.transfer_blocks(2, 3, 4, np.array([14]), tables, num_blocks=10)
    assert tb["status"] == -1 and tb["blocks"][0, 0].tolist() == [7, -1]
    short = tables[:, :, :1].copy()                             # each rank needs two blocks
    tb = oracle.transfer_blocks(2, 3, 4, np.array([14]), short, num_blocks=10)
    assert tb["status"] == -1 and tb["counts"][:, 0].tolist() == [1, 1]
    assert tb["totals"].tolist() == [16, 14]


# ------------------------------------------------------ PCP head-tail partition

def test_pcp_partition_page_examples():
    for ln in _read("pcp_zigzag.txt"):
        head, *ranks = ln.split("|")
        K, n = map(int, head.split())
        for ctx in (0, 37):
            r = oracle.pcp_partition(K, [ctx], [n], n)
            assert r["status"] == 0 and r["padded_len"].tolist() == [n]
            per = n // K
            for k, toks in enumerate(ranks):
                want = [ctx + int(x) for x in toks.split()]
                assert r["pos"][0, k * per:(k + 1) * per].tolist() == want


@pytest.mark.parametrize("K", [1, 2, 3, 4, 8])
def test_pcp_partition_balances_causal_work(K):
    """Aligned lengths: every rank's causal work (keys its queries see, with
    the cached context in front) is the same, as the head-tail pairing intends;
    rows form a permutation of the new positions."""
    for n in [2 * K, 6 * K, 2 * K * 17]:
        for ctx in [0, 1000]:
            r = oracle.pcp_partition(K, [ctx], [n], n)
            pos = r["pos"][0]
            assert sorted(pos.tolist()) == list(range(ctx, ctx + n))
            per = n // K
            work = [int((pos[k * per:(k + 1) * per].astype(np.int64) + 1).sum()) for k in range(K)]
            assert len(set(work)) == 1


def test_pcp_partition_padding_and_overflow():
    r = oracle.pcp_partition(2, [10, 0, 5], [5, 0, 4], 12)
    assert r["status"] == 0 and r["padded_len"].tolist() == [8, 0, 4]
    assert r["pos"][0].tolist() == [10, 11, -1, -1, 12, 13, 14, -1, -1, -1, -1, -1]
    assert (r["pos"][1] == -1).all()
    assert r["pos"][2].tolist()[:4] == [5, 8, 6, 7]
    bad = oracle.pcp_partition(4, [0], [9], 8)   # aligned to 16 > 8 rows
    assert bad["status"] == -1 and (bad["pos"] == -1).all()


# ------------------------------------------------ sparse (top-k) attention

from dcp_workloads import sparse_candidates  # noqa: E402


@pytest.mark.parametrize("name,kw", [
    ("mla_fp8_mixed", dict(B=2, lengths=("list", [40, 90]))),
    ("gqa_llama8b", dict(B=2, Tq=3, lengths=("list", [30, 70]))),
])
def test_sparse_with_every_position_is_dense(name, kw):
    """A candidate set holding every visible position reduces to the pinned
    dense (causal) attention."""
    wl = make_workload(config(name, **kw), seed=4)
    cand = sparse_candidates(wl, 4096)            # k above every length: all visible positions
    so, sl = oracle.sparse_attention(wl, cand)
    do, dl = oracle.attention(wl)
    assert np.allclose(so, do, atol=1e-12, rtol=0) and np.allclose(sl, dl, atol=1e-12, rtol=0)


@pytest.mark.parametrize("N,I", [(2, 1), (8, 1), (4, 64), (3, 5)])
def test_sparse_rank_partials_merge_to_sparse(N, I):
    wl = make_workload(config("mla_fp8_mixed", B=2, N=N, I=I, lengths=("list", [700, 1500])), seed=5)
    cand = sparse_candidates(wl, 200)
    full_o, full_l = oracle.sparse_attention(wl, cand)
    parts = [oracle.sparse_attention(wl, cand, rank=r) for r in range(N)]
    mo, ml = oracle.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.allclose(mo, full_o, atol=1e-12, rtol=0) and np.allclose(ml, full_l, atol=1e-12, rtol=0)


def test_sparse_single_candidate_and_order():
    wl = make_workload(config("gqa_llama8b", B=1, lengths=("list", [50])), seed=6)
    c = wl.cfg
    cand = np.full((1, 4), -1, dtype=np.int32)
    cand[0, 0] = 17
    o, l = oracle.sparse_attention(wl, cand)
    q = oracle.decode(wl.q[0, 0], "bf16")
    k = oracle.decode(wl.k[17], "bf16")
    v = oracle.decode(wl.v[17], "bf16")
    G = int(c["Hq"]) // int(c["Hkv"])
    for h in range(int(c["Hq"])):
        assert np.allclose(o[h], v[h // G], atol=1e-12)
        assert abs(l[h] - float(c["softmax_scale"]) * float(q[h] @ k[h // G])) < 1e-12
    # the candidate order does not matter
    base = sparse_candidates(wl, 20)
    shuffled = base.copy()
    np.random.default_rng(0).shuffle(shuffled[0, :20])
    a, la = oracle.sparse_attention(wl, base)
    b, lb = oracle.sparse_attention(wl, shuffled)
    assert np.allclose(a, b, atol=1e-12) and np.allclose(la, lb, atol=1e-12)


@pytest.mark.parametrize("N,I", [(8, 1), (4, 16), (3, 5)])
def test_sparse_localize_matches_closed_form(N, I):
    """Per rank, the candidates it owns in list order, at their local
    positions; checked against the closed form floor(t / (N I)) I + t mod I
    (the oracle uses the running-count definition)."""
    seq_lens = np.array([1000, 37], dtype=np.int32)
    rng = np.random.default_rng(1)
    cand = np.full((2, 64), -1, dtype=np.int32)
    for i, L in enumerate(seq_lens):
        n = min(64, int(L))
        cand[i, :n] = rng.choice(int(L), size=n, replace=False)
    local, counts = oracle.sparse_localize(cand, N, I, seq_lens, 1)
    for i in range(2):
        c = cand[i][cand[i] >= 0].astype(np.int64)
        assert int(counts[:, i].sum()) == c.size
        for r in range(N):
            mine = c[(c // I) % N == r]
            assert np.array_equal(local[r, i, :counts[r, i]], (mine // (N * I)) * I + mine % I)
            assert np.all(local[r, i, counts[r, i]:] == -1)


def test_one_million_tokens_on_dcp8_store_an_eighth_each():
    for ln in _read("capacity_1m_dcp8.txt"):
        shard, gib = ln.split("|")
        L, N, I, each = map(int, shard.split())
        total_gib, per_gpu_gib = map(float, gib.split())
        lens = [oracle.local_len(L, r, N, I) for r in range(N)]
        assert lens == [each] * N and sum(lens) == L
        # every rank keeps the same share of the request's KV bytes: the page's
        # per-GPU figure is its total over N, to its rounding of 0.1 GiB
        assert abs(total_gib * max(lens) / L - per_gpu_gib) <= 0.05


def test_merge_of_only_empty_partials_is_zero_and_minus_inf():
    """A row no rank holds a token of: its LSE is the log of an empty sum, -inf,
    and its output is the empty weighted mean, 0 by the empty-shard reading
    (a rank with no visible token contributes o = 0, L = -inf, weight 0).
    Rows beside it with one non-empty partial merge to that partial."""
    rng = np.random.default_rng(5)
    o = rng.normal(size=(3, 4, 8))
    lse = np.full((3, 4), -np.inf)
    lse[1, 2:] = rng.normal(size=2)  # rows 2 and 3: only rank 1 holds tokens
    o[:, :2] = 0.0                   # empty partials carry zeros
    out, l = oracle.merge(o, lse)
    assert np.all(out[:2] == 0) and np.all(np.isneginf(l[:2]))
    np.testing.assert_allclose(out[2:], o[1, 2:], rtol=0, atol=1e-15)
    np.testing.assert_allclose(l[2:], lse[1, 2:], rtol=0, atol=1e-15)


def test_slot_mapping_reports_a_missing_block():
    """A token whose local block has no id in its owner's table (-1) gets no
    slot on any rank and the call reports it; the other tokens are unaffected.
    N = 2, I = 1, bs = 4, L = 10: rank 0 owns tokens 0, 2, ..., 8 at local
    positions 0..4, so token 8 is in its second block and token 2 in its first;
    token 3 is rank 1's local position 1."""
    seq_lens = np.array([10], dtype=np.int32)
    tables, _ = _random_tables(2, 1, 4, seq_lens, seed=2)
    tables[0, 0, 1] = -1
    sm = oracle.slot_mapping(2, 1, 4, seq_lens, np.array([0, 0, 0], np.int32), np.array([8, 2, 3]), tables)
    assert sm["status"] == -1
    assert sm["owner"].tolist() == [0, 0, 1]
    assert np.all(sm["slots"][:, 0] == -1)
    assert sm["slots"][:, 1].tolist() == [int(tables[0, 0, 0]) * 4 + 1, -1]
    assert sm["slots"][:, 2].tolist() == [-1, int(tables[1, 0, 0]) * 4 + 1]


def test_transfer_blocks_pool_bound_is_exclusive():
    """Block ids run from 0 to num_blocks - 1: an id equal to num_blocks is
    outside the pool and is reported; num_blocks - 1 is not."""
    for last, bad in ((9, False), (10, True)):
        tables = np.array([[[7, last]], [[2, 5]]], dtype=np.int32)
        tb = oracle.transfer_blocks(2, 3, 4, np.array([14]), tables, num_blocks=10)
        assert (tb["status"] == -1) == bad
        assert tb["blocks"][0, 0].tolist() == [7, -1 if bad else last]
