"""CPU oracle for DCP decode attention (plain C, fp64) -- TEST INFRASTRUCTURE.

Only tests/, the package's smoke() check and bench.py's CPU-baseline leg may
import this module.  The CUDA path never imports, links or calls it, and the
two share no code: the oracle reads the dense per-request keys/values that the
seeded generator produced, never the paged cache.

Functions (all numpy in, numpy out):
  rank_of(t, N, I)                       interleave owner of token t
  local_layout(L, N, I)                  (rank[L], local_pos[L]) by running count
  local_len(L, r, N, I)                  tokens of the first L that rank r owns
  slot_mapping(...)                      owner/slots/local_lens/virt/rank blocks
  transfer_blocks(...)                   per-rank non-empty blocks, fills, totals
  pcp_partition(K, ctx_lens, q_lens, max_q)  head-tail prefill partition
  attention(wl, rank=-1, rows=None)      (out [rows, Dv], lse [rows]) in fp64
  merge(o_parts, lse_parts)              exact LSE merge of per-rank partials
  sparse_localize(cand, N, I, seq_lens, Tq)  per-rank local positions of candidates
  sparse_attention(wl, cand, rank=-1)    attention over each query's candidate set
  decode(raw, dtype, scale)              stored values -> float64

Every function follows one passage of the pages; the C source's header lists
them.  Parity status: all functions are pinned by tests/test_oracle_pins.py.
"""

import ctypes
import os

import numpy as np

from . import build as _build

_DT = {"f32": 0, "bf16": 1, "fp8": 2}
_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.orc_rank_of.restype = i64
        lib.orc_rank_of.argtypes = [i64, i64, i64]
        lib.orc_local_len.restype = i64
        lib.orc_local_len.argtypes = [i64, i64, i64, i64]
        lib.orc_local_layout.restype = None
        lib.orc_local_layout.argtypes = [i64, i64, i64, p, p]
        lib.orc_decode.restype = None
        lib.orc_decode.argtypes = [p, i64, i64, ctypes.c_double, p]
        lib.orc_slot_mapping.restype = ctypes.c_int
        lib.orc_slot_mapping.argtypes = [i64, i64, i64, i64, p, i64, p, p, p, i64, p, p, p, p, p]
        lib.orc_pcp_partition.restype = ctypes.c_int
        lib.orc_pcp_partition.argtypes = [i64, i64, p, p, i64, p, p]
        lib.orc_transfer_blocks.restype = ctypes.c_int
        lib.orc_transfer_blocks.argtypes = [i64, i64, i64, i64, p, p, i64, i64, p, p, p, p]
        lib.orc_attention.restype = None
        lib.orc_attention.argtypes = [i64, i64, i64, i64, i64, i64, i64, p, p, p, i64, p, p, i64,
                                      ctypes.c_double, ctypes.c_double, i64, i64, i64, i64, p, p, p, i64]
        lib.orc_merge.restype = None
        lib.orc_merge.argtypes = [i64, i64, i64, p, p, p, p]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def threads():
    """Threads the oracle uses: every host core."""
    return os.cpu_count() or 1


def rank_of(t, N, I):
    return int(_load().orc_rank_of(int(t), int(N), int(I)))


def local_len(L, r, N, I):
    return int(_load().orc_local_len(int(L), int(r), int(N), int(I)))


def local_layout(L, N, I):
    rank = np.empty(max(1, L), dtype=np.int32)
    lpos = np.empty(max(1, L), dtype=np.int64)
    _load().orc_local_layout(int(L), int(N), int(I), _ptr(rank), _ptr(lpos))
    return rank[:L], lpos[:L]


def decode(raw, dtype, scale=1.0):
    raw = np.ascontiguousarray(raw)
    out = np.empty(raw.size, dtype=np.float64)
    _load().orc_decode(_ptr(raw), raw.size, _DT[dtype], float(scale), _ptr(out))
    return out.reshape(raw.shape)


def slot_mapping(N, I, bs, seq_lens, tok_req, tok_pos, block_tables=None):
    """Returns dict(owner, slots or None, local_lens, virt_blocks, rank_blocks, status)."""
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    tok_req = np.ascontiguousarray(tok_req, dtype=np.int32)
    tok_pos = np.ascontiguousarray(tok_pos, dtype=np.int64)
    B, T = seq_lens.size, tok_req.size
    owner = np.empty(max(1, T), dtype=np.int8)
    local_lens = np.empty((N, max(1, B)), dtype=np.int32)
    virt = np.empty(max(1, B), dtype=np.int32)
    rblk = np.empty((N, max(1, B)), dtype=np.int32)
    slots, max_blocks, bt = None, 0, None
    if block_tables is not None:
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        max_blocks = bt.shape[-1]
        slots = np.empty((N, max(1, T)), dtype=np.int64)
    st = _load().orc_slot_mapping(N, I, bs, B, _ptr(seq_lens), T, _ptr(tok_req), _ptr(tok_pos),
                                  _ptr(bt), max_blocks, _ptr(owner), _ptr(slots), _ptr(local_lens),
                                  _ptr(virt), _ptr(rblk))
    return dict(owner=owner[:T], slots=None if slots is None else slots[:, :T],
                local_lens=local_lens[:, :B], virt_blocks=virt[:B], rank_blocks=rblk[:, :B], status=st)


def transfer_blocks(N, I, bs, seq_lens, block_tables, num_blocks):
    """Blocks moved under PD disaggregation.  Returns dict(counts [N, B],
    blocks [N, B, max_blocks], fills [N, B, max_blocks], totals [2], status)."""
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    B = seq_lens.size
    max_blocks = bt.shape[-1]
    counts = np.empty((N, max(1, B)), dtype=np.int32)
    blocks = np.empty((N, max(1, B), max_blocks), dtype=np.int32)
    fills = np.empty((N, max(1, B), max_blocks), dtype=np.int32)
    totals = np.zeros(2, dtype=np.int64)
    st = _load().orc_transfer_blocks(N, I, bs, B, _ptr(seq_lens), _ptr(bt), max_blocks, int(num_blocks),
                                     _ptr(counts), _ptr(blocks), _ptr(fills), _ptr(totals))
    return dict(counts=counts[:, :B], blocks=blocks[:, :B], fills=fills[:, :B], totals=totals, status=st)


def pcp_partition(K, ctx_lens, q_lens, max_q):
    """Head-tail prefill partition over K PCP ranks.  Returns dict(pos [B,
    max_q] (global positions in gathered rank order, -1 = padding),
    padded_len [B], status)."""
    ctx = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    ql = np.ascontiguousarray(q_lens, dtype=np.int32)
    B = ctx.size
    pos = np.empty((max(1, B), max_q), dtype=np.int32)
    plen = np.empty(max(1, B), dtype=np.int32)
    st = _load().orc_pcp_partition(K, B, _ptr(ctx), _ptr(ql), max_q, _ptr(pos), _ptr(plen))
    return dict(pos=pos[:B], padded_len=plen[:B], status=st)


def attention(wl, rank=-1, rows=None, nthreads=None):
    """Attention of the workload's query rows in fp64 (rank < 0: unsharded).

    rows: flat ids ((b * Tq + t) * Hq + h) or None for all.  Returns (out, lse).
    """
    c = wl.cfg
    B, Tq, Hq, Hkv, Dk, Dv = (int(c[k]) for k in ("B", "Tq", "Hq", "Hkv", "Dk", "Dv"))
    layout = 1 if c["layout"] == "mla" else 0
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = B * Tq * Hq if rows_arr is None else rows_arr.size
    out = np.empty((max(1, n), Dv), dtype=np.float64)
    lse = np.empty(max(1, n), dtype=np.float64)
    seq_lens = np.ascontiguousarray(wl.seq_lens, dtype=np.int32)
    req_start = np.ascontiguousarray(wl.req_start, dtype=np.int64)
    q = np.ascontiguousarray(wl.q)
    k = np.ascontiguousarray(wl.k)
    v = None if wl.v is None else np.ascontiguousarray(wl.v)
    _load().orc_attention(layout, B, Tq, Hq, Hkv, Dk, Dv, _ptr(seq_lens), _ptr(req_start),
                          _ptr(q), _DT[c["q_dtype"]], _ptr(k), _ptr(v), _DT[c["kv_dtype"]],
                          float(wl.kv_scale), float(c["softmax_scale"]), int(c["N"]), int(c["I"]),
                          int(rank), n if rows_arr is not None else 0, _ptr(rows_arr),
                          _ptr(out), _ptr(lse), int(nthreads or threads()))
    return out[:n], lse[:n]


def merge(o_parts, lse_parts):
    """o_parts [N, rows, Dv], lse_parts [N, rows] -> (out [rows, Dv], lse [rows])."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    N, rows, Dv = o_parts.shape
    out = np.empty((max(1, rows), Dv), dtype=np.float64)
    lse = np.empty(max(1, rows), dtype=np.float64)
    _load().orc_merge(N, rows, Dv, _ptr(o_parts), _ptr(lse_parts), _ptr(out), _ptr(lse))
    return out[:rows], lse[:rows]


def sparse_localize(cand, N, I, seq_lens, Tq):
    """Candidate localization under DCP ("vLLM DCP and PCP", the indexer
    localisation tests in its source-and-test table; the GLM-5.3
    context-parallelism page, "What DP and TP leave unresolved": sparse MLA
    attends to a selected token set).  For every query row's
    candidate list (global positions, -1 unused), each rank's candidates in
    list order, as its local positions (ownership by the rank equation, local
    positions by the running count of local_layout).  Returns (local [N, rows,
    k] int32 padded with -1, counts [N, rows] int32)."""
    cand = np.asarray(cand, dtype=np.int64)
    rows, k = cand.shape
    local = np.full((N, rows, k), -1, dtype=np.int32)
    counts = np.zeros((N, rows), dtype=np.int32)
    layouts = {}
    for i in range(rows):
        b = i // Tq
        L = int(seq_lens[b])
        if L not in layouts:
            layouts[L] = local_layout(L, N, I)
        rk, lp = layouts[L]
        for t in cand[i]:
            if t < 0:
                continue
            r = int(rk[t])
            local[r, i, counts[r, i]] = lp[t]
            counts[r, i] += 1
    return local, counts


def sparse_attention(wl, cand, rank=-1, N=None, I=None):
    """Attention of every query token's heads over its candidate set only, in
    fp64: s_j = scale * q . k_j over the candidates, o = softmax(s) V,
    L = logsumexp(s).  rank >= 0 keeps the candidates that rank owns (a
    rank's partial; empty: zeros and -inf).  Returns (out [rows*Hq, Dv],
    lse [rows*Hq]) with rows = B * Tq, row order (b, t, h)."""
    c = wl.cfg
    B, Tq, Hq, Hkv, Dk, Dv = (int(c[x]) for x in ("B", "Tq", "Hq", "Hkv", "Dk", "Dv"))
    N = int(c["N"]) if N is None else N
    I = int(c["I"]) if I is None else I
    G = Hq // Hkv
    mla = c["layout"] == "mla"
    scale = float(c["softmax_scale"])
    cand = np.asarray(cand, dtype=np.int64)
    out = np.zeros((B * Tq * Hq, Dv))
    lse = np.full(B * Tq * Hq, -np.inf)
    layouts = {}
    for b in range(B):
        L = int(wl.seq_lens[b])
        if rank >= 0 and L not in layouts:
            layouts[L] = local_layout(L, N, I)
        for t in range(Tq):
            i = b * Tq + t
            C = cand[i][cand[i] >= 0]
            if rank >= 0:
                C = C[layouts[L][0][C] == rank]
            if C.size == 0:
                continue
            rows_kv = wl.req_start[b] + C
            q = decode(wl.q[b, t], c["q_dtype"])                      # [Hq, Dk]
            kk = decode(wl.k[rows_kv], c["kv_dtype"], wl.kv_scale)    # [n, Hkv, Dk]
            vv = kk[:, :, :Dv] if mla else decode(wl.v[rows_kv], c["kv_dtype"], wl.kv_scale)
            for h in range(Hq):
                g = h // G
                s = scale * (kk[:, g, :] @ q[h])
                m = s.max()
                w = np.exp(s - m)
                l = w.sum()
                r = (i * Hq) + h
                lse[r] = m + np.log(l)
                out[r] = (w @ vv[:, g, :]) / l
    return out, lse
