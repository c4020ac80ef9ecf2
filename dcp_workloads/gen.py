"""Seeded input generation.

Recipe (every config):
  * lengths: fixed, an explicit list, or lognormal(log(median), sigma) clipped
    to [lo, hi] and rounded to integers;
  * q, k, v (or the MLA latent) ~ N(0, 1) drawn in fp32 from numpy's PCG64
    (k and v in fixed-size row chunks, chunk c seeded by child c of the
    tensor's SeedSequence, so threads do not change the values),
    then rounded to the storage dtype: bf16 by round-to-nearest-even (torch
    cast), fp8 e4m3fn with one per-tensor scale = amax / 448 (fp32), values
    divided by the scale, clamped to +-448 and cast (torch cast, RNE);
  * keys/values are laid out densely per request, request b occupying rows
    req_start[b] .. req_start[b+1]-1 in token order (no paging);
  * physical blocks: once a caller knows how many blocks each (rank, request)
    needs, allocate_blocks() hands out ids from a seeded random permutation of
    the pool, so every rank owns disjoint, scattered blocks.

Raw storage is returned as numpy arrays of the storage type: float32 for f32,
uint16 bit patterns for bf16, uint8 bit patterns for fp8.
"""

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

_CHUNK_VALUES = 1 << 24  # values per independently seeded chunk (fixed: results do not depend on threads)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (RNE, torch cast); return the uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def fp8_bits(x: np.ndarray, scale: float) -> np.ndarray:
    """Encode x / scale as fp8 e4m3fn (clamped to +-448, torch cast); uint8 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = torch.clamp(t / torch.tensor(scale, dtype=torch.float32), -448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _round(x: np.ndarray, dtype: str, scale: float = 1.0) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits(x)
    if dtype == "fp8":
        return fp8_bits(x, scale)
    raise ValueError(f"unknown dtype {dtype}")


def _np_dtype(dtype: str):
    return {"f32": np.float32, "bf16": np.uint16, "fp8": np.uint8}[dtype]


@dataclass
class Workload:
    cfg: dict
    seed: int
    seq_lens: np.ndarray            # [B] int32, global length incl. the Tq new tokens
    req_start: np.ndarray           # [B+1] int64 row offsets into k/v
    q: np.ndarray                   # [B, Tq, Hq, Dk] raw
    k: np.ndarray                   # [T_total, Hkv, Dk] raw (MLA: the latent rows)
    v: Optional[np.ndarray]         # [T_total, Hkv, Dv] raw (None for MLA)
    kv_scale: float = 1.0           # fp8 per-tensor scale (1.0 otherwise)
    extra: dict = field(default_factory=dict)

    @property
    def B(self):
        return int(self.cfg["B"])

    @property
    def total_tokens(self):
        return int(self.req_start[-1])

    def token_lists(self):
        """(tok_req [T] int32, tok_pos [T] int64) for every cached token, request-major."""
        L = self.seq_lens.astype(np.int64)
        tok_req = np.repeat(np.arange(self.B, dtype=np.int32), L)
        tok_pos = np.concatenate([np.arange(n, dtype=np.int64) for n in L]) if len(L) else np.zeros(0, np.int64)
        return tok_req, tok_pos

    def new_token_lists(self):
        """(tok_req, tok_pos) of the Tq newest tokens of every request (one decode step)."""
        Tq = int(self.cfg["Tq"])
        L = self.seq_lens.astype(np.int64)
        tok_req = np.repeat(np.arange(self.B, dtype=np.int32), Tq)
        tok_pos = np.concatenate([np.arange(n - Tq, n, dtype=np.int64) for n in L])
        return tok_req, tok_pos


def draw_lengths(cfg, rng) -> np.ndarray:
    spec = cfg["lengths"]
    B = int(cfg["B"])
    kind = spec[0]
    if kind == "fixed":
        out = np.full(B, int(spec[1]), dtype=np.int64)
    elif kind == "list":
        out = np.asarray(spec[1], dtype=np.int64)
        assert out.shape == (B,)
    elif kind == "lognormal":
        median, sigma, lo, hi = spec[1], spec[2], spec[3], spec[4]
        x = rng.lognormal(mean=np.log(median), sigma=sigma, size=B)
        out = np.rint(np.clip(x, lo, hi)).astype(np.int64)
    else:
        raise ValueError(kind)
    return out.astype(np.int32)


def _chunks(rows, shape_tail):
    per_row = int(np.prod(shape_tail)) if len(shape_tail) else 1
    step = max(1, _CHUNK_VALUES // max(1, per_row))
    return [(s, min(rows, s + step)) for s in range(0, rows, step)]


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


def _draw_rows(seedseq, rows, shape_tail, dtype, scale):
    """Draw rows x shape_tail standard normals chunk by chunk and round each chunk."""
    out = np.empty((rows,) + tuple(shape_tail), dtype=_np_dtype(dtype))
    chunks = _chunks(rows, shape_tail)
    seeds = seedseq.spawn(len(chunks))

    def work(i):
        s, e = chunks[i]
        x = np.random.Generator(np.random.PCG64(seeds[i])).standard_normal(
            (e - s,) + tuple(shape_tail), dtype=np.float32)
        out[s:e] = _round(x, dtype, scale)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(len(chunks))))
    return out


def _amax_rows(seedseq, rows, shape_tail):
    chunks = _chunks(rows, shape_tail)
    seeds = seedseq.spawn(len(chunks))

    def work(i):
        s, e = chunks[i]
        x = np.random.Generator(np.random.PCG64(seeds[i])).standard_normal(
            (e - s,) + tuple(shape_tail), dtype=np.float32)
        return float(np.abs(x).max()) if x.size else 0.0

    with ThreadPoolExecutor(_threads()) as ex:
        return max([0.0] + list(ex.map(work, range(len(chunks)))))


def make_workload(cfg: dict, seed: Optional[int] = None, zero_q: bool = False) -> Workload:
    """Draw one workload for cfg with the given seed (default: the config's index)."""
    seed = int(cfg.get("index", 0) if seed is None else seed)
    ss = np.random.SeedSequence(seed)
    s_len, s_q, s_k, s_v = ss.spawn(4)
    B, Tq, Hq, Hkv = (int(cfg[k]) for k in ("B", "Tq", "Hq", "Hkv"))
    Dk, Dv = int(cfg["Dk"]), int(cfg["Dv"])
    seq_lens = draw_lengths(cfg, np.random.Generator(np.random.PCG64(s_len)))
    if np.any(seq_lens < Tq):
        raise ValueError("every request needs at least Tq tokens")
    req_start = np.zeros(B + 1, dtype=np.int64)
    np.cumsum(seq_lens.astype(np.int64), out=req_start[1:])
    T = int(req_start[-1])

    rq = np.random.Generator(np.random.PCG64(s_q))
    qf = rq.standard_normal((B, Tq, Hq, Dk), dtype=np.float32)
    if zero_q:
        qf[...] = 0.0
    q = _round(qf, cfg["q_dtype"])

    kv_dtype = cfg["kv_dtype"]
    scale = 1.0
    if kv_dtype == "fp8":
        # per-tensor scale over everything the cache will hold (keys and values)
        amax = _amax_rows(np.random.SeedSequence(s_k.entropy, spawn_key=s_k.spawn_key), T, (Hkv, Dk))
        if cfg["layout"] == "gqa":
            amax = max(amax, _amax_rows(np.random.SeedSequence(s_v.entropy, spawn_key=s_v.spawn_key), T, (Hkv, Dv)))
        scale = float(np.float32(amax) / np.float32(448.0))
    k = _draw_rows(np.random.SeedSequence(s_k.entropy, spawn_key=s_k.spawn_key), T, (Hkv, Dk), kv_dtype, scale)
    v = None
    if cfg["layout"] == "gqa":
        v = _draw_rows(np.random.SeedSequence(s_v.entropy, spawn_key=s_v.spawn_key), T, (Hkv, Dv), kv_dtype, scale)
    return Workload(cfg=dict(cfg), seed=seed, seq_lens=seq_lens, req_start=req_start,
                    q=q, k=k, v=v, kv_scale=scale)


def allocate_blocks(rank_blocks: np.ndarray, seed: int, spare: int = 0):
    """Hand out physical block ids for per-(rank, request) block counts.

    rank_blocks: [N, B] number of blocks each rank needs for each request.
    Returns (block_tables [N, B, max_blocks] int32 padded with -1, num_blocks).
    Ids come from a seeded random permutation of the pool, dealt in (rank,
    request) order, so ranks hold disjoint, scattered blocks.
    """
    rank_blocks = np.asarray(rank_blocks, dtype=np.int64)
    N, B = rank_blocks.shape
    total = int(rank_blocks.sum())
    num_blocks = total + int(spare)
    max_blocks = max(1, int(rank_blocks.max()) if rank_blocks.size else 1)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), 0xB10C])))
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.full((N, B, max_blocks), -1, dtype=np.int32)
    pos = 0
    for r in range(N):
        for b in range(B):
            n = int(rank_blocks[r, b])
            tables[r, b, :n] = perm[pos:pos + n]
            pos += n
    return tables, num_blocks


def sparse_candidates(wl: Workload, k: int, seed: int = 0) -> np.ndarray:
    """A synthetic top-k indexer: for every query token (b, t) -- position
    L_b - Tq + t -- k distinct positions drawn uniformly from the ones it may
    attend to (0 .. its own position), sorted ascending; all of them when
    fewer are visible, -1 after the last.  Returns int32 [B * Tq, k]."""
    Tq = int(wl.cfg["Tq"])
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(wl.seed), int(seed), 0x70C])))
    out = np.full((wl.B * Tq, k), -1, dtype=np.int32)
    for b in range(wl.B):
        L = int(wl.seq_lens[b])
        for t in range(Tq):
            vis = L - Tq + t + 1
            pick = np.arange(vis) if vis <= k else np.sort(rng.choice(vis, size=k, replace=False))
            out[b * Tq + t, :len(pick)] = pick
    return out


def sink_tail_workload(cfg: dict, sink_positions, gaps_nats, seed: int = 0) -> Workload:
    """A peaked long-context input for the MLA layout (one request, Tq = 1):
    one strongly attended key (an "attention sink") at each of
    sink_positions, and a long flat tail of identical keys whose values have
    a nonzero mean, so that the tail's many small weights carry a share of
    the softmax mass that an output must not lose.

    Recipe (values before rounding to the storage dtype):
      * tail row: value columns c < Dv hold 0.5 + 0.25 cos(c), RoPE columns 0;
      * sink row: value columns -1 + 0.25 sin(c), RoPE columns 1.5;
      * query head h: latent columns 0, RoPE columns g_h with
        g_h = gaps_nats[h] / (softmax_scale * 1.5 * (Dk - Dv)), so that head h
        scores a sink about gaps_nats[h] nats above every tail token.
    fp8 uses one per-tensor scale amax / 448 = 1.5 / 448 (the sink's RoPE
    columns store 448 exactly).  `seed` only labels the workload (block
    permutation); nothing here is random.
    """
    B, Tq, Hq, Hkv = (int(cfg[k]) for k in ("B", "Tq", "Hq", "Hkv"))
    Dk, Dv = int(cfg["Dk"]), int(cfg["Dv"])
    assert cfg["layout"] == "mla" and B == 1 and Tq == 1 and Hkv == 1
    seq_lens = draw_lengths(cfg, None)
    L = int(seq_lens[0])
    gaps = np.asarray(gaps_nats, dtype=np.float64)
    assert gaps.shape == (Hq,)
    c = np.arange(Dk)
    tail = np.where(c < Dv, 0.5 + 0.25 * np.cos(c), 0.0).astype(np.float32)
    sink = np.where(c < Dv, -1.0 + 0.25 * np.sin(c), 1.5).astype(np.float32)
    kv_dtype = cfg["kv_dtype"]
    scale = float(np.float32(1.5) / np.float32(448.0)) if kv_dtype == "fp8" else 1.0
    tail_raw = _round(tail[None, None, :], kv_dtype, scale)[0, 0]
    sink_raw = _round(sink[None, None, :], kv_dtype, scale)[0, 0]
    k = np.empty((L, 1, Dk), dtype=_np_dtype(kv_dtype))
    k[:, 0, :] = tail_raw
    for p in sink_positions:
        assert 0 <= int(p) < L
        k[int(p), 0, :] = sink_raw
    g = gaps / (float(cfg["softmax_scale"]) * 1.5 * (Dk - Dv))
    qf = np.zeros((B, Tq, Hq, Dk), dtype=np.float32)
    qf[0, 0, :, Dv:] = g[:, None].astype(np.float32)
    q = _round(qf, cfg["q_dtype"])
    req_start = np.array([0, L], dtype=np.int64)
    return Workload(cfg=dict(cfg), seed=int(seed), seq_lens=seq_lens, req_start=req_start, q=q, k=k, v=None,
                    kv_scale=scale, extra={"sink_positions": [int(p) for p in sink_positions]})
