"""Parity at the full workload sizes, in the launch configuration the bench
times: metadata and slots bit-exact against the oracle, attention compared on
rows the oracle computes one by one, plus properties that hold at any size."""

import numpy as np
import pytest
import torch

import oracle
from dcp_workloads import CONFIG_ORDER, config, make_workload

from gpu_common import assert_close_rows, f64, tol_for

pytestmark = pytest.mark.gpu


def _sample_rows(wl, n, seed):
    c = wl.cfg
    B, Tq, Hq = int(c["B"]), int(c["Tq"]), int(c["Hq"])
    rng = np.random.default_rng(seed)
    rows = set()
    # the longest request, the shortest, and random others; every query token
    b_long, b_short = int(np.argmax(wl.seq_lens)), int(np.argmin(wl.seq_lens))
    for b in [b_long, b_short] + list(rng.integers(0, B, size=n)):
        t = int(rng.integers(0, Tq))
        h = int(rng.integers(0, Hq))
        rows.add((int(b) * Tq + t) * Hq + h)
        if len(rows) >= n:
            break
    if Tq > 1:
        for t in range(Tq):
            rows.add((b_long * Tq + t) * Hq + 5 % Hq)
    return np.array(sorted(rows), dtype=np.int64)


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
    rows = _sample_rows(wl, 12, seed=7)
    ref_o, ref_l = oracle.attention(wl, rows=rows)
    assert_close_rows(out_h[rows], lse_h[rows], ref_o, ref_l, tol_for(c), f"{name} sampled rows")
