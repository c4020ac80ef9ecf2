"""Host-side logic of the work split, checked on the CPU.

The attention kernels deal P chunks to We = min(W, P) workers as equal
contiguous ranges [w P / We, (w + 1) P / We) and give each merge group one
partial slot per worker that touches it.  These tests check the arithmetic the
planner and kernels share (worker_of / worker_begin in dcp_internal.cuh): every
worker in play owns at least one chunk, worker_of inverts the ranges, and the
segment count of a group equals the number of distinct workers touching it,
including when there are fewer chunks than workers.  The last test runs the
header code itself (compiled as host code) over random unit layouts.
"""

import os
import shutil
import subprocess

import numpy as np
import pytest

_HERE = os.path.dirname(os.path.abspath(__file__))


def worker_begin(w, W, P):
    return w * P // W


def worker_of(x, W, P):
    return ((x + 1) * W - 1) // P


@pytest.mark.parametrize("P,W", [(1, 1), (1, 1216), (7, 1216), (300, 1216), (1216, 1216), (131072, 1216),
                                 (5, 3), (1000003, 608)])
def test_ranges_cover_and_invert(P, W):
    We = min(W, P)
    starts = np.array([worker_begin(w, We, P) for w in range(We + 1)])
    assert starts[0] == 0 and starts[-1] == P
    assert np.all(np.diff(starts) >= 1)  # every worker in play owns >= 1 chunk
    xs = np.unique(np.concatenate([np.arange(min(P, 2000)), np.random.default_rng(0).integers(0, P, 2000)]))
    for x in xs:
        w = worker_of(int(x), We, P)
        assert starts[w] <= x < starts[w + 1]


def test_segment_counts_match_distinct_workers():
    rng = np.random.default_rng(1)
    for trial in range(200):
        groups = rng.integers(0, 6, size=rng.integers(1, 40))
        P = int(groups.sum())
        if P == 0:
            continue
        W = int(rng.integers(1, 3 * P + 5))
        We = min(W, P)
        bounds = np.concatenate([[0], np.cumsum(groups)])
        total = 0
        for g in range(len(groups)):
            a, e = bounds[g], bounds[g + 1]
            if e == a:
                continue
            cnt = worker_of(int(e - 1), We, P) - worker_of(int(a), We, P) + 1
            owners = {worker_of(int(x), We, P) for x in range(a, e)}
            assert cnt == len(owners)
            total += cnt
        assert total <= We + len(groups)


def test_tile_walk_and_worker_ranges_on_the_header_code(tmp_path):
    """The header code itself (worker ranges, unit lookup, the MLA kernels'
    tile walk), compiled by nvcc as host code and run on random unit layouts
    (tests/host/tile_walk_check.cu states the properties checked)."""
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "tile_walk_check")
    src = os.path.join(_HERE, "host", "tile_walk_check.cu")
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-x", "cu", src, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_closed_forms_of_the_cuda_path_match_the_oracle(tmp_path):
    """owner_rank / local_pos / local_len / local_len32 of dcp_internal.cuh,
    compiled as host code (tests/host/closed_forms_dump.cu), against the
    oracle bit-exactly where the oracle's brute-force count finishes quickly
    (the local position of token t is the count of its rank's tokens before
    it); at every size, the local lengths partition L with a spread <= I and
    the 32-bit form equals the 64-bit one."""
    import oracle
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "closed_forms_dump")
    src = os.path.join(_HERE, "host", "closed_forms_dump.cu")
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-x", "cu", src, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60).stdout.split("\n")
    small = 200000
    lens = {}
    n_t = n_l = 0
    for line in out:
        f = line.split()
        if not f:
            continue
        if f[0] == "T":
            N, I, t, owner, lpos = (int(x) for x in f[1:])
            assert owner == oracle.rank_of(t, N, I), line
            if t < small:
                assert lpos == oracle.local_len(t, owner, N, I), line
            n_t += 1
        else:
            N, I, L, rr, l64, l32 = (int(x) for x in f[1:])
            if L < small:
                assert l64 == oracle.local_len(L, rr, N, I), line
            if l32 >= 0:
                assert l32 == l64, line
            lens.setdefault((N, I, L), {})[rr] = l64  # (the case list repeats some L)
            n_l += 1
    assert n_t > 300 and n_l > 300
    for (N, I, L), by_rank in lens.items():
        v = [by_rank[r] for r in range(N)]
        assert sum(v) == L and max(v) - min(v) <= I, (N, I, L, v)
