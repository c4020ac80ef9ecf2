"""Error bounds of the two-term e4m3 split that the fp8-cache MLA kernel uses.

The fp8-cache kernel multiplies on kind::f8f6f4, so its bf16 query and its
fp32 probabilities are each carried as a sum of two e4m3 values, hi + lo, with
hi = e4m3(x) and lo = e4m3(x - hi), both rounded to nearest even.  These
tests check the stated bounds of that arithmetic, exhaustively where the
input type is small, using torch's float8_e4m3fn casts as the rounding.  They
do not run the kernel (the GPU parity tests do); they pin the numerical claim
that its tolerance rests on.

Query: a row is scaled by 2^-e so that its largest magnitude lies in
(224, 448].  A bf16 value has 8 significant bits and hi keeps 4, so the
residual is a multiple of the value's last-place unit with at most 4
significant bits: hi + lo is exact whenever the residual is an e4m3 normal
(>= 2^-6), and otherwise off by at most half the subnormal spacing, 2^-10.

Probabilities: p <= 2^8 goes through fp16 first, so the residual fp16(p) - hi
is exact in fp16; hi + lo then keeps about 8 significant bits: the error is
at most (2^-8 + 2^-11) p + 2^-10, and p below 2^-10 vanishes.
"""

import numpy as np
import torch

E4M3 = torch.float8_e4m3fn


def _e4m3(x):
    return x.to(E4M3).to(torch.float64)


def _all_finite_bf16():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).to(torch.float64)
    return x[torch.isfinite(x)]


def test_query_row_scale_puts_the_maximum_in_224_448():
    rng = np.random.default_rng(7)
    for amax in np.concatenate([rng.lognormal(0, 6, 2000), [2.0 ** k for k in range(-60, 60)]]):
        # the smallest e with amax * 2^-e <= 448; then amax * 2^-e > 224
        e = int(np.ceil(np.log2(amax / 448.0)))
        while amax * 2.0 ** -e > 448.0:
            e += 1
        while amax * 2.0 ** (1 - e) <= 448.0:
            e -= 1
        y = amax * 2.0 ** -e
        assert 224.0 < y <= 448.0, (amax, e, y)


def test_query_split_exact_unless_the_residual_is_subnormal():
    x = _all_finite_bf16()
    # every power-of-two scale that can occur: the row maximum lands in (224, 448],
    # so a value of the row lies at or below 448 after scaling
    for e in range(-140, 130):
        y = x * 2.0 ** -e
        y = y[y.abs() <= 448.0]
        hi = _e4m3(y)
        r = y - hi  # exact in fp64 (and in the kernel's fp32)
        lo = _e4m3(r)
        err = (y - (hi + lo)).abs()
        normal = r.abs() >= 2.0 ** -6
        assert torch.all(err[normal] == 0), e
        assert torch.all(err <= 2.0 ** -10), e
        # hi never saturates below 448 (448 is an e4m3 value)
        assert torch.all(hi.abs() <= 448.0)


def test_query_split_error_is_tiny_against_the_row_maximum():
    # the largest absolute error, 2^-10, against a row maximum above 224
    assert 2.0 ** -10 / 224.0 < 4.4e-6


def test_probability_split_bound():
    # probabilities as the kernel forms them, p = 2^(s - m_ref + 5) <= 2^8
    k = torch.arange(-14 * 4096, 8 * 4096 + 1, dtype=torch.float64) / 4096.0
    p = (2.0 ** k).to(torch.float32).to(torch.float64)
    ph = p.to(torch.float16).to(torch.float64)
    hi = _e4m3(ph)
    r = ph - hi
    assert torch.all(r.to(torch.float16).to(torch.float64) == r)  # the residual is exact in fp16
    lo = _e4m3(r)
    err = (p - (hi + lo)).abs()
    assert torch.all(err <= (2.0 ** -8 + 2.0 ** -11) * p + 2.0 ** -10)
    # below 2^-10 a probability rounds to zero in both terms
    tiny = p < 2.0 ** -10
    assert torch.all((hi + lo)[tiny] == 0)
    # about bf16's precision where the residual stays normal
    big = p >= 2.0 ** -2
    assert torch.all(err[big] <= (2.0 ** -8 + 2.0 ** -11) * p[big])


# ---------------------------------------------------------------------------
# The softmax reference across tiles.  A model of the fp8 kernel's per-tile
# step (its constants: tiles of 256 tokens, p' = 2^(s - m_ref + 5), the
# reference raised when a tile's maximum passes it by more than 3 binades and
# lowered to the tile's maximum when that lies more than 4 binades below it),
# with hi + lo formed as above; l sums the fp32 p'.  Scores are in log2 units.

TILE, UP, DOWN, BIAS = 256, 3.0, 4.0, 5.0


def _split_sum(p):
    ph = torch.from_numpy(p.astype(np.float32)).to(torch.float16).to(torch.float64)
    hi = _e4m3(ph)
    return (hi + _e4m3(ph - hi)).numpy()


def _tiled_softmax_weights(s2, lower):
    """Represented weights (what P.V sees) and fp32 row sum, both relative to
    the final reference, for scores s2 walked tile by tile."""
    m_ref, m_top = -np.inf, -np.inf
    rep, lsum = [], 0.0
    for t0 in range(0, len(s2), TILE):
        s = s2[t0:t0 + TILE]
        mx = s.max()
        m_top = max(m_top, mx)
        corr = 1.0
        if m_ref == -np.inf:
            m_ref, corr = mx, 0.0
        elif mx > m_ref + UP or (mx < m_ref - lower and m_top - mx <= 64.0):
            corr, m_ref = 2.0 ** (m_ref - mx), mx
        rep = [r * corr for r in rep]
        lsum = lsum * corr
        p = (2.0 ** (s - m_ref + BIAS)).astype(np.float32).astype(np.float64)
        rep.append(_split_sum(p))
        lsum += p.sum()
    return np.concatenate(rep), lsum


def test_one_way_reference_loses_a_flat_tail_two_way_keeps_it():
    # a sink 12 nats above 32K identical tail tokens: the tail carries ~17 % of
    # the mass, each tail token 2^-17.3 of the sink.  One-way, every tail tile
    # stays at the sink's reference and vanishes; two-way, only the TILE - 1
    # tail tokens that share the sink's tile do (plus the split's rounding)
    n = 32768
    s2 = np.zeros(n)
    s2[0] = 12.0 * np.log2(np.e)
    for lower, lost_at_least, lost_at_most in [(np.inf, 0.15, 1.0), (DOWN, 0.0, (TILE - 1) / (n - 1) + 2.0 ** -8)]:
        rep, lsum = _tiled_softmax_weights(s2, lower)
        tail_share_true = (n - 1) * np.exp(-12.0) / (1 + (n - 1) * np.exp(-12.0))
        tail_share_rep = rep[1:].sum() / lsum
        lost = (tail_share_true - tail_share_rep) / tail_share_true
        assert lost_at_least <= lost <= lost_at_most, (lower, lost)


def test_two_way_reference_aggregate_bound():
    """Against the row sum, the weight that P.V misses (or gets wrong) stays
    below the per-tile bound: a token is off by at most 2^-10 (p' units) below
    p' = 2^-6 and by (2^-8 + 2^-11) p' above, and a tile whose maximum sits at
    p' >= 2^(5 - DOWN) holds TILE - 1 = 255 other tokens at most, so the missing
    share is below 255 * 2^-10 / 2^(5 - DOWN) + 2^-8 + 2^-11 of the row sum."""
    rng = np.random.default_rng(11)
    bound = (TILE - 1) * 2.0 ** -10 / 2.0 ** (BIAS - DOWN) + 2.0 ** -8 + 2.0 ** -11
    worst = 0.0
    for trial in range(60):
        ntiles = int(rng.integers(2, 40))
        s2 = []
        for _ in range(ntiles):
            # adversarial tiles: one maximum, the rest just under the vanishing
            # point relative to a maximum that sits anywhere within the window
            top = rng.uniform(-DOWN, UP) + (0.0 if trial % 3 else rng.uniform(-30, 30))
            depth = rng.uniform(10.0, 16.0, TILE - 1)
            s2.append(np.concatenate([[top], top - depth]))
        s2 = np.concatenate(s2)
        rep, lsum = _tiled_softmax_weights(s2, DOWN)
        # both sides relative to the final reference: the fp32 row sum is exact enough here
        miss = abs(lsum - rep.sum()) / lsum
        worst = max(worst, miss)
        assert miss <= bound, (trial, miss, bound)
    assert worst > 0.0
