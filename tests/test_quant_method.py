"""The device NVFP4 activation quantizer decides each E2M1 code without a
division per value: q = float32(x * float32(1 / eff)), and where the codes of
q (1 - 2^-20) and q (1 + 2^-20) agree that code is taken, else x / eff is
divided.  The premise: q lies within 3 * 2^-24 (relative) of float32(x / eff)
and the E2M1 rounding is monotone, so whenever the two nudged codes agree they
equal the code of float32(x / eff); an exact tie always lands between them.
This checks the premise in float32 arithmetic on the CPU, over random values
and values placed exactly on the grid's midpoints (no GPU)."""
import numpy as np

from oracle import codec

EPS = np.float32(2.0 ** -20)


def _decide(x, eff):
    with np.errstate(all="ignore"):
        r = (np.float32(1.0) / eff).astype(np.float32)
        q = (x * r).astype(np.float32)
        lo = (q * (np.float32(1.0) - EPS)).astype(np.float32)
        hi = (q * (np.float32(1.0) + EPS)).astype(np.float32)
        exact = (x / eff).astype(np.float32)
    fin = np.isfinite(q)
    code = lambda v: codec.encode_rne_sat(np.where(fin, v, np.float32(0)), "e2m1")  # noqa: E731
    take = (code(lo) == code(hi)) & fin
    return take, code(lo), codec.encode_rne_sat(np.where(np.isfinite(exact), exact, np.float32(0)), "e2m1")


def test_agreeing_neighbours_give_the_exact_quotients_code():
    rng = np.random.default_rng(0)
    n = 400_000
    x = (rng.standard_normal(n) * np.exp2(rng.integers(-30, 30, n))).astype(np.float32)
    eff = (np.abs(rng.standard_normal(n)) * np.exp2(rng.integers(-30, 30, n)) + np.float32(1e-30)).astype(np.float32)
    take, fast, exact = _decide(x, eff)
    assert not np.any(take & (fast != exact))
    assert take.mean() > 0.99                     # the division is the rare path


def test_midpoints_always_take_the_division():
    # x / eff exactly on a midpoint between two E2M1 values (a tie): the two
    # nudged codes differ, so the exact quotient decides (ties to even)
    rng = np.random.default_rng(1)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    eff = np.exp2(rng.integers(-20, 20, 20_000)).astype(np.float32) * np.float32(1.5)
    x = (mids[rng.integers(0, 7, eff.size)] * eff * rng.choice([-1.0, 1.0], eff.size)).astype(np.float32)
    assert np.array_equal((x / eff).astype(np.float32), (mids[np.argmin(np.abs(np.abs(x / eff)[:, None] - mids), axis=1)]
                                                         * np.sign(x)).astype(np.float32))
    take, fast, exact = _decide(x, eff)
    assert not np.any(take)
