"""The quantised-entry parity checks themselves, on the CPU: the oracle's own
quantisation passes them, and the mistakes they exist to catch -- a scale
rounded the wrong way, codes truncated instead of rounded, a lost sign of
zero -- fail them.  The "GPU" side here is the oracle's output with the
mistake planted in it."""
import numpy as np
import pytest

import oracle
from _util import check_e4m3_rows, check_fp4_rows


def _entries(seed, rows, d):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((rows, d)) * rng.uniform(0.01, 4.0, (rows, 1))


def _pack(nib):
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def test_fp4_check_accepts_the_oracle_and_rejects_planted_mistakes():
    y = _entries(1, 64, 64)
    codes, scales = oracle.quantize_fp4_rows(y)
    check_fp4_rows(codes, scales, y)
    # scale rounded up instead of to nearest: some block's byte moves
    x = np.abs(y.reshape(64, 4, 16)).max(-1) / 6.0
    up = oracle.e4m3_encode(x)
    dec = oracle.e4m3_decode(up)
    up = np.where(dec < x, up + 1, up).astype(np.uint8)
    assert (up != scales).any()
    with pytest.raises(AssertionError):
        check_fp4_rows(codes, up, y)
    # codes truncated toward zero instead of rounded
    s = np.repeat(oracle.e4m3_decode(scales), 16, -1)
    r = y / s
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    trunc = np.searchsorted(grid, np.minimum(np.abs(r), 6), side="right") - 1
    nib = (trunc | np.where(np.signbit(r), 8, 0)).astype(np.uint8)
    with pytest.raises(AssertionError):
        check_fp4_rows(_pack(nib), scales, y)
    # -0 written as +0
    want = oracle.e2m1_encode(r)
    assert (want == 8).any()
    with pytest.raises(AssertionError):
        check_fp4_rows(_pack(np.where(want == 8, 0, want).astype(np.uint8)), scales, y)


def test_e4m3_check_accepts_the_oracle_and_rejects_planted_mistakes():
    y = _entries(2, 32, 128)
    codes, scales = oracle.quantize_e4m3_rows(y)
    check_e4m3_rows(codes, scales, y)
    # one code one step off, away from any midpoint
    bad = codes.copy()
    i = np.argmax(np.abs(y[0]))
    bad[0, (i + 1) % 128] ^= 1
    with pytest.raises(AssertionError):
        check_e4m3_rows(bad, scales, y)
    # scales 1e-5 off
    with pytest.raises(AssertionError):
        check_e4m3_rows(codes, scales * np.float32(1 + 1e-5), y)
