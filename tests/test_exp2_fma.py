"""The FMA-pipe exp2 that takes part of the softmax exponentials off the
special-function unit: its polynomial is the Remez minimax fit, and on the GPU
it stays within that fit's relative error of 2^x (Cody-Waite reduction is
exact, so the only error is the polynomial's and the float32 rounding)."""
import math
import os
import re

import numpy as np
import pytest
import torch

from kv_cache_compression_flash_b300.exp2_fit import remez_exp2, rounded

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _device_coefficients():
    text = open(os.path.join(ROOT, "kv_cache_compression_flash_b300", "csrc", "common.cuh")).read()
    return [float.fromhex(re.search(rf"kExp2C{i} = (0x[0-9a-fA-Fp.+-]+)f;", text).group(1)) for i in range(4)]


def test_coefficients_are_the_remez_fit():
    c32, err = rounded(remez_exp2(3))
    assert _device_coefficients() == [float(v) for v in c32]
    assert err < 1e-4
    # the fit equioscillates: its error is the same at both ends of the interval and at an interior extremum
    f = np.linspace(-0.5, 0.5, 200001)
    e = np.polyval(c32.astype(np.float64)[::-1], f) / np.exp2(f) - 1.0
    assert abs(abs(e[0]) - abs(e[-1])) < 0.05 * err and abs(e).max() <= err * 1.0001


def test_remez_is_exact_for_low_degree_limits():
    # degree 1 minimax of 2^f on [-1/2, 1/2] has a closed-form error level; a
    # higher degree is always at least as good
    errs = [rounded(remez_exp2(d))[1] for d in (2, 3, 4)]
    assert errs[0] > errs[1] > errs[2]
    assert errs[2] < 3e-6


@pytest.mark.gpu
def test_device_exp2_within_the_fit_error():
    from kv_cache_compression_flash_b300 import _lib as L
    x = np.concatenate([np.linspace(-125.0, 0.0, 1_000_001), np.linspace(-1.0, 1.0, 100_001),
                        -np.arange(0, 126, dtype=np.float64), [-125.5, -126.0, -200.0, -np.inf]]).astype(np.float32)
    y = L.debug_exp2(torch.from_numpy(x).cuda()).cpu().numpy().astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    ok = x >= -125.0
    rel = np.abs(y[ok] / ref[ok] - 1.0)
    _, err = rounded(remez_exp2(3))
    assert rel.max() <= err + 2.0 ** -22, rel.max()                 # the fit's error plus float32 rounding
    assert (y[~ok] == 0.0).all()
    assert y[x == 0.0][0] == pytest.approx(1.0, rel=err + 2.0 ** -22)
    # integers: the reduction leaves f = 0, so 2^n is the constant term scaled exactly
    ints = -np.arange(0, 126, dtype=np.float64)
    yi = L.debug_exp2(torch.from_numpy(ints.astype(np.float32)).cuda()).cpu().numpy().astype(np.float64)
    c0 = _device_coefficients()[0]
    assert np.array_equal(yi, c0 * np.exp2(ints))
