"""The cubic behind the prefill kernel's FMA-pipe exponentials: its constants
are the minimax fit, and the kernel's fp32 steps stay within the fit's bound."""
import pathlib
import re

import numpy as np
import pytest

scipy = pytest.importorskip("scipy")

from masked_flash_attention_gb300 import exp2_fit

SRC = pathlib.Path(__file__).resolve().parents[1] / "masked_flash_attention_gb300" / "csrc" / "prefill_sm103.cu"


def kernel_coeffs():
    text = SRC.read_text()
    return [float(re.search(r"kExp2C%d = ([0-9.e+-]+)f;" % k, text).group(1)) for k in (1, 2, 3)]


def test_constants_are_the_fit():
    cs, err = exp2_fit.fit()
    assert err < 1e-4
    np.testing.assert_allclose(kernel_coeffs(), cs, rtol=1e-7)


def test_relative_error_bound():
    cs = np.array(kernel_coeffs(), dtype=np.float32)
    v = np.linspace(-126.0, 8.0, 2_000_001).astype(np.float32)
    got = exp2_fit.exp2_fp32(v, cs).astype(np.float64)
    want = np.exp2(v.astype(np.float64))
    rel = np.abs(got / want - 1.0)
    assert rel.max() < 1.0e-4, rel.max()


def test_special_values():
    cs = np.array(kernel_coeffs(), dtype=np.float32)
    n = np.arange(-126, 9).astype(np.float32)
    np.testing.assert_array_equal(exp2_fit.exp2_fp32(n, cs), np.exp2(n))  # integers: exact powers of two
    low = np.array([-127.0, -150.0, -1e30, -np.inf], dtype=np.float32)
    np.testing.assert_array_equal(exp2_fit.exp2_fp32(low, cs), np.zeros(4, np.float32))
