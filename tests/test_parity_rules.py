"""The comparison rule itself (CPU only): it accepts what the stated tolerance
allows and rejects a planted error just beyond it."""
import numpy as np
import pytest
import torch

from tests import parity

F16, BF16, F32 = 0, 1, 2


def _bits(x, dt):
    t = torch.tensor(x, dtype={F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32}[dt])
    return parity.bits_of(t)


@pytest.mark.parametrize("dt", [F16, BF16])
def test_one_ulp_passes_two_ulp_fails_for_typical_elements(dt):
    c64 = np.array([10.0, -3.0, 0.75])
    want = _bits(c64, dt)
    sigma = np.full(3, 1.0)
    got = want.copy()
    got[0] += 1                                    # one ulp away
    parity.check(got, want, dt, c64=c64, sigma=sigma, K=64)
    got[0] += 1                                    # two ulps away
    with pytest.raises(AssertionError):
        parity.check(got, want, dt, c64=c64, sigma=sigma, K=64)


def test_cancellation_element_uses_accumulation_scale():
    # |exact| tiny, sigma large: an error of a few fp16 ulps but far below tau passes
    c64 = np.array([1e-4])
    sigma = np.array([15.0])
    K = 2048
    tau = parity.tau_of(sigma, K)[0]
    got = _bits([1e-4 + 0.5 * tau], F16)
    parity.check(got, _bits(c64, F16), F16, c64=c64, sigma=sigma, K=K)
    got = _bits([1e-4 + 3 * tau], F16)
    with pytest.raises(AssertionError):
        parity.check(got, _bits(c64, F16), F16, c64=c64, sigma=sigma, K=K)


def test_fp32_frobenius_and_max_abs():
    w = np.linspace(-5, 5, 101)
    want = _bits(w, F32)
    parity.check(want.copy(), want, F32)
    bad = _bits(w + 0.02, F32)
    with pytest.raises(AssertionError):
        parity.check(bad, want, F32)


def test_ordinal_is_monotone_and_signed_zero_equal():
    x = np.array([-2.0, -1.0, -0.0, 0.0, 1e-7, 1.0, 2.0])
    o = parity.ordinal(_bits(x, F16))
    assert np.all(np.diff(o) >= 0) and o[2] == o[3] == 0


def test_check_pair_allows_two_roundings_but_not_more():
    c64 = np.array([10.0, 1e-4])
    sigma = np.array([1.0, 15.0])
    a = _bits([10.0, 1e-4], F16)
    b = a.copy()
    b[0] += 2                                    # two ulps apart at 10.0
    parity.check_pair(a, b, F16, c64, sigma, 64)
    b[0] += 2                                    # four ulps apart
    with pytest.raises(AssertionError):
        parity.check_pair(a, b, F16, c64, sigma, 64)
