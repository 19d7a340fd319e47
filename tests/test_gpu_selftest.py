"""The arithmetic the quantizer kernels rely on, run on the device through
the C ABI (include/kvq_selftest.h) over exhaustive or adversarial inputs and
compared with IEEE division; and the kernels' bounded wait, made to give up.

The codes are rne((x - z) / s) in fp32 (TurboQuant 3-bit KV quantization
page, dpshk.com/news/6341316, §3.1); the kernels avoid the division on the
common path, so their arithmetic must reproduce the IEEE quotient exactly."""
import math

import pytest
import torch

import bit_quantized_kv_kvq_gb300 as kvq
from bit_quantized_kv_kvq_gb300 import workloads as W
from bit_quantized_kv_kvq_gb300.synth import LayerSource
from tests import kvq_check as K

pytestmark = pytest.mark.gpu

NONE = 2 ** 64 - 1
TWO_17 = 0x48000000  # bit pattern of 2^17 (fp16 max - min is at most 131008)


@pytest.mark.parametrize("levels", [3, 7, 15, 127, 255])
def test_scale_division_is_ieee_for_every_range_up_to_2_17(levels):
    """Every fp32 a in [0, 2^17] (1.2e9 values): the prefill's scale
    (max - min) / L equals __fdiv_rn(a, L) bit for bit."""
    mism, first = kvq.selftest_div_levels(levels, 0, TWO_17)
    assert (mism, first) == (0, NONE), "L=%d: %d mismatches, first a bits %#x" % (levels, mism, first)


@pytest.mark.parametrize("k_first,k_last", [(-256, 255), (-4096, -3840), (3840, 4096)])
def test_quant_step_near_ties(k_first, k_last):
    """The append and per-token kernels' quant_step(d, s, RN(1/s)) against
    rne(__fdiv_rn(d, s)) for every positive finite fp16 scale (subnormal
    ones included), codes k in the range, and dividends within 8 ulps of
    (k + 1/2) s."""
    mism, first = kvq.selftest_code_rounding(0, k_first, k_last, 8)
    assert (mism, first) == (0, NONE), "%d mismatches, first key %#x" % (mism, first)


def test_bracketed_codes_near_ties():
    """The prefill's bracketed reciprocal with the exact-residual settle
    against rne(__fdiv_rn(d, s)) for every normal fp16 scale, codes 0..255
    and dividends within 16 ulps of (k + 1/2) s."""
    mism, first = kvq.selftest_code_rounding(1, 0, 255, 16)
    assert (mism, first) == (0, NONE), "%d mismatches, first key %#x" % (mism, first)


def test_codebook_quotient_is_ieee_for_every_fp16_pair():
    """The codebook quantizer's x / s without a division (RN(x RN(1/s))
    corrected once by an fma) equals __fdiv_rn(x, s) for every finite fp16 x
    and every positive finite fp16 s (2.0e9 pairs)."""
    mism, first = kvq.selftest_codebook_quotient()
    assert (mism, first) == (0, NONE), "%d mismatches, first key %#x" % (mism, first)


def test_selftest_arguments_are_checked():
    with pytest.raises(kvq.KVQError):
        kvq.selftest_div_levels(5, 0, 10)
    with pytest.raises(kvq.KVQError):
        kvq.selftest_code_rounding(1, -1, 10, 4)
    with pytest.raises(kvq.KVQError):
        kvq.selftest_code_rounding(0, 0, 10, 65)


def test_bounded_wait_gives_up_and_reports_timeout():
    """A wait on a barrier that nothing completes gives up after its polls,
    raises the timeout bit, and the kernel returns: kvq_cache_status reports
    KVQ_ERR_TIMEOUT once, the word is then clear, and the context still
    runs a decode that matches the oracle."""
    wl = W.TINY_Q8
    cache = K.make_gpu_cache(wl, 300)
    src = LayerSource(wl, 0, device="cuda")
    k, v = src.kv(257)
    cache.prefill(0, k, v)
    assert cache.status() == 0
    cache.selftest_wait_timeout(200)  # at most 200 polls of 10 us
    with pytest.raises(kvq.KVQError) as ei:
        cache.status()
    assert ei.value.status == 6  # KVQ_ERR_TIMEOUT
    assert cache.status() == 0
    q, _, _ = src.step(0)
    out = cache.decode(0, q, 1.0 / math.sqrt(wl.head_dim))
    torch.cuda.synchronize()
    assert cache.status() == 0
    assert torch.isfinite(out).all()
    with pytest.raises(kvq.KVQError):
        cache.selftest_wait_timeout(0)
