"""End-to-end error of the quantized decode: the CUDA path's attention output
against fp64 attention on the unquantized fp16 K/V the cache was built from,
per workload codec (bit widths), on sampled streams. Reported, not gated by
a parity tolerance: quantization error is the method's own, not a kernel
defect. The checks are sanity bounds and the ordering more bits -> less
error on one shared set of keys and values."""
import math
from dataclasses import replace

import numpy as np
import pytest
import torch

from bit_quantized_kv_kvq_gb300 import workloads as W
from bit_quantized_kv_kvq_gb300.synth import LayerSource
from oracle import kvq_oracle as O
from tests import kvq_check as K

pytestmark = pytest.mark.gpu

SEQ = 8192


def _small(wl, seq=SEQ, **kw):
    hkv = min(wl.num_kv_heads, 2)
    return replace(wl, num_layers=1, batch=1, num_kv_heads=hkv, num_q_heads=hkv * wl.gqa, seq_len=seq, **kw)


def _e2e_error(wl, src_wl=None):
    """Max row error over every query head of the sampled streams, and the
    codec label."""
    src = LayerSource(src_wl or wl, 0, device="cuda")
    S = wl.seq_len
    k, v = src.kv(S)
    q, k1, v1 = src.step(0)
    cache = K.make_gpu_cache(wl, S + 1)
    cache.prefill(0, k, v)
    cache.append(0, k1, v1)
    scale = 1.0 / math.sqrt(wl.head_dim)
    o = cache.decode(0, q, scale)
    torch.cuda.synchronize()
    assert cache.status() == 0
    kf = np.concatenate([K.streams_of(k, wl), K.streams_of(k1[:, :, None], wl)], axis=1).astype(np.float64)
    vf = np.concatenate([K.streams_of(v, wl), K.streams_of(v1[:, :, None], wl)], axis=1).astype(np.float64)
    ref = O.attend(K.q_streams(q, wl), kf, vf, scale)
    got = o.detach().cpu().double().numpy().reshape(ref.shape)
    return float(O.row_relative_error(got, ref).max())


@pytest.mark.parametrize("wl", [W.TINY_Q8, W.LLAMA7B_16K, W.LLAMA70B_32K, W.DENSE_SPARSE_128K, W.LLAMA8B_FULL],
                         ids=lambda w: w.name)
def test_e2e_error_per_workload(wl, record_property):
    w = _small(wl)
    e = _e2e_error(w)
    label = "k%dv%d" % (w.k_bits, w.v_bits)
    record_property("e2e_error_" + label, e)
    print("\ne2e_error %s %s (%d tokens, %d streams): %.5f" % (wl.name, label, SEQ + 1, w.num_kv_heads, e))
    assert np.isfinite(e)
    bound = 0.05 if min(w.k_bits, w.v_bits) == 8 else 0.6
    assert e < bound


def test_more_bits_less_error():
    """One set of keys and values (lognormal key channels, 8192 tokens) under
    3-, 4- and 8-bit codes with the same groups (T = G = 128): the error
    falls as the bit width grows ([TurboQuant-3bit] §3.1: the quantization
    step is (max - min) / (2^b - 1))."""
    base = _small(W.LLAMA7B_16K)
    errs = {}
    for b in (3, 4, 8):
        w = replace(base, k_bits=b, v_bits=b, k_group=128, v_group=128)
        errs[b] = _e2e_error(w, src_wl=base)
    print("\ne2e_error by bits (T = G = 128):", {k: round(v, 5) for k, v in errs.items()})
    assert errs[8] < errs[4] < errs[3]
