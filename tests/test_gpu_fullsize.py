"""Parity at the full sizes of the five workloads (and the codebook layer), in the launch
configuration bench.py times: one prefill of the whole context, one append
and one decode, on the whole batch. The first and the last (batch, kv-head)
stream are then checked against the oracle run on those streams' inputs
alone: codes, scales, zero points, outlier lists and fp16 residual keys
bit-exact, attention of their query heads within 1e-3 of the fp64 oracle.
(The 32-layer workload runs one of its layers.)"""
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

FULL = [(w.name, w) for w in W.ALL + W.EXTRA]


@pytest.mark.parametrize("name,wl", FULL, ids=[f[0] for f in FULL])
def test_full_size_sampled_streams(name, wl):
    wl = replace(wl, num_layers=1)
    S, N = wl.seq_len, wl.batch * wl.num_kv_heads
    src = LayerSource(wl, 0, device="cuda")
    k, v = src.kv(S)
    _, k1, v1 = src.step(1)
    q, _, _ = src.step(2)
    scale = 1.0 / math.sqrt(wl.head_dim)
    cache = K.make_gpu_cache(wl, S + 1)
    cache.prefill(0, k, v)
    cache.append(0, k1, v1)
    out = cache.decode(0, q, scale)
    torch.cuda.synchronize()
    assert cache.status() == 0

    picks = sorted({0, N - 1})
    oc = O.OracleCache(K.spec_of(wl), len(picks))
    oc.prefill(K.streams_of(k, wl)[picks], K.streams_of(v, wl)[picks])
    oc.append(K.streams_of(k1, wl)[picks], K.streams_of(v1, wl)[picks])
    for i, n in enumerate(picks):
        K.assert_state_equal(K.gpu_state(cache, 0, n), K.oracle_state(oc, i), "stream %d" % n)
    ref = oc.decode(K.q_streams(q, wl)[picks], scale)
    got = out.cpu().double().reshape(N, wl.gqa, wl.head_dim).numpy()[picks]
    K.assert_attention_close(got, ref, where=name)
