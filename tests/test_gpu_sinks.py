"""Attention sinks (KVQuant page, cf-1.com/news/2306543, §4.1: the first
5-10 tokens keep their fp16 keys and values): the CUDA path against the
oracle with the same sink count — fp16 sink rows and the coded rows after
them bit-exact, attention within 1e-3 — through prefills shorter and longer
than the sinks, appends that cross the sink boundary and a key-block flush,
and every decode kernel family (stream-K at 8 query heads per kv-head,
token-row at 4, one head, the symmetric int8 GQA kernel and the generic
kernel with outliers)."""
import math
from dataclasses import replace

import pytest
import torch

import bit_quantized_kv_kvq_gb300 as kvq
from bit_quantized_kv_kvq_gb300 import workloads as W
from bit_quantized_kv_kvq_gb300.synth import LayerSource
from oracle import kvq_oracle as O
from tests import kvq_check as K

pytestmark = pytest.mark.gpu

CASES = [
    # (name, workload, q heads per kv-head, sinks, prefill length, appends)
    ("stream-K k3v3", replace(W.LLAMA70B_32K, batch=2, num_kv_heads=2), 8, 5, 360, 30),
    ("token-row k4v8", replace(W.LLAMA8B_FULL, batch=1, num_kv_heads=2), 4, 8, 3, 70),
    ("one head k4v4", replace(W.LLAMA7B_16K, batch=2, num_kv_heads=2), 1, 64, 200, 5),
    ("sym int8 gqa", replace(W.TINY_Q8, batch=1, num_kv_heads=2), 4, 10, 130, 3),
    ("generic, outliers", replace(W.DENSE_SPARSE_128K, batch=1, num_kv_heads=2, k_mode=W.ASYM_PER_TOKEN,
                                  k_group=32), 2, 5, 90, 12),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_sinks_against_the_oracle(case):
    name, wl0, g, ns, s, steps = case
    wl = replace(wl0, num_layers=1, num_q_heads=g * wl0.num_kv_heads, seq_len=s)
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(s)
    cache = K.make_gpu_cache(wl, s + steps + 1, sink_tokens=ns)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl, ns), wl.batch * wl.num_kv_heads)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    scale = 1.0 / math.sqrt(wl.head_dim)
    for t in range(steps + 1):
        q, k1, v1 = src.step(t)
        if t:
            cache.append(0, k1.cuda(), v1.cuda())
            oc.append(K.streams_of(k1[:, :, None], wl)[:, 0], K.streams_of(v1[:, :, None], wl)[:, 0])
        if t in (0, 1, steps // 2, steps):
            o = cache.decode(0, q.cuda(), scale).cpu().double()
            ref = oc.decode(K.q_streams(q, wl), scale)
            K.assert_attention_close(o.reshape(ref.shape).numpy(), ref, where="%s t=%d" % (name, t))
    torch.cuda.synchronize()
    assert cache.layout(0).sink_len == min(ns, s + steps)
    for n in range(wl.batch * wl.num_kv_heads):
        K.assert_state_equal(K.gpu_state(cache, 0, n), K.oracle_state(oc, n), "%s n=%d" % (name, n))
    assert cache.status() == 0


def test_sink_count_is_checked():
    with pytest.raises(kvq.KVQError):
        K.make_gpu_cache(replace(W.TINY_Q8, num_layers=1), 100, sink_tokens=65)
