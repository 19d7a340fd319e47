"""Mixed precision by layer (TurboQuant KV-cache page, demingchina.com/news/57821,
§5.3: the sensitive layers get more bits; KVQuant page, cf-1.com/news/2306543,
§4.2): one cache whose layers hold different code widths, each layer checked
against the oracle built with that layer's codec (state bit-exact, attention
within 1e-3), through prefill with a key residual, appends across a key-block
flush, and decode with 8 and with 4 query heads per kv-head."""
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

PAIRS = [(8, 8), (4, 8), (4, 4), (3, 3), (8, 4)]


@pytest.mark.parametrize("hq", [16, 8])
def test_layers_with_different_code_widths(hq):
    base = replace(W.LLAMA8B_FULL, num_layers=len(PAIRS), batch=1, num_kv_heads=2, num_q_heads=hq,
                   seq_len=300, v_group=128)
    S, steps = base.seq_len, 22  # 300 + 22 crosses the key block at 320
    cache = kvq.QuantizedKVCache(base.num_layers, base.batch, base.num_kv_heads, base.head_dim, S + steps,
                                 4, 4, base.k_mode, base.v_mode, base.k_group, base.v_group, 0,
                                 device="cuda", layer_bits=PAIRS)
    scale = 1.0 / math.sqrt(base.head_dim)
    for l, (kb, vb) in enumerate(PAIRS):
        wl = replace(base, k_bits=kb, v_bits=vb)
        assert cache.layout(l).k_words_per_row == O.words_per_row(kb, 128)
        assert cache.layout(l).v_words_per_row == O.words_per_row(vb, 128)
        src = LayerSource(wl, l, device="cpu")
        k, v = src.kv(S)
        cache.prefill(l, k.cuda(), v.cuda())
        oc = O.OracleCache(K.spec_of(wl), wl.batch * wl.num_kv_heads)
        oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
        for t in range(1, steps + 1):
            q, k1, v1 = src.step(t)
            cache.append(l, k1.cuda(), v1.cuda())
            oc.append(K.streams_of(k1[:, :, None], wl)[:, 0], K.streams_of(v1[:, :, None], wl)[:, 0])
            if t in (1, steps):
                o = cache.decode(l, q.cuda(), scale).cpu().double()
                ref = oc.decode(K.q_streams(q, wl), scale)
                K.assert_attention_close(o.reshape(ref.shape).numpy(), ref, where="layer %d k%dv%d step %d" % (l, kb, vb, t))
        torch.cuda.synchronize()
        for n in range(wl.batch * wl.num_kv_heads):
            K.assert_state_equal(K.gpu_state(cache, l, n), K.oracle_state(oc, n), "layer %d n=%d" % (l, n))
    assert cache.status() == 0
