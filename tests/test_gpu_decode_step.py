"""kvq_decode_step: one append + decode per layer, with the appends on a
second stream so that they overlap the decodes of earlier layers (the pages
run quantization and attention on separate streams: NIAH q8_0 page,
cf-1.com/news/5482713, §4.3). It must give what the same calls give one
after another on one stream: the same cache bytes and, for the deterministic
split decode, the same output bits (the stream-K decode merges its warps in
arrival order, so there the outputs agree to rounding)."""
import math
from dataclasses import replace

import pytest
import torch

from bit_quantized_kv_kvq_gb300 import workloads as W
from bit_quantized_kv_kvq_gb300.synth import LayerSource
from tests import kvq_check as K

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hq", [8, 16])
def test_two_stream_step_matches_the_serial_calls(hq):
    wl = replace(W.LLAMA8B_FULL, num_layers=4, batch=1, num_kv_heads=2, num_q_heads=hq, seq_len=300)
    S, steps = wl.seq_len, 20
    a = K.make_gpu_cache(wl, S + steps + 1)
    b = K.make_gpu_cache(wl, S + steps + 1)
    srcs = [LayerSource(wl, l, device="cuda") for l in range(wl.num_layers)]
    for l, src in enumerate(srcs):
        k, v = src.kv(S)
        a.prefill(l, k, v)
        b.prefill(l, k, v)
    scale = 1.0 / math.sqrt(wl.head_dim)
    aux = torch.cuda.Stream()
    outs_a = [torch.empty((1, hq, 128), dtype=torch.float32, device="cuda") for _ in range(wl.num_layers)]
    for t in range(1, steps + 1):
        qs, k1s, v1s = zip(*[src.step(t) for src in srcs])
        a.decode_step(list(qs), list(k1s), list(v1s), scale, outs_a, aux_stream=aux)
        outs_b = []
        for l in range(wl.num_layers):
            b.append(l, k1s[l], v1s[l])
            outs_b.append(b.decode(l, qs[l], scale))
        torch.cuda.synchronize()
        for l in range(wl.num_layers):
            if hq // wl.num_kv_heads == 8:
                torch.testing.assert_close(outs_a[l], outs_b[l], rtol=1e-6, atol=1e-6)
            else:
                assert torch.equal(outs_a[l], outs_b[l]), "step %d layer %d" % (t, l)
    assert a.status() == 0 and b.status() == 0
    assert torch.equal(a.buffer, b.buffer)
