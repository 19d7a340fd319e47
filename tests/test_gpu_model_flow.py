"""The full 8B-shaped decode flow as the workload defines it: 32 layers x 8
kv-heads (32 query heads), head_dim 128, batch 1, a 131072-token context
prefill-quantized on every layer, then 64 decode steps that each append one
token to every layer and run decode attention on every layer (4-bit
per-channel keys, 8-bit per-token values).

Checked against the oracle on sampled (batch, kv-head) streams, layer by
layer after the GPU flow: the packed state (codes, scales, zero points, fp16
key residual) bit-exact at steps 1, 32 and 64 on every layer; attention
within 1e-3 of the fp64 oracle at steps 1, 32 and 64 on every layer and at
every step on layer 0."""
import math

import numpy as np
import pytest
import torch

from bit_quantized_kv_kvq_gb300 import workloads as W
from bit_quantized_kv_kvq_gb300.synth import LayerSource
from oracle import kvq_oracle as O
from tests import kvq_check as K

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

STEPS = 64
PICKS = [0, 7]           # sampled streams (batch 1: kv-heads 0 and 7)
STATE_STEPS = (1, 32, 64)


def _picked(x, wl):
    """[B][H][S][D] device tensor -> the sampled streams [picks][S][D] numpy."""
    return x.reshape(wl.batch * wl.num_kv_heads, *x.shape[2:])[PICKS].cpu().numpy()


def test_8b_32_layer_prefill_then_64_decode_steps():
    wl = W.LLAMA8B_FULL
    S, Lyr = wl.seq_len, wl.num_layers
    scale = 1.0 / math.sqrt(wl.head_dim)
    cache = K.make_gpu_cache(wl, S + STEPS)
    srcs = [LayerSource(wl, l, device="cuda") for l in range(Lyr)]
    for l in range(Lyr):
        k, v = srcs[l].kv(S)
        cache.prefill(l, k, v)
        del k, v
    steps = [[srcs[l].step(t) for l in range(Lyr)] for t in range(1, STEPS + 1)]
    out = torch.empty((Lyr, wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    got = {}      # (t, l) -> GPU output rows of the sampled streams [picks][g][D]
    states = {}   # (t, l) -> new rows of the sampled streams' state
    for t in range(1, STEPS + 1):
        for l in range(Lyr):
            _, k1, v1 = steps[t - 1][l]
            cache.append(l, k1, v1)
        for l in range(Lyr):
            q, _, _ = steps[t - 1][l]
            cache.decode(l, q, scale, out=out[l])
        torch.cuda.synchronize()
        o = out.cpu().double().reshape(Lyr, wl.batch * wl.num_kv_heads, wl.gqa, wl.head_dim)
        for l in range(Lyr):
            if t in STATE_STEPS or l == 0:
                got[(t, l)] = o[l, PICKS].numpy().copy()
        if t in STATE_STEPS and t < STEPS:
            # the rows a step adds: value rows S .. S + t - 1, the key residual
            for l in range(Lyr):
                for i, n in enumerate(PICKS):
                    st = K.gpu_state(cache, l, n)
                    states[(t, l, i)] = {"v_words": st["v_words"][S:].copy(), "v_meta": st["v_meta"][S:].copy(),
                                         "k_resid": st["k_resid"].copy()}
    assert cache.status() == 0

    for l in range(Lyr):
        k, v = srcs[l].kv(S)
        ks, vs = _picked(k, wl), _picked(v, wl)
        del k, v
        oc = O.OracleCache(K.spec_of(wl), len(PICKS))
        oc.prefill(ks, vs)
        for t in range(1, STEPS + 1):
            q, k1, v1 = steps[t - 1][l]
            oc.append(_picked(k1[:, :, None], wl)[:, 0], _picked(v1[:, :, None], wl)[:, 0])
            if (t, l) in got:
                ref = oc.decode(K.q_streams(q, wl)[PICKS], scale)
                K.assert_attention_close(got[(t, l)], ref, where="layer %d step %d" % (l, t))
            if t in STATE_STEPS:
                for i, n in enumerate(PICKS):
                    want = K.oracle_state(oc, i)
                    if t == STEPS:
                        K.assert_state_equal(K.gpu_state(cache, l, n), want, "layer %d step %d n=%d" % (l, t, n))
                    else:
                        want_new = {"v_words": want["v_words"][S:], "v_meta": want["v_meta"][S:],
                                    "k_resid": want["k_resid"]}
                        K.assert_state_equal(states[(t, l, i)], want_new, "layer %d step %d n=%d" % (l, t, n))
