"""Prefill attention over the quantized cache (the NIAH q8_0 page,
cf-1.com/news/5482713, §4.2: the prefill behind the time to first token; the
KVQuant page, cf-1.com/news/2306543, §3.4: attention on the dequantized
cache): the queries of the last C cached positions attend the cache causally.
The CUDA kernel against the oracle's causal attention on the same dequantized
cache, within 1e-3 per row, for every codec family (per-channel keys with an
fp16 residual, 3/4/8-bit per-token values, outliers, symmetric int8, codebook
codes, sinks), one to eight query heads per kv-head, whole prefills and
chunks after appends, several CTAs per stream with a ragged last one."""
import math
from dataclasses import replace

import numpy as np
import pytest
import torch

import bit_quantized_kv_kvq_gb300 as kvq
from bit_quantized_kv_kvq_gb300 import workloads as W
from bit_quantized_kv_kvq_gb300.synth import LayerSource
from oracle import kvq_oracle as O
from tests import kvq_check as K

pytestmark = pytest.mark.gpu

CB = W.CODEBOOK_PER_TOKEN

CASES = [
    # (name, workload, q heads per kv-head, prefill, appends, chunk, sinks)
    ("8b k4v8 whole prefill", W.LLAMA8B_FULL, 4, 300, 0, 300, 0),
    ("8b k4v8 chunk of 37", W.LLAMA8B_FULL, 4, 300, 0, 37, 0),
    ("70b k3v3 g8", W.LLAMA70B_32K, 8, 200, 0, 200, 0),
    ("dense-sparse outliers g1", W.DENSE_SPARSE_128K, 1, 150, 0, 150, 0),
    ("7b k4v4 g2 appends", W.LLAMA7B_16K, 2, 100, 30, 30, 0),
    ("tiny sym int8", W.TINY_Q8, 4, 130, 3, 133, 0),
    ("codebook e2m1 g2", replace(W.LLAMA8B_E2M1), 2, 90, 5, 40, 0),
    ("sinks k4v8", W.LLAMA8B_FULL, 4, 100, 4, 104, 5),
]


def q_streams(q, wl, g):
    """q [B][C][Hq][D] -> [B*Hkv][C][g][D] numpy (query head h reads kv-head h // g)."""
    b, c = q.shape[0], q.shape[1]
    t = q.detach().cpu().double().reshape(b, c, wl.num_kv_heads, g, wl.head_dim).permute(0, 2, 1, 3, 4)
    return t.reshape(b * wl.num_kv_heads, c, g, wl.head_dim).numpy()


def build(wl, s, steps, ns):
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(s)
    cache = K.make_gpu_cache(wl, s + steps + 1, sink_tokens=ns)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl, ns), wl.batch * wl.num_kv_heads)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    for t in range(1, steps + 1):
        _, k1, v1 = src.step(t)
        cache.append(0, k1.cuda(), v1.cuda())
        oc.append(K.streams_of(k1[:, :, None], wl)[:, 0], K.streams_of(v1[:, :, None], wl)[:, 0])
    return cache, oc


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_prefill_attention_against_the_oracle(case):
    name, wl0, g, s, steps, chunk, ns = case
    wl = replace(wl0, num_layers=1, batch=2, num_kv_heads=2, num_q_heads=2 * g, seq_len=s)
    cache, oc = build(wl, s, steps, ns)
    gen = torch.Generator().manual_seed(7 + s + chunk)
    q = torch.randn((wl.batch, chunk, wl.num_q_heads, wl.head_dim), generator=gen).half()
    scale = 1.0 / math.sqrt(wl.head_dim)
    o = cache.prefill_attention(0, q.cuda(), scale)
    torch.cuda.synchronize()
    ref = oc.prefill_attention(q_streams(q, wl, g), scale)
    got = q_streams(o.float(), wl, g)
    K.assert_attention_close(got.reshape(-1, wl.head_dim), ref.reshape(-1, wl.head_dim), where=name)
    assert cache.status() == 0


def test_prefill_attention_fp16_output_and_last_row_is_the_decode():
    wl = replace(W.LLAMA8B_FULL, num_layers=1, batch=1, num_kv_heads=2, num_q_heads=8, seq_len=257)
    cache, oc = build(wl, 257, 0, 0)
    q = torch.randn((1, 64, 8, 128), generator=torch.Generator().manual_seed(3)).half().cuda()
    o32 = cache.prefill_attention(0, q, 0.09)
    o16 = cache.prefill_attention(0, q, 0.09, out_dtype=torch.float16)
    torch.cuda.synchronize()
    assert o16.dtype == torch.float16
    assert float((o16.float() - o32).abs().max()) <= 2e-3 * float(o32.abs().max())
    dec = cache.decode(0, q[:, -1].contiguous(), 0.09)
    err = O.row_relative_error(o32[:, -1].cpu().numpy(), dec.cpu().numpy())
    assert float(err.max()) <= 1e-4


def test_prefill_attention_arguments_are_checked():
    wl = replace(W.LLAMA7B_16K, num_layers=1, batch=1, num_kv_heads=2, num_q_heads=2, seq_len=10)
    cache, _ = build(wl, 10, 0, 0)
    q = torch.zeros((1, 11, 2, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KVQError):
        cache.prefill_attention(0, q, 1.0)                    # more queries than cached tokens
    with pytest.raises(kvq.KVQError):
        cache.prefill_attention(0, q[:, :0].contiguous(), 1.0)  # empty chunk
    with pytest.raises(kvq.KVQError):
        cache.prefill_attention(0, torch.zeros((1, 4, 3, 128), dtype=torch.float16, device="cuda"), 1.0)
    assert cache.status() == 0


def test_prefill_attention_full_size_sampled_streams():
    """One 8B-shaped layer at its full 131072-token context (8 kv-heads, 32
    query heads, the launch bench.py times with a shorter chunk): the last
    64 positions' queries, checked on the first and last stream against the
    oracle run on those streams alone."""
    wl = replace(W.LLAMA8B_FULL, num_layers=1)
    S, N = wl.seq_len, wl.batch * wl.num_kv_heads
    src = LayerSource(wl, 0, device="cuda")
    k, v = src.kv(S)
    cache = K.make_gpu_cache(wl, S + 1)
    cache.prefill(0, k, v)
    q = torch.randn((1, 64, wl.num_q_heads, 128), generator=torch.Generator().manual_seed(5)).half()
    o = cache.prefill_attention(0, q.cuda(), 1.0 / math.sqrt(128))
    torch.cuda.synchronize()
    assert cache.status() == 0
    picks = [0, N - 1]
    oc = O.OracleCache(K.spec_of(wl), len(picks))
    oc.prefill(K.streams_of(k, wl)[picks], K.streams_of(v, wl)[picks])
    del k, v
    ref = oc.prefill_attention(q_streams(q, wl, wl.gqa)[picks], 1.0 / math.sqrt(128))
    got = q_streams(o.float(), wl, wl.gqa)[picks]
    K.assert_attention_close(got.reshape(-1, 128), ref.reshape(-1, 128), where="full size")
