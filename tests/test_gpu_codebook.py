"""Codebook (non-uniform) 4-bit codes for keys and values (KVQuant page,
cf-1.com/news/2306543, §2.2 item 2; the minifloat levels of the TurboQuant
3-bit KV-cache page, dpshk.com/news/6341316, §3.3): the CUDA path against the
oracle with the same 16 levels. Codes and fp16 scales are bit-exact after a
prefill and after appends, including groups that are all zero; attention is
within 1e-3 of the fp64 oracle for one, two, four and eight query heads per
kv-head, with and without attention sinks, through both decode entry points."""
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


def random_levels(seed):
    """16 sorted levels of unequal spacing and sign balance, exact in fp16."""
    r = np.random.default_rng(seed)
    return tuple(float(x) for x in np.sort(r.standard_normal(16) * 1.5 + 0.2).astype(np.float16))


CASES = [
    # (name, base workload, q heads per kv-head, group, levels, prefill, appends, sinks)
    ("e2m1 g8 G32", W.LLAMA8B_FULL, 8, 32, kvq.E2M1_LEVELS, 300, 20, 0),
    ("e2m1 g1 G128", W.LLAMA7B_16K, 1, 128, kvq.E2M1_LEVELS, 70, 9, 0),
    ("random g4 G16", W.LLAMA70B_32K, 4, 16, random_levels(7), 129, 66, 0),
    ("random g2 G64 sinks", W.DENSE_SPARSE_128K, 2, 64, random_levels(8), 200, 12, 5),
]


def codebook_workload(wl0, g, group, seq):
    return replace(wl0, num_layers=1, batch=2, num_kv_heads=2, num_q_heads=2 * g, seq_len=seq,
                   k_bits=4, v_bits=4, k_mode=CB, v_mode=CB, k_group=group, v_group=group,
                   outliers_per_row=0, decode_steps=1)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_codebook_against_the_oracle(case):
    name, wl0, g, group, levels, s, steps, ns = case
    wl = codebook_workload(wl0, g, group, s)
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(s)
    k, v = k.clone(), v.clone()
    k[0, 1, 3, :group] = 0          # a key group that is all zero stores scale 0 and code 0
    v[1, 0, s - 1, -group:] = 0     # and a value group
    # a group at scale 1 (absmax = max|level|) holding the midpoints of adjacent
    # levels and the levels themselves: ties and near-ties of the nearest level
    lv = sorted(set(np.float16(x).item() for x in levels))
    cbmax = max(abs(x) for x in lv)
    mids = [cbmax] + [(a + b) / 2 for a, b in zip(lv, lv[1:])] + lv
    row = torch.tensor((mids * group)[:group], dtype=torch.float16)
    k[1, 0, 7, :group] = row
    if group < 128:
        v[0, 1, 2, group:2 * group] = row.flip(0)
    else:
        v[0, 1, 2, :] = row.flip(0)
    cache = K.make_gpu_cache(wl, s + steps + 1, sink_tokens=ns, codebook=levels)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl, ns, levels), wl.batch * wl.num_kv_heads)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    scale = 1.0 / math.sqrt(wl.head_dim)
    for t in range(steps + 1):
        q, k1, v1 = src.step(t)
        if t:
            cache.append(0, k1.cuda(), v1.cuda())
            oc.append(K.streams_of(k1[:, :, None], wl)[:, 0], K.streams_of(v1[:, :, None], wl)[:, 0])
        if t in (0, 1, steps):
            ref = oc.decode(K.q_streams(q, wl), scale)
            o = cache.decode(0, q.cuda(), scale).cpu().double()
            K.assert_attention_close(o.reshape(ref.shape).numpy(), ref, where="%s t=%d" % (name, t))
            o2 = cache.decode_static(0, q.cuda(), scale).cpu().double()
            K.assert_attention_close(o2.reshape(ref.shape).numpy(), ref, where="%s static t=%d" % (name, t))
    torch.cuda.synchronize()
    for n in range(wl.batch * wl.num_kv_heads):
        K.assert_state_equal(K.gpu_state(cache, 0, n), K.oracle_state(oc, n), "%s n=%d" % (name, n))
    assert cache.status() == 0


def test_codebook_state_at_full_head_count():
    """Prefill of one 8B-shaped layer at 32 query / 8 kv heads and 4096 tokens:
    codes and scales bit-exact on every stream, attention within tolerance."""
    wl = replace(codebook_workload(W.LLAMA8B_FULL, 4, 32, 4096), batch=1, num_kv_heads=8, num_q_heads=32)
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(wl.seq_len)
    cache = K.make_gpu_cache(wl, wl.seq_len + 1, codebook=kvq.E2M1_LEVELS)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl, 0, kvq.E2M1_LEVELS), wl.batch * wl.num_kv_heads)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    q, _, _ = src.step(0)
    scale = 1.0 / math.sqrt(wl.head_dim)
    o = cache.decode(0, q.cuda(), scale).cpu().double()
    ref = oc.decode(K.q_streams(q, wl), scale)
    K.assert_attention_close(o.reshape(ref.shape).numpy(), ref, where="8 kv heads")
    for n in range(wl.num_kv_heads):
        K.assert_state_equal(K.gpu_state(cache, 0, n), K.oracle_state(oc, n), "n=%d" % n)
