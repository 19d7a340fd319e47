"""Variable per-sequence lengths in a batch (per-token key codecs): a padded
prefill in which every batch row keeps its own number of tokens, appends at
each row's own length, and decodes over each row's own tokens. The CUDA path
against one oracle cache per stream built from that stream's tokens alone:
codes, scales and outliers of each stream's rows bit-exact, attention within
1e-3, through the GQA tensor-core kernel and the generic kernel, the
two-stream decode step, per-channel keys whose residual fills and flushes
a block at each row's own appends, prefill attention over ragged rows, and
the refusals (sinks, lengths out of range)."""
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

PT = W.ASYM_PER_TOKEN

CASES = [
    # (name, workload, q heads per kv-head, per-token overrides)
    ("q8_0 int8 g4", W.TINY_Q8, 4, {}),
    ("asym k4v4 g1", W.LLAMA7B_16K, 1, dict(k_mode=PT, k_group=32, v_group=32)),
    ("asym k4v8 g2 outliers", W.DENSE_SPARSE_128K, 2, dict(k_mode=PT, k_group=64, v_bits=8, v_group=64)),
    ("codebook e2m1 g8", W.LLAMA8B_E2M1, 8, {}),
    ("asym k3v3 g4", W.LLAMA70B_32K, 4, dict(k_mode=PT)),
]
LENS = [37, 200, 1, 130]
# per-channel keys: rows whose key residual fills (and flushes a block) during the appends
PC_CASES = [
    ("per-channel k4v8 T64 g4", W.LLAMA8B_FULL, 4, [62, 200, 1, 127]),
    ("per-channel k3v3 T128 g8", W.LLAMA70B_32K, 8, [126, 200, 1, 130]),
    ("per-channel k4v4 outliers g1", W.DENSE_SPARSE_128K, 1, [62, 150, 3, 64]),
]


def state_rows(cache, wl, n, rows):
    """The arrays of stream n holding its first `rows` tokens (per-channel
    keys: its own key blocks and fp16 residual)."""
    lo = cache.layout(0)
    D = wl.head_dim
    st = K.gpu_state(cache, 0, n)
    out = {key: st[key][:rows] for key in ("v_words", "v_meta")}
    kout = wl.outliers_per_row
    if wl.k_mode == W.ASYM_PER_CHANNEL:
        kq = rows // wl.k_group * wl.k_group
        wk = lo.k_words_per_row
        out["k_words"] = K._bytes(cache, lo.k_codes + n * lo.k_codes_stream_bytes, kq * wk * 4).view(
            np.uint32).reshape(kq, wk)
        nb = kq // wl.k_group
        out["k_meta"] = K._bytes(cache, lo.k_meta + n * lo.k_meta_stream_bytes, nb * D * 4).view(
            np.uint16).reshape(nb, D, 2)
        r = rows - kq
        out["k_resid"] = K._bytes(cache, lo.k_resid + n * lo.k_resid_stream_bytes, r * D * 2).view(
            np.float16).reshape(r, D)
        krows = kq
    else:
        out["k_words"] = st["k_words"][:rows]
        out["k_meta"] = st["k_meta"][:rows]
        krows = rows
    if kout:
        for t, nr in (("k", krows), ("v", rows)):
            rp = getattr(lo, t + "_out_rowptr")
            col = getattr(lo, t + "_out_col")
            val = getattr(lo, t + "_out_val")
            out[t + "_rowptr"] = K._bytes(cache, rp + n * lo.out_rowptr_stream_bytes, (nr + 1) * 4).view(np.int32)
            out[t + "_col"] = K._bytes(cache, col + n * lo.out_col_stream_bytes, nr * kout * 2).view(np.uint16)
            out[t + "_val"] = K._bytes(cache, val + n * lo.out_val_stream_bytes, nr * kout * 2).view(np.float16)
    return out


def run_case(wl0, g, over, steps=3, use_step=False, lens=LENS):
    LENS = lens
    wl = replace(wl0, num_layers=1, batch=len(LENS), num_kv_heads=2, num_q_heads=2 * g,
                 seq_len=max(LENS), **over)
    S, H = wl.seq_len, wl.num_kv_heads
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(S)
    cache = K.make_gpu_cache(wl, S + steps + 1)
    cache.prefill_varlen(0, k.cuda(), v.cuda(), LENS)
    assert cache.seq_lengths(0) == LENS and cache.length(0) == max(LENS)
    spec = K.spec_of(wl)
    ocs = []
    for n in range(wl.batch * H):
        b, h = divmod(n, H)
        oc = O.OracleCache(spec, 1)
        oc.prefill(k[b, h, :LENS[b]].numpy()[None], v[b, h, :LENS[b]].numpy()[None])
        ocs.append(oc)
    scale = 1.0 / math.sqrt(wl.head_dim)
    ws = cache.workspace(wl.num_q_heads)
    aux = torch.cuda.Stream() if use_step else None
    for t in range(1, steps + 1):
        q, k1, v1 = src.step(t)
        if use_step:
            out = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), device="cuda")
            cache.decode_step([q.cuda()], [k1.cuda()], [v1.cuda()], scale, [out], workspace=ws, aux_stream=aux)
        else:
            cache.append(0, k1.cuda(), v1.cuda())
            out = cache.decode(0, q.cuda(), scale, workspace=ws)
        torch.cuda.synchronize()
        got = out.cpu().double().numpy()
        for n, oc in enumerate(ocs):
            b, h = divmod(n, H)
            oc.append(k1[b, h].numpy()[None], v1[b, h].numpy()[None])
            ref = oc.decode(q[b, h * g:(h + 1) * g].double().numpy()[None], scale)
            K.assert_attention_close(got[b, h * g:(h + 1) * g], ref[0], where="stream %d t=%d" % (n, t))
    assert cache.seq_lengths(0) == [x + steps for x in LENS]
    for n, oc in enumerate(ocs):
        b = n // H
        K.assert_state_equal(state_rows(cache, wl, n, LENS[b] + steps), K.oracle_state(oc, 0), "stream %d" % n)
    assert cache.status() == 0


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_varlen_against_per_stream_oracles(case):
    name, wl0, g, over = case
    run_case(wl0, g, over)


@pytest.mark.parametrize("case", PC_CASES, ids=lambda c: c[0])
def test_varlen_per_channel_keys(case):
    name, wl0, g, lens = case
    run_case(wl0, g, {}, lens=lens)


def test_varlen_through_the_two_stream_step():
    run_case(W.TINY_Q8, 4, {}, steps=2, use_step=True)


def test_uniform_prefill_ends_variable_lengths():
    wl = replace(W.TINY_Q8, num_layers=1, batch=4, num_kv_heads=2, num_q_heads=8, seq_len=64)
    k, v = LayerSource(wl, 0, device="cpu").kv(64)
    cache = K.make_gpu_cache(wl, 80)
    cache.prefill_varlen(0, k.cuda(), v.cuda(), [3, 64, 9, 10])
    with pytest.raises(kvq.KVQError):  # a chunk longer than the shortest row
        cache.prefill_attention(0, torch.zeros((4, 4, 8, 128), dtype=torch.float16, device="cuda"), 1.0)
    cache.prefill(0, k.cuda(), v.cuda())
    assert cache.seq_lengths(0) == [64, 64, 64, 64]


def test_varlen_refusals():
    wl = replace(W.LLAMA8B_FULL, num_layers=1, batch=2, num_kv_heads=2, num_q_heads=4, seq_len=16)
    k, v = LayerSource(wl, 0, device="cpu").kv(16)
    tok = replace(W.TINY_Q8, num_layers=1, batch=2, num_kv_heads=2, num_q_heads=4, seq_len=16)
    cache = K.make_gpu_cache(tok, 32)
    with pytest.raises(kvq.KVQError):
        cache.prefill_varlen(0, k.cuda(), v.cuda(), [0, 16])             # an empty row
    with pytest.raises(kvq.KVQError):
        cache.prefill_varlen(0, k.cuda(), v.cuda(), [4, 17])             # past the padded rows
    sinks = K.make_gpu_cache(tok, 32, sink_tokens=2)
    with pytest.raises(kvq.KVQError):
        sinks.prefill_varlen(0, k.cuda(), v.cuda(), [4, 16])             # with sink tokens
    assert cache.status() == 0


@pytest.mark.parametrize("case", [("q8_0 int8 g4", W.TINY_Q8, 4, [37, 200, 20, 130]),
                                  ("per-channel k4v8 g4", W.LLAMA8B_FULL, 4, [62, 200, 20, 127]),
                                  ("per-channel k3v3 g8", W.LLAMA70B_32K, 8, [129, 200, 20, 140])],
                         ids=lambda c: c[0])
def test_prefill_attention_over_ragged_rows(case):
    """Each batch row's chunk is its own last positions: the queries of row
    b attend row b's tokens causally (one oracle cache per stream)."""
    name, wl0, g, lens = case
    wl = replace(wl0, num_layers=1, batch=len(lens), num_kv_heads=2, num_q_heads=2 * g, seq_len=max(lens))
    H, chunk = wl.num_kv_heads, 19
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(wl.seq_len)
    cache = K.make_gpu_cache(wl, wl.seq_len + 1)
    cache.prefill_varlen(0, k.cuda(), v.cuda(), lens)
    q = torch.randn((wl.batch, chunk, wl.num_q_heads, 128), generator=torch.Generator().manual_seed(9)).half()
    o = cache.prefill_attention(0, q.cuda(), 1.0 / math.sqrt(128)).cpu().double().numpy()
    for n in range(wl.batch * H):
        b, h = divmod(n, H)
        oc = O.OracleCache(K.spec_of(wl), 1)
        oc.prefill(k[b, h, :lens[b]].numpy()[None], v[b, h, :lens[b]].numpy()[None])
        ref = oc.prefill_attention(q[b, :, h * g:(h + 1) * g].double().numpy()[None], 1.0 / math.sqrt(128))
        K.assert_attention_close(o[b, :, h * g:(h + 1) * g].reshape(-1, 128), ref[0].reshape(-1, 128),
                                 where="%s stream %d" % (name, n))
    assert cache.status() == 0
