"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded fp16 inputs, at sizes the oracle finishes in seconds that still
span several tiles and a ragged tail. Codes, scales, zero points, outlier
lists and the fp16 key residual must be bit-exact; attention must be within
1e-3 (per-row max relative error) of the fp64 oracle on the same dequantized
cache."""
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

# Small versions of the five workloads: same codec and distribution, fewer
# streams, lengths with a ragged last tile / residual.
SMALL = [
    ("tiny_q8", replace(W.TINY_Q8, seq_len=1000), 70),
    ("tiny_q8_full", W.TINY_Q8, 3),
    ("llama7b", replace(W.LLAMA7B_16K, batch=2, num_q_heads=4, num_kv_heads=4, seq_len=357), 30),
    ("llama70b", replace(W.LLAMA70B_32K, batch=1, num_q_heads=16, num_kv_heads=2, seq_len=461), 60),
    ("dense_sparse", replace(W.DENSE_SPARSE_128K, num_q_heads=4, num_kv_heads=4, seq_len=269), 60),
    ("llama8b", replace(W.LLAMA8B_FULL, num_layers=2, num_q_heads=8, num_kv_heads=2, seq_len=242), 20),
]


def _run_case(wl, appends, check_every=7, layer=None):
    torch.manual_seed(0)
    layers = list(range(wl.num_layers)) if layer is None else [layer]
    cache = K.make_gpu_cache(wl, wl.seq_len + appends + 5)
    scale = 1.0 / math.sqrt(wl.head_dim)
    worst = 0.0
    for li in layers:
        src = LayerSource(wl, li, device="cpu")
        k, v = src.kv(wl.seq_len)
        oc = O.OracleCache(K.spec_of(wl), wl.batch * wl.num_kv_heads)
        oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
        cache.prefill(li, k.cuda(), v.cuda())
        torch.cuda.synchronize()
        for n in range(wl.batch * wl.num_kv_heads):
            K.assert_state_equal(K.gpu_state(cache, li, n), K.oracle_state(oc, n), "prefill n=%d" % n)
        for step in range(appends + 1):
            if step > 0:
                _, k1, v1 = src.step(step)
                oc.append(K.streams_of(k1, wl), K.streams_of(v1, wl))
                cache.append(li, k1.cuda(), v1.cuda())
            if step % check_every == 0 or step == appends:
                q, _, _ = src.step(10_000 + step)
                o = cache.decode(li, q.cuda(), scale)
                ref = oc.decode(K.q_streams(q, wl), scale)
                got = o.cpu().double().reshape(ref.shape).numpy()
                worst = max(worst, K.assert_attention_close(got, ref, where="step %d" % step))
        torch.cuda.synchronize()
        for n in range(wl.batch * wl.num_kv_heads):
            K.assert_state_equal(K.gpu_state(cache, li, n), K.oracle_state(oc, n),
                                 "after %d appends n=%d" % (appends, n))
    assert cache.status() == 0
    return worst


@pytest.mark.parametrize("name,wl,appends", SMALL, ids=[s[0] for s in SMALL])
def test_parity_small(name, wl, appends):
    _run_case(wl, appends)


@pytest.mark.parametrize("splits", [1, 2, 7, 0])
def test_split_count_invariance(splits):
    wl = replace(W.LLAMA70B_32K, batch=1, num_q_heads=16, num_kv_heads=2, seq_len=1000)
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(wl.seq_len)
    q, _, _ = src.step(1)
    cache = K.make_gpu_cache(wl, wl.seq_len)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl), wl.batch * wl.num_kv_heads)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    ref = oc.decode(K.q_streams(q, wl), 0.088)
    cache.set_decode_splits(splits)
    o = cache.decode(0, q.cuda(), 0.088).cpu().double().reshape(ref.shape).numpy()
    K.assert_attention_close(o, ref)


@pytest.mark.parametrize("seq", [1, 2, 63, 64, 65, 127, 128, 129])
@pytest.mark.parametrize("kmode", [W.ASYM_PER_CHANNEL, W.ASYM_PER_TOKEN])
def test_short_and_boundary_lengths(seq, kmode):
    wl = replace(W.DENSE_SPARSE_128K, num_q_heads=4, num_kv_heads=2, seq_len=seq, k_mode=kmode,
                 k_group=64 if kmode == W.ASYM_PER_CHANNEL else 32)
    _run_case(wl, appends=3, check_every=1)


@pytest.mark.parametrize("bits", [3, 4, 8])
@pytest.mark.parametrize("gqa", [1, 2, 4, 8])
def test_codec_and_gqa_grid(bits, gqa):
    wl = replace(W.LLAMA7B_16K, batch=1, num_kv_heads=2, num_q_heads=2 * gqa, seq_len=200,
                 k_bits=bits, v_bits=bits, k_group=128 if bits == 3 else 64,
                 v_group=128 if bits == 3 else 32)
    _run_case(wl, appends=2, check_every=1)


def test_sym_group16_and_fp16_output():
    wl = replace(W.TINY_Q8, seq_len=300, k_group=16, v_group=16)
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(wl.seq_len)
    q, _, _ = src.step(0)
    cache = K.make_gpu_cache(wl, 400)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl), wl.batch * wl.num_kv_heads)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    torch.cuda.synchronize()
    for n in range(2):
        K.assert_state_equal(K.gpu_state(cache, 0, n), K.oracle_state(oc, n))
    o16 = cache.decode(0, q.cuda(), 0.1, out_dtype=torch.float16)
    ref = oc.decode(K.q_streams(q, wl), 0.1)
    K.assert_attention_close(o16.cpu().double().reshape(ref.shape).numpy(), ref, tol=2e-3)


def test_degenerate_groups_on_gpu():
    """Constant rows, all-zero rows and a row of equal magnitudes (outlier
    ties) quantize exactly as the oracle does."""
    wl = replace(W.DENSE_SPARSE_128K, num_q_heads=2, num_kv_heads=2, seq_len=130)
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(wl.seq_len)
    k[0, 0, :64] = 1.5          # a whole constant key block
    v[0, 0, 3] = 0.0            # an all-zero value row
    v[0, 1, 5] = -2.0           # every entry ties in magnitude
    v[0, 1, 5, ::2] = 2.0
    k[0, 1, 70, :] = 0.0
    cache = K.make_gpu_cache(wl, 200)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl), 2)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    torch.cuda.synchronize()
    for n in range(2):
        K.assert_state_equal(K.gpu_state(cache, 0, n), K.oracle_state(oc, n))
    q, _, _ = src.step(0)
    o = cache.decode(0, q.cuda(), 0.09).cpu().double().reshape(2, 1, 128).numpy()
    K.assert_attention_close(o, oc.decode(K.q_streams(q, wl), 0.09))


def test_errors_are_reported_not_raised_on_device():
    import bit_quantized_kv_kvq_gb300 as kvq
    wl = replace(W.LLAMA7B_16K, batch=1, num_q_heads=2, num_kv_heads=2, seq_len=10)
    cache = K.make_gpu_cache(wl, 11)
    q = torch.zeros((1, 2, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        cache.decode(0, q, 1.0)          # empty layer
    assert e.value.status == 1
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(11)
    with pytest.raises(kvq.KVQError) as e:
        cache.prefill(0, torch.cat([k, k], 2).cuda(), torch.cat([v, v], 2).cuda())
    assert e.value.status == 4
    cache.prefill(0, k.cuda(), v.cuda())
    _, k1, v1 = src.step(1)
    with pytest.raises(kvq.KVQError) as e:
        cache.append(0, k1.cuda(), v1.cuda())   # full
    assert e.value.status == 4
    with pytest.raises(kvq.KVQError) as e:
        cache.decode(0, torch.zeros((1, 3, 128), dtype=torch.float16, device="cuda"), 1.0)
    assert e.value.status == 1
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        cache.decode(0, q, 1.0, workspace=ws)
    assert e.value.status == 3
    assert cache.status() == 0


def test_launch_counter_matches_the_work_enqueued():
    """prefill, append and decode enqueue one kernel each. The stream-K decode
    (per-channel keys, 8 query heads per kv-head) and the split decodes of the
    common codecs merge their splits inside their one kernel; only the
    generic decode adds a combine launch (also with one split)."""
    import bit_quantized_kv_kvq_gb300 as kvq
    cases = ((W.ASYM_PER_CHANNEL, 32, 0, 1, 1),  # stream-K
             (W.ASYM_PER_CHANNEL, 16, 0, 1, 1),  # token-row tensor-core split decode
             (W.ASYM_PER_TOKEN, 4, 0, 1, 1),     # one query head per kv-head
             (W.ASYM_PER_TOKEN, 8, 2, 2, 2))     # outliers with per-token keys: generic kernel + combine
    for kmode, hq, outl, extra_one, extra_split in cases:
        wl = replace(W.LLAMA7B_16K, batch=1, num_q_heads=hq, num_kv_heads=4, seq_len=300, k_mode=kmode,
                     k_group=64 if kmode == W.ASYM_PER_CHANNEL else 32, outliers_per_row=outl)
        src = LayerSource(wl, 0, device="cpu")
        k, v = src.kv(wl.seq_len)
        q, k1, v1 = src.step(0)
        cache = K.make_gpu_cache(wl, 400)
        n0 = kvq.kernel_launches()
        cache.prefill(0, k.cuda(), v.cuda())
        cache.append(0, k1.cuda(), v1.cuda())
        assert kvq.kernel_launches() - n0 == 2
        for splits, extra in ((1, extra_one), (3, extra_split)):
            cache.set_decode_splits(splits)
            n1 = kvq.kernel_launches()
            cache.decode(0, q.cuda(), 0.1)
            assert kvq.kernel_launches() - n1 == extra
        torch.cuda.synchronize()
        assert cache.status() == 0


@pytest.mark.parametrize("ctas", [1, 2, 3, 5, 8, 13, 0])
@pytest.mark.parametrize("seq,batch,hkv", [(70, 3, 4), (1000, 1, 2), (333, 2, 3), (200, 4, 5)])
def test_stream_k_partitions(ctas, seq, batch, hkv):
    """The stream-K decode (per-channel keys, 8 query heads per kv-head) cuts
    the key blocks of all streams into one range per CTA: one CTA holding many whole streams, streams cut across several
    CTAs, and ranges that start and end mid-stream must all agree with the
    oracle (the split-merge counters are reused across the calls). With 16
    streams or more the ranges are cut in a space that weighs each stream
    switch as extra blocks, so some CTAs hold no block at all."""
    wl = replace(W.LLAMA8B_FULL, num_layers=1, batch=batch, num_kv_heads=hkv, num_q_heads=8 * hkv,
                 seq_len=seq)
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(seq)
    cache = K.make_gpu_cache(wl, seq + 2)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl), wl.batch * wl.num_kv_heads)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    cache.set_decode_splits(ctas)
    for call in range(3):
        q, _, _ = src.step(50 + call)
        ref = oc.decode(K.q_streams(q, wl), 0.088)
        o = cache.decode(0, q.cuda(), 0.088).cpu().double().reshape(ref.shape).numpy()
        K.assert_attention_close(o, ref, where="ctas %d call %d" % (ctas, call))
    assert cache.status() == 0


NO_OUTLIER_CODECS = [
    ("k4c64_v4g64", dict(k_bits=4, v_bits=4, k_mode=W.ASYM_PER_CHANNEL, v_mode=W.ASYM_PER_TOKEN,
                         k_group=64, v_group=64)),
    ("k8c128_v8g32", dict(k_bits=8, v_bits=8, k_mode=W.ASYM_PER_CHANNEL, v_mode=W.ASYM_PER_TOKEN,
                          k_group=128, v_group=32)),
    ("k4c128_v8g128", dict(k_bits=4, v_bits=8, k_mode=W.ASYM_PER_CHANNEL, v_mode=W.ASYM_PER_TOKEN,
                           k_group=128, v_group=128)),
    ("k4t16_v4g16", dict(k_bits=4, v_bits=4, k_mode=W.ASYM_PER_TOKEN, v_mode=W.ASYM_PER_TOKEN,
                         k_group=16, v_group=16)),
    ("q8_g64", dict(k_bits=8, v_bits=8, k_mode=W.SYM_PER_TOKEN, v_mode=W.SYM_PER_TOKEN,
                    k_group=64, v_group=64)),
    ("k3c64_v3g128", dict(k_bits=3, v_bits=3, k_mode=W.ASYM_PER_CHANNEL, v_mode=W.ASYM_PER_TOKEN,
                          k_group=64, v_group=128)),
    ("k3t128_v4g64", dict(k_bits=3, v_bits=4, k_mode=W.ASYM_PER_TOKEN, v_mode=W.ASYM_PER_TOKEN,
                          k_group=128, v_group=64)),
    ("k8c64_v3g128", dict(k_bits=8, v_bits=3, k_mode=W.ASYM_PER_CHANNEL, v_mode=W.ASYM_PER_TOKEN,
                          k_group=64, v_group=128)),
]


@pytest.mark.parametrize("seq", [1, 63, 64, 65, 127, 128, 129, 300])
@pytest.mark.parametrize("name,codec", NO_OUTLIER_CODECS, ids=[c[0] for c in NO_OUTLIER_CODECS])
def test_lengths_without_outliers(seq, name, codec):
    wl = replace(W.LLAMA7B_16K, batch=1, num_q_heads=2, num_kv_heads=2, seq_len=seq,
                 outliers_per_row=0, **codec)
    _run_case(wl, appends=2, check_every=1)


def _tie_inputs(wl, seed):
    """fp16 K/V whose groups make many quotients exact ties k + 1/2: every
    group holds multiples of step/2 (one power-of-two step per group) with
    its extremes at 0 and lev * step (symmetric: -lev * step and lev * step),
    so the scale is step. Plus a constant stretch (zero scales) and a
    tiny-range stretch (subnormal fp16 scales)."""
    g = torch.Generator().manual_seed(seed)
    B, H, S, D = wl.batch, wl.num_kv_heads, wl.seq_len, wl.head_dim
    out = []
    for which in range(2):
        mode = wl.k_mode if which == 0 else wl.v_mode
        bits = wl.k_bits if which == 0 else wl.v_bits
        grp = wl.k_group if which == 0 else wl.v_group
        sym = mode == W.SYM_PER_TOKEN
        lev = 2 ** (bits - 1) - 1 if sym else 2 ** bits - 1
        half = torch.randint(0, 2 * lev + 1, (B, H, S, D), generator=g).double() / 2
        if sym:
            half = half * torch.where(torch.rand((B, H, S, D), generator=g) < 0.5, -1.0, 1.0)
        if mode == W.ASYM_PER_CHANNEL:
            nb = -(-S // grp)
            step = 2.0 ** torch.randint(-6, 3, (B, H, nb, 1, D), generator=g).double()
            step = step.expand(B, H, nb, grp, D).reshape(B, H, nb * grp, D)[:, :, :S]
            x = half * step
            x[:, :, 0::grp] = 0.0
            x[:, :, 1::grp] = lev * step[:, :, 1::grp]
        else:
            step = 2.0 ** torch.randint(-6, 3, (B, H, S, D // grp, 1), generator=g).double()
            x = half.reshape(B, H, S, D // grp, grp) * step
            x[..., 0] = -lev * step[..., 0] if sym else 0.0
            x[..., 1] = lev * step[..., 0]
            x = x.reshape(B, H, S, D)
        x16 = x.to(torch.float16)
        x16[:, :, : S // 4] = torch.where(torch.arange(D) % 2 == 0, x16[:, :, : S // 4], 1.25)
        tiny = torch.randint(0, lev + 1, (B, H, 128, D), generator=g).double() * 2.0 ** -20
        x16[:, :, 256:384] = tiny.to(torch.float16)
        x16[:, 1:, 256:384] += torch.tensor(0.5, dtype=torch.float16)
        out.append(x16)
    return out


@pytest.mark.parametrize("name,codec", NO_OUTLIER_CODECS, ids=[c[0] for c in NO_OUTLIER_CODECS])
def test_exact_ties_and_tiny_scales(name, codec):
    wl = replace(W.LLAMA7B_16K, batch=1, num_q_heads=2, num_kv_heads=2, seq_len=400,
                 outliers_per_row=0, **codec)
    k, v = _tie_inputs(wl, 7)
    cache = K.make_gpu_cache(wl, 420)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl), 2)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    torch.cuda.synchronize()
    for n in range(2):
        K.assert_state_equal(K.gpu_state(cache, 0, n), K.oracle_state(oc, n), "n=%d" % n)
    assert cache.status() == 0


def _outlier_inputs(wl, seed):
    """Seeded K/V with rows that stress the top-k selection: a row of equal
    magnitudes (ties go to the lower channel), a row of signed zeros, two
    channels far above the rest over the first 128 tokens (every key block
    there has channels whose members are all outliers), and a row whose
    largest magnitudes occur with both signs."""
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(wl.seq_len)
    g = torch.Generator().manual_seed(seed)
    for x in (k, v):
        sgn = torch.where(torch.rand(x.shape[-1], generator=g) < 0.5, -1.0, 1.0).to(x.dtype)
        x[:, :, 5] = 0.75 * sgn
        x[:, :, 6] = torch.where(torch.arange(x.shape[-1]) % 2 == 0, 0.0, -0.0).to(x.dtype)
        x[:, :, :128, 17] = 100.0
        x[:, :, :128, 90] = -100.0
        x[:, :, 7, 3] = 9.0
        x[:, :, 7, 40] = -9.0
        x[:, :, 7, 41] = 9.0
    return k, v


@pytest.mark.parametrize("kout", [1, 3, 8])
@pytest.mark.parametrize("seq", [65, 300])
@pytest.mark.parametrize("name,codec", NO_OUTLIER_CODECS, ids=[c[0] for c in NO_OUTLIER_CODECS])
def test_outlier_split_prefill(name, codec, seq, kout):
    """The dense-and-sparse split at every supported codec: CSR lists, the
    statistics over the remaining members and the zeroed outlier codes."""
    wl = replace(W.LLAMA7B_16K, batch=1, num_q_heads=2, num_kv_heads=2, seq_len=seq,
                 outliers_per_row=kout, **codec)
    k, v = _outlier_inputs(wl, 11)
    cache = K.make_gpu_cache(wl, seq + 8)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl), 2)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    torch.cuda.synchronize()
    for n in range(2):
        K.assert_state_equal(K.gpu_state(cache, 0, n), K.oracle_state(oc, n), "n=%d" % n)
    assert cache.status() == 0


@pytest.mark.parametrize("name,codec", NO_OUTLIER_CODECS[:4], ids=[c[0] for c in NO_OUTLIER_CODECS[:4]])
def test_outlier_split_with_exact_ties(name, codec):
    wl = replace(W.LLAMA7B_16K, batch=1, num_q_heads=2, num_kv_heads=2, seq_len=400,
                 outliers_per_row=2, **codec)
    k, v = _tie_inputs(wl, 9)
    cache = K.make_gpu_cache(wl, 420)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl), 2)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    torch.cuda.synchronize()
    for n in range(2):
        K.assert_state_equal(K.gpu_state(cache, 0, n), K.oracle_state(oc, n), "n=%d" % n)
    assert cache.status() == 0


TC_CODECS = [
    ("k3v3g128", dict(k_bits=3, v_bits=3, k_group=128, v_group=128)),
    ("k4v4g64", dict(k_bits=4, v_bits=4, k_group=64, v_group=64)),
    ("k4v4g128", dict(k_bits=4, v_bits=4, k_group=128, v_group=128)),
    ("k4v8g64", dict(k_bits=4, v_bits=8, k_group=64, v_group=64)),
    ("k8v4g64", dict(k_bits=8, v_bits=4, k_group=256, v_group=64)),
    ("k8v8g128", dict(k_bits=8, v_bits=8, k_group=64, v_group=128)),
]


@pytest.mark.parametrize("outliers", [0, 2])
@pytest.mark.parametrize("gqa", [1, 2, 4, 8])
@pytest.mark.parametrize("name,codec", TC_CODECS, ids=[c[0] for c in TC_CODECS])
def test_tensor_core_decode_grid(name, codec, gqa, outliers):
    """Per-channel keys with per-token values at every query-group size, with
    and without outliers, lengths with a ragged last tile and a key residual."""
    wl = replace(W.LLAMA7B_16K, batch=1, num_kv_heads=2, num_q_heads=2 * gqa, seq_len=333,
                 k_mode=W.ASYM_PER_CHANNEL, v_mode=W.ASYM_PER_TOKEN,
                 outliers_per_row=outliers, **codec)
    _run_case(wl, appends=2, check_every=1)


@pytest.mark.parametrize("kout", [1, 3, 8])
@pytest.mark.parametrize("gqa", [1, 4])
@pytest.mark.parametrize("vg", [64, 128])
def test_tensor_core_decode_outlier_counts(kout, gqa, vg):
    """Outlier counts other than two: an unpaired last entry (1, 3) and more
    channels per lane than the value-correction register cache holds (8),
    with one query head (register cache) and a group (shared atomics)."""
    wl = replace(W.DENSE_SPARSE_128K, batch=1, num_kv_heads=2, num_q_heads=2 * gqa, seq_len=333,
                 outliers_per_row=kout, v_group=vg)
    _run_case(wl, appends=2, check_every=1)


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 0])
@pytest.mark.parametrize("seq", [335, 1000])
@pytest.mark.parametrize("vg", [64, 128])
def test_one_head_outlier_split_counts(splits, seq, vg):
    """One query head, eight outliers per row (half of each lane's value
    corrections go through the shared atomics): the same attention for every
    split layout, the last split ragged and the key residual non-empty."""
    wl = replace(W.DENSE_SPARSE_128K, batch=1, num_q_heads=2, num_kv_heads=2, seq_len=seq,
                 outliers_per_row=8, v_group=vg)
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(wl.seq_len)
    q, _, _ = src.step(3)
    cache = K.make_gpu_cache(wl, wl.seq_len)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl), wl.batch * wl.num_kv_heads)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    ref = oc.decode(K.q_streams(q, wl), 0.088)
    cache.set_decode_splits(splits)
    for _ in range(3):  # repeated: the atomics' order varies between launches
        o = cache.decode(0, q.cuda(), 0.088).cpu().double().reshape(ref.shape).numpy()
        K.assert_attention_close(o, ref, where="splits %d" % splits)
    assert cache.status() == 0


@pytest.mark.parametrize("outliers", [0, 2])
def test_one_head_late_max_rescale(outliers):
    """One query head, one split: keys of every other 32-token tile scaled by
    10, so a warp's running max jumps by more than the lazy threshold after
    its first tile and every accumulator (zero-point sums kept per token
    lane, outlier corrections) must follow the rescale."""
    wl = replace(W.DENSE_SPARSE_128K, batch=1, num_q_heads=2, num_kv_heads=2, seq_len=333,
                 outliers_per_row=outliers, dist="normal")
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(wl.seq_len)
    big = (torch.arange(wl.seq_len) // 32) % 2 == 1
    k[:, :, big] = k[:, :, big] * 10
    q, _, _ = src.step(0)
    cache = K.make_gpu_cache(wl, 340)
    cache.prefill(0, k.cuda(), v.cuda())
    cache.set_decode_splits(1)
    oc = O.OracleCache(K.spec_of(wl), 2)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    ref = oc.decode(K.q_streams(q, wl), 0.088)
    o = cache.decode(0, q.cuda(), 0.088).cpu().double().reshape(ref.shape).numpy()
    K.assert_attention_close(o, ref)


def test_tensor_core_decode_wide_value_scales():
    """Value groups whose scales span many powers of two (the fp16 operand
    keeps its precision through the running exponent)."""
    wl = replace(W.LLAMA7B_16K, batch=1, num_q_heads=8, num_kv_heads=2, seq_len=700,
                 k_bits=4, v_bits=4, k_group=64, v_group=64, outliers_per_row=0)
    src = LayerSource(wl, 0, device="cpu")
    k, v = src.kv(wl.seq_len)
    g = torch.Generator().manual_seed(3)
    span = 2.0 ** torch.randint(-12, 9, (1, 2, wl.seq_len, 1), generator=g).double()
    v = (v.double() * span).clamp(-60000, 60000).to(torch.float16)
    k = (k.double() * 2.0 ** torch.randint(-6, 6, (1, 2, 1, 128), generator=g).double()).to(torch.float16)
    q, _, _ = src.step(0)
    cache = K.make_gpu_cache(wl, wl.seq_len)
    cache.prefill(0, k.cuda(), v.cuda())
    oc = O.OracleCache(K.spec_of(wl), 2)
    oc.prefill(K.streams_of(k, wl), K.streams_of(v, wl))
    torch.cuda.synchronize()
    for n in range(2):
        K.assert_state_equal(K.gpu_state(cache, 0, n), K.oracle_state(oc, n))
    for splits in (1, 3):
        cache.set_decode_splits(splits)
        o = cache.decode(0, q.cuda(), 0.088).cpu().double().reshape(2, 4, 128).numpy()
        K.assert_attention_close(o, oc.decode(K.q_streams(q, wl), 0.088))
