"""Glue for the parity tests: drives the CUDA path through the C ABI and the
oracle on the same fp16 inputs, and compares them (codes, scales, zero
points, outliers and fp16 residual bit-exact; attention within 1e-3 of the
per-row max, fp32 accumulation against the fp64 oracle)."""
from __future__ import annotations

import math

import numpy as np
import torch

import bit_quantized_kv_kvq_gb300 as kvq
from oracle import kvq_oracle as O

ATTN_TOL = 1e-3


def spec_of(wl, sink_tokens=0, codebook=None):
    codebook = wl.codebook if codebook is None else codebook
    return O.CodecSpec(wl.head_dim, wl.k_bits, wl.v_bits, wl.k_mode, wl.v_mode,
                       wl.k_group, wl.v_group, wl.outliers_per_row, sink_tokens,
                       None if codebook is None else tuple(float(x) for x in codebook))


def make_gpu_cache(wl, max_seq, num_layers=None, device="cuda", sink_tokens=0, codebook=None):
    codebook = wl.codebook if codebook is None else codebook
    return kvq.QuantizedKVCache(num_layers or wl.num_layers, wl.batch, wl.num_kv_heads,
                                wl.head_dim, max_seq, wl.k_bits, wl.v_bits, wl.k_mode, wl.v_mode,
                                wl.k_group, wl.v_group, wl.outliers_per_row, device=device,
                                sink_tokens=sink_tokens, codebook=codebook)


def streams_of(x, wl):
    """[B][H][...] -> [B*H][...] numpy."""
    t = x.detach().cpu()
    return t.reshape((wl.batch * wl.num_kv_heads,) + tuple(t.shape[2:])).numpy()


def q_streams(q, wl):
    """q [B][Hq][D] -> [B*Hkv][g][D] numpy (query head h reads kv-head h // g)."""
    t = q.detach().cpu().float().double()
    return t.reshape(wl.batch * wl.num_kv_heads, wl.gqa, wl.head_dim).numpy()


def _bytes(cache, ptr, nbytes):
    return cache.view(ptr, nbytes, torch.uint8).cpu().numpy()


def gpu_state(cache, layer, n):
    """Arrays of stream n of one layer, copied from the device cache."""
    c = cache.cfg
    lo = cache.layout(layer)
    D = c.head_dim
    L = lo.length - lo.sink_len  # coded rows (after the fp16 sinks)
    kq = lo.k_quantized_len
    out = {}
    if lo.sink_tokens:
        ns = lo.sink_len
        out["k_sink"] = _bytes(cache, lo.k_sink + n * lo.sink_stream_bytes, ns * D * 2).view(np.float16).reshape(ns, D)
        out["v_sink"] = _bytes(cache, lo.v_sink + n * lo.sink_stream_bytes, ns * D * 2).view(np.float16).reshape(ns, D)
    kr = kq if c.k_mode == O.ASYM_PER_CHANNEL else L
    wk, wv = lo.k_words_per_row, lo.v_words_per_row
    out["k_words"] = _bytes(cache, lo.k_codes + n * lo.k_codes_stream_bytes, kr * wk * 4).view(np.uint32).reshape(kr, wk)
    out["v_words"] = _bytes(cache, lo.v_codes + n * lo.v_codes_stream_bytes, L * wv * 4).view(np.uint32).reshape(L, wv)
    if c.k_mode == O.ASYM_PER_CHANNEL:
        nb = kq // c.k_group
        out["k_meta"] = _bytes(cache, lo.k_meta + n * lo.k_meta_stream_bytes, nb * D * 4).view(np.uint16).reshape(nb, D, 2)
        r = lo.k_resid_len
        out["k_resid"] = _bytes(cache, lo.k_resid + n * lo.k_resid_stream_bytes, r * D * 2).view(np.float16).reshape(r, D)
    else:
        g = D // c.k_group
        eb = lo.k_meta_entry_bytes
        m = _bytes(cache, lo.k_meta + n * lo.k_meta_stream_bytes, L * g * eb).view(np.uint16)
        out["k_meta"] = m.reshape(L, g, eb // 2)
    g = D // c.v_group
    eb = lo.v_meta_entry_bytes
    out["v_meta"] = _bytes(cache, lo.v_meta + n * lo.v_meta_stream_bytes, L * g * eb).view(np.uint16).reshape(L, g, eb // 2)
    k = c.outliers_per_row
    if k:
        for name, rows in (("k", kr), ("v", L)):
            rp = getattr(lo, name + "_out_rowptr")
            col = getattr(lo, name + "_out_col")
            val = getattr(lo, name + "_out_val")
            out[name + "_rowptr"] = _bytes(cache, rp + n * lo.out_rowptr_stream_bytes, (rows + 1) * 4).view(np.int32)
            out[name + "_col"] = _bytes(cache, col + n * lo.out_col_stream_bytes, rows * k * 2).view(np.uint16)
            out[name + "_val"] = _bytes(cache, val + n * lo.out_val_stream_bytes, rows * k * 2).view(np.float16)
    return out


def oracle_state(oc: O.OracleCache, i):
    """The same arrays for oracle stream i."""
    sp = oc.spec
    out = {"k_words": oc.k_words()[i], "v_words": oc.v_words()[i]}
    if sp.sink_tokens:
        out["k_sink"] = oc.sink_k[i]
        out["v_sink"] = oc.sink_v[i]
    if sp.k_mode == O.ASYM_PER_CHANNEL:
        out["k_meta"] = np.stack([oc.k.scale16[i].view(np.uint16), oc.k.zero16[i].view(np.uint16)], -1)
        out["k_resid"] = oc.k.resid[i]
    elif sp.k_mode in (O.SYM_PER_TOKEN, O.CODEBOOK_PER_TOKEN):
        out["k_meta"] = oc.k.scale16[i].view(np.uint16)[..., None]
    else:
        out["k_meta"] = np.stack([oc.k.scale16[i].view(np.uint16), oc.k.zero16[i].view(np.uint16)], -1)
    if sp.v_mode in (O.SYM_PER_TOKEN, O.CODEBOOK_PER_TOKEN):
        out["v_meta"] = oc.v.scale16[i].view(np.uint16)[..., None]
    else:
        out["v_meta"] = np.stack([oc.v.scale16[i].view(np.uint16), oc.v.zero16[i].view(np.uint16)], -1)
    if sp.outliers_per_row:
        for name, st in (("k", oc.k), ("v", oc.v)):
            rp, col, val = O.OracleCache.csr(st)
            out[name + "_rowptr"] = rp[i]
            out[name + "_col"] = col[i]
            out[name + "_val"] = val[i]
    return out


def assert_state_equal(gpu, ref, where=""):
    assert set(gpu) == set(ref), (sorted(gpu), sorted(ref))
    for key in ref:
        a, b = np.asarray(gpu[key]), np.asarray(ref[key])
        assert a.shape == b.shape, "%s %s: shape %s vs %s" % (where, key, a.shape, b.shape)
        if a.dtype == np.float16:
            a, b = a.view(np.uint16), b.view(np.uint16)
        if not np.array_equal(a, b):
            bad = np.argwhere(a != b)
            raise AssertionError("%s %s: %d mismatches, first at %s: gpu %s oracle %s" % (
                where, key, len(bad), bad[0].tolist(), a[tuple(bad[0])], b[tuple(bad[0])]))


def assert_attention_close(o_gpu, o_ref, tol=ATTN_TOL, where=""):
    err = O.row_relative_error(o_gpu, o_ref)
    worst = float(err.max())
    assert math.isfinite(worst) and worst <= tol, "%s attention row error %.3e > %.1e" % (where, worst, tol)
    return worst
