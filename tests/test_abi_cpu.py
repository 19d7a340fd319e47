"""Host-only checks of the C-ABI library (no GPU needed): it loads, exports
every entry point include/kvq.h declares, sizes caches, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

import bit_quantized_kv_kvq_gb300 as kvq
from bit_quantized_kv_kvq_gb300 import workloads as W
from oracle import kvq_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return kvq.lib()


def declared_entry_points():
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    return sorted(set(re.findall(r"KVQ_API\s+[\w\s\*]+?\b(kvq_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert len(names) >= 16 and "kvq_selftest_wait_timeout" in names
    for n in names:
        assert hasattr(lib, n), n


def test_version(lib):
    assert lib.kvq_version() == 100


def test_launch_counter_counts_nothing_without_work(lib):
    before = kvq.kernel_launches()
    with pytest.raises(kvq.KVQError):
        kvq.check(lib.kvq_prefill_quantize(None, 0, None, None, 0, None))
    assert kvq.kernel_launches() == before


def _cfg(**kw):
    base = dict(num_layers=1, batch=2, num_kv_heads=4, head_dim=128, max_seq=1000, k_bits=4,
                v_bits=4, k_mode=kvq.ASYM_PER_CHANNEL, v_mode=kvq.ASYM_PER_TOKEN, k_group=64,
                v_group=64, outliers_per_row=0)
    base.update(kw)
    return kvq.make_config(**base)


@pytest.mark.parametrize("wl", W.ALL + W.EXTRA, ids=lambda w: w.name)
def test_cache_bytes_cover_the_algorithmic_footprint(lib, wl):
    max_seq = wl.seq_len + wl.decode_steps
    cfg = kvq.make_config(wl.num_layers, wl.batch, wl.num_kv_heads, wl.head_dim, max_seq,
                          wl.k_bits, wl.v_bits, wl.k_mode, wl.v_mode, wl.k_group, wl.v_group,
                          wl.outliers_per_row, codebook=wl.codebook)
    got = kvq.cache_bytes(cfg)
    algo = O.packed_cache_bytes(wl.num_layers, wl.batch, wl.num_kv_heads, wl.head_dim, max_seq,
                                wl.k_bits, wl.v_bits, wl.k_mode, wl.v_mode, wl.k_group,
                                wl.v_group, wl.outliers_per_row)
    assert got >= algo
    # capacity rounding to 64 tokens + the fp16 residual block + alignment
    slack = wl.num_layers * wl.batch * wl.num_kv_heads * (64 + wl.k_group) * 600 + 4096 * wl.num_layers
    assert got <= algo + slack, (got, algo)


BAD = [
    (dict(head_dim=64), 2), (dict(k_bits=5), 1), (dict(v_mode=kvq.ASYM_PER_CHANNEL), 2),
    (dict(k_mode=kvq.SYM_PER_TOKEN, k_bits=4, k_group=32), 2), (dict(v_group=48), 1),
    (dict(v_bits=3, v_group=64), 2), (dict(outliers_per_row=9), 1), (dict(k_group=32), 2),
    (dict(max_seq=0), 1), (dict(batch=0), 1), (dict(k_mode=7), 1),
]
_CB = dict(k_mode=kvq.CODEBOOK_PER_TOKEN, v_mode=kvq.CODEBOOK_PER_TOKEN, k_group=32, v_group=32,
           codebook=kvq.E2M1_LEVELS)
BAD += [
    (dict(_CB, v_mode=kvq.ASYM_PER_TOKEN), 2),          # keys and values together only
    (dict(_CB, k_bits=3, v_bits=3, k_group=128, v_group=128), 2),  # 4-bit codes only
    (dict(_CB, outliers_per_row=2), 2),                 # no outliers beside codebook codes
    (dict(_CB, codebook=[0.0] * 16), 1),                # no nonzero level
    (dict(_CB, codebook=[float("inf")] + [1.0] * 15), 1),
    (dict(_CB, codebook=[float("nan")] + [1.0] * 15), 1),
    (dict(_CB, codebook=[0.0, 2.0 ** -20] + [1.0] * 14), 2),  # levels closer than max|level| / 65536
]


@pytest.mark.parametrize("kw,status", BAD, ids=[str(b[0]) for b in BAD])
def test_bad_configs_are_rejected(lib, kw, status):
    n = ctypes.c_size_t()
    assert lib.kvq_cache_bytes(ctypes.byref(_cfg(**kw)), ctypes.byref(n)) == status
    assert lib.kvq_last_error()


@pytest.mark.parametrize("group", [16, 32, 64, 128])
def test_codebook_cache_bytes(lib, group):
    """A codebook cache holds 4-bit codes and one fp16 scale per group."""
    cfg = _cfg(**dict(_CB, k_group=group, v_group=group))
    got = kvq.cache_bytes(cfg)
    algo = O.packed_cache_bytes(1, 2, 4, 128, 1000, 4, 4, O.CODEBOOK_PER_TOKEN, O.CODEBOOK_PER_TOKEN,
                                group, group)
    assert algo == 2 * 2 * 4 * 1000 * (64 + 2 * 128 // group)
    assert algo <= got <= algo + 2 * 4 * 64 * 600 + 4096, (got, algo)


def test_create_rejects_bad_buffers_on_the_host(lib):
    cfg = _cfg()
    h = ctypes.c_void_p()
    assert lib.kvq_cache_create(ctypes.byref(cfg), None, 1 << 30, None, ctypes.byref(h)) == 1
    assert lib.kvq_cache_create(ctypes.byref(cfg), ctypes.c_void_p(0x1008), 1 << 30, None,
                                ctypes.byref(h)) == 1
    assert lib.kvq_cache_create(ctypes.byref(cfg), ctypes.c_void_p(0x10000), 100, None,
                                ctypes.byref(h)) == 3
    assert b"needs" in lib.kvq_last_error()
    assert h.value is None


def test_null_handle_is_rejected(lib):
    assert lib.kvq_prefill_quantize(None, 0, None, None, 0, None) == 1
    assert lib.kvq_append_quantize(None, 0, None, None, None) == 1
    assert lib.kvq_decode_attention(None, 0, None, 1, 1.0, None, 0, None, 0, None) == 1
    n = ctypes.c_int32()
    assert lib.kvq_cache_length(None, 0, ctypes.byref(n)) == 1
    assert lib.kvq_cache_status(None, None, None) == 1


def test_per_layer_code_widths_size_the_cache(lib):
    """A per-layer map of code widths (mixed precision by layer) sizes the
    cache as the header plus each layer's own size; NULL is the uniform cache."""
    def nbytes(fn, cfg, arr):
        n = ctypes.c_size_t()
        kvq.check(fn(ctypes.byref(cfg), arr, ctypes.byref(n)))
        return n.value
    base = dict(batch=2, num_kv_heads=4, head_dim=128, max_seq=1000, k_mode=kvq.ASYM_PER_CHANNEL,
                v_mode=kvq.ASYM_PER_TOKEN, k_group=64, v_group=128, outliers_per_row=0)
    pairs = [(8, 8), (4, 8), (4, 4), (3, 3)]
    cfg = kvq.make_config(num_layers=4, k_bits=4, v_bits=4, **base)
    arr = (ctypes.c_int32 * 8)(*[b for p in pairs for b in p])
    uniform = ctypes.c_size_t()
    kvq.check(lib.kvq_cache_bytes(ctypes.byref(cfg), ctypes.byref(uniform)))
    assert nbytes(lib.kvq_cache_bytes_per_layer, cfg, None) == uniform.value
    header = 256
    want = header
    for kb, vb in pairs:
        one = kvq.make_config(num_layers=1, k_bits=kb, v_bits=vb, **base)
        want += nbytes(lib.kvq_cache_bytes_per_layer, one, None) - header
    assert nbytes(lib.kvq_cache_bytes_per_layer, cfg, arr) == want
    # a pair that the modes and groups do not allow: 3-bit values need whole-row groups
    bad = kvq.make_config(num_layers=2, k_bits=4, v_bits=4, **dict(base, v_group=64))
    arr2 = (ctypes.c_int32 * 4)(4, 4, 4, 3)
    with pytest.raises(kvq.KVQError) as e:
        nbytes(lib.kvq_cache_bytes_per_layer, bad, arr2)
    assert "layer 1" in str(e.value)


def test_package_e2m1_levels_match_the_oracle_bit_fields():
    """The package's minifloat codebook equals the oracle's, which derives
    each level from the code's sign, exponent and mantissa bits."""
    import numpy as np
    a = np.array(kvq.E2M1_LEVELS, np.float16).view(np.uint16)
    assert np.array_equal(a, O.e2m1_codebook().view(np.uint16))
