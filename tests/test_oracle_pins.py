"""Pins for the CPU oracle: each test ties an oracle function to something
other than itself -- a value printed on the pages (tests/golden), a closed
form, brute force on tiny inputs, or a library routine.

Pages are cited by short name, address and section:
[TurboQuant-3bit] dpshk.com/news/6341316, [KVQuant] cf-1.com/news/2306543,
[TurboQuant-mem] demingchina.com/news/57821, [W4A8-FA3]
discosf.com/news/4854722, [NIAH-q8_0] cf-1.com/news/5482713.
"""
import itertools
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append([c.strip() for c in line.split("|")])
    return out


def _fact(name):
    for row in _rows("page_facts.txt"):
        if row[0] == name:
            return int(row[1])
    raise KeyError(name)


# ---------------------------------------------------------------------------
# Footprint: values printed on the pages
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("row", _rows("footprint_pins.txt"), ids=lambda r: r[0])
def test_footprint_matches_pages(row):
    _, L, H, D, S, nb, expected, tol = row
    got = O.fp16_kv_cache_bytes(int(L), int(H), int(D), int(S), int(nb))
    expected = float(expected)
    if float(tol) == 0:
        assert got == int(expected)
    else:
        assert abs(got - expected) <= float(tol) * expected, (got, expected)


def test_one_head_context_bytes():
    # one head, one tensor: half of the K+V footprint
    assert O.fp16_kv_cache_bytes(1, 1, 128, 4096) // 2 == _fact("one_head_4096_fp16_bytes")


def test_position_groups_of_64():
    rng = np.random.default_rng(0)
    spec = O.CodecSpec(128, 4, 4, O.ASYM_PER_CHANNEL, O.ASYM_PER_TOKEN, 64, 64)
    c = O.OracleCache(spec, 1)
    x = rng.standard_normal((1, 2048, 128)).astype(np.float16)
    c.prefill(x, x)
    assert c.k.scale16.shape[1] == _fact("groups_of_64_in_2048")
    assert c.k.zero16.shape[1] == _fact("groups_of_64_in_2048")
    assert c.k.resid.shape[1] == 0


# ---------------------------------------------------------------------------
# Quantizer: ranges, grid values, error bound, brute force
# ---------------------------------------------------------------------------

def test_sym_int8_range_and_extremes():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 4, 32)) * 3).astype(np.float16)
    c, s16 = O.quantize_sym(x, 8)
    assert c.min() >= _fact("int8_code_min") and c.max() <= _fact("int8_code_max")
    # the largest-magnitude member of every group lands on +-127
    idx = np.abs(x.astype(np.float32)).argmax(-1)
    top = np.take_along_axis(c, idx[..., None], -1)[..., 0]
    assert np.all(np.abs(top) == 127)


@pytest.mark.parametrize("bits", [3, 4, 8])
def test_asym_range_ends(bits):
    rng = np.random.default_rng(bits)
    x = rng.standard_normal((200, 64)).astype(np.float16)
    c, s16, z16 = O.quantize_asym(x, bits)
    assert c.min() >= 0 and c.max() <= 2 ** bits - 1
    if bits == 3:
        assert c.max() == _fact("asym_3bit_code_max")
    # offset = group minimum: the minimum maps to code 0 and z16 is exactly it
    xm = x.astype(np.float32)
    assert np.all(z16.astype(np.float32) == xm.min(-1))
    assert np.all(np.take_along_axis(c, xm.argmin(-1)[:, None], -1) == 0)
    # the maximum maps to the top code (the scale spans max - min)
    assert np.all(np.take_along_axis(c, xm.argmax(-1)[:, None], -1) == 2 ** bits - 1)


@pytest.mark.parametrize("bits", [3, 4, 8])
def test_grid_values_reconstruct_exactly(bits):
    """x = z16 + k*s16 built exactly in fp16 must give code k and x_hat = x."""
    rng = np.random.default_rng(10 + bits)
    top = 2 ** bits - 1
    for trial in range(40):
        e = int(rng.integers(-8, -2))
        s = 2.0 ** e                       # power of two: z + k*s exact in fp16
        z = float(rng.integers(-64, 0)) * s
        ks = rng.integers(0, top + 1, size=32)
        ks[0], ks[1] = 0, top              # min and max present
        x = (z + ks * s).astype(np.float16)
        assert np.all(x.astype(np.float64) == z + ks * s)
        c, s16, z16 = O.quantize_asym(x[None], bits)
        assert float(s16[0]) == s and float(z16[0]) == z
        assert np.array_equal(c[0], ks)
        xh = z16.astype(np.float64)[0] + c[0] * s16.astype(np.float64)[0]
        assert np.array_equal(xh, x.astype(np.float64))


def test_sym_grid_values_reconstruct_exactly():
    rng = np.random.default_rng(5)
    for trial in range(40):
        s = 2.0 ** int(rng.integers(-10, -3))
        ks = rng.integers(-127, 128, size=32)
        ks[0] = 127 if trial % 2 else -127
        x = (ks * s).astype(np.float16)
        c, s16 = O.quantize_sym(x[None], 8)
        assert float(s16[0]) == s
        assert np.array_equal(c[0], ks)


@pytest.mark.parametrize("bits", [3, 4, 8])
def test_error_bound(bits):
    """|x - x_hat| <= s16/2 inside the grid; at the top end the fp16 rounding
    of the scale may leave max above the last grid point by that rounding."""
    rng = np.random.default_rng(20 + bits)
    x = (rng.standard_normal((500, 64)) * np.exp(rng.standard_normal((500, 1)))).astype(np.float16)
    c, s16, z16 = O.quantize_asym(x, bits)
    s = s16.astype(np.float64)[:, None]
    z = z16.astype(np.float64)[:, None]
    xh = z + c * s
    err = np.abs(x.astype(np.float64) - xh)
    top = z + (2 ** bits - 1) * s
    over = np.maximum(x.astype(np.float64) - top, 0)
    assert np.all(err <= s / 2 + over + 1e-12 * np.abs(z))
    # the slack is needed only at the top end, and only by fp16 rounding of s
    assert np.all(over <= 2.0 ** -11 * (2 ** bits - 1) * s + 1e-30)


def _nearest_code_bruteforce(x, s16, z16, lo, hi):
    """argmin_c |x - (z + c*s)| over c in [lo, hi], exact rationals, ties to
    the even code."""
    xs = Fraction(float(x))
    s = Fraction(float(s16))
    z = Fraction(float(z16))
    best, bestd = None, None
    for c in range(lo, hi + 1):
        d = abs(xs - (z + c * s))
        if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
            best, bestd = c, d
    return best


def _near_half(x, s16, z16):
    s = Fraction(float(s16))
    if s == 0:
        return False
    q = (Fraction(float(x)) - Fraction(float(z16))) / s
    frac = q - int(q)
    return abs(frac - Fraction(1, 2)) < Fraction(1, 2 ** 18)


@pytest.mark.parametrize("bits", [3, 4, 8])
def test_codes_are_nearest_grid_points_bruteforce(bits):
    rng = np.random.default_rng(30 + bits)
    x = (rng.standard_normal((60, 16)) * 2).astype(np.float16)
    c, s16, z16 = O.quantize_asym(x, bits)
    mism = 0
    for g in range(x.shape[0]):
        for j in range(x.shape[1]):
            bf = _nearest_code_bruteforce(x[g, j], s16[g], z16[g], 0, 2 ** bits - 1)
            if bf != c[g, j] and not _near_half(x[g, j], s16[g], z16[g]):
                mism += 1
    assert mism == 0


def test_sym_codes_are_nearest_bruteforce():
    rng = np.random.default_rng(40)
    x = (rng.standard_normal((40, 32))).astype(np.float16)
    c, s16 = O.quantize_sym(x, 8)
    for g in range(x.shape[0]):
        for j in range(x.shape[1]):
            bf = _nearest_code_bruteforce(x[g, j], s16[g], np.float16(0), -127, 127)
            if bf != c[g, j]:
                assert _near_half(x[g, j], s16[g], np.float16(0))


def test_degenerate_groups():
    # constant group: scale 0, every code 0, x_hat = z = the constant
    x = np.full((1, 64), 1.5, np.float16)
    c, s16, z16 = O.quantize_asym(x, 4)
    assert float(s16[0]) == 0 and float(z16[0]) == 1.5 and not c.any()
    xs = np.zeros((1, 32), np.float16)
    c, s16 = O.quantize_sym(xs, 8)
    assert float(s16[0]) == 0 and not c.any()
    # every member an outlier: scale = zero point = 0, codes 0
    m = np.ones((1, 64), bool)
    c, s16, z16 = O.quantize_asym(np.arange(64, dtype=np.float16)[None], 4, m)
    assert float(s16[0]) == 0 and float(z16[0]) == 0 and not c.any()


# ---------------------------------------------------------------------------
# Packing
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits,words", [(3, 13), (4, 16), (8, 32)])
def test_words_per_row(bits, words):
    assert O.words_per_row(bits, 128) == words


@pytest.mark.parametrize("bits", [3, 4, 8])
def test_pack_isolated_code_bit_positions(bits):
    """A row with a single nonzero code c at channel j sets exactly the bits
    of c at offset (j % cpw) * b inside word j // cpw."""
    cpw = O.codes_per_word(bits)
    top = 2 ** bits - 1
    for j in range(128):
        codes = np.zeros(128, np.int64)
        codes[j] = top
        w = O.pack_row_codes(codes, bits)
        expect = np.zeros_like(w)
        expect[j // cpw] = np.uint32(top << ((j % cpw) * bits))
        assert np.array_equal(w, expect), j


def test_pack_3bit_spare_bits_and_worked_word():
    # ten codes 1..7,0,1,2 in one word: written out bit by bit in the fixture
    codes = np.array([1, 2, 3, 4, 5, 6, 7, 0, 1, 2] + [0] * 118)
    w = O.pack_row_codes(codes, 3)
    # binary, high bits first: 00 | 010 001 000 111 110 101 100 011 010 001
    assert int(w[0]) == 0b00_010_001_000_111_110_101_100_011_010_001
    rng = np.random.default_rng(7)
    allc = rng.integers(0, 8, size=(100, 128))
    ws = O.pack_row_codes(allc, 3)
    assert np.all((ws >> 30) == 0)
    assert np.all(ws[:, -1] >> 24 == 0)   # last word holds 8 codes only


@pytest.mark.parametrize("bits", [3, 4, 8])
@pytest.mark.parametrize("signed", [False, True])
def test_pack_roundtrip(bits, signed):
    rng = np.random.default_rng(bits + 10 * signed)
    if signed:
        lo, hi = -(2 ** (bits - 1) - 1), 2 ** (bits - 1) - 1
    else:
        lo, hi = 0, 2 ** bits - 1
    c = rng.integers(lo, hi + 1, size=(17, 5, 128))
    back = O.unpack_row_codes(O.pack_row_codes(c, bits), bits, 128, signed=signed)
    assert np.array_equal(back, c)


# ---------------------------------------------------------------------------
# Outliers
# ---------------------------------------------------------------------------

def _dominant_subset_bruteforce(row, k):
    """The unique k-subset S such that every member beats every non-member
    under (|x| larger, then lower channel)."""
    d = len(row)
    key = [(abs(float(row[i])), -i) for i in range(d)]
    winners = []
    for sub in itertools.combinations(range(d), k):
        rest = [i for i in range(d) if i not in sub]
        if all(key[a] > key[b] for a in sub for b in rest):
            winners.append(sub)
    assert len(winners) == 1
    return list(winners[0])


def test_outliers_bruteforce_with_ties():
    rng = np.random.default_rng(50)
    for trial in range(200):
        # few distinct magnitudes so ties are common
        row = (rng.integers(-3, 4, size=8)).astype(np.float16)
        for k in (1, 2, 3):
            mask, cols, vals = O.select_outliers(row[None], k)
            bf = _dominant_subset_bruteforce(row, k)
            assert list(cols[0]) == bf
            assert np.array_equal(vals[0], row[bf])
            assert mask[0].sum() == k


def test_outlier_tie_break_is_lowest_channel_under_permutation():
    row = np.array([1, -5, 5, 2, -5, 0, 5, 1], np.float16)
    _, cols, _ = O.select_outliers(row[None], 2)
    assert list(cols[0]) == [1, 2]
    rng = np.random.default_rng(3)
    for _ in range(50):
        perm = rng.permutation(8)
        prow = row[perm]
        _, c, _ = O.select_outliers(prow[None], 2)
        five = [i for i in range(8) if abs(float(prow[i])) == 5]
        assert list(c[0]) == five[:2]


def test_outliers_leave_group_stats_and_restore_exactly():
    x = np.linspace(-1, 1, 64).astype(np.float16)
    x[10] = 300.0
    x[20] = -250.0
    spec = O.CodecSpec(64, 4, 4, O.ASYM_PER_TOKEN, O.ASYM_PER_TOKEN, 64, 64, outliers_per_row=2)
    c = O.OracleCache(spec, 1)
    c.prefill(x[None, None], x[None, None])
    assert float(c.v.zero16[0, 0, 0]) == float(np.float16(-1.0))
    assert list(c.v.out_cols[0, 0]) == [10, 20]
    vh = c.dequant_v()[0, 0]
    assert vh[10] == 300.0 and vh[20] == -250.0
    assert c.v.codes[0, 0, 10] == 0 and c.v.codes[0, 0, 20] == 0
    # the dense part still meets its error bound
    s = float(c.v.scale16[0, 0, 0])
    keep = np.ones(64, bool)
    keep[[10, 20]] = False
    assert np.all(np.abs(vh[keep] - x[keep].astype(np.float64)) <= s / 2 + 1e-9)


def test_outliers_only_affect_their_own_group():
    """Group-wise scaling confines an outlier's damage to its own group
    ([TurboQuant-mem] §2.3)."""
    rng = np.random.default_rng(60)
    x = rng.standard_normal((1, 1, 1, 128)).astype(np.float16)
    spec = O.CodecSpec(128, 4, 4, O.ASYM_PER_TOKEN, O.ASYM_PER_TOKEN, 32, 32)
    a = O.OracleCache(spec, 1)
    a.prefill(x[0], x[0])
    y = x.copy()
    y[..., 5] = 80.0
    b = O.OracleCache(spec, 1)
    b.prefill(y[0], y[0])
    assert np.array_equal(a.v.codes[..., 32:], b.v.codes[..., 32:])
    assert not np.array_equal(a.v.codes[..., :32], b.v.codes[..., :32])


# ---------------------------------------------------------------------------
# Cache: prefill/append consistency and the key residual
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kmode", [O.ASYM_PER_CHANNEL, O.ASYM_PER_TOKEN, O.SYM_PER_TOKEN])
def test_prefill_equals_token_by_token_appends(kmode):
    rng = np.random.default_rng(70 + kmode)
    d, s = 128, 64 * 3 + 17
    kbits = 8 if kmode == O.SYM_PER_TOKEN else 4
    spec = O.CodecSpec(d, kbits, 8, kmode, O.ASYM_PER_TOKEN,
                       64 if kmode == O.ASYM_PER_CHANNEL else 32, 64, outliers_per_row=2)
    k = rng.standard_normal((3, s, d)).astype(np.float16)
    v = rng.standard_normal((3, s, d)).astype(np.float16)
    a = O.OracleCache(spec, 3)
    a.prefill(k, v)
    b = O.OracleCache(spec, 3)
    b.prefill(k[:, :40], v[:, :40])
    for t in range(40, s):
        b.append(k[:, t], v[:, t])
    for f in ("codes", "scale16", "out_cols", "out_vals"):
        assert np.array_equal(getattr(a.k, f), getattr(b.k, f)), f
        assert np.array_equal(getattr(a.v, f), getattr(b.v, f)), f
    assert np.array_equal(a.dequant_k(), b.dequant_k())
    if kmode == O.ASYM_PER_CHANNEL:
        assert a.k.resid.shape[1] == 17
        assert np.array_equal(a.k.resid, k[:, -17:])


# ---------------------------------------------------------------------------
# Attention: library routine, closed forms
# ---------------------------------------------------------------------------

def test_attention_matches_torch_sdpa_fp64():
    rng = np.random.default_rng(80)
    n, g, s, d = 3, 4, 33, 16
    q = rng.standard_normal((n, g, d))
    k = rng.standard_normal((n, s, d))
    v = rng.standard_normal((n, s, d))
    scale = 0.37
    o = O.attend(q, k, v, scale)
    tq = torch.from_numpy(q)[:, :, None, :]
    tk = torch.from_numpy(k)[:, None].expand(n, g, s, d)
    tv = torch.from_numpy(v)[:, None].expand(n, g, s, d)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[:, :, 0]
    assert np.allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(81)
    d = 8
    v = rng.standard_normal((1, 5, d))
    k = rng.standard_normal((1, 5, d))
    # one token: the output is that token's value
    assert np.allclose(O.attend(rng.standard_normal((1, 1, d)), k[:, :1], v[:, :1], 1.0)[0, 0], v[0, 0])
    # zero query: all scores equal, output is the mean value
    assert np.allclose(O.attend(np.zeros((1, 1, d)), k, v, 1.0)[0, 0], v[0].mean(0))
    # two tokens whose scores differ by delta: weights are a logistic function
    kk = np.zeros((1, 2, d))
    kk[0, 0, 0] = 1.0
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 1.3
    w = 1.0 / (1.0 + np.exp(-1.3 * 0.5))
    assert np.allclose(O.attend(q, kk, v[:, :2], 0.5)[0, 0], w * v[0, 0] + (1 - w) * v[0, 1])
    # one dominant score: the output is that token's value
    kd = k.copy()
    kd[0, 3] = 50 * np.ones(d)
    assert np.allclose(O.attend(np.ones((1, 1, d)), kd, v, 1.0)[0, 0], v[0, 3], atol=1e-12)


def test_attention_shift_and_permutation_invariance():
    rng = np.random.default_rng(82)
    q = rng.standard_normal((2, 3, 16))
    k = rng.standard_normal((2, 20, 16))
    v = rng.standard_normal((2, 20, 16))
    o = O.attend(q, k, v, 0.25)
    perm = rng.permutation(20)
    assert np.allclose(O.attend(q, k[:, perm], v[:, perm], 0.25), o, atol=1e-13)


def test_dense_only_cache_is_plain_group_codec():
    rng = np.random.default_rng(83)
    x = rng.standard_normal((2, 128, 64)).astype(np.float16)
    spec = O.CodecSpec(64, 4, 4, O.ASYM_PER_TOKEN, O.ASYM_PER_TOKEN, 32, 32)
    c = O.OracleCache(spec, 2)
    c.prefill(x, x)
    codes, s16, z16 = O.quantize_asym(x.reshape(2, 128, 2, 32), 4)
    xh = z16.astype(np.float64)[..., None] + codes * s16.astype(np.float64)[..., None]
    assert np.array_equal(c.dequant_v(), xh.reshape(2, 128, 64))


def test_empty_cache_decode_is_rejected():
    spec = O.CodecSpec(64, 4, 4, O.ASYM_PER_TOKEN, O.ASYM_PER_TOKEN, 32, 32)
    c = O.OracleCache(spec, 1)
    c.prefill(np.zeros((1, 0, 64), np.float16), np.zeros((1, 0, 64), np.float16))
    with pytest.raises(ValueError):
        c.decode(np.zeros((1, 1, 64)), 1.0)


# ---------------------------------------------------------------------------
# Packed footprint of the layout (layout arithmetic, cross-checked by hand)
# ---------------------------------------------------------------------------

def test_packed_bytes_by_hand():
    # Llama-2-7B-shaped layer, B=8, 32 heads, S=16384, 4-bit K per channel (T=64),
    # 4-bit V per token (G=64): codes 2 x 256 MiB, metadata 2 x 32 MiB.
    got = O.packed_cache_bytes(1, 8, 32, 128, 16384, 4, 4, O.ASYM_PER_CHANNEL,
                               O.ASYM_PER_TOKEN, 64, 64)
    assert got == 2 * 256 * 2 ** 20 + 2 * 32 * 2 ** 20
    # Llama-2-70B-shaped layer, 3-bit, 13 words per row: 52 B codes + 4 B meta
    # per token and tensor (T = G = 128).
    got = O.packed_cache_bytes(1, 4, 8, 128, 32768, 3, 3, O.ASYM_PER_CHANNEL,
                               O.ASYM_PER_TOKEN, 128, 128)
    assert got == 4 * 8 * 32768 * 2 * (52 + 4)


def test_zero_extremes_are_positive_zero():
    x = np.array([[-0.0, 0.0, 1.0, 2.0]], np.float16)
    _, s16, z16 = O.quantize_asym(x, 4)
    assert z16.view(np.uint16)[0] == 0
    x = np.array([[-0.0, -0.0, -0.0, -0.0], [0.0, -0.0, 0.0, -0.0]], np.float16)
    _, s16, z16 = O.quantize_asym(x, 4)
    assert np.all(s16.view(np.uint16) == 0) and np.all(z16.view(np.uint16) == 0)


# ---------------------------------------------------------------------------
# Per-channel key blocks: each (block, channel) holds its own grid
# ---------------------------------------------------------------------------

def _channel_grid_keys(bits, block, nb, d, seed):
    """Keys whose channel c in block b takes the grid values z_bc + k s_bc,
    k = 0 .. 2^b - 1 (both ends present), in a token order that differs per
    channel. s_bc and z_bc are integers times 2^-q_bc, with q_bc, s_bc and z_bc
    different across blocks and channels, and every key is an integer below
    2048 times a power of two, so it is exact in fp16."""
    rng = np.random.default_rng(seed)
    levels = 2 ** bits - 1
    x = np.zeros((1, nb * block, d), np.float16)
    s = np.zeros((nb, d))
    z = np.zeros((nb, d))
    k = np.zeros((nb, block, d), np.int64)
    for b in range(nb):
        for c in range(d):
            q = 3 + (b + 2 * c) % 6
            s_int = 1 + (3 * b + c) % 3
            z_int = (c * 7 + b * 11) % (2047 - levels * s_int) - 300
            s[b, c] = s_int * 2.0 ** -q
            z[b, c] = z_int * 2.0 ** -q
            ks = rng.integers(0, levels + 1, size=block)
            ks[rng.permutation(block)[:2]] = [0, levels]  # both extremes somewhere
            k[b, :, c] = ks
            x[0, b * block:(b + 1) * block, c] = (z[b, c] + ks * s[b, c]).astype(np.float16)
            assert np.array_equal(x[0, b * block:(b + 1) * block, c].astype(np.float64), z[b, c] + ks * s[b, c])
    return x, s, z, k


@pytest.mark.parametrize("bits", [3, 4, 8])
def test_per_channel_blocks_recover_each_channels_grid(bits):
    """[KVQuant] §2.2 item 1 and [W4A8-FA3] §2.4: a key group is one channel
    over T consecutive tokens. With channel c of block b built on its own grid
    z_bc + k s_bc, the block's metadata must be exactly (s_bc, z_bc) at
    [stream][b][c] and the codes must be the grid indices k; grouping over
    channels instead, or a transposed block, gives other extremes."""
    block, nb, d = 64, 3, 128
    x, s, z, k = _channel_grid_keys(bits, block, nb, d, seed=500 + bits)
    spec = O.CodecSpec(d, bits, 8, O.ASYM_PER_CHANNEL, O.ASYM_PER_TOKEN, block, 64)
    c = O.OracleCache(spec, 1)
    c.prefill(x, x)
    assert c.k.scale16.shape == (1, nb, d)
    assert np.array_equal(c.k.scale16[0].astype(np.float64), s)
    assert np.array_equal(c.k.zero16[0].astype(np.float64), z)
    assert np.array_equal(c.k.codes[0], k.reshape(nb * block, d))
    assert c.k.resid.shape[1] == 0


def test_per_channel_perturbation_stays_in_its_block_and_channel():
    """Raising one key of channel c in block b above the channel's maximum
    changes that block-channel's scale and no other metadata or codes outside
    it (the per-channel counterpart of group confinement, [TurboQuant-mem]
    §2.3)."""
    bits, block, nb, d = 4, 64, 3, 128
    x, s, z, _ = _channel_grid_keys(bits, block, nb, d, seed=77)
    spec = O.CodecSpec(d, bits, 8, O.ASYM_PER_CHANNEL, O.ASYM_PER_TOKEN, block, 64)
    a = O.OracleCache(spec, 1)
    a.prefill(x, x.copy())
    bb, cc, tt = 1, 37, 5
    y = x.copy()
    y[0, bb * block + tt, cc] = np.float16(z[bb, cc] + 20 * s[bb, cc])
    b = O.OracleCache(spec, 1)
    b.prefill(y, x.copy())
    ds = a.k.scale16 != b.k.scale16
    assert ds[0, bb, cc] and ds.sum() == 1
    assert np.array_equal(a.k.zero16, b.k.zero16)
    dc = a.k.codes != b.k.codes
    rows = np.nonzero(dc[0])[0]
    assert set(np.nonzero(dc[0])[1]) == {cc}
    assert rows.min() >= bb * block and rows.max() < (bb + 1) * block
    assert np.array_equal(a.v.codes, b.v.codes)


# ---------------------------------------------------------------------------
# Footprint: CSR outliers and the fp16 key residual, by hand
# ---------------------------------------------------------------------------

def test_packed_bytes_csr_by_hand():
    # dense-and-sparse 128K layer: 32 streams, 4-bit K per channel (T=64) and
    # V per token (G=64), 2 outliers per row. Per stream and tensor: codes
    # 131072 * 64 B, metadata 1 MiB, CSR 4 (131072 + 1) + 131072 * 2 * 4 B.
    got = O.packed_cache_bytes(1, 1, 32, 128, 131072, 4, 4, O.ASYM_PER_CHANNEL,
                               O.ASYM_PER_TOKEN, 64, 64, outliers_per_row=2)
    per = 131072 * 64 + 2 ** 20 + 4 * 131073 + 131072 * 8
    assert per == 11010052
    assert got == 32 * 2 * per == 704643328


def test_packed_bytes_key_residual_by_hand():
    # S = 1000 with T = 64: 960 key rows as codes in 15 blocks, 40 fp16 keys.
    got = O.packed_cache_bytes(1, 1, 1, 128, 1000, 4, 8, O.ASYM_PER_CHANNEL,
                               O.ASYM_PER_TOKEN, 64, 64)
    k = 960 * 64 + 15 * 128 * 4 + 40 * 128 * 2
    v = 1000 * (128 + 2 * 4)
    assert (k, v) == (79360, 136000)
    assert got == k + v
    # with 3 outliers per row: the key CSR covers the 960 coded rows only,
    # the value CSR all 1000 rows
    got = O.packed_cache_bytes(1, 1, 1, 128, 1000, 4, 8, O.ASYM_PER_CHANNEL,
                               O.ASYM_PER_TOKEN, 64, 64, outliers_per_row=3)
    assert got == k + v + (4 * 961 + 960 * 12) + (4 * 1001 + 1000 * 12)


@pytest.mark.parametrize("length", [1, 63, 64, 1000, 4097])
def test_bench_accounting_matches_oracle_footprint(length):
    """bench.py's byte counts (the package's accounting module) equal the
    oracle's footprint for every workload and ragged lengths."""
    from bit_quantized_kv_kvq_gb300 import accounting as A, workloads as W
    for wl in W.ALL + W.EXTRA:
        want = O.packed_cache_bytes(1, wl.batch, wl.num_kv_heads, wl.head_dim, length, wl.k_bits,
                                    wl.v_bits, wl.k_mode, wl.v_mode, wl.k_group, wl.v_group,
                                    wl.outliers_per_row)
        assert A.cache_read_bytes(wl, length) == want, wl.name


# ---------------------------------------------------------------------------
# The error measure of the attention gate
# ---------------------------------------------------------------------------

def test_row_relative_error_closed_form():
    """Reading R13: max_d |o - o_ref| / max_d |o_ref| per row."""
    o_ref = np.array([[1.0, -4.0, 2.0], [-8.0, 1.0, 0.5], [0.0, 0.0, 0.0]])
    o = np.array([[1.5, -4.0, 2.0], [-6.0, 1.0, 0.25], [0.0, 0.0, 0.0]])
    got = O.row_relative_error(o, o_ref)
    assert np.array_equal(got, [0.5 / 4.0, 2.0 / 8.0, 0.0])
    # rows along the last axis only; the denominator is the reference's
    assert O.row_relative_error(o_ref, o)[1] == 2.0 / 6.0
    x = np.arange(24.0).reshape(2, 3, 4) + 1
    e = O.row_relative_error(x * (1 + 1e-3), x)
    assert e.shape == (2, 3) and np.allclose(e, 1e-3, rtol=1e-12)


# ---------------------------------------------------------------------------
# Attention sinks ([KVQuant] §4.1): the first tokens kept in fp16
# ---------------------------------------------------------------------------

def _sink_spec(ns, kmode=O.ASYM_PER_CHANNEL, bits=3):
    return O.CodecSpec(128, bits, bits, kmode, O.ASYM_PER_TOKEN, 64 if kmode == O.ASYM_PER_CHANNEL else 32,
                       128, 0, ns)


def test_all_sink_cache_is_exact_attention():
    """When the sinks cover the whole sequence nothing is quantized: the
    decode is fp64 attention on the fp16 inputs themselves."""
    rng = np.random.default_rng(91)
    k = rng.standard_normal((2, 7, 128)).astype(np.float16)
    v = rng.standard_normal((2, 7, 128)).astype(np.float16)
    q = rng.standard_normal((2, 3, 128))
    c = O.OracleCache(_sink_spec(8), 2)
    c.prefill(k, v)
    assert c.coded_length == 0 and c.sink_k.shape[1] == 7
    assert np.array_equal(c.decode(q, 0.1), O.attend(q, k.astype(np.float64), v.astype(np.float64), 0.1))


@pytest.mark.parametrize("kmode", [O.ASYM_PER_CHANNEL, O.ASYM_PER_TOKEN])
def test_sinks_shift_quantization_past_them(kmode):
    """With sinks, the quantized state is that of a cache without sinks fed
    the tokens after them (per-channel key blocks start after the sinks), by
    prefill and by appends crossing the sink boundary alike."""
    rng = np.random.default_rng(92 + kmode)
    ns, s = 5, 200
    k = rng.standard_normal((2, s, 128)).astype(np.float16)
    v = rng.standard_normal((2, s, 128)).astype(np.float16)
    a = O.OracleCache(_sink_spec(ns, kmode), 2)
    a.prefill(k, v)
    b = O.OracleCache(_sink_spec(0, kmode), 2)
    b.prefill(k[:, ns:], v[:, ns:])
    assert np.array_equal(a.sink_k, k[:, :ns]) and np.array_equal(a.sink_v, v[:, :ns])
    for f in ("codes", "scale16", "zero16"):
        assert np.array_equal(getattr(a.k, f), getattr(b.k, f)), f
        assert np.array_equal(getattr(a.v, f), getattr(b.v, f)), f
    c = O.OracleCache(_sink_spec(ns, kmode), 2)
    c.prefill(k[:, :3], v[:, :3])
    for t in range(3, s):
        c.append(k[:, t], v[:, t])
    assert np.array_equal(c.k.codes, b.k.codes) and np.array_equal(c.v.codes, b.v.codes)
    assert np.array_equal(c.sink_k, a.sink_k)
    q = rng.standard_normal((2, 2, 128))
    assert np.array_equal(c.decode(q, 0.09), a.decode(q, 0.09))


def test_sinks_keep_a_dominant_first_token_exact():
    """A first token that draws most of the attention (the pattern that
    motivates sinks) is reproduced better with it kept in fp16."""
    rng = np.random.default_rng(93)
    s = 256
    k = rng.standard_normal((1, s, 128)).astype(np.float16)
    v = rng.standard_normal((1, s, 128)).astype(np.float16)
    q = rng.standard_normal((1, 1, 128))
    k[0, 0] = (q[0, 0] * 0.8).astype(np.float16)  # a large score for token 0
    ref = O.attend(q, k.astype(np.float64), v.astype(np.float64), 0.3)
    errs = []
    for ns in (0, 5):
        c = O.OracleCache(_sink_spec(ns, O.ASYM_PER_TOKEN), 1)
        c.prefill(k, v)
        errs.append(float(O.row_relative_error(c.decode(q, 0.3), ref).max()))
    assert errs[1] < errs[0]


# ---------------------------------------------------------------------------
# Codebook codes: the 4-bit minifloat ([TurboQuant-3bit] §3.3) and NUQ
# levels ([KVQuant] §2.2 item 2)
# ---------------------------------------------------------------------------

def test_e2m1_codebook_from_its_bit_fields():
    """1 sign | 2 exponent | 1 mantissa: the positive half is 0, 0.5, 1, 1.5,
    2, 3, 4, 6 and the sign bit negates (reading R20: bias 1, subnormal at
    exponent 0)."""
    cb = O.e2m1_codebook().astype(np.float64)
    assert cb[:8].tolist() == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert np.array_equal(cb[8:], -cb[:8])
    assert cb.dtype == np.float64 and np.array_equal(O.e2m1_codebook().astype(np.float64), cb)


def test_codebook_codes_are_nearest_levels_bruteforce():
    """Every code is the index of the level nearest to x / s16 (exact
    rationals over all 16 levels), the lowest index on exact ties; the scale
    is absmax / max |level| rounded to fp16."""
    from fractions import Fraction
    rng = np.random.default_rng(101)
    for cb in (O.e2m1_codebook(), np.sort(rng.standard_normal(16)).astype(np.float16)):
        x = (rng.standard_normal((40, 32)) * rng.uniform(0.01, 100, (40, 1))).astype(np.float16)
        codes, s16 = O.quantize_codebook(x, cb)
        cbmax = max(abs(float(v)) for v in cb)
        for r in range(x.shape[0]):
            am = max(abs(float(v)) for v in x[r])
            assert s16[r] == np.float16(np.float32(am) / np.float32(cbmax))
            s = Fraction(float(s16[r]))
            for j in range(x.shape[1]):
                y = np.float32(x[r, j]) / np.float32(s16[r])  # the quotient the codec rounds
                dist = [abs(Fraction(float(y)) - Fraction(float(v))) for v in cb]
                best = min(dist)
                assert codes[r, j] == dist.index(best), (r, j)


def test_codebook_levels_reconstruct_exactly_and_zero_groups():
    """Values that are levels times the scale come back exactly; a zero group
    stores scale 0 and code 0."""
    cb = O.e2m1_codebook()
    s = np.float16(0.125)
    idx = np.array([[0, 1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15, 7]])
    x = (cb.astype(np.float32)[idx] * np.float32(s)).astype(np.float16)  # max |x| = 6 s
    codes, s16 = O.quantize_codebook(x, cb)
    assert s16[0] == s
    assert np.array_equal(cb[codes].astype(np.float64) * float(s16[0]), x.astype(np.float64))
    codes, s16 = O.quantize_codebook(np.zeros((1, 32), np.float16), cb)
    assert s16[0] == 0 and np.all(codes == 0)


def test_codebook_cache_dequantizes_through_the_levels():
    """A cache in codebook mode dequantizes x_hat = cb[code] * s16, so its
    attention equals attention on those values."""
    rng = np.random.default_rng(102)
    cb = tuple(float(v) for v in O.e2m1_codebook())
    spec = O.CodecSpec(128, 4, 4, O.CODEBOOK_PER_TOKEN, O.CODEBOOK_PER_TOKEN, 32, 32, 0, 0, cb)
    k = rng.standard_normal((2, 50, 128)).astype(np.float16)
    v = rng.standard_normal((2, 50, 128)).astype(np.float16)
    c = O.OracleCache(spec, 2)
    c.prefill(k, v)
    kc, ks = O.quantize_codebook(k.reshape(2, 50, 4, 32), np.array(cb, np.float16))
    want = np.array(cb)[kc] * ks.astype(np.float64)[..., None]
    assert np.array_equal(c.dequant_k(), want.reshape(2, 50, 128))
    assert c.k.zero16 is None


# ---------------------------------------------------------------------------
# Prefill attention (causal chunk of queries over the cache, reading R22)
# ---------------------------------------------------------------------------

def test_causal_attention_of_equal_keys_is_the_running_mean():
    """With every key equal the weights are uniform: query i returns the mean
    of the values 0 .. positions[i] (a closed form, no softmax involved)."""
    rng = np.random.default_rng(11)
    n, s, d = 2, 9, 8
    k = np.broadcast_to(rng.standard_normal(d), (n, s, d)).copy()
    v = rng.standard_normal((n, s, d))
    q = rng.standard_normal((n, 4, 3, d))
    pos = np.array([0, 3, 5, 8])
    o = O.causal_attend(q, k, v, pos, 0.7)
    run_mean = np.cumsum(v, axis=1) / np.arange(1, s + 1)[None, :, None]
    for i, p in enumerate(pos):
        for h in range(3):
            np.testing.assert_allclose(o[:, i, h], run_mean[:, p], rtol=0, atol=1e-13)


def test_causal_attention_hides_later_tokens():
    """A later token with an overwhelming score changes nothing for queries
    before it, and takes over the query at its own position."""
    rng = np.random.default_rng(12)
    n, s, d = 1, 12, 16
    k = rng.standard_normal((n, s, d)) * 0.1
    v = rng.standard_normal((n, s, d))
    q = rng.standard_normal((n, s, 2, d))
    k[:, 7] = q[:, 7, 0] * 50.0            # token 7: huge score for head 0 of query 7 onward
    pos = np.arange(s)
    o1 = O.causal_attend(q, k, v, pos, 1.0)
    v2 = v.copy()
    v2[:, 7] += 100.0
    o2 = O.causal_attend(q, k, v2, pos, 1.0)
    np.testing.assert_array_equal(o1[:, :7], o2[:, :7])
    assert np.abs(o2[:, 7:] - o1[:, 7:]).max() > 1.0
    np.testing.assert_allclose(o1[:, 7, 0], v[:, 7], rtol=0, atol=1e-9)


def test_prefill_attention_last_query_is_the_decode():
    """The chunk's last query attends the whole cache: the decode of the same
    cache; a one-query chunk is exactly the decode."""
    rng = np.random.default_rng(13)
    spec = O.CodecSpec(128, 4, 4, O.ASYM_PER_CHANNEL, O.ASYM_PER_TOKEN, 64, 32)
    oc = O.OracleCache(spec, 2)
    oc.prefill(rng.standard_normal((2, 150, 128)).astype(np.float16),
               rng.standard_normal((2, 150, 128)).astype(np.float16))
    q = rng.standard_normal((2, 5, 4, 128))
    o = oc.prefill_attention(q, 0.1)
    np.testing.assert_allclose(o[:, -1], oc.decode(q[:, -1], 0.1), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(oc.prefill_attention(q[:, -1:], 0.1)[:, 0], oc.decode(q[:, -1], 0.1))
    with pytest.raises(ValueError):
        oc.prefill_attention(rng.standard_normal((2, 151, 4, 128)), 0.1)


def test_ragged_decode_bytes_are_the_rows_own():
    """A ragged batch's decode bytes are the footprint of each row's own
    tokens (one-row caches of those lengths) plus the queries and outputs."""
    from bit_quantized_kv_kvq_gb300 import accounting as A, workloads as W
    wl = W.RAGGED_Q8
    for extra in (0, 1, 64):
        L = max(wl.lens) + extra
        want = sum(O.packed_cache_bytes(1, 1, wl.num_kv_heads, wl.head_dim, n + extra, wl.k_bits, wl.v_bits,
                                        wl.k_mode, wl.v_mode, wl.k_group, wl.v_group) for n in wl.lens)
        want += wl.batch * wl.num_q_heads * wl.head_dim * 6
        assert A.decode_bytes(wl, L) == want
