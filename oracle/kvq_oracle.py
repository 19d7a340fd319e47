"""Plain CPU oracle for group-wise low-bit KV-cache quantization and
single-token decode attention over the quantized cache.

TEST INFRASTRUCTURE. This module is the checker, not the product: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it. The CUDA library
never calls it, and it shares no code, constant table or helper with the
CUDA path.

What it computes, and where the pages fix it. Pages are cited by a short
name, their address and the section on the page:

* [TurboQuant-3bit] "TurboQuant 3-bit KV-cache quantization",
  dpshk.com/news/6341316
* [KVQuant] "KVQuant: breaking the KV-cache memory wall",
  cf-1.com/news/2306543
* [TurboQuant-mem] "TurboQuant: the KV cache as memory killer",
  demingchina.com/news/57821
* [W4A8-FA3] "W8A8/W4A8, sparsity, FlashAttention-3 and KV-cache
  quantization in practice", discosf.com/news/4854722
* [NIAH-q8_0] "TurboQuant NIAH single-needle q8_0 KV-cache measurements",
  cf-1.com/news/5482713

Precision. The codec decides integer codes, so it runs in fp32 with IEEE
round-to-nearest-even at every step (numpy float32 ufuncs do not contract
to FMA): a code is an integer decided by floating point, and both sides take
that decision in the same precision. Dequantization and attention run in
fp64. Where the pages leave a point open, the reading taken is numbered
(R1, R2, ...) and stated in the function that uses it.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
values the pages print, closed forms, brute force or library routines.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

SYM_PER_TOKEN = 0
ASYM_PER_TOKEN = 1
ASYM_PER_CHANNEL = 2
CODEBOOK_PER_TOKEN = 3


# ---------------------------------------------------------------------------
# Footprint
# ---------------------------------------------------------------------------

def fp16_kv_cache_bytes(num_layers, num_kv_heads, head_dim, seq_len,
                        bytes_per_elem=2, batch=1):
    """Unquantized KV-cache size: K and V (factor 2) for every layer, KV head,
    channel and cached token.

    [TurboQuant-3bit] §2.1 gives the per-token form 2 x L x d_head x h x bytes;
    [TurboQuant-mem] §1.2 gives the element count 2 x L x H x D x S.
    """
    return 2 * num_layers * num_kv_heads * head_dim * seq_len * bytes_per_elem * batch


def codes_per_word(bits):
    """Codes held by one 32-bit word: 32/b for b in {4, 8}; for b = 3 the
    word holds ten codes and its top two bits stay zero (the 3-bit layout
    of ten codes per word with two spare bits)."""
    if bits == 3:
        return 10
    if bits in (4, 8):
        return 32 // bits
    raise ValueError("bits must be 3, 4 or 8")


def words_per_row(bits, head_dim):
    return -(-head_dim // codes_per_word(bits))


def packed_cache_bytes(num_layers, batch, num_kv_heads, head_dim, seq_len,
                       k_bits, v_bits, k_mode, v_mode, k_group, v_group,
                       outliers_per_row=0):
    """Algorithmic bytes of a quantized cache holding ``seq_len`` tokens per
    layer: packed codes + fp16 metadata + CSR outliers (int32 row pointers,
    uint16 columns, fp16 values). Keys in per-channel mode hold floor(S/T)
    quantized blocks plus an fp16 residual of S mod T keys (reading R7).

    Metadata per group: an fp16 scale for symmetric groups (zero point 0,
    [NIAH-q8_0] §1.2); an fp16 scale and an fp16 zero point for asymmetric
    groups ([TurboQuant-3bit] §3.1, [W4A8-FA3] §2.4); an fp16 scale for
    codebook groups, whose levels carry their own signs (reading R20).
    """
    streams = num_layers * batch * num_kv_heads
    total = 0
    for bits, mode, group, is_k in ((k_bits, k_mode, k_group, True),
                                    (v_bits, v_mode, v_group, False)):
        rowb = 4 * words_per_row(bits, head_dim)
        if mode == ASYM_PER_CHANNEL:
            nq = (seq_len // group) * group
            total += streams * (nq * rowb + (nq // group) * head_dim * 4
                                + (seq_len - nq) * head_dim * 2)
            rows = nq
        else:
            meta = 2 if mode in (SYM_PER_TOKEN, CODEBOOK_PER_TOKEN) else 4
            total += streams * seq_len * (rowb + (head_dim // group) * meta)
            rows = seq_len
        if outliers_per_row:
            total += streams * (4 * (rows + 1) + rows * outliers_per_row * 4)
    return total


# ---------------------------------------------------------------------------
# Dense-and-sparse split: per-row top-k outliers
# ---------------------------------------------------------------------------

def select_outliers(rows16, k):
    """Largest-magnitude entries of each row, kept aside in fp16.

    [KVQuant] §2.2 item 3 splits each vector into a dense low-bit part and a
    few full-precision outliers whose count per token is bounded; §3.3 sets
    the ratio near 1 %. Reading R9: exactly ``k`` entries per (token, head)
    row, ranked by |x| descending, ties to the lower channel, stored sorted
    by channel.

    Returns (mask [..., D] bool, cols [..., k] int64 ascending, vals [..., k]
    float16).
    """
    rows16 = np.asarray(rows16, dtype=np.float16)
    shape = rows16.shape
    d = shape[-1]
    flat = rows16.reshape(-1, d)
    mask = np.zeros(flat.shape, dtype=bool)
    if k == 0:
        return (mask.reshape(shape), np.zeros(shape[:-1] + (0,), np.int64),
                np.zeros(shape[:-1] + (0,), np.float16))
    mag = np.abs(flat.astype(np.float32))
    # stable sort on -|x| keeps equal magnitudes in channel order
    order = np.argsort(-mag, axis=1, kind="stable")[:, :k]
    cols = np.sort(order, axis=1)
    np.put_along_axis(mask, cols, True, axis=1)
    vals = np.take_along_axis(flat, cols, axis=1)
    return (mask.reshape(shape), cols.reshape(shape[:-1] + (k,)),
            vals.reshape(shape[:-1] + (k,)))


# ---------------------------------------------------------------------------
# Group quantizers (groups along the LAST axis)
# ---------------------------------------------------------------------------

def quantize_asym(x16, bits, mask=None):
    """Asymmetric min/max quantizer over groups laid along the last axis.

    [TurboQuant-3bit] §3.1: offset = group minimum, code =
    clamp(round((x - offset) / scale), 0, 2^b - 1). Reading R1: scale =
    (max - min) / (2^b - 1). Reading R4/R5: scale and offset are rounded to
    fp16 (RNE) first and the codes are computed from the stored fp16 values,
    in fp32: subtract, IEEE divide, round half to even, clamp. Reading R6: a
    group whose scale is 0 (constant group, or fp16 underflow) gets code 0
    everywhere; a group whose members are all outliers stores scale = zero
    point = 0. Masked (outlier) slots are left out of the statistics and get
    code 0 (reading R10).

    Returns codes (int64, same shape), s16 and z16 (float16, shape[:-1]).
    """
    x16 = np.asarray(x16, dtype=np.float16)
    x = x16.astype(np.float32)
    if mask is None:
        mask = np.zeros(x.shape, dtype=bool)
    live = ~mask
    any_live = live.any(axis=-1)
    mn = np.where(live, x, np.float32(np.inf)).min(axis=-1)
    mx = np.where(live, x, np.float32(-np.inf)).max(axis=-1)
    mn = np.where(any_live, mn, np.float32(0))
    mx = np.where(any_live, mx, np.float32(0))
    # reading R15: zero extremes are taken as +0 (-0 + +0 = +0 under RNE), so
    # the stored zero point and scale never carry a negative zero
    mn = mn + np.float32(0)
    mx = mx + np.float32(0)
    levels = np.float32(2 ** bits - 1)
    s32 = (mx - mn) / levels
    s16 = s32.astype(np.float16)
    z16 = mn.astype(np.float16)
    s = s16.astype(np.float32)[..., None]
    z = z16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint((x - z) / s)
    q = np.where(s > 0, q, np.float32(0))
    q = np.clip(q, 0, 2 ** bits - 1)
    q = np.where(mask, 0, q)
    return q.astype(np.int64), s16, z16


def quantize_sym(x16, bits, mask=None):
    """Symmetric quantizer with zero point 0 over groups along the last axis.

    [NIAH-q8_0] §1.2: the q8_0 cache is int8 with zero point fixed at 0.
    Reading R2: one fp16 scale per group of G channels, scale =
    absmax / (2^(b-1) - 1). Reading R3: codes are clamped to the symmetric
    range [-(2^(b-1) - 1), 2^(b-1) - 1] (inside the int8 range [-128, 127]).
    Codes are computed from the stored fp16 scale in fp32 (IEEE divide,
    round half to even).
    """
    x16 = np.asarray(x16, dtype=np.float16)
    x = x16.astype(np.float32)
    if mask is None:
        mask = np.zeros(x.shape, dtype=bool)
    qmax = 2 ** (bits - 1) - 1
    am = np.where(mask, np.float32(0), np.abs(x)).max(axis=-1)
    s32 = am / np.float32(qmax)
    s16 = s32.astype(np.float16)
    s = s16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(x / s)
    q = np.where(s > 0, q, np.float32(0))
    q = np.clip(q, -qmax, qmax)
    q = np.where(mask, 0, q)
    return q.astype(np.int64), s16


def e2m1_codebook():
    """The 4-bit minifloat code `1 sign | 2 exponent | 1 mantissa`
    ([TurboQuant-3bit] §3.3) as a 16-entry codebook indexed by the code's
    bits s e1 e0 m. Reading R20: exponent bias 1 with e = 0 subnormal, so the
    magnitudes are m/2 for e = 0 and 2^(e-1) (1 + m/2) otherwise: 0, 0.5, 1,
    1.5, 2, 3, 4, 6; the sign bit negates. Every value is exact in fp16."""
    vals = []
    for code in range(16):
        sgn, e, m = code >> 3, (code >> 1) & 3, code & 1
        v = 2.0 ** (e - 1) * (1 + m / 2) if e else m / 2
        vals.append(-v if sgn else v)
    return np.array(vals, np.float16)


def quantize_codebook(x16, codebook16):
    """Codebook (non-uniform) quantizer over groups along the last axis
    ([KVQuant] §2.2 item 2: levels placed where the values are dense;
    [TurboQuant-3bit] §3.3 for the minifloat levels). Reading R20: one fp16
    scale per group, s = absmax / max_i |cb_i| (fp32, stored RNE as fp16);
    y = x / s16 in fp32 (IEEE divide); the code is the index i with the
    smallest |y - cb_i| in fp32, the lowest index on ties; a group whose
    scale is 0 stores code 0 everywhere. x_hat = cb[code] * s16.

    Returns codes (int64, same shape as x16) and s16 (float16, shape[:-1])."""
    x16 = np.asarray(x16, dtype=np.float16)
    x = x16.astype(np.float32)
    cb = np.asarray(codebook16, np.float16).astype(np.float32)
    cbmax = np.float32(np.abs(cb).max())
    am = np.abs(x).max(axis=-1)
    s16 = (am / cbmax).astype(np.float16)
    s = s16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        y = x / s
    d = np.abs(y[..., None] - cb)                       # [..., 16] in fp32
    codes = np.argmin(d, axis=-1)                        # first minimum: lowest index on ties
    codes = np.where(s > 0, codes, 0)
    return codes.astype(np.int64), s16


# ---------------------------------------------------------------------------
# Bit packing along a (token, head) row
# ---------------------------------------------------------------------------

def pack_row_codes(codes, bits):
    """Pack integer codes laid along the last axis into uint32 words.

    Code j of a row goes to word j // cpw at bit offset (j % cpw) * b, with
    cpw = 32/b for b in {4, 8} and cpw = 10 for b = 3 (ten codes per word,
    the top two bits zero). Signed codes are stored as b-bit two's
    complement. Rows shorter than a whole word leave the unused bits zero.
    """
    codes = np.asarray(codes, dtype=np.int64)
    cpw = codes_per_word(bits)
    d = codes.shape[-1]
    nw = -(-d // cpw)
    padded = np.zeros(codes.shape[:-1] + (nw * cpw,), dtype=np.uint64)
    padded[..., :d] = (codes & ((1 << bits) - 1)).astype(np.uint64)
    padded = padded.reshape(codes.shape[:-1] + (nw, cpw))
    shifts = (np.arange(cpw, dtype=np.uint64) * np.uint64(bits))
    words = (padded << shifts).sum(axis=-1)
    return words.astype(np.uint32)


def unpack_row_codes(words, bits, head_dim, signed=False):
    """Inverse of :func:`pack_row_codes`."""
    words = np.asarray(words, dtype=np.uint32).astype(np.uint64)
    cpw = codes_per_word(bits)
    shifts = np.arange(cpw, dtype=np.uint64) * np.uint64(bits)
    c = (words[..., None] >> shifts) & np.uint64((1 << bits) - 1)
    c = c.reshape(words.shape[:-1] + (-1,))[..., :head_dim].astype(np.int64)
    if signed:
        c = np.where(c >= (1 << (bits - 1)), c - (1 << bits), c)
    return c


# ---------------------------------------------------------------------------
# Cache state for a batch of independent (batch, kv-head) streams
# ---------------------------------------------------------------------------

@dataclass
class CodecSpec:
    head_dim: int
    k_bits: int
    v_bits: int
    k_mode: int
    v_mode: int
    k_group: int
    v_group: int
    outliers_per_row: int = 0
    sink_tokens: int = 0
    codebook: tuple = None  # 16 fp16 values for CODEBOOK_PER_TOKEN tensors


class TensorState:
    """Quantized rows of one tensor (K or V) for N streams.

    codes: int64 [N][R][D]; scale16/zero16: float16 metadata, per token
    [N][R][D/G] or per channel block [N][R/T][D]; out_cols/out_vals:
    [N][R][k]; resid: float16 [N][r][D] keys awaiting a full block.

    Rows arrive in pieces (a prefill, then one token per append); the pieces
    are kept in lists and joined along the row axis when an array is read, so
    that an append costs the size of its own rows (a data structure only:
    the arrays read back are exactly the concatenation of what was added).
    """

    _FIELDS = ("codes", "scale16", "zero16", "out_cols", "out_vals")

    def __init__(self, codes, scale16, zero16, out_cols, out_vals, resid=None):
        self._parts = {f: [] for f in self._FIELDS}
        self._joined = {}
        self._has_zero = zero16 is not None
        self.add(codes=codes, scale16=scale16, zero16=zero16, out_cols=out_cols, out_vals=out_vals)
        self.resid = resid

    def add(self, **rows):
        for f, a in rows.items():
            if a is None:
                continue
            self._parts[f].append(np.asarray(a))
            self._joined.pop(f, None)

    def _get(self, f):
        if f == "zero16" and not self._has_zero:
            return None
        if f not in self._joined:
            parts = self._parts[f]
            self._joined[f] = parts[0] if len(parts) == 1 else np.concatenate(parts, axis=1)
            self._parts[f] = [self._joined[f]]
        return self._joined[f]

    codes = property(lambda self: self._get("codes"))
    scale16 = property(lambda self: self._get("scale16"))
    zero16 = property(lambda self: self._get("zero16"))
    out_cols = property(lambda self: self._get("out_cols"))
    out_vals = property(lambda self: self._get("out_vals"))


def _quantize_rows_per_token(x16, bits, mode, group, k_out, codebook=None):
    n, r, d = x16.shape
    mask, cols, vals = select_outliers(x16, k_out)
    xg = x16.reshape(n, r, d // group, group)
    mg = mask.reshape(n, r, d // group, group)
    if mode == SYM_PER_TOKEN:
        c, s16 = quantize_sym(xg, bits, mg)
        z16 = None
    elif mode == CODEBOOK_PER_TOKEN:
        assert k_out == 0 and codebook is not None
        c, s16 = quantize_codebook(xg, codebook)
        z16 = None
    else:
        c, s16, z16 = quantize_asym(xg, bits, mg)
    return c.reshape(n, r, d), s16, z16, cols, vals


def _quantize_blocks_per_channel(x16, bits, block, k_out):
    """Keys grouped per channel over ``block`` consecutive tokens
    ([KVQuant] §2.2 item 1: per-channel key quantization; [W4A8-FA3] §2.4:
    per-head groups of 64 positions, each with its own scale and zero point).
    x16: [N][nb*T][D]."""
    n, r, d = x16.shape
    nb = r // block
    mask, cols, vals = select_outliers(x16, k_out)
    xt = x16.reshape(n, nb, block, d).transpose(0, 1, 3, 2)      # [N][nb][D][T]
    mt = mask.reshape(n, nb, block, d).transpose(0, 1, 3, 2)
    c, s16, z16 = quantize_asym(xt, bits, mt)                     # s16: [N][nb][D]
    c = c.transpose(0, 1, 3, 2).reshape(n, r, d)
    return c, s16, z16, cols, vals


class OracleCache:
    """Quantized KV cache of N independent streams (one per (batch, kv-head))
    of one layer, built by the same steps the pages describe for a decode
    loop ([KVQuant] §3.4: quantize the new key/value, store codes plus fp16
    outliers, dequantize on read and attend).

    Keys in per-channel mode (reading R7): a prefill of S tokens quantizes
    floor(S/T) whole blocks and keeps the last S mod T keys in fp16; appended
    keys join that fp16 residual and a block is quantized once it holds T
    keys; codes already written are never requantized. Values (and keys in
    per-token modes) are quantized row by row as they arrive ([NIAH-q8_0]
    §2.2: only the newly written row is quantized).

    Attention sinks ([KVQuant] §4.1: the first 5-10 tokens keep full
    precision; reading R18): the first ``spec.sink_tokens`` tokens of every
    stream keep their fp16 keys and values, take part in attention as they
    are, and are never quantized; quantization, and the per-channel key
    blocks, start at the token after them.
    """

    def __init__(self, spec: CodecSpec, n_streams: int):
        self.spec = spec
        self.n = n_streams
        self.length = 0
        self.k = None
        self.v = None
        d = spec.head_dim
        self.sink_k = np.zeros((n_streams, 0, d), np.float16)
        self.sink_v = np.zeros((n_streams, 0, d), np.float16)

    @property
    def coded_length(self):
        """Tokens after the sinks (the quantized rows and the key residual)."""
        return self.length - self.sink_k.shape[1]

    # -- helpers --------------------------------------------------------
    def _empty_state(self, bits, mode, group):
        d = self.spec.head_dim
        n = self.n
        ko = self.spec.outliers_per_row
        if mode == ASYM_PER_CHANNEL:
            meta_shape = (n, 0, d)
        else:
            meta_shape = (n, 0, d // group)
        return TensorState(
            codes=np.zeros((n, 0, d), np.int64),
            scale16=np.zeros(meta_shape, np.float16),
            zero16=None if mode in (SYM_PER_TOKEN, CODEBOOK_PER_TOKEN) else np.zeros(meta_shape, np.float16),
            out_cols=np.zeros((n, 0, ko), np.int64),
            out_vals=np.zeros((n, 0, ko), np.float16),
            resid=np.zeros((n, 0, d), np.float16) if mode == ASYM_PER_CHANNEL else None)

    def _append_rows(self, st, x16, bits, mode, group):
        ko = self.spec.outliers_per_row
        if mode == ASYM_PER_CHANNEL:
            pend = np.concatenate([st.resid, x16], axis=1)
            nfull = (pend.shape[1] // group) * group
            if nfull:
                c, s16, z16, cols, vals = _quantize_blocks_per_channel(
                    pend[:, :nfull], bits, group, ko)
                st.add(codes=c, scale16=s16, zero16=z16, out_cols=cols, out_vals=vals)
            st.resid = pend[:, nfull:].copy()
        else:
            c, s16, z16, cols, vals = _quantize_rows_per_token(x16, bits, mode, group, ko, self.spec.codebook)
            st.add(codes=c, scale16=s16, zero16=z16, out_cols=cols, out_vals=vals)

    # -- the decode-loop steps -------------------------------------------
    def prefill(self, k16, v16):
        """Quantize a whole prompt: k16, v16 float16 [N][S][D]."""
        sp = self.spec
        k16 = np.asarray(k16, np.float16)
        v16 = np.asarray(v16, np.float16)
        assert k16.shape == v16.shape and k16.shape[0] == self.n
        assert k16.shape[2] == sp.head_dim
        self.k = self._empty_state(sp.k_bits, sp.k_mode, sp.k_group)
        self.v = self._empty_state(sp.v_bits, sp.v_mode, sp.v_group)
        ns = min(k16.shape[1], sp.sink_tokens)
        self.sink_k = k16[:, :ns].copy()
        self.sink_v = v16[:, :ns].copy()
        self._append_rows(self.k, k16[:, ns:], sp.k_bits, sp.k_mode, sp.k_group)
        self._append_rows(self.v, v16[:, ns:], sp.v_bits, sp.v_mode, sp.v_group)
        self.length = k16.shape[1]

    def append(self, k1, v1):
        """Quantize one new token per stream: k1, v1 float16 [N][D]."""
        sp = self.spec
        if self.k is None:
            self.k = self._empty_state(sp.k_bits, sp.k_mode, sp.k_group)
            self.v = self._empty_state(sp.v_bits, sp.v_mode, sp.v_group)
        k1 = np.asarray(k1, np.float16)[:, None, :]
        v1 = np.asarray(v1, np.float16)[:, None, :]
        if self.length < sp.sink_tokens:
            self.sink_k = np.concatenate([self.sink_k, k1], axis=1)
            self.sink_v = np.concatenate([self.sink_v, v1], axis=1)
        else:
            self._append_rows(self.k, k1, sp.k_bits, sp.k_mode, sp.k_group)
            self._append_rows(self.v, v1, sp.v_bits, sp.v_mode, sp.v_group)
        self.length += 1

    # -- dequantization (fp64) --------------------------------------------
    def _dequant(self, st, mode, group):
        """x_hat = z16 + c * s16 (asymmetric), c * s16 (symmetric) or
        cb[c] * s16 (codebook), exact in fp64; outlier slots take their stored fp16 value (reading R10);
        fp16 residual keys are used as they are."""
        d = self.spec.head_dim
        c = st.codes.astype(np.float64)
        n, r, _ = c.shape
        if mode == ASYM_PER_CHANNEL:
            s = np.repeat(st.scale16.astype(np.float64), group, axis=1)
            z = np.repeat(st.zero16.astype(np.float64), group, axis=1)
            xh = z + c * s
        else:
            s = np.repeat(st.scale16.astype(np.float64), group, axis=2)
            if mode == CODEBOOK_PER_TOKEN:  # the code indexes the codebook (reading R20)
                c = np.asarray(self.spec.codebook, np.float16).astype(np.float64)[st.codes]
            xh = c * s
            if mode == ASYM_PER_TOKEN:
                xh = np.repeat(st.zero16.astype(np.float64), group, axis=2) + xh
        if st.out_cols.shape[-1]:
            np.put_along_axis(xh, st.out_cols, st.out_vals.astype(np.float64), axis=2)
        if st.resid is not None and st.resid.shape[1]:
            xh = np.concatenate([xh, st.resid.astype(np.float64)], axis=1)
        assert xh.shape == (n, self.coded_length, d)
        return xh

    def dequant_k(self):
        """Every cached key in fp64: the fp16 sinks, then the dequantized rows."""
        return np.concatenate([self.sink_k.astype(np.float64),
                               self._dequant(self.k, self.spec.k_mode, self.spec.k_group)], axis=1)

    def dequant_v(self):
        return np.concatenate([self.sink_v.astype(np.float64),
                               self._dequant(self.v, self.spec.v_mode, self.spec.v_group)], axis=1)

    def decode(self, q, softmax_scale):
        """Decode attention of q [N][g][D] (g query heads per KV stream)
        over every cached token of each stream, on the dequantized cache."""
        if self.length == 0:
            raise ValueError("attention over an empty cache is undefined")
        return attend(q, self.dequant_k(), self.dequant_v(), softmax_scale)

    def prefill_attention(self, q, softmax_scale):
        """Prefill attention over the quantized cache (reading R22): q is
        [N][C][g][D], the queries of the last C cached positions of every
        stream; query i sits at position length - C + i and attends the
        dequantized tokens 0 .. length - C + i."""
        q = np.asarray(q, dtype=np.float64)
        c = q.shape[1]
        if not 0 < c <= self.length:
            raise ValueError("the chunk must hold 1 .. length queries")
        positions = np.arange(self.length - c, self.length)
        return causal_attend(q, self.dequant_k(), self.dequant_v(), positions, softmax_scale)

    # -- packed views in the storage format --------------------------------
    def k_words(self):
        return pack_row_codes(self.k.codes, self.spec.k_bits)

    def v_words(self):
        return pack_row_codes(self.v.codes, self.spec.v_bits)

    @staticmethod
    def csr(st):
        """(row_ptr int32 [R+1], col uint16 [nnz], val float16 [nnz]) for
        every stream, as arrays with a leading stream axis."""
        n, r, k = st.out_cols.shape
        row_ptr = np.broadcast_to((np.arange(r + 1) * k).astype(np.int32), (n, r + 1))
        return (np.ascontiguousarray(row_ptr),
                st.out_cols.reshape(n, r * k).astype(np.uint16),
                st.out_vals.reshape(n, r * k))


# ---------------------------------------------------------------------------
# Attention (fp64)
# ---------------------------------------------------------------------------

def attend(q, k_hat, v_hat, softmax_scale):
    """Single-token softmax attention per KV stream, in fp64.

    q: [N][g][D]; k_hat, v_hat: [N][S][D]. For each query head,
    e_t = scale * <q, k_t>, p = softmax(e) (shifted by max e), o = sum_t p_t v_t
    ([KVQuant] §3.4 step 3: attention on the dequantized cache; reading R14
    maps query head h to KV head h // (H_q / H_kv)).
    """
    q = np.asarray(q, dtype=np.float64)
    k_hat = np.asarray(k_hat, dtype=np.float64)
    v_hat = np.asarray(v_hat, dtype=np.float64)
    e = np.einsum("ngd,nsd->ngs", q, k_hat) * float(softmax_scale)
    e = e - e.max(axis=-1, keepdims=True)
    p = np.exp(e)
    p /= p.sum(axis=-1, keepdims=True)
    return np.einsum("ngs,nsd->ngd", p, v_hat)


def causal_attend(q, k_hat, v_hat, positions, softmax_scale):
    """Causal attention of a chunk of queries over a cache, in fp64 (reading
    R22; the prefill of [NIAH-q8_0] §4.2, whose time to first token the
    chunked queries make up). q: [N][C][g][D]; k_hat, v_hat: [N][S][D];
    positions: [C] cache positions of the queries. Query i attends tokens
    0 .. positions[i] (its own token included) exactly as `attend` attends a
    whole cache. Returns [N][C][g][D]."""
    q = np.asarray(q, dtype=np.float64)
    out = np.empty(q.shape, dtype=np.float64)
    for i, p in enumerate(np.asarray(positions)):
        out[:, i] = attend(q[:, i], k_hat[:, :int(p) + 1], v_hat[:, :int(p) + 1], softmax_scale)
    return out


def row_relative_error(o, o_ref):
    """Per-row error: max_d |o - o_ref| / max_d |o_ref| (reading R13)."""
    o = np.asarray(o, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    num = np.abs(o - o_ref).max(axis=-1)
    den = np.maximum(np.abs(o_ref).max(axis=-1), 1e-30)
    return num / den

