"""Group-wise low-bit KV cache with fused dequant decode attention on GB300.

A thin ctypes binding over ``libkvq.so`` (C ABI in ``include/kvq.h``). The
binding only marshals arguments: every step of quantization and attention
runs in the library's CUDA kernels. PyTorch provides device memory and
streams. There is no CPU fallback: if the library is missing the import of
:func:`lib` raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import workloads as _W

__all__ = [
    "KVQError", "QuantizedKVCache", "lib", "library_path",
    "SYM_PER_TOKEN", "ASYM_PER_TOKEN", "ASYM_PER_CHANNEL", "CODEBOOK_PER_TOKEN", "F32", "F16",
    "E2M1_LEVELS",
]

SYM_PER_TOKEN = 0
ASYM_PER_TOKEN = 1
ASYM_PER_CHANNEL = 2
CODEBOOK_PER_TOKEN = 3
F32 = 0
F16 = 1

# The 4-bit minifloat `1 sign | 2 exponent | 1 mantissa` as codebook levels.
E2M1_LEVELS = _W.E2M1

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libkvq.so")

STATUS_NAMES = {
    0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_UNSUPPORTED",
    3: "KVQ_ERR_BUFFER_TOO_SMALL", 4: "KVQ_ERR_CAPACITY", 5: "KVQ_ERR_CUDA",
    6: "KVQ_ERR_TIMEOUT", 7: "KVQ_ERR_DEVICE_STATUS",
}


class KVQError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, str(status)), message))


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "batch", "num_kv_heads", "head_dim", "max_seq", "k_bits", "v_bits",
        "k_mode", "v_mode", "k_group", "v_group", "outliers_per_row")] + [
        ("codebook", ctypes.c_uint16 * 16), ("sink_tokens", ctypes.c_int32)]


class Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "capacity", "length", "k_quantized_len", "k_resid_len", "k_words_per_row",
        "v_words_per_row", "k_meta_entry_bytes", "v_meta_entry_bytes")] + [
        (n, ctypes.c_int64) for n in (
            "k_codes_stream_bytes", "v_codes_stream_bytes", "k_meta_stream_bytes",
            "v_meta_stream_bytes", "k_resid_stream_bytes", "out_rowptr_stream_bytes",
            "out_col_stream_bytes", "out_val_stream_bytes")] + [
        (n, ctypes.c_void_p) for n in (
            "k_codes", "k_meta", "k_resid", "v_codes", "v_meta", "k_out_rowptr", "k_out_col",
            "k_out_val", "v_out_rowptr", "v_out_col", "v_out_val")] + [
        ("sink_tokens", ctypes.c_int32), ("sink_len", ctypes.c_int32), ("sink_stream_bytes", ctypes.c_int64),
        ("k_sink", ctypes.c_void_p), ("v_sink", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_SIGNATURES = {
    "kvq_cache_bytes": [ctypes.POINTER(Config), ctypes.POINTER(ctypes.c_size_t)],
    "kvq_cache_create": [ctypes.POINTER(Config), _P, ctypes.c_size_t, _P, ctypes.POINTER(_P)],
    "kvq_cache_bytes_per_layer": [ctypes.POINTER(Config), ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_size_t)],
    "kvq_cache_create_per_layer": [ctypes.POINTER(Config), ctypes.POINTER(_I), _P, ctypes.c_size_t, _P,
                                   ctypes.POINTER(_P)],
    "kvq_cache_destroy": [_P],
    "kvq_prefill_quantize": [_P, _I, _P, _P, _I, _P],
    "kvq_append_quantize": [_P, _I, _P, _P, _P],
    "kvq_decode_workspace_bytes": [_P, _I, ctypes.POINTER(ctypes.c_size_t)],
    "kvq_decode_attention": [_P, _I, _P, _I, ctypes.c_float, _P, _I, _P, ctypes.c_size_t, _P],
    "kvq_decode_attention_static": [_P, _I, _P, _I, ctypes.c_float, _P, _I, _P],
    "kvq_cache_set_decode_splits": [_P, _I],
    "kvq_decode_step": [_P, ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P), _I, ctypes.c_float,
                        ctypes.POINTER(_P), _I, _P, ctypes.c_size_t, _P, _P],
    "kvq_cache_get_layout": [_P, _I, ctypes.POINTER(Layout)],
    "kvq_cache_length": [_P, _I, ctypes.POINTER(_I)],
    "kvq_prefill_quantize_varlen": [_P, _I, _P, _P, _I, ctypes.POINTER(_I), _P],
    "kvq_cache_seq_lengths": [_P, _I, ctypes.POINTER(_I)],
    "kvq_cache_status": [_P, _P, ctypes.POINTER(ctypes.c_uint32)],
    "kvq_selftest_div_levels": [_I, ctypes.c_uint32, ctypes.c_uint32, _P, _P],
    "kvq_selftest_code_rounding": [_I, _I, _I, _I, _P, _P],
    "kvq_selftest_codebook_quotient": [_P, _P],
    "kvq_prefill_attention": [_P, _I, _P, _I, _I, ctypes.c_float, _P, _I, _P],
    "kvq_selftest_wait_timeout": [_P, _I, _P],
}

_lib = None


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise ImportError("libkvq.so is not built (run __graft_entry__.build()); "
                              "there is no fallback implementation")
        L = ctypes.CDLL(library_path)
        for name, args in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.kvq_last_error.argtypes = []
        L.kvq_last_error.restype = ctypes.c_char_p
        L.kvq_version.argtypes = []
        L.kvq_version.restype = ctypes.c_int32
        L.kvq_kernel_launches.argtypes = []
        L.kvq_kernel_launches.restype = ctypes.c_uint64
        _lib = L
    return _lib


def _selftest_result(run, device):
    res = torch.empty(2, dtype=torch.int64, device=device)
    check(run(ctypes.c_void_p(res.data_ptr())))
    mism, first = (int(x) & 0xFFFFFFFFFFFFFFFF for x in res.cpu().tolist())
    return mism, first


def selftest_div_levels(levels, a_first, a_last, device="cuda", stream=None):
    """(mismatches, smallest mismatching fp32 bit pattern or 2^64 - 1) of the
    prefill's scale division against IEEE division (kvq_selftest.h)."""
    return _selftest_result(lambda r: lib().kvq_selftest_div_levels(levels, a_first, a_last, r,
                                                                    _stream_ptr(stream)), device)


def selftest_code_rounding(method, k_first, k_last, ulps, device="cuda", stream=None):
    """(mismatches, smallest mismatching input key or 2^64 - 1) of the code
    rounding near ties against IEEE division (kvq_selftest.h)."""
    return _selftest_result(lambda r: lib().kvq_selftest_code_rounding(method, k_first, k_last, ulps, r,
                                                                       _stream_ptr(stream)), device)


def selftest_codebook_quotient(device="cuda", stream=None):
    """(mismatches, smallest mismatching (s bits << 16 | x bits) or 2^64 - 1)
    of the codebook quantizer's division-free quotient against IEEE
    division over every finite fp16 x and positive finite fp16 s."""
    return _selftest_result(lambda r: lib().kvq_selftest_codebook_quotient(r, _stream_ptr(stream)), device)


def kernel_launches() -> int:
    """Device kernels this process has enqueued through the library."""
    return int(lib().kvq_kernel_launches())


def check(status):
    if status != 0:
        raise KVQError(status, lib().kvq_last_error().decode(errors="replace"))


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_config(num_layers, batch, num_kv_heads, head_dim, max_seq, k_bits, v_bits, k_mode,
                v_mode, k_group, v_group, outliers_per_row=0, sink_tokens=0, codebook=None):
    """codebook: 16 levels (floats, stored as fp16) for CODEBOOK_PER_TOKEN tensors."""
    cb = (ctypes.c_uint16 * 16)()
    if codebook is not None:
        bits = torch.tensor([float(x) for x in codebook], dtype=torch.float16).view(torch.int16)
        if bits.numel() != 16:
            raise ValueError("a codebook has 16 levels")
        for i, b in enumerate(bits.tolist()):
            cb[i] = b & 0xFFFF
    return Config(num_layers, batch, num_kv_heads, head_dim, max_seq, k_bits, v_bits, k_mode,
                  v_mode, k_group, v_group, outliers_per_row, cb, sink_tokens)


def cache_bytes(cfg: Config) -> int:
    n = ctypes.c_size_t()
    check(lib().kvq_cache_bytes(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def _check_half(t, shape, name):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float16 or not t.is_cuda:
        raise TypeError("%s must be a CUDA float16 tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))


class QuantizedKVCache:
    """A packed KV cache of ``num_layers`` layers in one torch-owned device
    buffer, driven through the C ABI."""

    def __init__(self, num_layers, batch, num_kv_heads, head_dim, max_seq, k_bits, v_bits,
                 k_mode, v_mode, k_group, v_group, outliers_per_row=0, device=None,
                 stream=None, layer_bits=None, sink_tokens=0, codebook=None):
        """layer_bits: None, or one (k_bits, v_bits) pair per layer overriding
        k_bits / v_bits (kvq_cache_create_per_layer)."""
        self.cfg = make_config(num_layers, batch, num_kv_heads, head_dim, max_seq, k_bits,
                               v_bits, k_mode, v_mode, k_group, v_group, outliers_per_row, sink_tokens,
                               codebook)
        self.layer_bits = None
        lb = None
        if layer_bits is not None:
            pairs = [tuple(int(b) for b in p) for p in layer_bits]
            if len(pairs) != num_layers or any(len(p) != 2 for p in pairs):
                raise ValueError("layer_bits needs one (k_bits, v_bits) pair per layer")
            self.layer_bits = pairs
            lb = (_I * (2 * num_layers))(*[b for p in pairs for b in p])
        n = ctypes.c_size_t()
        check(lib().kvq_cache_bytes_per_layer(ctypes.byref(self.cfg), lb, ctypes.byref(n)))
        self.nbytes = n.value
        self.device = torch.device(device if device is not None else "cuda")
        self.buffer = torch.empty(self.nbytes, dtype=torch.uint8, device=self.device)
        h = ctypes.c_void_p()
        check(lib().kvq_cache_create_per_layer(ctypes.byref(self.cfg), lb, ctypes.c_void_p(self.buffer.data_ptr()),
                                               self.nbytes, _stream_ptr(stream), ctypes.byref(h)))
        self.handle = h
        self._ws = {}

    # -- hot path -----------------------------------------------------------
    def prefill(self, layer, k, v, stream=None):
        c = self.cfg
        s = k.shape[2] if k.dim() == 4 else 0
        _check_half(k, (c.batch, c.num_kv_heads, s, c.head_dim), "k")
        _check_half(v, (c.batch, c.num_kv_heads, s, c.head_dim), "v")
        check(lib().kvq_prefill_quantize(self.handle, layer, ctypes.c_void_p(k.data_ptr()),
                                         ctypes.c_void_p(v.data_ptr()), s, _stream_ptr(stream)))

    def prefill_varlen(self, layer, k, v, lens, stream=None):
        """Prefill from a padded batch in which batch row b holds lens[b] of
        the k.shape[2] rows (kvq_prefill_quantize_varlen); later appends and
        decodes of the layer use each row's own length."""
        c = self.cfg
        s = k.shape[2] if k.dim() == 4 else 0
        _check_half(k, (c.batch, c.num_kv_heads, s, c.head_dim), "k")
        _check_half(v, (c.batch, c.num_kv_heads, s, c.head_dim), "v")
        if len(lens) != c.batch:
            raise ValueError("one length per batch row")
        arr = (ctypes.c_int32 * c.batch)(*[int(x) for x in lens])
        check(lib().kvq_prefill_quantize_varlen(self.handle, layer, ctypes.c_void_p(k.data_ptr()),
                                                ctypes.c_void_p(v.data_ptr()), s, arr, _stream_ptr(stream)))

    def seq_lengths(self, layer):
        arr = (ctypes.c_int32 * self.cfg.batch)()
        check(lib().kvq_cache_seq_lengths(self.handle, layer, arr))
        return list(arr)

    def append(self, layer, k1, v1, stream=None):
        c = self.cfg
        _check_half(k1, (c.batch, c.num_kv_heads, c.head_dim), "k1")
        _check_half(v1, (c.batch, c.num_kv_heads, c.head_dim), "v1")
        check(lib().kvq_append_quantize(self.handle, layer, ctypes.c_void_p(k1.data_ptr()),
                                        ctypes.c_void_p(v1.data_ptr()), _stream_ptr(stream)))

    def workspace_bytes(self, num_q_heads):
        n = ctypes.c_size_t()
        check(lib().kvq_decode_workspace_bytes(self.handle, num_q_heads, ctypes.byref(n)))
        return n.value

    def workspace(self, num_q_heads):
        ws = self._ws.get(num_q_heads)
        if ws is None:
            ws = torch.empty(self.workspace_bytes(num_q_heads), dtype=torch.uint8, device=self.device)
            self._ws[num_q_heads] = ws
        return ws

    def decode(self, layer, q, softmax_scale, out=None, out_dtype=torch.float32, workspace=None,
               stream=None):
        c = self.cfg
        hq = q.shape[1]
        _check_half(q, (c.batch, hq, c.head_dim), "q")
        if out is None:
            out = torch.empty((c.batch, hq, c.head_dim), dtype=out_dtype, device=q.device)
        code = {torch.float32: F32, torch.float16: F16}[out.dtype]
        ws = self.workspace(hq) if workspace is None else workspace
        check(lib().kvq_decode_attention(self.handle, layer, ctypes.c_void_p(q.data_ptr()), hq,
                                         float(softmax_scale), ctypes.c_void_p(out.data_ptr()),
                                         code, ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                         _stream_ptr(stream)))
        return out

    def decode_static(self, layer, q, softmax_scale, out=None, out_dtype=torch.float32,
                      stream=None):
        """decode() without a workspace: the split scratch is the library's own
        device array (for callers that cannot allocate; see kvq.h)."""
        c = self.cfg
        hq = q.shape[1]
        _check_half(q, (c.batch, hq, c.head_dim), "q")
        if out is None:
            out = torch.empty((c.batch, hq, c.head_dim), dtype=out_dtype, device=q.device)
        code = {torch.float32: F32, torch.float16: F16}[out.dtype]
        check(lib().kvq_decode_attention_static(self.handle, layer, ctypes.c_void_p(q.data_ptr()),
                                                hq, float(softmax_scale),
                                                ctypes.c_void_p(out.data_ptr()), code,
                                                _stream_ptr(stream)))
        return out

    def prefill_attention(self, layer, q, softmax_scale, out=None, out_dtype=torch.float32, stream=None):
        """Causal attention of the queries of the layer's last q.shape[1]
        positions over the cache (kvq_prefill_attention): q fp16
        [B][chunk][H_q][D] -> out [B][chunk][H_q][D]."""
        c = self.cfg
        if q.dim() != 4:
            raise ValueError("q must be [batch][chunk][query heads][head_dim]")
        chunk, hq = q.shape[1], q.shape[2]
        _check_half(q, (c.batch, chunk, hq, c.head_dim), "q")
        if out is None:
            out = torch.empty((c.batch, chunk, hq, c.head_dim), dtype=out_dtype, device=q.device)
        code = {torch.float32: F32, torch.float16: F16}[out.dtype]
        check(lib().kvq_prefill_attention(self.handle, layer, ctypes.c_void_p(q.data_ptr()), chunk, hq,
                                          float(softmax_scale), ctypes.c_void_p(out.data_ptr()), code,
                                          _stream_ptr(stream)))
        return out

    def decode_step(self, qs, k1s, v1s, softmax_scale, outs, workspace=None, stream=None, aux_stream=None):
        """Append one token and decode on every layer (kvq_decode_step): qs,
        k1s, v1s, outs are per-layer tensors; with aux_stream the appends run
        there, overlapping the decodes of earlier layers."""
        c = self.cfg
        nl = c.num_layers
        if not (len(qs) == len(k1s) == len(v1s) == len(outs) == nl):
            raise ValueError("one q, k1, v1 and out per layer")
        hq = qs[0].shape[1]
        for l in range(nl):
            _check_half(qs[l], (c.batch, hq, c.head_dim), "q")
            _check_half(k1s[l], (c.batch, c.num_kv_heads, c.head_dim), "k1")
            _check_half(v1s[l], (c.batch, c.num_kv_heads, c.head_dim), "v1")
        code = {torch.float32: F32, torch.float16: F16}[outs[0].dtype]
        ws = self.workspace(hq) if workspace is None else workspace
        arr = lambda ts: (_P * nl)(*[t.data_ptr() for t in ts])
        check(lib().kvq_decode_step(self.handle, arr(qs), arr(k1s), arr(v1s), hq, float(softmax_scale), arr(outs),
                                    code, ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream_ptr(stream),
                                    ctypes.c_void_p(aux_stream.cuda_stream) if aux_stream is not None else None))

    # -- inspection ---------------------------------------------------------
    def set_decode_splits(self, splits):
        check(lib().kvq_cache_set_decode_splits(self.handle, splits))

    def length(self, layer):
        n = ctypes.c_int32()
        check(lib().kvq_cache_length(self.handle, layer, ctypes.byref(n)))
        return n.value

    def layout(self, layer):
        lo = Layout()
        check(lib().kvq_cache_get_layout(self.handle, layer, ctypes.byref(lo)))
        return lo

    def status(self, stream=None):
        w = ctypes.c_uint32()
        check(lib().kvq_cache_status(self.handle, _stream_ptr(stream), ctypes.byref(w)))
        return w.value

    def selftest_wait_timeout(self, polls, stream=None):
        """Runs the bounded-wait self-test on this cache (kvq_selftest.h)."""
        check(lib().kvq_selftest_wait_timeout(self.handle, polls, _stream_ptr(stream)))

    def view(self, ptr, nbytes, dtype):
        """A tensor view of ``nbytes`` of the cache buffer starting at device
        pointer ``ptr`` (for inspection and checkpoints)."""
        off = int(ptr) - self.buffer.data_ptr()
        if off < 0 or off + nbytes > self.nbytes:
            raise ValueError("pointer outside the cache buffer")
        return self.buffer[off:off + nbytes].view(dtype)

    def close(self):
        if getattr(self, "handle", None):
            lib().kvq_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
