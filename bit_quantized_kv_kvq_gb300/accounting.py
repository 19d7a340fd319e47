"""Algorithmic byte counts of each hot-path step (the roofline numerators).

Decode reads every cached token once: packed codes, fp16 scale/zero per
group, CSR outliers (int32 row pointer, uint16 column, fp16 value), fp16
residual keys, plus the fp16 query; it writes the fp32 output. Prefill reads
the fp16 K and V and writes the packed cache. Append reads one fp16 K/V row
per stream and writes one packed value row (and one fp16 residual key row or
packed key row; a full key block of codes when the residual fills).
Split-K partials are workspace traffic, not algorithmic bytes.
"""
from __future__ import annotations

from dataclasses import replace

from .workloads import ASYM_PER_CHANNEL, CODEBOOK_PER_TOKEN, SYM_PER_TOKEN


def _cpw(bits):
    return 10 if bits == 3 else 32 // bits


def row_bytes(bits, head_dim=128):
    return 4 * (-(-head_dim // _cpw(bits)))


def meta_entry_bytes(mode):
    """fp16 scale (symmetric and codebook groups) or fp16 scale + zero point."""
    return 2 if mode in (SYM_PER_TOKEN, CODEBOOK_PER_TOKEN) else 4


def cache_read_bytes(wl, length):
    """Packed bytes of one layer holding ``length`` tokens per stream."""
    n = wl.batch * wl.num_kv_heads
    d = wl.head_dim
    k = wl.outliers_per_row
    total = 0
    for bits, mode, group, is_k in ((wl.k_bits, wl.k_mode, wl.k_group, True),
                                    (wl.v_bits, wl.v_mode, wl.v_group, False)):
        if mode == ASYM_PER_CHANNEL:
            nq = length // group * group
            total += n * (nq * row_bytes(bits, d) + (nq // group) * d * 4 + (length - nq) * d * 2)
            rows = nq
        else:
            total += n * length * (row_bytes(bits, d) + (d // group) * meta_entry_bytes(mode))
            rows = length
        if k:
            total += n * (4 * (rows + 1) + rows * k * 4)
    return total


def row_lengths(wl, length):
    """Tokens of each batch row when the longest holds `length` (a ragged
    batch's rows all grow by one token per append)."""
    if not wl.lens:
        return [length] * wl.batch
    return [x + length - max(wl.lens) for x in wl.lens]


def decode_bytes(wl, length):
    """One decode over every batch row's own tokens (the longest: `length`)."""
    if wl.lens:
        one = replace(wl, batch=1, lens=None)
        cache = sum(cache_read_bytes(one, n) for n in row_lengths(wl, length))
    else:
        cache = cache_read_bytes(wl, length)
    return cache + wl.batch * wl.num_q_heads * wl.head_dim * 2 + wl.batch * wl.num_q_heads * wl.head_dim * 4


def prefill_bytes(wl, length):
    return 2 * wl.batch * wl.num_kv_heads * length * wl.head_dim * 2 + cache_read_bytes(wl, length)


def append_bytes(wl, length_before):
    """One appended token per stream (flushes a key block when it fills)."""
    return (2 * wl.batch * wl.num_kv_heads * wl.head_dim * 2
            + cache_read_bytes(wl, length_before + 1) - cache_read_bytes(wl, length_before))
