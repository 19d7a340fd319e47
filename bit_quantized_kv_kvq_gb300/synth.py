"""Seeded synthetic inputs (fp16 Q, K, V) shared by the CUDA path and the
oracle.

This module draws numbers and nothing else: it holds none of the codec's or
the attention's arithmetic. Both sides read the same generated fp16 bytes.

Distributions (all seeded with ``torch.Generator``; values are clamped to
+-60000 before the fp16 cast so every input is finite):

* ``normal``: K, V, Q ~ N(0, 1).
* ``k_lognormal_channels``: K = N(0, 1) * sigma_c with one sigma_c =
  exp(0.5 * N(0, 1)) per (layer, kv-head, channel); V, Q ~ N(0, 1).
* ``k_heavy15``: K ~ N(0, 1) with 4 channels per (layer, kv-head), chosen
  by the seeded generator, multiplied by 15; V, Q ~ N(0, 1).
* ``t3_heavy20``: K and V ~ Student-t with 3 degrees of freedom
  (Z / sqrt(chi2_3 / 3)), with ceil(2 % of D) channels per (kv-head)
  multiplied by 20 in both K and V; Q ~ N(0, 1).
"""
from __future__ import annotations

import math

import torch

CLAMP = 60000.0


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _student_t3(shape, g, device):
    z = _normal(shape, g, device)
    chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(3):
        n = _normal(shape, g, device)
        chi2 += n * n
    return z / torch.sqrt(chi2 / 3.0)


def _heavy_channel_mask(num_kv_heads, head_dim, count, g, device):
    """[H][D] 0/1 mask with ``count`` distinct channels per head."""
    mask = torch.zeros((num_kv_heads, head_dim), device=device, dtype=torch.float32)
    for h in range(num_kv_heads):
        idx = torch.randperm(head_dim, generator=g, device=device)[:count]
        mask[h, idx] = 1.0
    return mask


def _to_fp16(x):
    return x.clamp_(-CLAMP, CLAMP).to(torch.float16)


class LayerSource:
    """Draws the K/V of one layer and the query/append tokens of each decode
    step, reproducibly from (workload seed, layer)."""

    def __init__(self, wl, layer, device="cpu", seed=None):
        self.wl = wl
        self.layer = layer
        self.device = torch.device(device)
        base = wl.seed if seed is None else seed
        self.seed = base * 1_000_003 + layer * 7919
        g = _gen(self.device, self.seed)
        d = wl.head_dim
        h = wl.num_kv_heads
        if wl.dist == "k_lognormal_channels":
            self.k_chan = torch.exp(0.5 * _normal((h, d), g, self.device))
            self.v_chan = None
        elif wl.dist == "k_heavy15":
            self.k_chan = 1.0 + 14.0 * _heavy_channel_mask(h, d, 4, g, self.device)
            self.v_chan = None
        elif wl.dist == "t3_heavy20":
            m = _heavy_channel_mask(h, d, math.ceil(0.02 * d), g, self.device)
            self.k_chan = 1.0 + 19.0 * m
            self.v_chan = self.k_chan
        elif wl.dist == "normal":
            self.k_chan = None
            self.v_chan = None
        else:
            raise ValueError(wl.dist)

    def _draw(self, shape, g, chan, heavy_tail):
        x = _student_t3(shape, g, self.device) if heavy_tail else _normal(shape, g, self.device)
        if chan is not None:
            # chan is [H][D]; shape is [B][H][..][D]
            view = chan.view(1, chan.shape[0], *([1] * (len(shape) - 3)), chan.shape[1])
            x = x * view
        return _to_fp16(x)

    def kv(self, seq_len, batch=None, stream=0):
        """K, V fp16 [B][H_kv][S][D] for ``seq_len`` tokens."""
        wl = self.wl
        b = wl.batch if batch is None else batch
        g = _gen(self.device, self.seed + 17 + 101 * stream)
        shape = (b, wl.num_kv_heads, seq_len, wl.head_dim)
        t3 = wl.dist == "t3_heavy20"
        k = self._draw(shape, g, self.k_chan, t3)
        v = self._draw(shape, g, self.v_chan, t3)
        return k, v

    def step(self, step, batch=None):
        """Decode step ``step``: (q [B][H_q][D], k1 [B][H_kv][D], v1 [B][H_kv][D])."""
        wl = self.wl
        b = wl.batch if batch is None else batch
        g = _gen(self.device, self.seed + 1_000_033 + 131 * step)
        q = _to_fp16(_normal((b, wl.num_q_heads, wl.head_dim), g, self.device))
        shape = (b, wl.num_kv_heads, 1, wl.head_dim)
        t3 = wl.dist == "t3_heavy20"
        k1 = self._draw(shape, g, self.k_chan, t3)[:, :, 0]
        v1 = self._draw(shape, g, self.v_chan, t3)[:, :, 0]
        return q, k1.contiguous(), v1.contiguous()
