"""The five seeded synthetic workloads, described by shape and codec, and
the codebook-codec layer and the ragged batch beside them.

Each entry names what it is: the tiny q8_0-style GQA layer, the
Llama-2-7B-shaped MHA layer (two contexts), the Llama-2-70B-shaped GQA layer
with 3-bit codes, the dense-and-sparse 128K MHA layer, and the full
8B-shaped 32-layer decode. Value distributions are produced by
``synth.py``; this file holds sizes and codec settings only.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

SYM_PER_TOKEN = 0
ASYM_PER_TOKEN = 1
ASYM_PER_CHANNEL = 2
CODEBOOK_PER_TOKEN = 3


@dataclass(frozen=True)
class Workload:
    name: str
    index: int            # 0..4, also picks the seed (1000 + index)
    num_layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seq_len: int
    k_bits: int
    v_bits: int
    k_mode: int
    v_mode: int
    k_group: int
    v_group: int
    outliers_per_row: int = 0
    decode_steps: int = 1
    dist: str = "normal"  # normal | k_lognormal_channels | k_heavy15 | t3_heavy20
    codebook: tuple = None  # 16 levels of CODEBOOK_PER_TOKEN tensors
    lens: tuple = None      # ragged batch: each row's tokens at the prefill (seq_len = the longest)

    @property
    def gqa(self):
        return self.num_q_heads // self.num_kv_heads

    @property
    def seed(self):
        return 1000 + self.index

    def with_seq(self, seq_len, **kw):
        return replace(self, seq_len=seq_len, **kw)

    def codec_kwargs(self):
        return dict(k_bits=self.k_bits, v_bits=self.v_bits, k_mode=self.k_mode,
                    v_mode=self.v_mode, k_group=self.k_group, v_group=self.v_group,
                    outliers_per_row=self.outliers_per_row, codebook=self.codebook)


# The 4-bit minifloat `1 sign | 2 exponent | 1 mantissa` as 16 codebook levels,
# indexed by the code's bits (exponent bias 1, subnormal at exponent 0).
E2M1 = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0)


TINY_Q8 = Workload("tiny-q8_0-gqa8x2-d128-s4096", 0, 1, 1, 8, 2, 128, 4096,
                   8, 8, SYM_PER_TOKEN, SYM_PER_TOKEN, 32, 32, dist="normal")
LLAMA7B_8K = Workload("llama2-7b-layer-b8-h32-s8192-int4", 1, 1, 8, 32, 32, 128, 8192,
                      4, 4, ASYM_PER_CHANNEL, ASYM_PER_TOKEN, 64, 64,
                      dist="k_lognormal_channels")
LLAMA7B_16K = LLAMA7B_8K.with_seq(16384, name="llama2-7b-layer-b8-h32-s16384-int4")
LLAMA70B_32K = Workload("llama2-70b-layer-b4-h64x8-s32768-int3", 2, 1, 4, 64, 8, 128, 32768,
                        3, 3, ASYM_PER_CHANNEL, ASYM_PER_TOKEN, 128, 128, dist="k_heavy15")
DENSE_SPARSE_128K = Workload("dense-sparse-b1-h32-s131072-int4-out2", 3, 1, 1, 32, 32, 128,
                             131072, 4, 4, ASYM_PER_CHANNEL, ASYM_PER_TOKEN, 64, 64,
                             outliers_per_row=2, dist="t3_heavy20")
LLAMA8B_FULL = Workload("8b-32layer-h32x8-s131072-k4v8-64steps", 4, 32, 1, 32, 8, 128, 131072,
                        4, 8, ASYM_PER_CHANNEL, ASYM_PER_TOKEN, 64, 64, decode_steps=64,
                        dist="k_lognormal_channels")

# Beyond the five: the 8B-shaped layer with 4-bit minifloat codebook codes for
# keys and values, one fp16 scale per 32 channels.
LLAMA8B_E2M1 = Workload("8b-layer-h32x8-s131072-e2m1-g32", 5, 1, 1, 32, 8, 128, 131072,
                        4, 4, CODEBOOK_PER_TOKEN, CODEBOOK_PER_TOKEN, 32, 32, decode_steps=64,
                        dist="k_lognormal_channels", codebook=E2M1)

# A ragged batch of eight q8_0-style sequences (int8 per-token keys and
# values, 8 kv-heads, 4 query heads per kv-head) from 512 to 32768 tokens.
RAGGED_Q8 = Workload("q8_0-gqa4-b8x8-ragged-s32768", 6, 1, 8, 32, 8, 128, 32768,
                     8, 8, SYM_PER_TOKEN, SYM_PER_TOKEN, 32, 32, decode_steps=64, dist="normal",
                     lens=(32768, 4096, 16384, 1024, 28672, 8192, 512, 20480))

ALL = [TINY_Q8, LLAMA7B_8K, LLAMA7B_16K, LLAMA70B_32K, DENSE_SPARSE_128K, LLAMA8B_FULL]
EXTRA = [LLAMA8B_E2M1, RAGGED_Q8]
BY_NAME = {w.name: w for w in ALL + EXTRA}
