"""The decode entry point for callers that cannot allocate device memory
(kvq_decode_attention_static): called through the C ABI, its output must
match kvq_decode_attention (which takes a caller workspace) within the
attention tolerance, on two calls in a row. Collected last on purpose: it
must pass both alone in a fresh process and after every other test."""
import ctypes
import math
from dataclasses import replace

import pytest
import torch

import bit_quantized_kv_kvq_gb300 as kvq
from bit_quantized_kv_kvq_gb300 import workloads as W
from bit_quantized_kv_kvq_gb300.synth import LayerSource
from oracle import kvq_oracle as O
from tests import kvq_check as K

pytestmark = pytest.mark.gpu


def _static_call(cache, layer, q, out):
    lib = kvq.lib()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.kvq_decode_attention_static(cache.handle, layer, ctypes.c_void_p(q.data_ptr()),
                                           q.shape[1], ctypes.c_float(1.0 / math.sqrt(128)),
                                           ctypes.c_void_p(out.data_ptr()), kvq.F32, st)


@pytest.mark.parametrize("wl", [
    replace(W.LLAMA7B_16K, batch=2, num_q_heads=4, num_kv_heads=4, seq_len=3000),
    replace(W.LLAMA8B_FULL, num_layers=2, num_q_heads=16, num_kv_heads=4, seq_len=5000),
], ids=["mha", "gqa"])
def test_static_scratch_matches_workspace_path(wl):
    torch.cuda.init()
    cache = K.make_gpu_cache(wl, wl.seq_len + 4)
    scale = 1.0 / math.sqrt(128)
    for layer in range(wl.num_layers):
        src = LayerSource(wl, layer, device="cuda")
        k, v = src.kv(wl.seq_len)
        cache.prefill(layer, k, v)
    for call in range(2):  # two calls in a row share the static scratch
        layer = call % wl.num_layers
        q, _, _ = LayerSource(wl, layer, device="cuda").step(100 + call)
        ref = cache.decode(layer, q, scale)
        got = torch.full_like(ref, float("nan"))
        status = _static_call(cache, layer, q, got)
        assert status == 0, kvq.lib().kvq_last_error()
        torch.cuda.synchronize()
        err = O.row_relative_error(got.cpu().double().numpy(), ref.cpu().double().numpy())
        assert float(err.max()) <= K.ATTN_TOL
    assert cache.status() == 0


def test_static_scratch_rejects_oversized_calls():
    # per-token keys decode through split partials: 512 rows x 64 splits of
    # fp32 partials is far above the 4 MiB maximum
    wl = replace(W.LLAMA7B_16K, batch=16, num_q_heads=32, num_kv_heads=32, seq_len=4096,
                 k_mode=W.ASYM_PER_TOKEN, k_group=32)
    cache = K.make_gpu_cache(wl, wl.seq_len)
    src = LayerSource(wl, 0, device="cuda")
    k, v = src.kv(wl.seq_len)
    cache.prefill(0, k, v)
    cache.set_decode_splits(64)
    q, _, _ = src.step(1)
    out = torch.empty((wl.batch, wl.num_q_heads, 128), dtype=torch.float32, device="cuda")
    assert _static_call(cache, 0, q, out) == 3
    assert b"static maximum" in kvq.lib().kvq_last_error()
