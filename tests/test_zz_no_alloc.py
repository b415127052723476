"""Decode attention without a caller-supplied workspace.

kvc_decode_attention_noalloc serves callers that cannot allocate device memory
when they run a step (fixed memory budgets, runtimes that forbid allocation
after start-up, hosts that own every allocation).  It must give the same
outputs as kvc_decode_attention with a caller workspace, call after call, since
every call reuses the same fixed scratch array in the library.  This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2  # the attention tolerance of the parity tests


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_cache_kvc_gb300.build import build_library
    build_library()


def _bf16(rng, shape):
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32))
    return x.to(torch.bfloat16).cuda()


@pytest.mark.parametrize("bits,hq,hkv,lengths,window", [(8, 8, 2, [300, 47], 0), (4, 40, 8, [700, 130, 9], 0),
                                                         (8, 16, 4, [400, 30], 64)])  # with a bf16 window
def test_noalloc_matches_workspace_entry_point(bits, hq, hkv, lengths, window):
    from compressed_kv_cache_kvc_gb300 import _lib as L
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits + hq)
    B = len(lengths)
    mbps = (max(lengths) + 15) // 16 + 2
    cache = KVCache(hq, hkv, bits, B * mbps, B, mbps, bf16_window=window)
    for b, n in enumerate(lengths):
        cache.quantize_append(_bf16(rng, (1, hkv, n, 128)), _bf16(rng, (1, hkv, n, 128)), seq_begin=b)
    lib = L.lib()
    assert cache.workspace_bytes(B) <= L.KVC_NOALLOC_SCRATCH_BYTES
    scale = 1.0 / 128 ** 0.5
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):  # two calls in a row share the same scratch
        q = _bf16(rng, (B, hq, 128))
        ref = cache.decode_attention(q, accumulate_h2o=False).float()
        out = torch.full_like(q, float("nan"))
        st = lib.kvc_decode_attention_noalloc(cache.handle, 0, B, ctypes.c_void_p(q.data_ptr()),
                                              ctypes.c_void_p(out.data_ptr()), ctypes.c_float(scale), 0, stream)
        assert st == L.KVC_OK, L.status_string(st)
        torch.cuda.synchronize()
        got = out.float()
        err = (got - ref).abs()
        assert torch.all(err <= ATOL + RTOL * ref.abs()), float(err.max())
    assert cache.read_status() == 0


def test_noalloc_rejects_slices_beyond_the_scratch():
    from compressed_kv_cache_kvc_gb300 import _lib as L
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    cache = KVCache(64, 8, 8, num_blocks=8, max_batch=64, max_blocks_per_seq=2048)
    assert cache.workspace_bytes(64) > L.KVC_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(64, 64, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    st = L.lib().kvc_decode_attention_noalloc(cache.handle, 0, 64, ctypes.c_void_p(q.data_ptr()),
                                              ctypes.c_void_p(out.data_ptr()), ctypes.c_float(0.08), 0,
                                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == L.KVC_ERR_CAPACITY
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(out)) == 0  # nothing ran
