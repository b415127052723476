"""CPU-only checks of the C ABI: the library builds and loads, exports every
symbol include/kvc.h declares, and its host-side validation rejects bad calls
before anything reaches a GPU (so these run without one)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from compressed_kv_cache_kvc_gb300.build import build_library
    build_library()
    from compressed_kv_cache_kvc_gb300 import _lib as L
    return L


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "kvc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 15
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(so, n), n
    # and the binding declares each of them
    assert set(names) == set(lib._SIGS)


def test_version_and_strings(lib):
    L = lib.lib()
    assert L.kvc_version() == lib.KVC_VERSION == 400
    assert L.kvc_status_string(lib.KVC_ERR_CAPACITY) == b"out of cache capacity"


def _cfg(lib, **kw):
    d = dict(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, bits=8, num_blocks=8, max_batch=2,
             max_blocks_per_seq=4)
    d.update(kw)
    return lib.KvcConfig(**d)


class _FakeState:
    """Host memory standing in for device memory: the calls below must fail
    validation before they could touch it."""

    def __init__(self, lib, cfg):
        self.n = lib.lib().kvc_state_bytes(ctypes.byref(cfg))
        self.buf = ctypes.create_string_buffer(self.n + 512)
        addr = ctypes.addressof(self.buf)
        self.ptr = ctypes.c_void_p(addr + (-addr) % 256)


def _create(lib, cfg):
    fs = _FakeState(lib, cfg)
    h = ctypes.c_void_p()
    st = lib.lib().kvc_cache_create(ctypes.byref(cfg), fs.ptr, fs.n, ctypes.byref(h))
    return st, h, fs


def test_state_bytes_layout(lib):
    L = lib.lib()
    cfg = _cfg(lib)
    n = L.kvc_state_bytes(ctypes.byref(cfg))
    # codes K+V, 4 per-slot fp32/int32 arrays, sinks, tables ... all 256-aligned
    slots = 8 * 2 * 16
    assert n >= 2 * slots * 128 + 4 * slots * 4 + 2 * 2 * 2 * 4 * 128 * 2
    assert n % 256 == 0
    cfg4 = _cfg(lib, bits=4)
    assert L.kvc_state_bytes(ctypes.byref(cfg4)) < n
    for bad in (dict(head_dim=64), dict(page_size=32), dict(bits=2), dict(num_q_heads=7),
                dict(num_q_heads=32, num_kv_heads=2), dict(num_blocks=0)):
        assert L.kvc_state_bytes(ctypes.byref(_cfg(lib, **bad))) == 0, bad


def test_create_validation(lib):
    L = lib.lib()
    st, h, fs = _create(lib, _cfg(lib, head_dim=64))
    assert st == lib.KVC_ERR_UNSUPPORTED
    st, h, fs = _create(lib, _cfg(lib, num_q_heads=72, num_kv_heads=8))
    assert st == lib.KVC_ERR_UNSUPPORTED
    cfg = _cfg(lib)
    fs = _FakeState(lib, cfg)
    h = ctypes.c_void_p()
    assert L.kvc_cache_create(ctypes.byref(cfg), fs.ptr, fs.n - 1, ctypes.byref(h)) == lib.KVC_ERR_INVALID_ARG
    mis = ctypes.c_void_p(fs.ptr.value + 8)
    assert L.kvc_cache_create(ctypes.byref(cfg), mis, fs.n, ctypes.byref(h)) == lib.KVC_ERR_INVALID_ARG
    st, h, fs = _create(lib, cfg)
    assert st == lib.KVC_OK and h.value
    ptr, nb = ctypes.c_void_p(), ctypes.c_size_t()
    assert L.kvc_cache_buffer(h, 0, ctypes.byref(ptr), ctypes.byref(nb)) == lib.KVC_OK
    assert ptr.value == fs.ptr.value and nb.value == 8 * 2 * 16 * 128
    assert L.kvc_cache_buffer(h, 99, ctypes.byref(ptr), ctypes.byref(nb)) == lib.KVC_ERR_INVALID_ARG
    L.kvc_cache_destroy(h)


def test_call_validation_before_any_launch(lib):
    L = lib.lib()
    cfg = _cfg(lib, num_blocks=3, max_blocks_per_seq=2)
    st, h, fs = _create(lib, cfg)
    assert st == lib.KVC_OK
    dummy = ctypes.c_void_p(fs.ptr.value)  # aligned, never dereferenced
    # bad ranges
    assert L.kvc_quantize_append(h, 1, 2, 1, dummy, dummy, None) == lib.KVC_ERR_INVALID_ARG
    assert L.kvc_quantize_append(h, 0, 1, -1, dummy, dummy, None) == lib.KVC_ERR_INVALID_ARG
    # n_new == 0 is a no-op
    assert L.kvc_quantize_append(h, 0, 1, 0, None, None, None) == lib.KVC_OK
    assert L.kvc_last_launch_count(h) == 0
    # per-sequence table overflow: 4 sinks + 33 slots needs 3 pages > 2
    assert L.kvc_quantize_append(h, 0, 1, 37, dummy, dummy, None) == lib.KVC_ERR_CAPACITY
    # misaligned inputs
    assert L.kvc_quantize_append(h, 0, 1, 1, ctypes.c_void_p(fs.ptr.value + 2), dummy, None) == \
        lib.KVC_ERR_INVALID_ARG
    s, p = ctypes.c_int32(), ctypes.c_int32()
    assert L.kvc_cache_lengths(h, 0, ctypes.byref(s), ctypes.byref(p)) == lib.KVC_OK
    assert (s.value, p.value) == (0, 0)
    # attention over an empty sequence is rejected
    ws = L.kvc_workspace_bytes(h, 1)
    assert ws > 0
    wsbuf = ctypes.create_string_buffer(ws + 512)
    wsp = ctypes.c_void_p(ctypes.addressof(wsbuf) + (-ctypes.addressof(wsbuf)) % 256)
    assert L.kvc_decode_attention(h, 0, 1, dummy, dummy, ctypes.c_float(0.088), 1, wsp, ws, None) == \
        lib.KVC_ERR_INVALID_ARG
    # workspace too small
    assert L.kvc_decode_attention(h, 0, 1, dummy, dummy, ctypes.c_float(0.088), 1, wsp, ws - 1, None) == \
        lib.KVC_ERR_INVALID_ARG
    # bad flags / scale
    assert L.kvc_decode_attention(h, 0, 1, dummy, dummy, ctypes.c_float(0.088), 4, wsp, ws, None) == \
        lib.KVC_ERR_INVALID_ARG
    assert L.kvc_decode_attention(h, 0, 1, dummy, dummy, ctypes.c_float(-1.0), 1, wsp, ws, None) == \
        lib.KVC_ERR_INVALID_ARG
    # eviction parameters
    mask = dummy
    bad = [lib.KvcEvictParams(0, 10, 8, 0), lib.KvcEvictParams(0, 10, -1, 0), lib.KvcEvictParams(1, 0, 0, 0),
           lib.KvcEvictParams(7, 100, 0, 0),
           # block-granular: retention in (0, 1], recent >= 0
           lib.KvcEvictParams(2, 0, 8, 0, 0.0), lib.KvcEvictParams(2, 0, 8, 0, 1.5),
           lib.KvcEvictParams(2, 0, -1, 0, 0.5), lib.KvcEvictParams(2, 0, 8, 0, float("nan"))]
    for prm in bad:
        assert L.kvc_h2o_select_evict(h, 0, 1, ctypes.byref(prm), mask, wsp, ws, None) == lib.KVC_ERR_INVALID_ARG
    # compaction needs a pending selection
    assert L.kvc_compact_blocks(h, 0, 1, mask, wsp, ws, None) == lib.KVC_ERR_STATE
    # the overlapped step checks its arguments as the one-call step does,
    # before anything is enqueued on either stream
    for prm in bad[:4]:
        assert L.kvc_decode_step_overlap(h, 0, 1, dummy, dummy, dummy, dummy, ctypes.c_float(0.088),
                                         ctypes.byref(prm), wsp, ws, None, None) == lib.KVC_ERR_INVALID_ARG
    ok = lib.KvcEvictParams(0, 100, 8, 0)
    assert L.kvc_decode_step_overlap(h, 0, 1, dummy, dummy, dummy, dummy, ctypes.c_float(0.088), ctypes.byref(ok),
                                     wsp, ws - 1, None, None) == lib.KVC_ERR_INVALID_ARG
    assert L.kvc_decode_step_overlap(h, 0, 1, dummy, dummy, dummy, dummy, ctypes.c_float(float("nan")),
                                     ctypes.byref(ok), wsp, ws, None, None) == lib.KVC_ERR_INVALID_ARG
    # tracing events come in pairs
    assert L.kvc_set_trace_events(h, dummy, None) == lib.KVC_ERR_INVALID_ARG
    assert L.kvc_set_trace_events(h, None, None) == lib.KVC_OK
    L.kvc_cache_destroy(h)


def test_block_eviction_page_limit(lib):
    """Block-granular eviction keeps a sequence's page keys in one CTA's
    shared memory: more than 4096 pages per sequence is refused before any
    launch, by the selection and by the one-call step."""
    L = lib.lib()
    st, h, fs = _create(lib, _cfg(lib, num_blocks=3, max_blocks_per_seq=4097))
    assert st == lib.KVC_OK
    dummy = ctypes.c_void_p(fs.ptr.value)
    ws = L.kvc_workspace_bytes(h, 1)
    wsbuf = ctypes.create_string_buffer(ws + 512)
    wsp = ctypes.c_void_p(ctypes.addressof(wsbuf) + (-ctypes.addressof(wsbuf)) % 256)
    blk = lib.KvcEvictParams(2, 0, 8, 0, 0.5)
    assert L.kvc_h2o_select_evict(h, 0, 1, ctypes.byref(blk), dummy, wsp, ws, None) == lib.KVC_ERR_UNSUPPORTED
    assert L.kvc_decode_step(h, 0, 1, dummy, dummy, dummy, dummy, ctypes.c_float(0.088), ctypes.byref(blk), wsp, ws,
                             None) == lib.KVC_ERR_UNSUPPORTED
    assert L.kvc_last_launch_count(h) == 0
    L.kvc_cache_destroy(h)


def test_prefill_context_validation(lib):
    """A prompt over a sequence with context: bad ranges, lengths, flags,
    scales and workspaces are refused and the capacity is checked, all before
    any launch."""
    L = lib.lib()
    st, h, fs = _create(lib, _cfg(lib, num_blocks=3, max_blocks_per_seq=2))
    assert st == lib.KVC_OK
    dummy = ctypes.c_void_p(fs.ptr.value)
    ws = L.kvc_prefill_context_workspace_bytes(h, 1, 5)
    ws37 = L.kvc_prefill_context_workspace_bytes(h, 1, 37)
    assert 0 < ws < ws37  # the row statistics grow with the prompt
    assert L.kvc_prefill_context_workspace_bytes(None, 1, 5) == 0
    assert L.kvc_prefill_context_workspace_bytes(h, 0, 5) == 0 and L.kvc_prefill_context_workspace_bytes(h, 1, 0) == 0
    wsbuf = ctypes.create_string_buffer(ws37 + 512)
    wsp = ctypes.c_void_p(ctypes.addressof(wsbuf) + (-ctypes.addressof(wsbuf)) % 256)

    def call(handle=h, seq_begin=0, batch=1, n=5, scale=0.088, flags=1, nbytes=ws37):
        return L.kvc_prefill_context(handle, seq_begin, batch, n, dummy, dummy, dummy, dummy, ctypes.c_float(scale),
                                     flags, wsp, nbytes, None)

    assert call(handle=None) == lib.KVC_ERR_INVALID_ARG
    for kw in [dict(seq_begin=1, batch=2), dict(n=0), dict(flags=4), dict(scale=-1.0), dict(scale=float("inf")),
               dict(nbytes=ws - 1), dict(n=37, nbytes=ws37 - 1)]:
        assert call(**kw) == lib.KVC_ERR_INVALID_ARG, kw
    assert call(n=37) == lib.KVC_ERR_CAPACITY  # 4 sinks + 33 slots need 3 pages > 2
    assert L.kvc_last_launch_count(h) == 0
    s, p = ctypes.c_int32(), ctypes.c_int32()
    assert L.kvc_cache_lengths(h, 0, ctypes.byref(s), ctypes.byref(p)) == lib.KVC_OK
    assert (s.value, p.value) == (0, 0)
    L.kvc_cache_destroy(h)
    # with a bf16 window the column sums cover the window's positions too
    st, h2, fs2 = _create(lib, _cfg(lib, num_blocks=3, max_blocks_per_seq=2, bf16_window=128))
    assert st == lib.KVC_OK
    st, h3, fs3 = _create(lib, _cfg(lib, num_blocks=3, max_blocks_per_seq=2))
    assert L.kvc_prefill_context_workspace_bytes(h2, 1, 5) > L.kvc_prefill_context_workspace_bytes(h3, 1, 5)
    L.kvc_cache_destroy(h2)
    L.kvc_cache_destroy(h3)


def test_header_is_c99_and_the_abi_works_from_c(lib, tmp_path):
    """include/kvc.h compiles as plain C99 (-pedantic, warnings as errors) and
    a C program linked against the library makes the host-side calls."""
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(lib.LIB_PATH)
    exe = str(tmp_path / "kvc_abi_c99")
    cmd = ["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "kvc_abi_c99.c"), "-o", exe, "-L", libdir, "-lkvc",
           "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from compressed_kv_cache_kvc_gb300 import _lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        L.lib()


def test_hybrid_window_validation(lib):
    """bf16_window: negative is invalid, above 4096 unsupported; the ring
    buffers take max_batch x Hkv x W rows of 128 bf16 for K and for V; the
    selection needs the recent window (H2O) or the StreamingLLM window to
    cover W, and block-granular eviction is unsupported with a window; the
    host capacity check counts only the tokens that leave the window."""
    L = lib.lib()
    assert L.kvc_state_bytes(ctypes.byref(_cfg(lib, bf16_window=-1))) == 0
    assert L.kvc_state_bytes(ctypes.byref(_cfg(lib, bf16_window=4097))) == 0
    cfg = _cfg(lib, bf16_window=16, num_blocks=3, max_blocks_per_seq=2)
    st, h, fs = _create(lib, cfg)
    assert st == lib.KVC_OK
    ptr, nb = ctypes.c_void_p(), ctypes.c_size_t()
    assert L.kvc_cache_buffer(h, lib.BUF["RING_K"], ctypes.byref(ptr), ctypes.byref(nb)) == lib.KVC_OK
    assert nb.value == 2 * 2 * 16 * 128 * 2
    assert L.kvc_cache_buffer(h, lib.BUF["RING_SCORE"], ctypes.byref(ptr), ctypes.byref(nb)) == lib.KVC_OK
    assert nb.value == 2 * 2 * 16 * 4
    dummy = ctypes.c_void_p(fs.ptr.value)
    ws = L.kvc_workspace_bytes(h, 1)
    wsbuf = ctypes.create_string_buffer(ws + 512)
    wsp = ctypes.c_void_p(ctypes.addressof(wsbuf) + (-ctypes.addressof(wsbuf)) % 256)
    for prm, want in [(lib.KvcEvictParams(0, 100, 8, 0), lib.KVC_ERR_INVALID_ARG),      # recent < W
                      (lib.KvcEvictParams(1, 0, 0, 8), lib.KVC_ERR_INVALID_ARG),        # window < W
                      (lib.KvcEvictParams(2, 0, 8, 0, 0.5), lib.KVC_ERR_UNSUPPORTED)]:  # block + window
        assert L.kvc_h2o_select_evict(h, 0, 1, ctypes.byref(prm), dummy, wsp, ws, None) == want
        assert L.kvc_decode_step(h, 0, 1, dummy, dummy, dummy, dummy, ctypes.c_float(0.088), ctypes.byref(prm),
                                 wsp, ws, None) == want
    # 4 sinks + 16 window + 33 pool slots need 3 pages > 2
    assert L.kvc_quantize_append(h, 0, 1, 53, dummy, dummy, None) == lib.KVC_ERR_CAPACITY
    L.kvc_cache_destroy(h)


def test_code_format_validation(lib):
    L = lib.lib()
    assert L.kvc_state_bytes(ctypes.byref(_cfg(lib, codes=2))) == 0
    assert L.kvc_state_bytes(ctypes.byref(_cfg(lib, codes=-1))) == 0
    assert L.kvc_state_bytes(ctypes.byref(_cfg(lib, codes=lib.KVC_CODES_E4M3, bits=4))) == 0
    st, h, fs = _create(lib, _cfg(lib, codes=lib.KVC_CODES_E4M3, bits=4))
    assert st == lib.KVC_ERR_UNSUPPORTED
    a = L.kvc_state_bytes(ctypes.byref(_cfg(lib, codes=lib.KVC_CODES_E4M3)))
    assert a > 0 and a == L.kvc_state_bytes(ctypes.byref(_cfg(lib)))  # same layout as INT8


def test_release_validation(lib):
    L = lib.lib()
    st, h, fs = _create(lib, _cfg(lib))
    assert st == lib.KVC_OK
    assert L.kvc_release_sequences(h, 1, 2, None) == lib.KVC_ERR_INVALID_ARG
    assert L.kvc_release_sequences(h, -1, 1, None) == lib.KVC_ERR_INVALID_ARG
    assert L.kvc_release_sequences(h, 0, 2, None) == lib.KVC_OK  # empty: nothing to launch
    assert L.kvc_last_launch_count(h) == 0
    L.kvc_cache_destroy(h)
