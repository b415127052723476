"""Thin Python binding of the compressed-KV C library.

``KVCache`` owns one layer's device state (a torch uint8 buffer used only as
device memory) and forwards each call to the C ABI with raw pointers and the
current torch CUDA stream.  Every step of the decode path runs in the
library's CUDA kernels; nothing here computes.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib as L

PAGE = 16
HEAD_DIM = 128
NUM_SINK = 4


def _stream_ptr(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t: torch.Tensor, dtype, name: str, device=None, shape=None):
    """Argument check before any pointer goes to the library: a contiguous
    CUDA tensor of `dtype` (on `device`, of `shape`, when given), since the
    kernels read and write exactly the extents the call's sizes imply."""
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of dtype {dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the cache on {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, not {tuple(t.shape)}")


class KVCache:
    """One layer's compressed, paged KV cache on the current CUDA device."""

    def __init__(self, num_q_heads: int, num_kv_heads: int, bits: int, num_blocks: int,
                 max_batch: int, max_blocks_per_seq: int, block_order=None, device=None, bf16_window: int = 0,
                 codes: str = "int"):
        """bf16_window = W > 0: hybrid precision, the last W positions of each
        sequence kept in bf16 (they enter the quantised pool when they leave
        the window).  codes = "int" (INT8/INT4) or "e4m3" (FP8, bits = 8)."""
        self.lib = L.lib()
        self.cfg = L.KvcConfig(num_q_heads, num_kv_heads, HEAD_DIM, PAGE, bits, num_blocks, max_batch,
                               max_blocks_per_seq, bf16_window,
                               {"int": L.KVC_CODES_INT, "e4m3": L.KVC_CODES_E4M3}[codes])
        self.bf16_window = bf16_window
        self.codes = codes
        self.num_q_heads, self.num_kv_heads, self.bits = num_q_heads, num_kv_heads, bits
        self.group = num_q_heads // num_kv_heads
        self.num_blocks, self.max_batch, self.max_blocks_per_seq = num_blocks, max_batch, max_blocks_per_seq
        self.s_cap = max_blocks_per_seq * PAGE
        nbytes = self.lib.kvc_state_bytes(ctypes.byref(self.cfg))
        if nbytes == 0:
            raise L.KvcError(L.KVC_ERR_UNSUPPORTED, "kvc_state_bytes")
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.state = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.state.data_ptr()) % 256
        self.state_view = self.state[off:off + nbytes]
        self.state_bytes = nbytes
        h = ctypes.c_void_p()
        L.check(self.lib.kvc_cache_create(ctypes.byref(self.cfg), ctypes.c_void_p(self.state_view.data_ptr()),
                                          nbytes, ctypes.byref(h)), "kvc_cache_create")
        self.handle = h
        self._ws = {}
        self.reset(block_order)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            try:
                self.lib.kvc_cache_destroy(h)
            except Exception:
                pass
            self.handle = None

    # -- state ---------------------------------------------------------------
    def reset(self, block_order=None, stream=None):
        arr = None
        if block_order is not None:
            vals = [int(x) for x in block_order]
            arr = (ctypes.c_int32 * len(vals))(*vals)
        L.check(self.lib.kvc_cache_reset(self.handle, arr, ctypes.c_void_p(_stream_ptr(stream))), "kvc_cache_reset")

    def release(self, seq_begin: int = 0, batch: int = 1, stream=None):
        """Free the sequences [seq_begin, seq_begin + batch): pages back to the
        pool, lengths to 0 (idempotent)."""
        L.check(self.lib.kvc_release_sequences(self.handle, seq_begin, batch, ctypes.c_void_p(_stream_ptr(stream))),
                "kvc_release_sequences")

    def buffer(self, name: str) -> torch.Tensor:
        """Device view of one state buffer (uint8, reinterpret with .view)."""
        ptr, nb = ctypes.c_void_p(), ctypes.c_size_t()
        L.check(self.lib.kvc_cache_buffer(self.handle, L.BUF[name], ctypes.byref(ptr), ctypes.byref(nb)),
                "kvc_cache_buffer")
        off = ptr.value - self.state_view.data_ptr()
        return self.state_view[off:off + nb.value]

    def lengths(self, seq: int):
        s, p = ctypes.c_int32(), ctypes.c_int32()
        L.check(self.lib.kvc_cache_lengths(self.handle, seq, ctypes.byref(s), ctypes.byref(p)), "kvc_cache_lengths")
        return s.value, p.value

    def sync_host(self, stream=None):
        L.check(self.lib.kvc_cache_sync_host(self.handle, ctypes.c_void_p(_stream_ptr(stream))), "kvc_cache_sync_host")

    def workspace_bytes(self, batch: int) -> int:
        return int(self.lib.kvc_workspace_bytes(self.handle, batch))

    def workspace(self, batch: int) -> torch.Tensor:
        nb = self.workspace_bytes(batch)
        ws = self._ws.get(nb)
        if ws is None:
            ws = torch.empty(nb + 256, dtype=torch.uint8, device=self.device)
            off = (-ws.data_ptr()) % 256
            ws = ws[off:off + nb]
            self._ws[nb] = ws
        return ws

    def read_status(self, stream=None) -> int:
        v = ctypes.c_int32()
        st = self.lib.kvc_read_status(self.handle, ctypes.byref(v), ctypes.c_void_p(_stream_ptr(stream)))
        if st not in (L.KVC_OK, L.KVC_ERR_DEVICE):
            L.check(st, "kvc_read_status")
        return v.value

    def set_trace_events(self, start=None, stop=None):
        a = ctypes.c_void_p(start.cuda_event) if start is not None else None
        b = ctypes.c_void_p(stop.cuda_event) if stop is not None else None
        L.check(self.lib.kvc_set_trace_events(self.handle, a, b), "kvc_set_trace_events")

    def last_launch_count(self) -> int:
        return int(self.lib.kvc_last_launch_count(self.handle))

    # -- the decode step -----------------------------------------------------
    def quantize_append(self, k: torch.Tensor, v: torch.Tensor, seq_begin: int = 0, stream=None):
        """k, v: bf16 [batch, Hkv, n_new, 128]."""
        _need(k, torch.bfloat16, "k", self.device)
        _need(v, torch.bfloat16, "v", self.device)
        if k.shape != v.shape or k.dim() != 4 or k.shape[1] != self.num_kv_heads or k.shape[3] != HEAD_DIM:
            raise ValueError("k, v must be [batch, num_kv_heads, n_new, 128]")
        L.check(self.lib.kvc_quantize_append(self.handle, seq_begin, k.shape[0], k.shape[2],
                                             ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                             ctypes.c_void_p(_stream_ptr(stream))), "kvc_quantize_append")

    def decode_attention(self, q: torch.Tensor, out: torch.Tensor | None = None, seq_begin: int = 0,
                         sm_scale: float | None = None, accumulate_h2o: bool = True, workspace=None,
                         stream=None) -> torch.Tensor:
        """q: bf16 [batch, Hq, 128] -> bf16 [batch, Hq, 128]."""
        _need(q, torch.bfloat16, "q", self.device)
        if q.dim() != 3 or q.shape[1] != self.num_q_heads or q.shape[2] != HEAD_DIM:
            raise ValueError("q must be [batch, num_q_heads, 128]")
        batch = q.shape[0]
        if out is None:
            out = torch.empty_like(q)
        _need(out, torch.bfloat16, "out", self.device, q.shape)
        ws = self.workspace(batch) if workspace is None else workspace
        _need(ws, torch.uint8, "workspace", self.device)
        scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
        flags = L.KVC_ATTN_ACCUM_H2O if accumulate_h2o else 0
        L.check(self.lib.kvc_decode_attention(self.handle, seq_begin, batch, ctypes.c_void_p(q.data_ptr()),
                                              ctypes.c_void_p(out.data_ptr()), ctypes.c_float(scale), flags,
                                              ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                              ctypes.c_void_p(_stream_ptr(stream))), "kvc_decode_attention")
        return out

    def new_keep_mask(self, batch: int) -> torch.Tensor:
        return torch.empty(batch, self.num_kv_heads, self.s_cap, dtype=torch.uint8, device=self.device)

    def h2o_select_evict(self, batch: int, mode: str = "h2o", budget: int = 0, recent: int = 0,
                         window: int = 0, seq_begin: int = 0, keep_mask=None, workspace=None,
                         stream=None, retention: float = 1.0) -> torch.Tensor:
        """mode "h2o", "streaming" or "block" (whole pages by mean H2O score;
        `retention` = fraction of the candidate pages kept)."""
        m = {"h2o": L.KVC_EVICT_H2O, "streaming": L.KVC_EVICT_STREAMING, "block": L.KVC_EVICT_BLOCK}[mode]
        params = L.KvcEvictParams(m, budget, recent, window, retention)
        mask = self.new_keep_mask(batch) if keep_mask is None else keep_mask
        _need(mask, torch.uint8, "keep_mask", self.device, (batch, self.num_kv_heads, self.s_cap))
        ws = self.workspace(batch) if workspace is None else workspace
        _need(ws, torch.uint8, "workspace", self.device)
        L.check(self.lib.kvc_h2o_select_evict(self.handle, seq_begin, batch, ctypes.byref(params),
                                              ctypes.c_void_p(mask.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                              ws.numel(), ctypes.c_void_p(_stream_ptr(stream))),
                "kvc_h2o_select_evict")
        return mask

    def compact_blocks(self, keep_mask: torch.Tensor, batch: int, seq_begin: int = 0, workspace=None,
                       stream=None):
        _need(keep_mask, torch.uint8, "keep_mask", self.device, (batch, self.num_kv_heads, self.s_cap))
        ws = self.workspace(batch) if workspace is None else workspace
        _need(ws, torch.uint8, "workspace", self.device)
        L.check(self.lib.kvc_compact_blocks(self.handle, seq_begin, batch, ctypes.c_void_p(keep_mask.data_ptr()),
                                            ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                            ctypes.c_void_p(_stream_ptr(stream))), "kvc_compact_blocks")

    def prefill(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_begin: int = 0, out=None,
                sm_scale: float | None = None, accumulate_h2o: bool = True, workspace=None, stream=None):
        """Prompt of fresh sequences: q bf16 [batch, Hq, n, 128], k/v bf16
        [batch, Hkv, n, 128] -> causal attention output bf16 [batch, Hq, n,
        128]; the tokens are appended and (accumulate_h2o) their H2O scores
        set to the prompt attention's column sums."""
        _need(q, torch.bfloat16, "q", self.device)
        _need(k, torch.bfloat16, "k", self.device)
        _need(v, torch.bfloat16, "v", self.device)
        if q.dim() != 4 or q.shape[1] != self.num_q_heads or q.shape[3] != HEAD_DIM:
            raise ValueError("q must be [batch, num_q_heads, n, 128]")
        batch, n = q.shape[0], q.shape[2]
        if tuple(k.shape) != (batch, self.num_kv_heads, n, HEAD_DIM) or k.shape != v.shape:
            raise ValueError("k, v must be [batch, num_kv_heads, n, 128]")
        if out is None:
            out = torch.empty_like(q)
        _need(out, torch.bfloat16, "out", self.device, q.shape)
        nbytes = self.lib.kvc_prefill_workspace_bytes(self.handle, batch, n)
        if workspace is None:
            raw = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
            off = (-raw.data_ptr()) % 256
            workspace = raw[off:off + nbytes]
        _need(workspace, torch.uint8, "workspace", self.device)
        scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
        L.check(self.lib.kvc_prefill_attention(self.handle, seq_begin, batch, n, ctypes.c_void_p(q.data_ptr()),
                                               ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                               ctypes.c_void_p(out.data_ptr()), ctypes.c_float(scale),
                                               L.KVC_ATTN_ACCUM_H2O if accumulate_h2o else 0,
                                               ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                               ctypes.c_void_p(_stream_ptr(stream))), "kvc_prefill_attention")
        return out

    def prefill_context_workspace(self, batch: int, n: int) -> torch.Tensor:
        nbytes = self.lib.kvc_prefill_context_workspace_bytes(self.handle, batch, n)
        raw = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        return raw[(-raw.data_ptr()) % 256:][:nbytes]

    def prefill_context(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, seq_begin: int = 0, out=None,
                        sm_scale: float | None = None, accumulate_h2o: bool = True, workspace=None, stream=None):
        """A prompt on sequences that may hold context: q bf16 [batch, Hq, n,
        128], k/v bf16 [batch, Hkv, n, 128] -> bf16 [batch, Hq, n, 128]; each
        prompt query attends causally to the compressed cache (the workspace,
        if given, from prefill_context_workspace(batch, n))."""
        _need(q, torch.bfloat16, "q", self.device)
        _need(k, torch.bfloat16, "k", self.device)
        _need(v, torch.bfloat16, "v", self.device)
        if q.dim() != 4 or q.shape[1] != self.num_q_heads or q.shape[3] != HEAD_DIM:
            raise ValueError("q must be [batch, num_q_heads, n, 128]")
        batch, n = q.shape[0], q.shape[2]
        if tuple(k.shape) != (batch, self.num_kv_heads, n, HEAD_DIM) or k.shape != v.shape:
            raise ValueError("k, v must be [batch, num_kv_heads, n, 128]")
        if out is None:
            out = torch.empty_like(q)
        _need(out, torch.bfloat16, "out", self.device, q.shape)
        ws = self.prefill_context_workspace(batch, n) if workspace is None else workspace
        _need(ws, torch.uint8, "workspace", self.device)
        scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
        L.check(self.lib.kvc_prefill_context(self.handle, seq_begin, batch, n, ctypes.c_void_p(q.data_ptr()),
                                             ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                             ctypes.c_void_p(out.data_ptr()), ctypes.c_float(scale),
                                             L.KVC_ATTN_ACCUM_H2O if accumulate_h2o else 0,
                                             ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                             ctypes.c_void_p(_stream_ptr(stream))), "kvc_prefill_context")
        return out

    def decode_step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, mode: str = "h2o",
                    budget: int = 0, recent: int = 0, window: int = 0, seq_begin: int = 0, out=None,
                    sm_scale: float | None = None, workspace=None, stream=None,
                    retention: float = 1.0) -> torch.Tensor:
        """The whole decode step of this layer in one library call (append one
        token, attention, selection, compaction); same results as `step`.
        mode "h2o", "streaming" or "block" (see `h2o_select_evict`)."""
        _need(q, torch.bfloat16, "q", self.device)
        _need(k_new, torch.bfloat16, "k_new", self.device)
        _need(v_new, torch.bfloat16, "v_new", self.device)
        batch = q.shape[0]
        if q.dim() != 3 or q.shape[1] != self.num_q_heads or q.shape[2] != HEAD_DIM:
            raise ValueError("q must be [batch, num_q_heads, 128]")
        if tuple(k_new.shape) != (batch, self.num_kv_heads, 1, HEAD_DIM) or k_new.shape != v_new.shape:
            raise ValueError("k_new, v_new must be [batch, num_kv_heads, 1, 128]")
        if out is None:
            out = torch.empty_like(q)
        _need(out, torch.bfloat16, "out", self.device, q.shape)
        ws = self.workspace(batch) if workspace is None else workspace
        _need(ws, torch.uint8, "workspace", self.device)
        scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
        m = {"h2o": L.KVC_EVICT_H2O, "streaming": L.KVC_EVICT_STREAMING, "block": L.KVC_EVICT_BLOCK}[mode]
        params = L.KvcEvictParams(m, budget, recent, window, retention)
        L.check(self.lib.kvc_decode_step(self.handle, seq_begin, batch, ctypes.c_void_p(q.data_ptr()),
                                         ctypes.c_void_p(k_new.data_ptr()), ctypes.c_void_p(v_new.data_ptr()),
                                         ctypes.c_void_p(out.data_ptr()), ctypes.c_float(scale), ctypes.byref(params),
                                         ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                         ctypes.c_void_p(_stream_ptr(stream))), "kvc_decode_step")
        return out

    def decode_step_overlap(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, evict_stream,
                            mode: str = "h2o", budget: int = 0, recent: int = 0, window: int = 0,
                            seq_begin: int = 0, out=None, sm_scale: float | None = None, workspace=None,
                            stream=None, retention: float = 1.0) -> torch.Tensor:
        """`decode_step` with the eviction (scores, selection, compaction) on
        `evict_stream`, after the output is ready on `stream`.  The workspace
        stays in use until the eviction has run (one per cache); later calls
        on this cache order themselves after it.  Inside a stream capture the
        caller joins `evict_stream` back into `stream` before the capture
        ends."""
        _need(q, torch.bfloat16, "q", self.device)
        _need(k_new, torch.bfloat16, "k_new", self.device)
        _need(v_new, torch.bfloat16, "v_new", self.device)
        batch = q.shape[0]
        if q.dim() != 3 or q.shape[1] != self.num_q_heads or q.shape[2] != HEAD_DIM:
            raise ValueError("q must be [batch, num_q_heads, 128]")
        if tuple(k_new.shape) != (batch, self.num_kv_heads, 1, HEAD_DIM) or k_new.shape != v_new.shape:
            raise ValueError("k_new, v_new must be [batch, num_kv_heads, 1, 128]")
        if out is None:
            out = torch.empty_like(q)
        _need(out, torch.bfloat16, "out", self.device, q.shape)
        ws = self.workspace(batch) if workspace is None else workspace
        _need(ws, torch.uint8, "workspace", self.device)
        scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
        m = {"h2o": L.KVC_EVICT_H2O, "streaming": L.KVC_EVICT_STREAMING, "block": L.KVC_EVICT_BLOCK}[mode]
        params = L.KvcEvictParams(m, budget, recent, window, retention)
        L.check(self.lib.kvc_decode_step_overlap(
            self.handle, seq_begin, batch, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k_new.data_ptr()),
            ctypes.c_void_p(v_new.data_ptr()), ctypes.c_void_p(out.data_ptr()), ctypes.c_float(scale),
            ctypes.byref(params), ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(_stream_ptr(stream)),
            ctypes.c_void_p(_stream_ptr(evict_stream))), "kvc_decode_step_overlap")
        return out

    def step(self, q, k_new, v_new, mode="h2o", budget=0, recent=0, window=0, seq_begin=0, out=None,
             keep_mask=None, stream=None, retention=1.0):
        """One decode step of this layer: append -> attention (+H2O) -> select -> compact."""
        batch = q.shape[0]
        self.quantize_append(k_new, v_new, seq_begin=seq_begin, stream=stream)
        out = self.decode_attention(q, out=out, seq_begin=seq_begin, accumulate_h2o=(mode != "streaming"),
                                    stream=stream)
        mask = self.h2o_select_evict(batch, mode=mode, budget=budget, recent=recent, window=window,
                                     seq_begin=seq_begin, keep_mask=keep_mask, stream=stream, retention=retention)
        self.compact_blocks(mask, batch, seq_begin=seq_begin, stream=stream)
        return out
