"""Thin ctypes binding of ``liboasis.so`` with the C ABI's names.

Argument marshalling only: every function takes torch tensors (or raw integer
pointers), passes their addresses, sizes and the current CUDA stream to the
library, and raises :class:`OasisError` when the library returns a non-OK
status.  No computation of the method happens here.  If the library is missing
the import of a function raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboasis.so")

OASIS_OK = 0
STATUS_NAMES = {0: "OK", 1: "ERR_INVALID", 2: "ERR_CUDA", 3: "ERR_TIMEOUT", 4: "ERR_UNSUPPORTED"}

EW_BAD_BLOCK = 0x1
EW_BAD_SLOT = 0x2
EW_NO_SLOT = 0x4
EW_BAD_COUNT = 0x8
EW_TIMEOUT = 0x10


class OasisError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "Hq", "Hkv", "d", "bs", "nb_max", "n_la", "Kb", "P")]

    @classmethod
    def of(cls, B, Hq, Hkv, nb_max, n_la, Kb, P, d=128, bs=16) -> "Shape":
        return cls(B, Hq, Hkv, d, bs, nb_max, n_la, Kb, P)

    @classmethod
    def from_workload(cls, w) -> "Shape":
        return cls(w.B, w.Hq, w.Hkv, w.d, w.bs, w.nb_max, w.n_la, w.Kb, w.P)

    def astuple(self):
        return tuple(getattr(self, n) for n, _ in self._fields_)


_VP = ctypes.c_void_p
_SIGS = {
    "oasis_version": ([], ctypes.c_char_p),
    "oasis_last_error": ([], ctypes.c_char_p),
    "oasis_score_blocks": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "oasis_score_blocks_dynamic": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, ctypes.c_int32, _VP],
                                   ctypes.c_int),
    "oasis_topk_select": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "oasis_fetch_diff_capped": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                 ctypes.c_int32, _VP, _VP, _VP], ctypes.c_int),
    "oasis_gather_h2d": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                          _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "oasis_assign_slots": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP],
                           ctypes.c_int),
    "oasis_copy_fetched": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "oasis_copy_fetched_wait": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_uint32,
                                 ctypes.c_int32, _VP, _VP], ctypes.c_int),
    "oasis_error_word_status": ([_VP, _VP, _VP], ctypes.c_int),
    "oasis_score_blocks_copy": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                 _VP, _VP, _VP], ctypes.c_int),
    "oasis_set_agreement": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "oasis_pool_keys": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP], ctypes.c_int),
    "oasis_pool_append": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "oasis_score_blocks_pooled": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                   _VP, _VP, _VP], ctypes.c_int),
    "oasis_topk_select_pooled": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "oasis_fetch_diff_capped_pooled": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                        ctypes.c_int32, _VP, _VP, _VP], ctypes.c_int),
    "oasis_attn_lookahead_workspace_bytes": ([ctypes.POINTER(Shape)], ctypes.c_size_t),
    "oasis_sparse_decode_attn_lookahead": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                            ctypes.c_float, _VP, ctypes.c_size_t, _VP, _VP, _VP], ctypes.c_int),
    "oasis_topk_select_diff": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, ctypes.c_int32, _VP, _VP, _VP,
                                _VP, _VP, _VP], ctypes.c_int),
    "oasis_topk_select_diff_pooled": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, ctypes.c_int32, _VP, _VP,
                                       _VP, _VP, _VP, _VP], ctypes.c_int),
    "oasis_touch_host": ([_VP, ctypes.c_size_t, _VP, _VP], ctypes.c_int),
    "oasis_set_option": ([ctypes.c_int32, ctypes.c_int32], ctypes.c_int),
    "oasis_trace_bytes": ([ctypes.c_int32], ctypes.c_size_t),
    "oasis_trace_set": ([_VP, ctypes.c_int32], ctypes.c_int),
    "oasis_sparse_decode_attn": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                  ctypes.c_float, _VP, ctypes.c_size_t, _VP, _VP], ctypes.c_int),
    "oasis_attn_workspace_bytes": ([ctypes.POINTER(Shape)], ctypes.c_size_t),
    "oasis_sparse_decode_attn_noalloc": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                          ctypes.c_float, _VP, _VP], ctypes.c_int),
    "oasis_append_kv": ([ctypes.POINTER(Shape), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_int32,
                         _VP, _VP], ctypes.c_int),
}

_lib = None


def load(path: Optional[str] = None):
    """Load liboasis.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with sparse_decode_attention_oasis_gb300.build.build()")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIGS.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    if path is None:
        _lib = lib
    return lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int):
    if st != OASIS_OK:
        raise OasisError(fn, st, load().oasis_last_error().decode())


def oasis_version() -> str:
    return load().oasis_version().decode()


def oasis_last_error() -> str:
    return load().oasis_last_error().decode()


def oasis_attn_workspace_bytes(shape: Shape) -> int:
    return int(load().oasis_attn_workspace_bytes(ctypes.byref(shape)))


def oasis_score_blocks(shape: Shape, k_hbm, ctx_len, q_la, scores, err_word=None, stream=None):
    _check("oasis_score_blocks", load().oasis_score_blocks(
        ctypes.byref(shape), _ptr(k_hbm), _ptr(ctx_len), _ptr(q_la), _ptr(scores), _ptr(err_word),
        _stream(stream)))


def oasis_score_blocks_dynamic(shape: Shape, k_hbm, ctx_len, q_la, scores, work, reserve_ctas: int = 0,
                               stream=None):
    """oasis_score_blocks with chunks from an atomic counter (work: device int32/uint32 [2],
    zero before the call and left zero after it); reserve_ctas thread-block slots stay free."""
    _check("oasis_score_blocks_dynamic", load().oasis_score_blocks_dynamic(
        ctypes.byref(shape), _ptr(k_hbm), _ptr(ctx_len), _ptr(q_la), _ptr(scores), _ptr(work), int(reserve_ctas),
        _stream(stream)))


def oasis_topk_select(shape: Shape, scores, k_hbm, q_la, ctx_len, sel, nsel, stream=None):
    _check("oasis_topk_select", load().oasis_topk_select(
        ctypes.byref(shape), _ptr(scores), _ptr(k_hbm), _ptr(q_la), _ptr(ctx_len), _ptr(sel),
        _ptr(nsel), _stream(stream)))


def oasis_fetch_diff_capped(shape: Shape, scores, k_hbm, q_la, ctx_len, sel, nsel, blk2slot,
                            fetch_cap: int, fetch, nfetch, stream=None):
    _check("oasis_fetch_diff_capped", load().oasis_fetch_diff_capped(
        ctypes.byref(shape), _ptr(scores), _ptr(k_hbm), _ptr(q_la), _ptr(ctx_len), _ptr(sel),
        _ptr(nsel), _ptr(blk2slot), int(fetch_cap), _ptr(fetch), _ptr(nfetch), _stream(stream)))


def oasis_gather_h2d(shape: Shape, host_kv, sel, nsel, fetch, nfetch, blk2slot, slot2blk,
                     last_used, step, k_pool, v_pool, err_word, stream=None):
    """``step`` is a device int32 tensor of one element (the LRU clock value)."""
    _check("oasis_gather_h2d", load().oasis_gather_h2d(
        ctypes.byref(shape), _ptr(host_kv), _ptr(sel), _ptr(nsel), _ptr(fetch), _ptr(nfetch),
        _ptr(blk2slot), _ptr(slot2blk), _ptr(last_used), _ptr(step), _ptr(k_pool), _ptr(v_pool),
        _ptr(err_word), _stream(stream)))


def oasis_assign_slots(shape: Shape, sel, nsel, fetch, nfetch, blk2slot, slot2blk, last_used, step,
                       err_word, stream=None):
    """Table half of the gather (slots, evictions, LRU clock); the pools are not touched."""
    _check("oasis_assign_slots", load().oasis_assign_slots(
        ctypes.byref(shape), _ptr(sel), _ptr(nsel), _ptr(fetch), _ptr(nfetch), _ptr(blk2slot),
        _ptr(slot2blk), _ptr(last_used), _ptr(step), _ptr(err_word), _stream(stream)))


def oasis_copy_fetched(shape: Shape, host_kv, fetch, nfetch, blk2slot, k_pool, v_pool, err_word,
                       stream=None):
    """Data half of the gather: host tier -> the slots oasis_assign_slots gave the fetch list."""
    _check("oasis_copy_fetched", load().oasis_copy_fetched(
        ctypes.byref(shape), _ptr(host_kv), _ptr(fetch), _ptr(nfetch), _ptr(blk2slot), _ptr(k_pool),
        _ptr(v_pool), _ptr(err_word), _stream(stream)))


def oasis_copy_fetched_wait(shape: Shape, host_kv, fetch, nfetch, blk2slot, k_pool, v_pool, ready_flag,
                            ready_value: int, max_polls: int, err_word, stream=None):
    """oasis_copy_fetched after a bounded wait for *ready_flag >= ready_value (a uint32 in
    page-locked mapped host memory); on expiry nothing is copied and err_word gets EW_TIMEOUT."""
    _check("oasis_copy_fetched_wait", load().oasis_copy_fetched_wait(
        ctypes.byref(shape), _ptr(host_kv), _ptr(fetch), _ptr(nfetch), _ptr(blk2slot), _ptr(k_pool),
        _ptr(v_pool), _ptr(ready_flag), int(ready_value), int(max_polls), _ptr(err_word), _stream(stream)))


def oasis_error_word_status(err_word, stream=None):
    """(status, bits): waits for the stream and reads the error word; status is
    ERR_TIMEOUT (3) when a bounded wait gave up, else OK (0).  Does not raise."""
    bits = ctypes.c_uint32(0)
    st = load().oasis_error_word_status(_ptr(err_word), _stream(stream), ctypes.byref(bits))
    return int(st), int(bits.value)


def oasis_score_blocks_copy(shape: Shape, k_hbm, ctx_len, q_la, scores, host_kv, fetch, nfetch,
                            blk2slot, k_pool, v_pool, err_word, stream=None):
    """Block scoring of one layer carrying the data half of another layer's gather."""
    _check("oasis_score_blocks_copy", load().oasis_score_blocks_copy(
        ctypes.byref(shape), _ptr(k_hbm), _ptr(ctx_len), _ptr(q_la), _ptr(scores), _ptr(host_kv),
        _ptr(fetch), _ptr(nfetch), _ptr(blk2slot), _ptr(k_pool), _ptr(v_pool), _ptr(err_word),
        _stream(stream)))


def oasis_set_agreement(shape: Shape, pred, npred, exact, nexact, blk2slot, counts, err_word=None,
                        stream=None):
    """Per head (|pred & exact|, |pred & exact & resident| or -1, |exact|) into counts [B][Hkv][3]."""
    _check("oasis_set_agreement", load().oasis_set_agreement(
        ctypes.byref(shape), _ptr(pred), _ptr(npred), _ptr(exact), _ptr(nexact), _ptr(blk2slot),
        _ptr(counts), _ptr(err_word), _stream(stream)))


def oasis_pool_keys(shape: Shape, k_hbm, ctx_len, k_pooled, stream=None):
    """Min/max pooled compressed keys bf16 [B][Hkv][nb_max][2][d] from the full keys."""
    _check("oasis_pool_keys", load().oasis_pool_keys(
        ctypes.byref(shape), _ptr(k_hbm), _ptr(ctx_len), _ptr(k_pooled), _stream(stream)))


def oasis_pool_append(shape: Shape, k_new, ctx_len, k_pooled, err_word=None, stream=None):
    """Fold each request's new key at position ctx_len[b] into its block's pooled rows."""
    _check("oasis_pool_append", load().oasis_pool_append(
        ctypes.byref(shape), _ptr(k_new), _ptr(ctx_len), _ptr(k_pooled), _ptr(err_word), _stream(stream)))


def oasis_score_blocks_pooled(shape: Shape, k_pooled, ctx_len, q_la, scores, host_kv=None, fetch=None,
                              nfetch=None, blk2slot=None, k_pool=None, v_pool=None, err_word=None,
                              stream=None):
    """Pooled block scores; with host_kv the launch also carries a gather's copy half."""
    _check("oasis_score_blocks_pooled", load().oasis_score_blocks_pooled(
        ctypes.byref(shape), _ptr(k_pooled), _ptr(ctx_len), _ptr(q_la), _ptr(scores), _ptr(host_kv),
        _ptr(fetch), _ptr(nfetch), _ptr(blk2slot), _ptr(k_pool), _ptr(v_pool), _ptr(err_word),
        _stream(stream)))


def oasis_topk_select_pooled(shape: Shape, scores, k_pooled, q_la, ctx_len, sel, nsel, stream=None):
    _check("oasis_topk_select_pooled", load().oasis_topk_select_pooled(
        ctypes.byref(shape), _ptr(scores), _ptr(k_pooled), _ptr(q_la), _ptr(ctx_len), _ptr(sel), _ptr(nsel),
        _stream(stream)))


def oasis_fetch_diff_capped_pooled(shape: Shape, scores, k_pooled, q_la, ctx_len, sel, nsel, blk2slot,
                                   fetch_cap: int, fetch, nfetch, stream=None):
    _check("oasis_fetch_diff_capped_pooled", load().oasis_fetch_diff_capped_pooled(
        ctypes.byref(shape), _ptr(scores), _ptr(k_pooled), _ptr(q_la), _ptr(ctx_len), _ptr(sel), _ptr(nsel),
        _ptr(blk2slot), int(fetch_cap), _ptr(fetch), _ptr(nfetch), _stream(stream)))


def oasis_attn_lookahead_workspace_bytes(shape: Shape) -> int:
    return int(load().oasis_attn_lookahead_workspace_bytes(ctypes.byref(shape)))


def oasis_sparse_decode_attn_lookahead(shape: Shape, q, q_la, k_pool, v_pool, sel, nsel, blk2slot, ctx_len,
                                       scale: float, workspace, ws_bytes: int, out, out_la, stream=None):
    """True and lookahead queries over the same sparse KV: out [B][Hq][d], out_la [B][n_la][Hq][d]."""
    _check("oasis_sparse_decode_attn_lookahead", load().oasis_sparse_decode_attn_lookahead(
        ctypes.byref(shape), _ptr(q), _ptr(q_la), _ptr(k_pool), _ptr(v_pool), _ptr(sel), _ptr(nsel),
        _ptr(blk2slot), _ptr(ctx_len), float(scale), _ptr(workspace), int(ws_bytes), _ptr(out), _ptr(out_la),
        _stream(stream)))


def oasis_topk_select_diff(shape: Shape, scores, k_hbm, q_la, ctx_len, blk2slot, fetch_cap: int, sel, nsel,
                           fetch, nfetch, host_kv=None, stream=None):
    """Top-K and the capped diff in one launch (host_kv: prefetch the fetched blocks into L2)."""
    _check("oasis_topk_select_diff", load().oasis_topk_select_diff(
        ctypes.byref(shape), _ptr(scores), _ptr(k_hbm), _ptr(q_la), _ptr(ctx_len), _ptr(blk2slot), int(fetch_cap),
        _ptr(sel), _ptr(nsel), _ptr(fetch), _ptr(nfetch), _ptr(host_kv), _stream(stream)))


def oasis_topk_select_diff_pooled(shape: Shape, scores, k_pooled, q_la, ctx_len, blk2slot, fetch_cap: int, sel,
                                  nsel, fetch, nfetch, host_kv=None, stream=None):
    _check("oasis_topk_select_diff_pooled", load().oasis_topk_select_diff_pooled(
        ctypes.byref(shape), _ptr(scores), _ptr(k_pooled), _ptr(q_la), _ptr(ctx_len), _ptr(blk2slot),
        int(fetch_cap), _ptr(sel), _ptr(nsel), _ptr(fetch), _ptr(nfetch), _ptr(host_kv), _stream(stream)))


def oasis_touch_host(host_tensor, nbytes: Optional[int] = None, sink=None, stream=None):
    """Read a pinned, mapped host range once through the SMs' load path (host-tier warm-up)."""
    n = host_tensor.numel() * host_tensor.element_size() if nbytes is None else int(nbytes)
    _check("oasis_touch_host", load().oasis_touch_host(_ptr(host_tensor), n, _ptr(sink), _stream(stream)))


OPT_SCORE_CTAS_PER_SM = 1
OPT_SCORE_KERNEL = 2
OPT_COPY_CTAS = 3
OPT_SCORE_STATIC_SHARE = 4
SCORE_KERNEL_MMA = 0
SCORE_KERNEL_TC = 1


def oasis_set_option(option: int, value: int):
    """Process-wide launch option (OPT_SCORE_CTAS_PER_SM: scorer CTAs per SM, 0 = as many as
    fit; OPT_SCORE_KERNEL: SCORE_KERNEL_MMA or SCORE_KERNEL_TC)."""
    _check("oasis_set_option", load().oasis_set_option(int(option), int(value)))


TRACE_KINDS = 7
TRACE_SCORE, TRACE_SCORE_POOLED, TRACE_SELECT, TRACE_GATHER, TRACE_COPY, TRACE_ATTN, TRACE_APPEND = range(7)
TRACE_HEADER_BYTES = 128


def oasis_trace_bytes(capacity: int) -> int:
    return int(load().oasis_trace_bytes(int(capacity)))


def oasis_trace_set(dev_buf, capacity: int = 0):
    """Make later launches record their spans into dev_buf (None: tracing off)."""
    _check("oasis_trace_set", load().oasis_trace_set(_ptr(dev_buf), int(capacity)))


def oasis_sparse_decode_attn(shape: Shape, q, k_pool, v_pool, sel, nsel, blk2slot, ctx_len,
                             scale: float, workspace, ws_bytes: int, out, stream=None):
    _check("oasis_sparse_decode_attn", load().oasis_sparse_decode_attn(
        ctypes.byref(shape), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(sel), _ptr(nsel),
        _ptr(blk2slot), _ptr(ctx_len), float(scale), _ptr(workspace), int(ws_bytes), _ptr(out),
        _stream(stream)))


def oasis_append_kv(shape: Shape, k_new, v_new, ctx_len, k_hbm, host_kv, blk2slot, k_pool, v_pool,
                    advance: bool = True, err_word=None, stream=None):
    _check("oasis_append_kv", load().oasis_append_kv(
        ctypes.byref(shape), _ptr(k_new), _ptr(v_new), _ptr(ctx_len), _ptr(k_hbm), _ptr(host_kv),
        _ptr(blk2slot), _ptr(k_pool), _ptr(v_pool), 1 if advance else 0, _ptr(err_word), _stream(stream)))


def oasis_sparse_decode_attn_noalloc(shape: Shape, q, k_pool, v_pool, sel, nsel, blk2slot, ctx_len,
                                     scale: float, out, stream=None):
    """Attention with the library's built-in device scratch instead of a workspace."""
    _check("oasis_sparse_decode_attn_noalloc", load().oasis_sparse_decode_attn_noalloc(
        ctypes.byref(shape), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(sel), _ptr(nsel),
        _ptr(blk2slot), _ptr(ctx_len), float(scale), _ptr(out), _stream(stream)))
