"""GB300 (sm_103a) paged MXFP4 index-K scorer: thin Python binding of the C ABI.

The computation runs entirely in the CUDA library ``_build/libmx4index.so``
(declared in ``include/mx4_index.h``); this module only marshals torch tensors
into pointers and sizes.  There is no CPU fallback: every entry point raises
if the library is missing or the call is rejected.

Entry points (same names as the C ABI):

* ``mx4_index_score_prefill`` / ``mx4_index_score_decode``: block scores
  ``[rows, 64, ceil(max_seq_len/128)]`` fp32.
* ``mx4_index_logits_prefill`` / ``mx4_index_logits_decode``: per-token
  logits ``[rows, 64, max_seq_len]`` fp32.
* ``mx4_quantize_q_e4m3``: the bf16 -> e4m3 query rounding on its own.
* ``mx4_index_get_device_status``: device-side error bits.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .buildlib import LIB_PATH, build  # noqa: F401

HEADS = 64
DIM = 128
PAGE = 128

MX4_OK = 0
MX4_ERR_INVALID_ARG = 1
MX4_ERR_MISALIGNED = 2
MX4_ERR_UNSUPPORTED = 3
MX4_ERR_CUDA = 4
MX4_DEV_BAD_PAGE = 0x1
MX4_DEV_TIMEOUT = 0x2

# exported symbols, in the order include/mx4_index.h declares them
EXPORTED_SYMBOLS = (
    "mx4_index_score_prefill",
    "mx4_index_score_decode",
    "mx4_index_logits_prefill",
    "mx4_index_logits_decode",
    "mx4_index_score_prefill_fp8",
    "mx4_index_score_decode_fp8",
    "mx4_index_logits_prefill_fp8",
    "mx4_index_logits_decode_fp8",
    "mx4_index_topk_prefill",
    "mx4_index_topk_decode",
    "mx4_sparse_pa_decode",
    "mx4_quantize_q_e4m3",
    "mx4_index_k_write",
    "mx4_index_get_device_status",
    "mx4_status_string",
    "mx4_abi_version",
)


class Mx4Error(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} ({status})")
        self.status = status


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"the CUDA library {path} is not built; run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        _lib = configure_library(ctypes.CDLL(path))
        return _lib


def configure_library(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the argument and result types of every exported entry point
    on a loaded copy of the library."""
    i32, i64, f32, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
    prefill_args = [vp, i32, vp, vp, i64, i64, vp, vp, vp, vp, i32, i32, f32, vp, vp, i32, i64, i64]
    decode_args = [vp, i32, vp, vp, i64, i64, vp, vp, i32, f32, vp, vp, i32, i64, i64]
    for name, args in (("mx4_index_score_prefill", prefill_args),
                       ("mx4_index_logits_prefill", prefill_args),
                       ("mx4_index_score_decode", decode_args),
                       ("mx4_index_logits_decode", decode_args)):
        f = getattr(lib, name)
        f.restype = i32
        f.argtypes = args
    prefill_fp8_args = [vp, i32, vp, i64, vp, vp, vp, vp, i32, i32, f32, vp, vp, i32, i64, i64]
    decode_fp8_args = [vp, i32, vp, i64, vp, vp, i32, f32, vp, vp, i32, i64, i64]
    for name, args in (("mx4_index_score_prefill_fp8", prefill_fp8_args),
                       ("mx4_index_logits_prefill_fp8", prefill_fp8_args),
                       ("mx4_index_score_decode_fp8", decode_fp8_args),
                       ("mx4_index_logits_decode_fp8", decode_fp8_args)):
        f = getattr(lib, name)
        f.restype = i32
        f.argtypes = args
    lib.mx4_index_topk_prefill.restype = i32
    lib.mx4_index_topk_prefill.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, i32, i64]
    lib.mx4_index_topk_decode.restype = i32
    lib.mx4_index_topk_decode.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, i32, i64]
    lib.mx4_sparse_pa_decode.restype = i32
    lib.mx4_sparse_pa_decode.argtypes = [vp, i64, i32, i32, vp, vp, i64, i64, i64, i64, vp, vp, i64, i64, i64,
                                         i64, vp, i32, vp, f32, vp, i64, vp]
    lib.mx4_quantize_q_e4m3.restype = i32
    lib.mx4_quantize_q_e4m3.argtypes = [vp, vp, i64, vp]
    lib.mx4_index_k_write.restype = i32
    lib.mx4_index_k_write.argtypes = [vp, i64, i64, vp, vp, vp, i64, i64, i64, vp]
    lib.mx4_index_get_device_status.restype = i32
    lib.mx4_index_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.mx4_status_string.restype = ctypes.c_char_p
    lib.mx4_status_string.argtypes = [i32]
    lib.mx4_abi_version.restype = i32
    lib.mx4_abi_version.argtypes = []
    return lib


def _check(fn: str, status: int):
    if status != MX4_OK:
        lib = load_library()
        raise Mx4Error(fn, status, lib.mx4_status_string(status).decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _out(out, shape, like):
    import torch
    if out is None:
        return torch.empty(shape, dtype=torch.float32, device=like.device)
    if out.dtype != torch.float32 or tuple(out.shape) != tuple(shape) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous float32 tensor of shape {tuple(shape)}")
    return out


def _q_info(q):
    import torch
    if q.dtype == torch.bfloat16:
        e4 = 0
    elif q.dtype in (torch.uint8, torch.float8_e4m3fn):
        e4 = 1
    else:
        raise ValueError("q must be bfloat16 or e4m3 (float8_e4m3fn / uint8 bytes)")
    if q.dim() != 3 or q.shape[1] != HEADS or q.shape[2] != DIM or not q.is_contiguous():
        raise ValueError("q must be a contiguous [rows, 64, 128] tensor")
    return e4


def mx4_index_score_prefill(q, k_data, k_scale, k_data_page_stride, k_scale_page_stride, block_table,
                            cu_seqlens_q, seq_lens, prefix_lens, max_query_len, max_seq_len, sm_scale,
                            out=None, *, num_pool_pages, stream=None, logits=False):
    """Block scores (or per-token logits with ``logits=True``) for prefill rows.

    ``k_data`` / ``k_scale`` are uint8 tensors whose first byte is page 0 of
    the respective view (e.g. a flat pool and the same pool offset by 8192);
    ``num_pool_pages`` is the number of pages both views address."""
    lib = load_library()
    e4 = _q_info(q)
    P = (max_seq_len + PAGE - 1) // PAGE
    ncols = max_seq_len if logits else P
    out = _out(out, (q.shape[0], HEADS, ncols), q)
    fn = "mx4_index_logits_prefill" if logits else "mx4_index_score_prefill"
    st = getattr(lib, fn)(
        _ptr(q), e4, _ptr(k_data), _ptr(k_scale), int(k_data_page_stride), int(k_scale_page_stride),
        _ptr(block_table), _ptr(cu_seqlens_q), _ptr(seq_lens), _ptr(prefix_lens), int(max_query_len),
        int(max_seq_len), float(sm_scale), _ptr(out), _stream(stream), int(seq_lens.shape[0]),
        int(block_table.stride(0)) if block_table.dim() == 2 else int(block_table.shape[-1]),
        int(num_pool_pages))
    _check(fn, st)
    return out


def mx4_index_score_decode(q, k_data, k_scale, k_data_page_stride, k_scale_page_stride, block_table,
                           seq_lens, max_seq_len, sm_scale, out=None, *, num_pool_pages, stream=None,
                           logits=False):
    """Block scores (or per-token logits with ``logits=True``) for decode rows
    (one query row per request)."""
    lib = load_library()
    e4 = _q_info(q)
    P = (max_seq_len + PAGE - 1) // PAGE
    ncols = max_seq_len if logits else P
    out = _out(out, (q.shape[0], HEADS, ncols), q)
    fn = "mx4_index_logits_decode" if logits else "mx4_index_score_decode"
    st = getattr(lib, fn)(
        _ptr(q), e4, _ptr(k_data), _ptr(k_scale), int(k_data_page_stride), int(k_scale_page_stride),
        _ptr(block_table), _ptr(seq_lens), int(max_seq_len), float(sm_scale), _ptr(out),
        _stream(stream), int(seq_lens.shape[0]),
        int(block_table.stride(0)) if block_table.dim() == 2 else int(block_table.shape[-1]),
        int(num_pool_pages))
    _check(fn, st)
    return out


def mx4_index_logits_prefill(*args, **kwargs):
    return mx4_index_score_prefill(*args, logits=True, **kwargs)


def mx4_index_logits_decode(*args, **kwargs):
    return mx4_index_score_decode(*args, logits=True, **kwargs)


def _bt_stride(block_table):
    return int(block_table.stride(0)) if block_table.dim() == 2 else int(block_table.shape[-1])


def mx4_index_score_prefill_fp8(q, k_fp8, k_page_stride, block_table, cu_seqlens_q, seq_lens, prefix_lens,
                                max_query_len, max_seq_len, sm_scale, out=None, *, num_pool_pages,
                                stream=None, logits=False):
    """Prefill block scores (or logits) over an fp8 index cache: ``k_fp8`` is
    a uint8 tensor whose first byte is page 0 (128 tokens x 128 e4m3 bytes)."""
    lib = load_library()
    e4 = _q_info(q)
    P = (max_seq_len + PAGE - 1) // PAGE
    out = _out(out, (q.shape[0], HEADS, max_seq_len if logits else P), q)
    fn = "mx4_index_logits_prefill_fp8" if logits else "mx4_index_score_prefill_fp8"
    st = getattr(lib, fn)(
        _ptr(q), e4, _ptr(k_fp8), int(k_page_stride), _ptr(block_table), _ptr(cu_seqlens_q), _ptr(seq_lens),
        _ptr(prefix_lens), int(max_query_len), int(max_seq_len), float(sm_scale), _ptr(out), _stream(stream),
        int(seq_lens.shape[0]), _bt_stride(block_table), int(num_pool_pages))
    _check(fn, st)
    return out


def mx4_index_score_decode_fp8(q, k_fp8, k_page_stride, block_table, seq_lens, max_seq_len, sm_scale,
                               out=None, *, num_pool_pages, stream=None, logits=False):
    """Decode block scores (or logits) over an fp8 index cache."""
    lib = load_library()
    e4 = _q_info(q)
    P = (max_seq_len + PAGE - 1) // PAGE
    out = _out(out, (q.shape[0], HEADS, max_seq_len if logits else P), q)
    fn = "mx4_index_logits_decode_fp8" if logits else "mx4_index_score_decode_fp8"
    st = getattr(lib, fn)(
        _ptr(q), e4, _ptr(k_fp8), int(k_page_stride), _ptr(block_table), _ptr(seq_lens), int(max_seq_len),
        float(sm_scale), _ptr(out), _stream(stream), int(seq_lens.shape[0]), _bt_stride(block_table),
        int(num_pool_pages))
    _check(fn, st)
    return out


def mx4_index_logits_prefill_fp8(*args, **kwargs):
    return mx4_index_score_prefill_fp8(*args, logits=True, **kwargs)


def mx4_index_logits_decode_fp8(*args, **kwargs):
    return mx4_index_score_decode_fp8(*args, logits=True, **kwargs)


def _topk_out(sel, count, rows, groups, topk, like):
    import torch
    if sel is None:
        sel = torch.empty((rows, groups, topk), dtype=torch.int32, device=like.device)
    if count is None:
        count = torch.empty((rows, groups), dtype=torch.int32, device=like.device)
    if sel.dtype != torch.int32 or tuple(sel.shape) != (rows, groups, topk) or not sel.is_contiguous():
        raise ValueError(f"sel must be a contiguous int32 tensor of shape {(rows, groups, topk)}")
    if count.dtype != torch.int32 or tuple(count.shape) != (rows, groups) or not count.is_contiguous():
        raise ValueError(f"count must be a contiguous int32 tensor of shape {(rows, groups)}")
    return sel, count


def _topk_tokens(tokens, want_tokens, rows, kv_groups, like):
    import torch
    if tokens is None and want_tokens:
        tokens = torch.empty((rows, kv_groups), dtype=torch.int32, device=like.device)
    if tokens is not None and (tokens.dtype != torch.int32 or tuple(tokens.shape) != (rows, kv_groups)
                               or not tokens.is_contiguous()):
        raise ValueError(f"tokens must be a contiguous int32 tensor of shape {(rows, kv_groups)}")
    return tokens


def mx4_index_topk_prefill(scores, block_table, cu_seqlens_q, seq_lens, prefix_lens, max_query_len, max_seq_len,
                           topk, *, local_pages=1, kv_groups=1, sel=None, count=None, tokens=None,
                           want_tokens=False, stream=None):
    """Top-k page selection over prefill block scores ``scores`` [rows, 64, P]
    (the scorer's output).  Returns (sel int32 [rows, kv_groups, topk],
    count int32 [rows, kv_groups]), plus tokens int32 [rows, kv_groups] (the
    live tokens of the selected pages) when ``tokens`` is given or
    ``want_tokens`` is set."""
    import torch
    lib = load_library()
    if scores.dtype != torch.float32 or scores.dim() != 3 or not scores.is_contiguous():
        raise ValueError("scores must be a contiguous float32 [rows, 64, P] tensor")
    sel, count = _topk_out(sel, count, scores.shape[0], kv_groups, topk, scores)
    tok = _topk_tokens(tokens, want_tokens, scores.shape[0], kv_groups, scores)
    fn = "mx4_index_topk_prefill"
    _check(fn, lib.mx4_index_topk_prefill(
        _ptr(scores), _ptr(block_table), _ptr(cu_seqlens_q), _ptr(seq_lens), _ptr(prefix_lens), int(max_query_len),
        int(max_seq_len), int(topk), int(local_pages), int(kv_groups), _ptr(sel), _ptr(count), _ptr(tok),
        _stream(stream), int(seq_lens.shape[0]), _bt_stride(block_table)))
    return (sel, count) if tok is None else (sel, count, tok)


def mx4_index_topk_decode(scores, block_table, seq_lens, max_seq_len, topk, *, local_pages=1, kv_groups=1,
                          sel=None, count=None, tokens=None, want_tokens=False, stream=None):
    """Top-k page selection over decode block scores (one row per request);
    returns as ``mx4_index_topk_prefill``."""
    import torch
    lib = load_library()
    if scores.dtype != torch.float32 or scores.dim() != 3 or not scores.is_contiguous():
        raise ValueError("scores must be a contiguous float32 [rows, 64, P] tensor")
    sel, count = _topk_out(sel, count, scores.shape[0], kv_groups, topk, scores)
    tok = _topk_tokens(tokens, want_tokens, scores.shape[0], kv_groups, scores)
    fn = "mx4_index_topk_decode"
    _check(fn, lib.mx4_index_topk_decode(
        _ptr(scores), _ptr(block_table), _ptr(seq_lens), int(max_seq_len), int(topk), int(local_pages),
        int(kv_groups), _ptr(sel), _ptr(count), _ptr(tok), _stream(stream), int(seq_lens.shape[0]),
        _bt_stride(block_table)))
    return (sel, count) if tok is None else (sel, count, tok)


def mx4_sparse_pa_decode(q, k_pool, v_pool, block_table, context_lens, softmax_scale, out=None, *,
                         stream=None):
    """Sparse paged-attention decode over MXFP4 K/V pools [pages, kv_heads,
    8704] (codes at byte 0, scales at byte 8192 of each page).  ``q``: e4m3
    bytes [rows, kv_heads, groups, 128]; ``block_table``: int32 [rows,
    kv_heads, width]; ``context_lens``: int32 [rows, kv_heads].  Returns bf16
    [rows, kv_heads, groups, 128]."""
    import torch
    lib = load_library()
    if q.dtype not in (torch.uint8, torch.float8_e4m3fn) or q.dim() != 4 or q.shape[3] != DIM \
            or not q.is_contiguous():
        raise ValueError("q must be a contiguous e4m3 [rows, kv_heads, groups, 128] tensor")
    rows, kvh, groups, _ = q.shape
    for pool in (k_pool, v_pool):
        if pool.dtype != torch.uint8 or pool.dim() != 3 or pool.shape[1] != kvh or pool.shape[2] != 8704 \
                or not pool.is_contiguous():
            raise ValueError("pools must be contiguous uint8 [pages, kv_heads, 8704] tensors")
    if v_pool.shape[0] != k_pool.shape[0]:
        raise ValueError("k_pool and v_pool must hold the same number of pages")
    if block_table.dtype != torch.int32 or block_table.dim() != 3 or not block_table.is_contiguous():
        raise ValueError("block_table must be a contiguous int32 [rows, kv_heads, width] tensor")
    if context_lens.dtype != torch.int32 or not context_lens.is_contiguous():
        raise ValueError("context_lens must be a contiguous int32 [rows, kv_heads] tensor")
    if out is None:
        out = torch.empty((rows, kvh, groups, DIM), dtype=torch.bfloat16, device=q.device)
    ps = kvh * 8704
    kd = k_pool.data_ptr()
    vd = v_pool.data_ptr()
    _check("mx4_sparse_pa_decode", lib.mx4_sparse_pa_decode(
        _ptr(q), rows, kvh, groups, kd, kd + 8192, ps, 8704, ps, 8704, vd, vd + 8192, ps, 8704, ps, 8704,
        _ptr(block_table), int(block_table.shape[2]), _ptr(context_lens), float(softmax_scale), _ptr(out),
        int(k_pool.shape[0]), _stream(stream)))
    return out


def mx4_quantize_q_e4m3(q_bf16, out=None, *, stream=None):
    """bf16 tensor -> uint8 tensor of e4m3 bytes (same shape)."""
    import torch
    lib = load_library()
    if q_bf16.dtype != torch.bfloat16 or not q_bf16.is_contiguous():
        raise ValueError("q_bf16 must be a contiguous bfloat16 tensor")
    if out is None:
        out = torch.empty(q_bf16.shape, dtype=torch.uint8, device=q_bf16.device)
    _check("mx4_quantize_q_e4m3",
           lib.mx4_quantize_q_e4m3(_ptr(q_bf16), _ptr(out), q_bf16.numel(), _stream(stream)))
    return out


def mx4_index_k_write(k, slot_mapping, k_data, k_scale, k_data_page_stride, k_scale_page_stride, *,
                      num_pool_pages=0, stream=None):
    """Quantise bf16 keys into MXFP4 page slots (``mx4_index_k_write``).

    ``k``: bfloat16 [num_tokens, >=128] with unit inner stride (the key is the
    first 128 elements of each row); ``slot_mapping``: int64 [num_tokens]
    (page * 128 + token-in-page, negative = padding); ``k_data`` /
    ``k_scale``: uint8 tensors whose first byte is page 0 of each view.
    Writes in place; returns nothing."""
    import torch
    lib = load_library()
    if k.dtype != torch.bfloat16 or k.dim() != 2 or k.stride(1) != 1:
        raise ValueError("k must be a 2-D bfloat16 tensor with unit inner stride")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_contiguous() \
            or tuple(slot_mapping.shape) != (k.shape[0],):
        raise ValueError("slot_mapping must be a contiguous int64 tensor of shape [num_tokens]")
    if k_data.dtype != torch.uint8 or k_scale.dtype != torch.uint8:
        raise ValueError("k_data and k_scale must be uint8 tensors")
    _check("mx4_index_k_write",
           lib.mx4_index_k_write(_ptr(k), k.shape[0], k.stride(0), _ptr(slot_mapping), _ptr(k_data),
                                 _ptr(k_scale), int(k_data_page_stride), int(k_scale_page_stride),
                                 int(num_pool_pages), _stream(stream)))


def mx4_index_get_device_status(stream=None) -> int:
    """Synchronise ``stream``, return and clear the device status bits."""
    lib = load_library()
    v = ctypes.c_uint32(0)
    _check("mx4_index_get_device_status", lib.mx4_index_get_device_status(_stream(stream), ctypes.byref(v)))
    return int(v.value)
