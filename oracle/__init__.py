"""fp64 CPU oracle for the paged MXFP4 index-K scorer (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package; the product path (``sparse_attention_mxfp4_gb300``) never does, and
this package imports nothing from it.

The arithmetic lives in ``mx4_oracle.c`` (plain C, fp64); this file only
compiles it with gcc and marshals numpy arrays.  Every function states the
passage it follows in the C source.

Parity unpinned: only the cosine-against-bf16 context figure
(``score(..., unquantized=True)``), which the pages report as quantisation
context, not as a pass criterion.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmx4oracle.so")

HEADS = 64
DIM = 128
PAGE = 128

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP) into oracle/_build/."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add, so every product and sum is
    # rounded as written in the source.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c_i64p = ctypes.POINTER(ctypes.c_int64)
        lib.orc_e2m1_value.restype = ctypes.c_double
        lib.orc_e2m1_value.argtypes = [ctypes.c_int]
        lib.orc_e8m0_value.restype = ctypes.c_double
        lib.orc_e8m0_value.argtypes = [ctypes.c_int]
        lib.orc_e4m3_value.restype = ctypes.c_double
        lib.orc_e4m3_value.argtypes = [ctypes.c_int]
        lib.orc_bf16_value.restype = ctypes.c_double
        lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
        lib.orc_e4m3_from_double.restype = ctypes.c_int
        lib.orc_e4m3_from_double.argtypes = [ctypes.c_double]
        lib.orc_bf16_to_e4m3.restype = ctypes.c_int
        lib.orc_bf16_to_e4m3.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_e4m3_n.restype = None
        lib.orc_bf16_to_e4m3_n.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.orc_e4m3_values_n.restype = None
        lib.orc_e4m3_values_n.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.orc_score.restype = ctypes.c_int
        lib.orc_score.argtypes = [
            ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int64,
            c_i64p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.orc_e2m1_from_double.restype = ctypes.c_int
        lib.orc_e2m1_from_double.argtypes = [ctypes.c_double]
        lib.orc_quantize_group.restype = ctypes.c_int
        lib.orc_quantize_group.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        lib.orc_write_index_k.restype = ctypes.c_int64
        lib.orc_write_index_k.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
        lib.orc_score_fp8.restype = ctypes.c_int
        lib.orc_score_fp8.argtypes = [
            ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int64,
            c_i64p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.orc_topk.restype = ctypes.c_int
        lib.orc_topk.argtypes = [
            ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, c_i64p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.orc_pa_decode.restype = ctypes.c_int
        lib.orc_pa_decode.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int]
        lib.orc_live_pairs.restype = ctypes.c_int64
        lib.orc_live_pairs.argtypes = [
            ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_int, c_i64p, ctypes.c_int64]
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u8(a):
    a = np.asarray(a)
    assert a.dtype == np.uint8, a.dtype
    return np.ascontiguousarray(a)


def _i32(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.int32))


# ------------------------------------------------------------------ codecs --
def e2m1_value(code: int) -> float:
    """Value of a 4-bit e2m1 code (MXFP4 element; aiter #7061, "Format")."""
    return _load().orc_e2m1_value(int(code))


def e8m0_value(byte: int) -> float:
    """2^(byte-127) (aiter #7061, "Format": value = e2m1 x 2^(byte-127))."""
    return _load().orc_e8m0_value(int(byte))


def e4m3_value(byte: int) -> float:
    """Value of an e4m3 (fn) byte."""
    return _load().orc_e4m3_value(int(byte))


def bf16_value(bits: int) -> float:
    return _load().orc_bf16_value(int(bits))


def e4m3_from_double(x: float) -> int:
    """RNE, satfinite rounding of a real to an e4m3 byte."""
    return _load().orc_e4m3_from_double(float(x))


def bf16_to_e4m3(bits) -> np.ndarray:
    """Round bf16 bit patterns (uint16 array) to e4m3 bytes, RNE-satfinite
    (aiter #7061, "Kernels": a bf16 query is rounded to e4m3)."""
    a = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    out = np.empty(a.shape, dtype=np.uint8)
    _load().orc_bf16_to_e4m3_n(_ptr(a), _ptr(out), a.size)
    return out


def e4m3_values(codes) -> np.ndarray:
    a = _u8(codes)
    out = np.empty(a.shape, dtype=np.float64)
    _load().orc_e4m3_values_n(_ptr(a), _ptr(out), a.size)
    return out


# ------------------------------------------------------------------ scorer --
def score(*, decode: bool, q: np.ndarray, q_is_e4m3: bool, k_data: np.ndarray,
          k_scale: np.ndarray, k_data_page_stride: int, k_scale_page_stride: int,
          block_table: np.ndarray, block_table_stride: int, seq_lens,
          max_seq_len: int, sm_scale: float, cu_seqlens_q=None, prefix_lens=None,
          rows=None, want_scores: bool = True, want_logits: bool = False,
          unquantized: bool = False, num_pool_pages: int = 0,
          num_threads: int = 0):
    """Block scores and/or per-token logits for the listed query rows, fp64.

    ``q``: [rows_total, 64, 128] uint16 (bf16 bits) or uint8 (e4m3).
    ``k_data`` / ``k_scale``: flat uint8 buffers; page p's data starts at byte
    ``p * k_data_page_stride`` and its scales at ``p * k_scale_page_stride``.
    ``block_table``: int32, request b's page j at ``b * block_table_stride + j``.
    Returns ``(scores, logits)``, each ``None`` unless requested;
    scores [n_rows, 64, ceil(max_seq_len/128)], logits [n_rows, 64, max_seq_len].
    """
    lib = _load()
    q = np.ascontiguousarray(q)
    if q_is_e4m3:
        assert q.dtype == np.uint8
    else:
        assert q.dtype == np.uint16
    k_data = _u8(k_data).reshape(-1)
    k_scale = _u8(k_scale).reshape(-1)
    bt = _i32(block_table).reshape(-1)
    sl = _i32(seq_lens)
    cu = _i32(cu_seqlens_q)
    pl = _i32(prefix_lens)
    num_seqs = int(sl.shape[0])
    if rows is None:
        n_total = num_seqs if decode else int(cu[-1])
        rows = np.arange(n_total, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    P = (max_seq_len + PAGE - 1) // PAGE
    sc = np.empty((n, HEADS, P), dtype=np.float64) if want_scores else None
    lg = np.empty((n, HEADS, max_seq_len), dtype=np.float64) if want_logits else None
    st = lib.orc_score(
        1 if decode else 0, _ptr(q), 1 if q_is_e4m3 else 0, 1 if unquantized else 0,
        _ptr(k_data), _ptr(k_scale), int(k_data_page_stride), int(k_scale_page_stride),
        _ptr(bt), int(block_table_stride), _ptr(cu), _ptr(sl), _ptr(pl),
        num_seqs, int(max_seq_len), float(sm_scale), int(num_pool_pages),
        rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n,
        _ptr(sc), _ptr(lg), int(num_threads))
    if st != 0:
        raise ValueError(f"oracle rejected the inputs (status {st})")
    return sc, lg


def score_fp8(*, decode: bool, q: np.ndarray, q_is_e4m3: bool, k_fp8: np.ndarray, k_page_stride: int,
              block_table: np.ndarray, block_table_stride: int, seq_lens, max_seq_len: int,
              sm_scale: float, cu_seqlens_q=None, prefix_lens=None, rows=None,
              want_scores: bool = True, want_logits: bool = False, num_pool_pages: int = 0,
              num_threads: int = 0):
    """The scorer over an fp8 index cache (the format the MXFP4 cache
    replaces): page p's token i holds 128 e4m3 bytes at
    ``k_fp8[p * k_page_stride + i * 128 :]``, no scale.  Otherwise as
    ``score``."""
    lib = _load()
    q = np.ascontiguousarray(q)
    assert q.dtype == (np.uint8 if q_is_e4m3 else np.uint16)
    k = _u8(k_fp8).reshape(-1)
    bt = _i32(block_table).reshape(-1)
    sl = _i32(seq_lens)
    cu = _i32(cu_seqlens_q)
    pl = _i32(prefix_lens)
    num_seqs = int(sl.shape[0])
    if rows is None:
        n_total = num_seqs if decode else int(cu[-1])
        rows = np.arange(n_total, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    P = (max_seq_len + PAGE - 1) // PAGE
    sc = np.empty((n, HEADS, P), dtype=np.float64) if want_scores else None
    lg = np.empty((n, HEADS, max_seq_len), dtype=np.float64) if want_logits else None
    st = lib.orc_score_fp8(
        1 if decode else 0, _ptr(q), 1 if q_is_e4m3 else 0, 0, _ptr(k), int(k_page_stride),
        _ptr(bt), int(block_table_stride), _ptr(cu), _ptr(sl), _ptr(pl),
        num_seqs, int(max_seq_len), float(sm_scale), int(num_pool_pages),
        rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n,
        _ptr(sc), _ptr(lg), int(num_threads))
    if st != 0:
        raise ValueError(f"oracle rejected the inputs (status {st})")
    return sc, lg


def live_pairs(*, decode: bool, seq_lens, max_seq_len: int, cu_seqlens_q=None,
               prefix_lens=None, rows=None) -> int:
    """Number of live (row, token) pairs under the causal limit."""
    lib = _load()
    sl = _i32(seq_lens)
    cu = _i32(cu_seqlens_q)
    pl = _i32(prefix_lens)
    if rows is None:
        n_total = sl.shape[0] if decode else int(cu[-1])
        rows = np.arange(n_total, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return int(lib.orc_live_pairs(1 if decode else 0, _ptr(cu), _ptr(sl), _ptr(pl),
                                  int(sl.shape[0]), int(max_seq_len),
                                  rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                  rows.shape[0]))


# ------------------------------------------------------------------ writer --
def e2m1_from_double(x: float) -> int:
    """Round a real to an e2m1 code: nearest value, ties to the even code,
    saturating at 6, sign kept (the writer reading in ``mx4_oracle.c``)."""
    return _load().orc_e2m1_from_double(float(x))


def quantize_group(x) -> tuple[int, np.ndarray]:
    """One 32-element group -> (e8m0 scale byte, 32 e2m1 codes), following the
    OCP MX conversion reading stated in ``mx4_oracle.c``."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    assert a.shape == (32,)
    codes = np.empty(32, dtype=np.uint8)
    byte = _load().orc_quantize_group(_ptr(a), _ptr(codes))
    return int(byte), codes


def write_index_k(*, k_bits: np.ndarray, slot_mapping, k_data: np.ndarray, k_scale: np.ndarray,
                  k_data_page_stride: int, k_scale_page_stride: int, num_pool_pages: int = 0) -> int:
    """Quantise bf16 keys (uint16 bit patterns [num_tokens, W], W >= 128; the
    key is the first 128 elements of each row) into the page slots of
    ``slot_mapping`` (int64; slot s = token s % 128 of page s // 128,
    negative = skip).  ``k_data`` / ``k_scale`` are flat uint8 buffers written
    in place.  Returns the count of slots outside the pool (skipped)."""
    k = np.ascontiguousarray(np.asarray(k_bits))
    assert k.dtype == np.uint16 and k.ndim == 2 and k.shape[1] >= DIM
    n = k.shape[0]
    assert k_data.dtype == np.uint8 and k_data.flags.c_contiguous
    assert k_scale.dtype == np.uint8 and k_scale.flags.c_contiguous
    sm = np.ascontiguousarray(np.asarray(slot_mapping, dtype=np.int64))
    assert sm.shape == (n,)
    return int(_load().orc_write_index_k(_ptr(k), n, int(k.shape[1]), _ptr(sm), _ptr(k_data),
                                         _ptr(k_scale), int(k_data_page_stride),
                                         int(k_scale_page_stride), int(num_pool_pages)))


# ------------------------------------------------------------------- top-k --
def topk(*, decode: bool, scores: np.ndarray, block_table: np.ndarray, block_table_stride: int, seq_lens,
         max_seq_len: int, topk: int, local: int = 1, kv_groups: int = 1, cu_seqlens_q=None,
         prefix_lens=None, rows=None, want_tokens: bool = False):
    """Top-k page selection after the scorer (the readings are stated in
    ``mx4_oracle.c``).  ``scores``: float32 [rows_total, 64, P] block scores.
    Returns (sel int32 [n_rows, kv_groups, topk] physical ids, -1 padded, in
    ascending page order; count int32 [n_rows, kv_groups]), and with
    ``want_tokens`` also tokens int32 [n_rows, kv_groups], the live tokens of
    the selected pages."""
    lib = _load()
    sc = np.ascontiguousarray(scores, dtype=np.float32)
    bt = _i32(block_table).reshape(-1)
    sl = _i32(seq_lens)
    cu = _i32(cu_seqlens_q)
    pl = _i32(prefix_lens)
    num_seqs = int(sl.shape[0])
    if rows is None:
        n_total = num_seqs if decode else int(cu[-1])
        rows = np.arange(n_total, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    sel = np.empty((n, kv_groups, topk), dtype=np.int32)
    cnt = np.empty((n, kv_groups), dtype=np.int32)
    tok = np.empty((n, kv_groups), dtype=np.int32)
    st = lib.orc_topk(1 if decode else 0, _ptr(sc), int(max_seq_len), _ptr(bt), int(block_table_stride),
                      _ptr(cu), _ptr(sl), _ptr(pl), num_seqs, int(topk), int(local), int(kv_groups),
                      rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n, _ptr(sel), _ptr(cnt), _ptr(tok))
    if st != 0:
        raise ValueError(f"oracle rejected the inputs (status {st})")
    return (sel, cnt, tok) if want_tokens else (sel, cnt)


# ------------------------------------------------ sparse paged attention --
def pa_decode(*, q: np.ndarray, k_data, k_scale, kd_ps: int, kd_hs: int, ks_ps: int, ks_hs: int,
              v_data, v_scale, vd_ps: int, vd_hs: int, vs_ps: int, vs_hs: int, block_table: np.ndarray,
              context_lens, softmax_scale: float, num_pool_pages: int = 0, num_threads: int = 0) -> np.ndarray:
    """Decode attention over each row's selected MXFP4 K/V pages, fp64 (the
    definition and readings are in ``mx4_oracle.c``).  ``q``: e4m3 bytes
    [rows, kv_heads, groups, 128]; ``block_table``: int32 [rows, kv_heads,
    width]; ``context_lens``: int32 [rows, kv_heads].  Returns float64
    [rows, kv_heads, groups, 128]."""
    lib = _load()
    q = _u8(q)
    assert q.ndim == 4 and q.shape[3] == DIM
    n, kvh, g, _ = q.shape
    bt = _i32(block_table)
    assert bt.ndim == 3 and bt.shape[:2] == (n, kvh)
    cl = _i32(context_lens).reshape(-1)
    out = np.empty((n, kvh, g, DIM), dtype=np.float64)
    st = lib.orc_pa_decode(_ptr(q), n, kvh, g,
                           _ptr(_u8(k_data).reshape(-1)), _ptr(_u8(k_scale).reshape(-1)), kd_ps, kd_hs, ks_ps, ks_hs,
                           _ptr(_u8(v_data).reshape(-1)), _ptr(_u8(v_scale).reshape(-1)), vd_ps, vd_hs, vs_ps, vs_hs,
                           _ptr(bt), int(bt.shape[2]), _ptr(cl), float(softmax_scale), int(num_pool_pages),
                           _ptr(out), int(num_threads))
    if st != 0:
        raise ValueError(f"oracle rejected the inputs (status {st})")
    return out
