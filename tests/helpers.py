"""Shared test helpers: run the oracle on a workload, compare results."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_attention_mxfp4_gb300 import workloads as W

# Tolerance for finite fp32 scores against the fp64 oracle: relative 1e-5,
# absolute 1e-6 (the accuracy the scorer is specified to).  -inf placement is
# compared exactly.
RTOL = 1e-5
ATOL = 1e-6

# Decode contexts (pages per row): 9 with a partial last page, 10 partial, 12
# full, 17 with the 17th partial, 2 partial, 32 partial, 16 full, 58 partial,
# 31 partial: the last page lands at every offset inside the scorer's 8-page
# work units and at the end of a CTA's range.  The garbage past each context
# holds e8m0 bytes 0 and 255 (MXFP4) or the e4m3 NaN codes (fp8).
RAGGED_DECODE_SEQ_LENS = [1029, 1200, 1536, 2055, 131, 4032, 2048, 7297, 3845]


def oracle_run(w: W.Workload, rows=None, logits=False, scores=True, real_pool=False,
               unquantized=False, num_threads=0):
    """Oracle block scores / logits of workload ``w`` for ``rows`` (default all).

    ``real_pool``: read the pages from a host pool in the workload's own
    layout (single-region or split, real page ids); otherwise from a compact
    copy of the used pages."""
    if real_pool:
        bufs, (dbuf, doff), (sbuf, soff) = W.build_pool(w, "cpu")
        kd = dbuf.numpy()[doff:]
        ks = sbuf.numpy()[soff:]
        sd, ss = w.k_data_page_stride, w.k_scale_page_stride
        bt = w.block_table.numpy()
        npool = w.num_pool_pages
    else:
        kd, ks, sd, ss, bt, npool = W.compact_host(w)
    if w.cache == "fp8":
        return oracle.score_fp8(
            decode=w.decode, q=W.q_numpy(w), q_is_e4m3=w.q_is_e4m3, k_fp8=kd, k_page_stride=sd,
            block_table=bt, block_table_stride=w.block_table_stride, seq_lens=w.seq_lens.numpy(),
            cu_seqlens_q=None if w.decode else w.cu_seqlens_q.numpy(),
            prefix_lens=None if w.decode else w.prefix_lens.numpy(),
            max_seq_len=w.max_seq_len, sm_scale=w.sm_scale, rows=rows,
            want_scores=scores, want_logits=logits, num_pool_pages=npool, num_threads=num_threads)
    return oracle.score(
        decode=w.decode, q=W.q_numpy(w), q_is_e4m3=w.q_is_e4m3, k_data=kd, k_scale=ks,
        k_data_page_stride=sd, k_scale_page_stride=ss, block_table=bt,
        block_table_stride=w.block_table_stride, seq_lens=w.seq_lens.numpy(),
        cu_seqlens_q=None if w.decode else w.cu_seqlens_q.numpy(),
        prefix_lens=None if w.decode else w.prefix_lens.numpy(),
        max_seq_len=w.max_seq_len, sm_scale=w.sm_scale, rows=rows,
        want_scores=scores, want_logits=logits, unquantized=unquantized,
        num_pool_pages=npool, num_threads=num_threads)


def compare(got, ref, rtol=RTOL, atol=ATOL, what="scores", extra=None):
    """Assert fp32 ``got`` matches fp64 ``ref``: -inf placement exactly,
    finite values within |got-ref| <= atol + rtol*|ref| (+ ``extra``, an
    elementwise allowance, when given).  Returns stats."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    ninf_ref = np.isneginf(ref)
    ninf_got = np.isneginf(got)
    bad_mask = ninf_ref != ninf_got
    if bad_mask.any():
        idx = np.argwhere(bad_mask)[:5]
        raise AssertionError(f"{what}: -inf placement differs at {idx.tolist()} "
                             f"(got {got[tuple(idx[0])]}, ref {ref[tuple(idx[0])]}); "
                             f"{int(bad_mask.sum())} cells")
    fin = ~ninf_ref
    assert np.isfinite(got[fin]).all(), f"{what}: non-finite value where a finite one is expected"
    err = np.abs(got[fin] - ref[fin])
    lim = atol + rtol * np.abs(ref[fin])
    if extra is not None:
        lim = lim + np.asarray(extra, dtype=np.float64)[fin]
    bad = err > lim
    if bad.any():
        i = int(np.argmax(err - lim))
        raise AssertionError(f"{what}: {int(bad.sum())} of {fin.sum()} cells out of tolerance; "
                             f"worst got {got[fin][i]!r} ref {ref[fin][i]!r}")
    exact = float((got[fin] == ref[fin].astype(np.float32).astype(np.float64)).mean()) if fin.any() else 1.0
    rel = float((err / np.maximum(np.abs(ref[fin]), 1e-30)).max()) if fin.any() else 0.0
    return {"cells": int(got.size), "finite": int(fin.sum()), "max_abs_err": float(err.max()) if fin.any() else 0.0,
            "max_rel_err": rel, "fp32_exact_fraction": exact}


def plain_tolerance_stats(got, ref, rtol=RTOL, atol=ATOL):
    """How far finite fp32 results sit from the plain tolerance
    |got - ref| <= atol + rtol*|ref|: the fraction of finite cells outside it,
    the worst absolute and relative error, and the worst error in units of the
    plain limit."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    err = np.abs(got[fin] - ref[fin])
    lim = atol + rtol * np.abs(ref[fin])
    rel = err / np.maximum(np.abs(ref[fin]), 1e-30)
    return {"finite_cells": int(fin.sum()), "outside_plain": int((err > lim).sum()),
            "outside_plain_fraction": float((err > lim).mean()) if fin.any() else 0.0,
            "max_abs_err": float(err.max()) if fin.any() else 0.0,
            "max_rel_err": float(rel.max()) if fin.any() else 0.0,
            "worst_over_plain_limit": float((err / lim).max()) if fin.any() else 0.0}


def e4m3_values_numpy(codes):
    """e4m3 (fn) values from the bit fields: bias 7, subnormal step 2^-9,
    S.1111.111 NaN."""
    c = np.asarray(codes).astype(np.int64)
    s, e, m = (c >> 7) & 1, (c >> 3) & 15, c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def dequant_numpy(w: W.Workload):
    """Independent dequantisation in numpy from the bit fields of each code
    (used to pin the oracle; shares nothing with the oracle's C code)."""
    if w.cache == "fp8":
        return e4m3_values_numpy(w.pages_fp8.numpy())       # [U, 128, 128]
    data = w.pages_data.numpy()
    scale = w.pages_scale.numpy().astype(np.float64)
    lo = data & 15
    hi = data >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(data.shape[0], W.PAGE, W.DIM)
    s = (codes >> 3) & 1
    e = (codes >> 1) & 3
    m = codes & 1
    mag = np.where(e > 0, np.exp2(e.astype(np.float64) - 1) * (1 + m / 2.0), m / 2.0)
    val = np.where(s == 1, -mag, mag)
    sc = np.exp2(np.repeat(scale, 32, axis=-1) - 127.0)
    return val * sc          # [U, 128, 128]


def q_values_numpy(w: W.Workload):
    """Independent e4m3 value of every Q element (bf16 inputs rounded by
    exhaustive nearest-even search)."""
    if w.q_is_e4m3:
        codes = w.q.numpy().astype(np.int64)
    else:
        bits = w.q.view(torch.int16).numpy().view(np.uint16).astype(np.uint32)
        x = (bits << 16).view(np.float32).astype(np.float64)
        grid_codes = np.array([c for c in range(127)], dtype=np.int64)
        e = (grid_codes >> 3) & 15
        m = grid_codes & 7
        grid = np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * np.exp2(e - 7.0))
        ax = np.minimum(np.abs(x), 448.0).reshape(-1)
        idx = np.searchsorted(grid, ax)          # grid[idx-1] < ax <= grid[idx]
        idx = np.clip(idx, 1, len(grid) - 1)
        lo_v, hi_v = grid[idx - 1], grid[idx]
        pick_hi = (hi_v - ax < ax - lo_v) | ((hi_v - ax == ax - lo_v) & (grid_codes[idx] % 2 == 0))
        mag_code = np.where(ax == 0, 0, np.where(pick_hi, idx, idx - 1))
        codes = (mag_code | (np.signbit(x.reshape(-1)).astype(np.int64) << 7)).reshape(x.shape)
    s = (codes >> 7) & 1
    e = (codes >> 3) & 15
    m = codes & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * np.exp2(e - 7.0))
    return np.where(s == 1, -mag, mag)       # [rows, 64, 128]


def scores_numpy(w: W.Workload, rows=None, logits=False):
    """Block scores by a different formulation: dense dequantised K gathered
    per request, one float64 matmul per request, a broadcast causal mask and a
    reshape-max per page."""
    kv = dequant_numpy(w)
    qv = q_values_numpy(w)
    ids = {int(p): u for u, p in enumerate(w.page_ids.tolist())}
    P = w.num_out_pages
    B = w.num_seqs
    total = w.total_rows
    rows = np.arange(total) if rows is None else np.asarray(rows)
    out = np.full((len(rows), W.HEADS, P), -np.inf)
    lg = np.full((len(rows), W.HEADS, w.max_seq_len), -np.inf) if logits else None
    for ri, r in enumerate(rows):
        if w.decode:
            b, pos = int(r), 0
            L = int(w.seq_lens[b])
        else:
            cu = w.cu_seqlens_q.numpy()
            b = int(np.searchsorted(cu, r, side="right") - 1)
            pos = int(r - cu[b])
            L = min(int(w.seq_lens[b]), int(w.prefix_lens[b]) + pos + 1)
        L = min(L, w.max_seq_len)
        if L <= 0:
            continue
        npg = (L + W.PAGE - 1) // W.PAGE
        k = np.concatenate([kv[ids[int(w.block_table[b, j])]] for j in range(npg)], axis=0)[:L]
        v = w.sm_scale * (qv[r] @ k.T)                       # [64, L]
        pad = np.full((W.HEADS, npg * W.PAGE), -np.inf)
        pad[:, :L] = v
        out[ri, :, :npg] = pad.reshape(W.HEADS, npg, W.PAGE).max(axis=2)
        if logits:
            lg[ri, :, :L] = v
    return out, lg


# Accumulation allowance for per-token logits.  The tensor core forms the
# 128 products exactly but accumulates them (within each 32-element block and
# across the four scaled blocks) with fp32-class precision in an order and
# width the hardware does not document.  The classical worst-case bound for
# summing n terms in any order with unit roundoff u = 2^-24 is
#     |computed - exact| <= gamma_n * sum_i |x_i|,  gamma_n = n*u / (1 - n*u)
# (Higham, Accuracy and Stability of Numerical Algorithms, eq. 4.4), here with
# n = 128 products, plus one rounding of the final sm_scale product:
#     allowance = gamma_128 * sm_scale * sum_d |q_d * k_d| + 2^-24 * |logit|.
# With scale bytes in [122, 127] every partial sum is exact in fp32 and the
# allowance never matters; it admits cancellation error when scale bytes span
# 2^-27 .. 2^23 (the wide-scale workload).  Block scores are held to the
# plain 1e-5 / 1e-6 tolerance.
_U = 2.0 ** -24
GAMMA_128 = 128 * _U / (1 - 128 * _U)


def logits_accum_allowance(w: W.Workload, rows=None):
    """gamma_128 * sm_scale * sum_d |q_d k_d| + u * |logit| for every
    (row, head, token), by the independent numpy dequantisation; 0 where the
    token has no page."""
    kv = dequant_numpy(w)
    qv = q_values_numpy(w)
    ids = {int(p): u for u, p in enumerate(w.page_ids.tolist())}
    total = w.total_rows
    rows = np.arange(total) if rows is None else np.asarray(rows)
    out = np.zeros((len(rows), W.HEADS, w.max_seq_len))
    for ri, r in enumerate(rows):
        if w.decode:
            b = int(r)
        else:
            cu = w.cu_seqlens_q.numpy()
            b = int(np.searchsorted(cu, r, side="right") - 1)
        n = int(w.seq_lens[b])
        npg = (n + W.PAGE - 1) // W.PAGE
        if npg == 0:
            continue
        k = np.concatenate([kv[ids[int(w.block_table[b, j])]] for j in range(npg)], axis=0)[:n]
        absum = np.abs(qv[r]) @ np.abs(k).T
        val = np.abs(qv[r] @ k.T)
        out[ri, :, :n] = w.sm_scale * (GAMMA_128 * absum + _U * val)
    return out


def e4m3_code_exact(v):
    """The e4m3 byte whose value is exactly v (exhaustive search over the 256
    codes, sign of zero kept), or -1 where no byte has that value."""
    vals = e4m3_values_numpy(np.arange(256))
    v = np.asarray(v, dtype=np.float64)
    out = np.full(v.shape, -1, dtype=np.int64)
    o = out.reshape(-1)
    for i, x in enumerate(v.reshape(-1)):
        hit = [c for c in np.nonzero(vals == x)[0] if np.signbit(vals[c]) == np.signbit(x)]
        if hit:
            o[i] = hit[0]
    return out


def mxfp4_as_fp8(w: W.Workload) -> W.Workload:
    """The MXFP4 workload's keys re-stored as an fp8 cache (every value must be
    an e4m3 value: scale bytes 119..133)."""
    import dataclasses
    vals = dequant_numpy(w)                       # [U, 128, 128]
    uniq, inv = np.unique(vals.reshape(-1), return_inverse=True)
    # np.unique merges -0.0 and +0.0; map zeros by their own sign below
    uc = e4m3_code_exact(uniq)
    assert (uc >= 0).all(), "a value outside e4m3"
    codes = uc[inv].reshape(vals.shape)
    codes = np.where(vals == 0, np.where(np.signbit(vals), 0x80, 0x00), codes).astype(np.uint8)
    return dataclasses.replace(w, cache="fp8", layout="fp8", pages_fp8=torch.from_numpy(codes),
                               k_data_page_stride=W.FP8_PAGE_BYTES, k_scale_page_stride=0)


def clamp_garbage_scales(w: W.Workload, lo=119, hi=133) -> W.Workload:
    """Scale bytes outside [lo, hi] (only in garbage tails) set to 127."""
    import dataclasses
    ps = w.pages_scale.clone()
    ps[(ps < lo) | (ps > hi)] = 127
    return dataclasses.replace(w, pages_scale=ps)
