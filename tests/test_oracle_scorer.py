"""Pins of the oracle's scorer: brute force on one-hot inputs, exact rational
arithmetic, an independent numpy formulation, invariances the pages state,
the masked special cases and closed-form live counts.  CPU only."""
import dataclasses
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_mxfp4_gb300 import workloads as W
from helpers import oracle_run, scores_numpy, q_values_numpy, dequant_numpy

SM = W.SM_SCALE


def _one_page_workload(seed=0, q_rows=1, seq=128, prefix=None):
    return W.make_workload("onehot", seed=seed, q_lens=[q_rows], seq_lens=[seq],
                           prefix_lens=[prefix if prefix is not None else seq - q_rows],
                           pool_pages=4)


@pytest.mark.parametrize("d0,code,sbyte,t0,qv", [
    (0, 3, 127, 5, 1.5),      # low nibble of byte 0, group 0
    (1, 7, 125, 0, -2.0),     # high nibble of byte 0
    (37, 13, 122, 127, 0.75), # odd element in group 1, last token
    (64, 9, 130, 64, 448.0),  # group 2, code 9 = -0.5
    (127, 15, 101, 99, -0.001953125),  # last element (high nibble), group 3, q = -2^-9
    (96, 8, 150, 17, 3.0),    # code 8 = -0: product is zero
])
def test_brute_force_one_hot(d0, code, sbyte, t0, qv):
    """One non-zero Q element and one non-zero K code: every output has a
    closed form, which also pins nibble order and scale-group indexing."""
    w = _one_page_workload()
    q = torch.zeros_like(w.q)
    h0 = 23
    q[0, h0, d0] = qv          # exactly representable in bf16 and e4m3
    data = torch.zeros_like(w.pages_data)
    scale = torch.full_like(w.pages_scale, 127)
    byte = code if d0 % 2 == 0 else code << 4
    data[0, t0, d0 // 2] = byte
    scale[0, t0, d0 // 32] = sbyte
    w = dataclasses.replace(w, q=q, pages_data=data, pages_scale=scale)
    sc, lg = oracle_run(w, logits=True)
    e2m1 = [0, .5, 1, 1.5, 2, 3, 4, 6][code & 7] * (-1 if code & 8 else 1)
    want = SM * (qv * e2m1 * 2.0 ** (sbyte - 127))
    exp_lg = np.zeros((1, 64, 128))
    exp_lg[0, h0, t0] = want
    np.testing.assert_array_equal(lg, exp_lg)
    exp_sc = np.zeros((1, 64, 1))
    exp_sc[0, h0, 0] = max(want, 0.0)
    np.testing.assert_array_equal(sc, exp_sc)


@pytest.mark.parametrize("scale_lo,scale_hi,exact", [(122, 127, True), (100, 150, False)])
def test_exact_rational_small_case(scale_lo, scale_hi, exact):
    """Logits and scores against exact rational arithmetic (Fractions) on a
    random two-page case.  With scale bytes in [122, 127] every product is a
    multiple of 2^-15 below 2^12, so the fp64 sum is exact and the oracle must
    equal the correctly rounded rational result; with bytes 100..150 it must
    lie within the recursive-summation bound (n-1) * 2^-53 * sum|terms|."""
    w = W.make_workload("exact", seed=3, q_lens=[2], seq_lens=[200], prefix_lens=[198],
                        pool_pages=4, scale_lo=scale_lo, scale_hi=scale_hi)
    sc, lg = oracle_run(w, logits=True)
    data = w.pages_data.numpy()
    scale = w.pages_scale.numpy()
    e2m1 = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    ids = {int(p): u for u, p in enumerate(w.page_ids.tolist())}
    qvals = q_values_numpy(w)
    sm = Fraction(SM)
    for r in range(2):
        L = min(200, 198 + r + 1)
        for h in (0, 31, 63):
            best = [None, None]
            for t in range(L):
                u = ids[int(w.block_table[0, t // 128])]
                i = t % 128
                acc = Fraction(0)
                absum = Fraction(0)
                for d in range(128):
                    byte = int(data[u, i, d // 2])
                    c = (byte >> 4) if d & 1 else (byte & 15)
                    kv = e2m1[c & 7] * (-1 if c & 8 else 1) * Fraction(2) ** (int(scale[u, i, d // 32]) - 127)
                    term = Fraction(qvals[r, h, d]) * kv
                    acc += term
                    absum += abs(term)
                val = sm * acc
                if exact:
                    assert lg[r, h, t] == float(val), (r, h, t)
                else:
                    bound = sm * absum * Fraction(128, 2 ** 53) + abs(val) * Fraction(1, 2 ** 52)
                    assert abs(Fraction(lg[r, h, t]) - val) <= bound, (r, h, t)
                j = t // 128
                if best[j] is None or val > best[j]:
                    best[j] = val
            for j in range(2):
                if exact:
                    assert sc[r, h, j] == float(best[j])
                else:
                    assert sc[r, h, j] == lg[r, h, j * 128:(j + 1) * 128].max()
            assert np.all(np.isneginf(lg[r, h, L:]))


@pytest.mark.parametrize("scale_lo,scale_hi,exact", [(122, 127, True), (100, 150, False)])
def test_matches_numpy_formulation_ragged(scale_lo, scale_hi, exact):
    """A ragged batch (odd row counts, an empty request, partial pages,
    prefix+q_len != seq_len) against the dense numpy formulation."""
    w = W.make_workload("ragged", seed=11, q_lens=[5, 0, 3, 9], seq_lens=[300, 64, 129, 1000],
                        prefix_lens=[295, 64, 100, 990], pool_pages=40,
                        scale_lo=scale_lo, scale_hi=scale_hi)
    sc, lg = oracle_run(w, logits=True)
    ref_sc, ref_lg = scores_numpy(w, logits=True)
    if exact:
        np.testing.assert_array_equal(sc, ref_sc)
        np.testing.assert_array_equal(lg, ref_lg)
    else:
        np.testing.assert_allclose(sc, ref_sc, rtol=1e-13, atol=0)
        np.testing.assert_allclose(lg, ref_lg, rtol=1e-13, atol=1e-300)


def test_matches_numpy_formulation_decode_e4m3_q():
    w = W.make_workload("dec", seed=5, q_lens=None, seq_lens=[1, 128, 129, 700, 0], decode=True,
                        pool_pages=16, q_e4m3=True, layout="split", k_data_page_stride=8320,
                        k_scale_page_stride=576)
    sc, _ = oracle_run(w, real_pool=True)
    ref, _ = scores_numpy(w)
    np.testing.assert_array_equal(sc, ref)
    assert np.all(np.isneginf(sc[4]))          # seq_len 0: every page -inf
    assert np.all(np.isneginf(sc[0, :, 1:]))   # one live token: only page 0 finite
    assert np.all(np.isfinite(sc[0, :, 0]))


def test_block_table_permutation_invariance():
    w = W.make_workload("perm", seed=7, q_lens=[4, 6], seq_lens=[500, 260], pool_pages=32)
    a, _ = oracle_run(w, real_pool=True)
    b, _ = oracle_run(W.permute_pages(w, seed=99), real_pool=True)
    np.testing.assert_array_equal(a, b)


def test_split_and_single_region_agree():
    w = W.make_workload("lay", seed=8, q_lens=[3], seq_lens=[777], pool_pages=12)
    a, la = oracle_run(w, real_pool=True, logits=True)
    s = W.relayout(w, "split", k_data_page_stride=8192 + 96, k_scale_page_stride=512 + 32)
    b, lb = oracle_run(s, real_pool=True, logits=True)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_garbage_past_live_limit_changes_nothing():
    w = W.make_workload("garb", seed=9, q_lens=[4], seq_lens=[300], pool_pages=8)
    a, la = oracle_run(w, logits=True)
    data = w.pages_data.clone()
    scale = w.pages_scale.clone()
    last = {int(p): u for u, p in enumerate(w.page_ids.tolist())}[int(w.block_table[0, 2])]
    data[last, 300 - 256:] = 0xFF
    scale[last, 300 - 256:] = 255
    scale[last, 300 - 256 + 1:] = 0
    g = dataclasses.replace(w, pages_data=data, pages_scale=scale)
    b, lb = oracle_run(g, logits=True)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_fully_masked_pages_are_neg_inf():
    # seq 1024 but prefix 100: row 0 sees tokens < 101, so pages 1..7 have no live token
    w = W.make_workload("mask", seed=10, q_lens=[3], seq_lens=[1024], prefix_lens=[100],
                        pool_pages=8)
    sc, lg = oracle_run(w, logits=True)
    assert np.all(np.isfinite(sc[:, :, 0]))
    assert np.all(np.isneginf(sc[:, :, 1:]))
    assert np.all(np.isneginf(lg[0, :, 101:])) and np.all(np.isfinite(lg[0, :, :101]))
    assert np.all(np.isneginf(lg[2, :, 103:])) and np.all(np.isfinite(lg[2, :, :103]))


def test_single_live_token_page_and_partial_last_page():
    # seq 257: page 2 holds one token; rows see up to the whole sequence
    w = W.make_workload("tail", seed=12, q_lens=[2], seq_lens=[257], prefix_lens=[255],
                        pool_pages=4)
    sc, lg = oracle_run(w, logits=True)
    # row 0: L = 256 -> page 2 masked; row 1: L = 257 -> page 2 is its token 256 alone
    assert np.all(np.isneginf(sc[0, :, 2]))
    np.testing.assert_array_equal(sc[1, :, 2], lg[1, :, 256])
    np.testing.assert_array_equal(sc[1, :, 0], lg[1, :, :128].max(axis=1))


def _closed_form_live(q_lens, seq_lens, prefix_lens):
    total = 0
    for ql, s, p in zip(q_lens, seq_lens, prefix_lens):
        for r in range(ql):
            total += max(0, min(s, p + r + 1))
    return total


@pytest.mark.parametrize("name,q_lens,seq,prefix,expected", [
    ("prefill-tiny", [32], [1024], [992], 32_272),
    ("prefill-long", [4096], [131072], [126976], 528_484_352),
    ("mtp", [8] * 32, [32768] * 32, [32760] * 32, 8_387_712),
    ("chunked", [32768], [132768], [100000], 3_813_687_296),
])
def test_live_pairs_closed_form(name, q_lens, seq, prefix, expected):
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    got = oracle.live_pairs(decode=False, seq_lens=seq, max_seq_len=max(seq), cu_seqlens_q=cu,
                            prefix_lens=prefix)
    # arithmetic series: sum over rows of (prefix + r + 1), all below seq_len here
    series = sum(ql * (p + 1) + ql * (ql - 1) // 2 for ql, p in zip(q_lens, prefix))
    assert got == series == expected
    if sum(q_lens) <= 4096:
        assert got == _closed_form_live(q_lens, seq, prefix)


def test_live_pairs_decode():
    got = oracle.live_pairs(decode=True, seq_lens=[131072] * 64, max_seq_len=131072)
    assert got == 64 * 131072


def test_unquantized_q_differs_and_cosine_close():
    """Context figure only: bf16 Q without e4m3 rounding gives other logits;
    their cosine against the quantised ones is close to 1."""
    w = W.make_workload("cos", seed=13, q_lens=[4], seq_lens=[512], pool_pages=6)
    _, a = oracle_run(w, logits=True, scores=False)
    _, b = oracle_run(w, logits=True, scores=False, unquantized=True)
    fin = np.isfinite(a)
    assert not np.array_equal(a[fin], b[fin])
    cos = float(np.dot(a[fin], b[fin]) / (np.linalg.norm(a[fin]) * np.linalg.norm(b[fin])))
    assert 0.99 < cos < 1.0
