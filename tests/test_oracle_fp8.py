"""Pins of the oracle's fp8-cache scorer (the format the MXFP4 cache replaces).

- Cross-format: MXFP4 values e2m1 x 2^(byte-127) are exact e4m3 values for
  scale bytes 119..133 (aiter #7061 "Format"); the same keys stored as fp8
  score bit for bit like the MXFP4 pages.  The window's edges are checked too.
- An independent numpy formulation (bit-field e4m3 decoding, one float64
  matmul per request) on a ragged batch whose garbage tails hold e4m3 NaN codes.
- One-hot closed forms.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_mxfp4_gb300 import workloads as W
from helpers import (clamp_garbage_scales, e4m3_code_exact as _e4m3_code_exact, e4m3_values_numpy,
                     mxfp4_as_fp8, oracle_run, scores_numpy)


def test_mxfp4_window_values_are_exact_e4m3():
    mags = np.array([0.5, 1, 1.5, 2, 3, 4, 6])
    for b in range(119, 134):
        v = mags * 2.0 ** (b - 127)
        assert (_e4m3_code_exact(v) >= 0).all(), b
    # just outside the window some values are not e4m3 values
    assert (_e4m3_code_exact(mags * 2.0 ** (118 - 127)) < 0).any()
    assert (_e4m3_code_exact(mags * 2.0 ** (134 - 127)) < 0).any()


@pytest.mark.parametrize("decode", [False, True])
def test_fp8_cache_scores_like_mxfp4_within_the_window(decode):
    if decode:
        w = W.make_workload("x8d", seed=60, q_lens=None, seq_lens=[700, 129, 1500], decode=True,
                            pool_pages=24, scale_lo=119, scale_hi=133)
    else:
        w = W.make_workload("x8p", seed=61, q_lens=[5, 9], seq_lens=[700, 1500], prefix_lens=[695, 1491],
                            pool_pages=24, scale_lo=119, scale_hi=133)
    # the garbage tails (bytes 0 and 255) are not e4m3-exact: clear them to a
    # representable byte; they are past every live limit
    w = clamp_garbage_scales(w)
    f = mxfp4_as_fp8(w)
    a, la = oracle_run(w, logits=True)
    b, lb = oracle_run(f, logits=True)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_fp8_oracle_matches_numpy_formulation_with_nan_garbage():
    w = W.make_workload("f8", seed=62, q_lens=[37, 0, 130, 5, 1], seq_lens=[1500, 300, 2049, 129, 1],
                        prefix_lens=[1463, 300, 1900, 124, 0], pool_pages=64, bt_width=20, cache="fp8")
    assert np.isnan(e4m3_values_numpy(w.pages_fp8.numpy())).any()      # NaN garbage is present
    ref, lg = oracle_run(w, logits=True)
    alt, alt_lg = scores_numpy(w, logits=True)
    np.testing.assert_allclose(ref, alt, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lg, alt_lg, rtol=1e-12, atol=1e-12)
    assert not np.isnan(ref).any() and not np.isnan(lg).any()


@pytest.mark.parametrize("h0,d0,t0,code", [(0, 0, 0, 0x38), (63, 127, 127, 0xB9), (7, 64, 31, 0x01),
                                           (40, 5, 100, 0x7E)])
def test_fp8_one_hot(h0, d0, t0, code):
    base = W.make_workload("o8", seed=63, q_lens=[1], seq_lens=[128], prefix_lens=[127], pool_pages=2,
                           cache="fp8")
    q = torch.zeros_like(base.q)
    q[0, h0, d0] = 2.0
    k = torch.zeros_like(base.pages_fp8)
    k[0, t0, d0] = code
    w = dataclasses.replace(base, q=q, pages_fp8=k)
    sc, lg = oracle_run(w, logits=True)
    want = W.SM_SCALE * 2.0 * float(e4m3_values_numpy(np.array([code]))[0])
    exp = np.zeros_like(lg)
    exp[0, h0, t0] = want
    np.testing.assert_array_equal(lg, exp)
    np.testing.assert_array_equal(sc[:, :, 0], exp.max(axis=2))
