"""GPU parity of the scorer over an fp8 index cache against the fp64 oracle,
and the cross-format identity with the MXFP4 scorer."""
import dataclasses

import numpy as np
import pytest
import torch

import sparse_attention_mxfp4_gb300 as mx4
from sparse_attention_mxfp4_gb300 import harness
from sparse_attention_mxfp4_gb300 import workloads as W
from helpers import (RAGGED_DECODE_SEQ_LENS, clamp_garbage_scales, compare, logits_accum_allowance, mxfp4_as_fp8,
                     oracle_run)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx4.build()
    mx4.load_library()
    mx4.mx4_index_get_device_status()
    yield
    assert mx4.mx4_index_get_device_status() == 0


def _gpu(w, logits=False):
    c = harness.to_device(w)
    out = c.run(logits=logits)
    torch.cuda.synchronize()
    st = mx4.mx4_index_get_device_status()
    assert st == 0, f"device status {st:#x}"
    return out.cpu().numpy()


def _check(w, rows=None, real_pool=False):
    got = _gpu(w)
    ref, _ = oracle_run(w, rows=rows, real_pool=real_pool)
    compare(got if rows is None else got[rows], ref, what=f"{w.name} scores")
    got_l = _gpu(w, logits=True)
    _, ref_l = oracle_run(w, rows=rows, logits=True, scores=False, real_pool=real_pool)
    compare(got_l if rows is None else got_l[rows], ref_l, what=f"{w.name} logits",
            extra=logits_accum_allowance(w, rows))


def test_fp8_prefill_ragged_with_nan_garbage():
    w = W.make_workload("f8r", seed=70, q_lens=[37, 0, 130, 5, 1], seq_lens=[1500, 300, 2049, 129, 1],
                        prefix_lens=[1463, 300, 1900, 124, 0], pool_pages=64, bt_width=20, cache="fp8")
    _check(w)


def test_fp8_decode_ragged_padded_stride_e4m3_q():
    w = W.make_workload("f8d", seed=71, q_lens=None, seq_lens=[1, 128, 129, 5000, 0, 16384, 77], decode=True,
                        pool_pages=300, cache="fp8", k_data_page_stride=16384 + 80, q_e4m3=True)
    _check(w, real_pool=True)


def test_fp8_decode_ragged_last_pages_with_nan_garbage():
    """Decode over an fp8 cache whose partial last pages hold the e4m3 NaN
    codes past the live limit, last pages at every offset of a work unit."""
    w = W.make_workload("f8ragged", seed=26, q_lens=None, seq_lens=RAGGED_DECODE_SEQ_LENS, decode=True,
                        pool_pages=300, cache="fp8")
    got = _gpu(w)
    ref, _ = oracle_run(w)
    compare(got, ref, what="fp8 ragged decode")


def test_fp8_block_table_permutation_bit_identical():
    w = W.make_workload("f8p", seed=72, q_lens=[4, 7], seq_lens=[900, 3000], pool_pages=64, cache="fp8")
    np.testing.assert_array_equal(_gpu(w), _gpu(W.permute_pages(w, seed=5)))


@pytest.mark.parametrize("decode", [False, True])
def test_fp8_cache_matches_mxfp4_cache_within_the_window(decode):
    """The same keys as MXFP4 (scale bytes 119..133) and as fp8 give the same
    scores on the GPU (both within tolerance of the one oracle result)."""
    if decode:
        w = W.make_workload("x8d", seed=73, q_lens=None, seq_lens=[700, 129, 3000], decode=True,
                            pool_pages=40, scale_lo=119, scale_hi=133)
    else:
        w = W.make_workload("x8p", seed=74, q_lens=[5, 9], seq_lens=[700, 1500], prefix_lens=[695, 1491],
                            pool_pages=24, scale_lo=119, scale_hi=133)
    w = clamp_garbage_scales(w)
    f = mxfp4_as_fp8(w)
    a, b = _gpu(w), _gpu(f)
    ref, _ = oracle_run(w)
    compare(a, ref, what="mxfp4")
    compare(b, ref, what="fp8")
    assert np.array_equal(np.isneginf(a), np.isneginf(b))


@pytest.mark.parametrize("name,n_rows", [("decode-fp8", 64), ("prefill-long-fp8", 256)])
def test_fp8_full_size_sampled(name, n_rows):
    w = W.make_config(name)
    c = harness.to_device(w)
    out = c.run()
    torch.cuda.synchronize()
    assert mx4.mx4_index_get_device_status() == 0
    rows = W.sample_rows(w, n_rows, 0)
    got = out[torch.from_numpy(rows).to(out.device)].cpu().numpy()
    ref, _ = oracle_run(w, rows=rows)
    compare(got, ref, what=name)
    del c, out
