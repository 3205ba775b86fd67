"""GPU top-k page selection against the oracle's, bit for bit: the oracle
runs on the same fp32 block scores the GPU selection reads."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mxfp4_gb300 as mx4
from sparse_attention_mxfp4_gb300 import harness
from sparse_attention_mxfp4_gb300 import workloads as W

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


def _topk_gpu(w, scores, k, local, groups, bt=None):
    bt = (w.block_table if bt is None else bt).cuda()
    if w.decode:
        return mx4.mx4_index_topk_decode(scores, bt, w.seq_lens.cuda(), w.max_seq_len, k, local_pages=local,
                                         kv_groups=groups, want_tokens=True)
    return mx4.mx4_index_topk_prefill(scores, bt, w.cu_seqlens_q.cuda(), w.seq_lens.cuda(), w.prefix_lens.cuda(),
                                      w.max_query_len, w.max_seq_len, k, local_pages=local, kv_groups=groups,
                                      want_tokens=True)


def _topk_oracle(w, scores_np, k, local, groups, rows=None):
    return oracle.topk(decode=w.decode, scores=scores_np, block_table=w.block_table.numpy(),
                       block_table_stride=w.block_table_stride, seq_lens=w.seq_lens.numpy(),
                       cu_seqlens_q=None if w.decode else w.cu_seqlens_q.numpy(),
                       prefix_lens=None if w.decode else w.prefix_lens.numpy(), max_seq_len=w.max_seq_len,
                       topk=k, local=local, kv_groups=groups, rows=rows, want_tokens=True)


def _check_chain(w, k, local, groups):
    c = harness.to_device(w)
    scores = c.run()
    sel, cnt, tok = _topk_gpu(w, scores, k, local, groups)
    torch.cuda.synchronize()
    ref_sel, ref_cnt, ref_tok = _topk_oracle(w, scores.cpu().numpy(), k, local, groups)
    np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
    np.testing.assert_array_equal(sel.cpu().numpy(), ref_sel)
    np.testing.assert_array_equal(tok.cpu().numpy(), ref_tok)


@pytest.mark.parametrize("k,local,groups", [(4, 1, 1), (1, 1, 1), (3, 0, 2), (16, 4, 4), (5, 5, 64)])
def test_scorer_then_topk_prefill_ragged(k, local, groups):
    w = W.make_workload("tk", seed=80, q_lens=[37, 0, 130, 5, 1], seq_lens=[1500, 300, 2049, 129, 1],
                        prefix_lens=[1463, 300, 1900, 124, 0], pool_pages=64, bt_width=20)
    _check_chain(w, k, local, groups)


@pytest.mark.parametrize("k,local,groups", [(8, 1, 1), (64, 2, 2), (4, 1, 64), (16, 2, 32)])
def test_scorer_then_topk_decode_ragged(k, local, groups):
    """Decode rows, including 32 and 64 head groups (one or two heads a
    group)."""
    w = W.make_workload("tkd", seed=81, q_lens=None, seq_lens=[1, 128, 129, 5000, 0, 16384, 77], decode=True,
                        pool_pages=300, layout="split", k_data_page_stride=8320, k_scale_page_stride=576)
    _check_chain(w, k, local, groups)


def test_scorer_then_topk_decode_many_rows():
    """400 decode rows of mixed lengths, one CTA each."""
    g = np.random.default_rng(84)
    lens = [int(x) for x in g.integers(0, 3000, size=400)]
    w = W.make_workload("tkm", seed=84, q_lens=None, seq_lens=lens, decode=True, pool_pages=10000)
    _check_chain(w, 6, 1, 1)


@pytest.mark.parametrize("P_tokens,offset", [(1100, 0), (4096, 1), (16384, 0), (131072, 0), (131072, 1)])
def test_ties_signed_zeros_and_scalar_path(P_tokens, offset):
    """Integer-valued scores (many ties) with +0 / -0 mixed; P not a multiple
    of 4 or a misaligned scores pointer take the scalar path.  Few items run
    as clusters: up to 32 chosen pages of at most 1024 candidates take the
    two-stage select (ties split across the cluster's CTAs), more take the
    radix select."""
    g = torch.Generator().manual_seed(82 + P_tokens)
    w = W.make_workload("ties", seed=83, q_lens=[3, 6], seq_lens=[P_tokens, P_tokens - 300],
                        prefix_lens=[P_tokens - 3, P_tokens - 306], pool_pages=2 * ((P_tokens + 127) // 128))
    P = w.num_out_pages
    vals = torch.randint(-2, 3, (w.total_rows, 64, P), generator=g).float()
    zeros = vals == 0
    vals[zeros & (torch.rand(vals.shape, generator=g) < 0.5)] = -0.0
    host = vals.numpy()
    base = torch.empty(vals.numel() + offset, dtype=torch.float32, device="cuda")
    scores = base[offset:].view(vals.shape)
    scores.copy_(vals.cuda())
    for k, local, groups in ((3, 1, 1), (7, 2, 2), (40, 1, 8), (33, 1, 1), (34, 1, 4), (1024, 1, 1)):
        sel, cnt, tok = _topk_gpu(w, scores, k, local, groups)
        torch.cuda.synchronize()
        ref_sel, ref_cnt, ref_tok = _topk_oracle(w, host, k, local, groups)
        np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
        np.testing.assert_array_equal(sel.cpu().numpy(), ref_sel)
        np.testing.assert_array_equal(tok.cpu().numpy(), ref_tok)


@pytest.mark.parametrize("name,k,rows", [("decode", 16, None), ("decode", 64, None), ("prefill-long", 16, 64)])
def test_topk_full_size(name, k, rows):
    w = W.make_config(name)
    c = harness.to_device(w)
    scores = c.run()
    sel, cnt, tok = _topk_gpu(w, scores, k, 1, 1)
    torch.cuda.synchronize()
    r = None if rows is None else W.sample_rows(w, rows, 1)
    sc_host = scores.cpu().numpy()
    ref_sel, ref_cnt, ref_tok = _topk_oracle(w, sc_host, k, 1, 1, rows=r)
    got_sel = sel.cpu().numpy() if r is None else sel.cpu().numpy()[r]
    got_cnt = cnt.cpu().numpy() if r is None else cnt.cpu().numpy()[r]
    got_tok = tok.cpu().numpy() if r is None else tok.cpu().numpy()[r]
    np.testing.assert_array_equal(got_cnt, ref_cnt)
    np.testing.assert_array_equal(got_sel, ref_sel)
    np.testing.assert_array_equal(got_tok, ref_tok)
    del c, scores
