"""One decode step of the whole path on one CUDA stream, with no host
synchronisation between the kernels: each request's new index key is
quantised into its pool slot (writer), every page of every request is scored
(scorer), the top pages are selected (top-k), and each row attends over its
selected pages, with the index pool as K and a V pool beside it (attention).
The kernels are programmatic dependent launches, so this also checks that
each one sees the previous one's writes.

Every stage is compared with the oracle fed the previous GPU stage's output:
the written pool bit for bit, the block scores within the scorer tolerance,
the selection bit for bit, the attention output within the bound of
tests/test_gpu_attn.py.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mxfp4_gb300 as mx4
from sparse_attention_mxfp4_gb300 import harness
from sparse_attention_mxfp4_gb300 import workloads as W
from helpers import compare
from test_gpu_attn import _abs_weighted_v
from test_oracle_attn import _run as oracle_attn

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


@pytest.mark.parametrize("topk", [4, 16])
def test_decode_step_chain_on_one_stream(topk):
    lens = [1, 128, 129, 1500, 3000, 2049, 700]
    B = len(lens)
    npool = 120
    w = W.make_workload("chain", seed=90, q_lens=None, seq_lens=lens, decode=True, pool_pages=npool)
    c = harness.to_device(w)
    pool = c.buffers[0]
    pool_host = pool.cpu().numpy().copy()            # the pool before this step's write

    g = torch.Generator().manual_seed(91)
    keys = torch.randn((B, W.DIM), generator=g).to(torch.bfloat16)
    slots = torch.tensor([int(w.block_table[b, (L - 1) // W.PAGE]) * W.PAGE + (L - 1) % W.PAGE
                          for b, L in enumerate(lens)], dtype=torch.int64)
    q_att = torch.randn((B, 1, 16, W.DIM), generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
    v_data = torch.randint(0, 256, (npool, 1, W.DATA_BYTES), generator=g, dtype=torch.uint8)
    v_scale = torch.randint(122, 128, (npool, 1, W.SCALE_BYTES), generator=g, dtype=torch.uint8)
    v_pool = torch.cat([v_data, v_scale], dim=2).contiguous()

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        mx4.mx4_index_k_write(keys.cuda(), slots.cuda(), c.k_data, c.k_scale, w.k_data_page_stride,
                              w.k_data_page_stride, num_pool_pages=npool, stream=stream)
        scores = c.run(stream=stream)
        # the selection and, for the attention, the live tokens of the selected
        # pages (listed in ascending order, the partial last page at the end)
        sel, cnt, ctx = mx4.mx4_index_topk_decode(scores, c.block_table, c.seq_lens, w.max_seq_len, topk,
                                                  local_pages=1, kv_groups=1, want_tokens=True, stream=stream)
        k_pool = pool[: npool * W.PAGE_BYTES].view(npool, 1, W.PAGE_BYTES)
        out = mx4.mx4_sparse_pa_decode(q_att.cuda(), k_pool, v_pool.cuda(), sel.view(B, 1, topk), ctx.view(B, 1),
                                       w.sm_scale, stream=stream)
    torch.cuda.synchronize()
    assert mx4.mx4_index_get_device_status() == 0

    # 1. the written pool, bit for bit
    oracle.write_index_k(k_bits=keys.view(torch.int16).numpy().view(np.uint16), slot_mapping=slots.numpy(),
                         k_data=pool_host, k_scale=pool_host[W.DATA_BYTES:],
                         k_data_page_stride=w.k_data_page_stride, k_scale_page_stride=w.k_data_page_stride,
                         num_pool_pages=npool)
    got_pool = pool.cpu().numpy()
    assert np.array_equal(got_pool, pool_host), "written pool differs from the oracle's"

    # 2. block scores over the written pool
    ref, _ = oracle.score(decode=True, q=W.q_numpy(w), q_is_e4m3=w.q_is_e4m3, k_data=pool_host,
                          k_scale=pool_host[W.DATA_BYTES:], k_data_page_stride=w.k_data_page_stride,
                          k_scale_page_stride=w.k_data_page_stride, block_table=w.block_table.numpy(),
                          block_table_stride=w.block_table_stride, seq_lens=w.seq_lens.numpy(),
                          max_seq_len=w.max_seq_len, sm_scale=w.sm_scale, num_pool_pages=npool)
    sc = scores.cpu().numpy()
    compare(sc, ref, what="chain scores")

    # 3. the selection over the GPU's scores, bit for bit
    ref_sel, ref_cnt, ref_tok = oracle.topk(decode=True, scores=sc, block_table=w.block_table.numpy(),
                                            block_table_stride=w.block_table_stride, seq_lens=w.seq_lens.numpy(),
                                            max_seq_len=w.max_seq_len, topk=topk, local=1, kv_groups=1,
                                            want_tokens=True)
    np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
    np.testing.assert_array_equal(sel.cpu().numpy(), ref_sel)
    np.testing.assert_array_equal(ctx.cpu().numpy(), ref_tok)

    # 4. attention over the GPU's selection, its context the selection's
    # live tokens
    case = W.AttnCase("chain", q=q_att, k_pool=torch.from_numpy(got_pool[: npool * W.PAGE_BYTES]).view(
        npool, 1, W.PAGE_BYTES), v_pool=v_pool, block_table=sel.cpu().view(B, 1, topk),
        context_lens=ctx.cpu().view(B, 1), softmax_scale=w.sm_scale)
    assert [int(x) for x in case.context_lens[:, 0]] == [
        min(L, (min(topk, (L + 127) // 128) - 1) * 128 + L - 128 * ((L + 127) // 128 - 1)) for L in lens]
    got = out.float().cpu().numpy()
    aref = oracle_attn(case)
    lim = 2.0 ** -8 * (_abs_weighted_v(case) + np.abs(aref)) + 2.0 ** -8 * np.abs(aref) + 1e-30
    err = np.abs(got - aref)
    assert not (err > lim).any(), f"{int((err > lim).sum())} outside; worst {err.max():.3e}"
    assert np.linalg.norm(got - aref) / np.linalg.norm(aref) < 4e-3
