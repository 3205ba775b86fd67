"""CUDA-graph capture and replay of the selection, attention and writer
entry points: every replay (outputs poisoned before it) reproduces the eager
result bit for bit, so the host-known launch configuration is stable."""
import numpy as np
import pytest
import torch

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


def _replay_matches(call, outs, poison):
    """``poison``: a fill value per output, or None to restore the output's
    contents from before the first call (for in-place writes)."""
    before = [o.clone() for o in outs]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call(s)                      # warm-up on the capture stream
    torch.cuda.synchronize()
    ref = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
    for _ in range(3):
        for o, v, b in zip(outs, poison, before):
            if v is None:
                o.copy_(b)
            else:
                o.fill_(v)
        g.replay()
        torch.cuda.synchronize()
        for o, r in zip(outs, ref):
            assert torch.equal(o, r)


def test_graph_topk_decode():
    w = W.make_workload("gtk", seed=120, q_lens=None, seq_lens=[700, 3000, 129], decode=True, pool_pages=40)
    c = harness.to_device(w)
    scores = c.run()
    sel = torch.empty((w.total_rows, 2, 6), dtype=torch.int32, device="cuda")
    cnt = torch.empty((w.total_rows, 2), dtype=torch.int32, device="cuda")
    tok = torch.empty((w.total_rows, 2), dtype=torch.int32, device="cuda")
    _replay_matches(lambda s: mx4.mx4_index_topk_decode(scores, c.block_table, c.seq_lens, w.max_seq_len, 6,
                                                        local_pages=2, kv_groups=2, sel=sel, count=cnt, tokens=tok,
                                                        stream=s),
                    [sel, cnt, tok], [-7, -7, -7])


def test_graph_sparse_attention():
    a = W.make_attn_case("gat", seed=121, rows=3, kv_heads=2, groups=8, width=5)
    q, kp, vp, bt, cl = a.q.cuda(), a.k_pool.cuda(), a.v_pool.cuda(), a.block_table.cuda(), a.context_lens.cuda()
    out = torch.empty((3, 2, 8, 128), dtype=torch.bfloat16, device="cuda")
    _replay_matches(lambda s: mx4.mx4_sparse_pa_decode(q, kp, vp, bt, cl, a.softmax_scale, out, stream=s),
                    [out], [float("nan")])


def test_graph_index_k_write():
    wc = W.make_write_case("gwr", seed=122, num_tokens=500, num_pool_pages=8, dist="wide")
    bufs, (db, do), (sb, so) = W.write_pool(wc, device="cuda")
    k, sm = wc.k.cuda(), wc.slot_mapping.cuda()
    _replay_matches(lambda s: mx4.mx4_index_k_write(k, sm, db[do:], sb[so:], wc.k_data_page_stride,
                                                    wc.k_scale_page_stride, num_pool_pages=8, stream=s),
                    bufs, [None] * len(bufs))
