"""GPU parity at the measured configurations' full sizes, in the launch
configuration bench.py times, on seeded samples of rows the oracle computes
one by one."""
import numpy as np
import pytest
import torch

import sparse_attention_mxfp4_gb300 as mx4
from sparse_attention_mxfp4_gb300 import harness
from sparse_attention_mxfp4_gb300 import workloads as W
from helpers import compare, oracle_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx4.build()
    mx4.load_library()
    mx4.mx4_index_get_device_status()
    yield
    torch.cuda.empty_cache()


def _run_full(w):
    c = harness.to_device(w)
    out = c.run()
    torch.cuda.synchronize()
    assert mx4.mx4_index_get_device_status() == 0
    return c, out


def _sampled(w, out, n_rows, seed=0):
    rows = W.sample_rows(w, n_rows, seed)
    got = out[torch.from_numpy(rows).to(out.device)].cpu().numpy()
    ref, _ = oracle_run(w, rows=rows)
    return compare(got, ref, what=w.name)


def test_decode_full_size_every_row():
    """The measured decode call, element by element: all 64 rows x 64 heads x
    1024 pages against the oracle."""
    w = W.make_config("decode")
    c, out = _run_full(w)
    assert out.shape == (64, 64, 1024)
    assert torch.isfinite(out).all()          # every page of every request is live
    ref, _ = oracle_run(w)
    compare(out.cpu().numpy(), ref, what="decode (all rows)")
    del c


def test_decode_graph_replay_with_poisoned_output():
    """The decode call as bench.py times it (captured in a CUDA graph on a side
    stream, host-known grid): each replay into a NaN-poisoned output gives the
    eager call's bits."""
    w = W.make_config("decode")
    c = harness.to_device(w)
    ref = c.run().clone()
    out = torch.empty_like(ref)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c.run(out=out, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.run(out=out, stream=s)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert mx4.mx4_index_get_device_status() == 0
    del c, g


def test_prefill_long_full_size():
    w = W.make_config("prefill-long")
    c, out = _run_full(w)
    assert out.shape == (4096, 64, 1024)
    # mask structure at any size: row r has ceil((126977 + r)/128) live pages
    live = torch.isfinite(out[:, 0, :]).sum(dim=1).cpu().numpy()
    exp = (126977 + np.arange(4096) + 127) // 128
    np.testing.assert_array_equal(live, exp)
    _sampled(w, out, 256)
    del c


def test_mtp_full_size_pool_past_4gib():
    w = W.make_config("mtp")
    assert W.STRADDLE_2_32_PAGE in set(w.page_ids.tolist())
    c, out = _run_full(w)
    assert out.shape == (256, 64, 256)
    # every row of every request: all 256 pages live
    assert torch.isfinite(out).all()
    _sampled(w, out, 256)
    del c


def test_chunked_full_size_256_sampled_rows():
    w = W.make_config("chunked")
    c, out = _run_full(w)
    assert out.shape == (32768, 64, 1038)
    live = torch.isfinite(out[:, 0, :]).sum(dim=1).cpu().numpy()
    exp = (100001 + np.arange(32768) + 127) // 128
    np.testing.assert_array_equal(live, exp)
    _sampled(w, out, 256)
    del c
