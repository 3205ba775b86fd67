"""The bounded waits of the scorer and attention kernels, run out on the GPU
without hanging anything.

Every mbarrier wait of the kernels gives up after a time limit; the waiting
role then sets MX4_DEV_TIMEOUT and the bit of its wait site in the device
status word and raises the CTA's abort flag, every other role leaves its loop
at its next wait, the CTA lets its copies and MMAs finish, frees its tensor
memory and returns.  The test uses a separate test build of the library
(compiled with MX4_STALL_TEST and a 2 ms limit) in which the waits of one
chosen site in CTA 0 never see their barrier complete, as if the arriving
side had stalled.  For every wait site: the call returns, the status word
names the timeout and the site, and the next normal call in the same CUDA
context (through the test build and through the product library) matches the
oracle.  Nothing traps, faults or waits without a limit.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mxfp4_gb300 as mx4
from sparse_attention_mxfp4_gb300 import buildlib, harness
from sparse_attention_mxfp4_gb300 import workloads as W
from helpers import compare, oracle_run

pytestmark = pytest.mark.gpu

STALL_LIB = os.path.join(buildlib.BUILD_DIR, "libmx4index_stalltest.so")
STALL_FLAGS = ("-DMX4_STALL_TEST", "-DMX4_WAIT_LIMIT_NS=2000000ull")

# wait sites (the MX4_DEV_TIMEOUT site numbers of include/mx4_index.h)
SCORER_SITES = (0, 1, 2, 3, 4, 5)
ATTN_SITES = (6, 7, 8)


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx4.build()
    product = mx4.load_library()
    path = buildlib.build(lib_path=STALL_LIB, extra_flags=STALL_FLAGS)
    test = mx4.configure_library(ctypes.CDLL(path))
    test.mx4_test_set_stall.restype = ctypes.c_int
    test.mx4_test_set_stall.argtypes = [ctypes.c_int, ctypes.c_int]
    yield product, test
    mx4._lib = product


def _status(lib) -> int:
    v = ctypes.c_uint32(0)
    assert lib.mx4_index_get_device_status(None, ctypes.byref(v)) == mx4.MX4_OK
    return int(v.value)


def _scorer_case(kind):
    if kind == "prefill":
        w = W.make_workload("stall-p", seed=41, q_lens=[37, 5], seq_lens=[1500, 300], prefix_lens=[1463, 295],
                            pool_pages=24)
    else:   # decode block scores, with a partial last page
        w = W.make_workload("stall-d", seed=42, q_lens=None, seq_lens=[2055, 1200, 131], decode=True,
                            pool_pages=40)
    return w, harness.to_device(w)


def _scorer_ok(w, case):
    out = case.run()
    torch.cuda.synchronize()
    assert mx4.mx4_index_get_device_status() == 0
    ref, _ = oracle_run(w)
    compare(out.cpu().numpy(), ref, what=f"{w.name} after a timeout")


@pytest.mark.parametrize("kind,site", [(k, s) for k in ("prefill", "decode") for s in SCORER_SITES])
def test_scorer_wait_runs_out_and_reports(libs, kind, site):
    product, test = libs
    w, case = _scorer_case(kind)
    mx4._lib = test
    try:
        assert _status(test) == 0
        assert test.mx4_test_set_stall(site, 0) == mx4.MX4_OK
        case.run()
        torch.cuda.synchronize()
        st = _status(test)
        assert test.mx4_test_set_stall(-1, 0) == mx4.MX4_OK
        assert st & mx4.MX4_DEV_TIMEOUT, f"status {st:#x}"
        assert st & (0x100 << site), f"status {st:#x}: site {site} not named"
        # the same context serves the next call: test build, then product
        _scorer_ok(w, case)
    finally:
        mx4._lib = product
    _scorer_ok(w, case)


def _attn_case(rows):
    ac = W.make_attn_case(f"stall-a{rows}", seed=43, rows=rows, kv_heads=1, groups=16, width=5)
    dev = dict(q=ac.q.cuda(), k=ac.k_pool.cuda(), v=ac.v_pool.cuda(), bt=ac.block_table.cuda(),
               ctx=ac.context_lens.cuda())
    return ac, dev


def _attn_run(ac, d):
    return mx4.mx4_sparse_pa_decode(d["q"], d["k"], d["v"], d["bt"], d["ctx"], ac.softmax_scale)


def _attn_ok(ac, d):
    out = _attn_run(ac, d)
    torch.cuda.synchronize()
    assert mx4.mx4_index_get_device_status() == 0
    kd, ks, kps, khs, sps, shs = ac.views(ac.k_pool)
    vd, vs, vps, vhs, vsps, vshs = ac.views(ac.v_pool)
    ref = oracle.pa_decode(q=ac.q.numpy(), k_data=kd.numpy(), k_scale=ks.numpy(), kd_ps=kps, kd_hs=khs, ks_ps=sps,
                           ks_hs=shs, v_data=vd.numpy(), v_scale=vs.numpy(), vd_ps=vps, vd_hs=vhs, vs_ps=vsps,
                           vs_hs=vshs, block_table=ac.block_table.numpy(), context_lens=ac.context_lens.numpy(),
                           softmax_scale=ac.softmax_scale, num_pool_pages=ac.num_pool_pages)
    got = out.float().cpu().numpy()
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 4e-3


# 3 rows: one item a cluster (single-group kernel); 120 and 200 rows: more
# items than clusters (the two-group kernel, on single CTAs for 120 items and
# on 2-CTA clusters for 200 on GB300)
@pytest.mark.parametrize("rows", [3, 120, 200])
@pytest.mark.parametrize("site", ATTN_SITES)
def test_attention_wait_runs_out_and_reports(libs, site, rows):
    product, test = libs
    ac, d = _attn_case(rows)
    mx4._lib = test
    try:
        assert _status(test) == 0
        assert test.mx4_test_set_stall(site, 0) == mx4.MX4_OK
        _attn_run(ac, d)
        torch.cuda.synchronize()
        st = _status(test)
        assert test.mx4_test_set_stall(-1, 0) == mx4.MX4_OK
        assert st & mx4.MX4_DEV_TIMEOUT, f"status {st:#x}"
        assert st & (0x100 << site), f"status {st:#x}: site {site} not named"
        _attn_ok(ac, d)
    finally:
        mx4._lib = product
    _attn_ok(ac, d)
