"""GPU parity of the MXFP4 index-K page writer against the oracle's writer:
the whole pool (every byte, touched or not) must be bit-identical."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
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


def _oracle_pool(case, num_pool_pages=0):
    bufs, (dbuf, doff), (sbuf, soff) = W.write_pool(case)
    kbits = case.k.view(torch.int16).numpy().view(np.uint16)
    kd = dbuf.numpy()
    ks = sbuf.numpy()
    bad = oracle.write_index_k(k_bits=kbits, slot_mapping=case.slot_mapping.numpy(), k_data=kd[doff:],
                               k_scale=ks[soff:], k_data_page_stride=case.k_data_page_stride,
                               k_scale_page_stride=case.k_scale_page_stride, num_pool_pages=num_pool_pages)
    return [b.numpy() for b in bufs], bad


def _gpu_pool(case, num_pool_pages=0, k=None):
    bufs, (dbuf, doff), (sbuf, soff) = W.write_pool(case, device="cuda")
    kk = case.k.cuda() if k is None else k
    mx4.mx4_index_k_write(kk, case.slot_mapping.cuda(), dbuf[doff:], sbuf[soff:], case.k_data_page_stride,
                          case.k_scale_page_stride, num_pool_pages=num_pool_pages)
    torch.cuda.synchronize()
    return [b.cpu().numpy() for b in bufs], mx4.mx4_index_get_device_status()


def _same(a, b):
    for x, y in zip(a, b):
        if not np.array_equal(x, y):
            idx = np.flatnonzero(x != y)
            raise AssertionError(f"{idx.size} bytes differ, first at {idx[:5].tolist()}: "
                                 f"gpu {x[idx[:5]].tolist()} oracle {y[idx[:5]].tolist()}")


@pytest.mark.parametrize("dist,layout,width,pad", [
    ("normal", "single", 128, 0),
    ("wide", "single", 128, 7),
    ("wide", "split", 136, 5),        # strided key rows, padded split views
    ("normal", "split", 256, 0),
])
def test_writer_bit_exact(dist, layout, width, pad):
    case = W.make_write_case(f"w-{dist}-{layout}", seed=40, num_tokens=3000, num_pool_pages=40, dist=dist,
                             layout=layout, row_width=width, pad_every=pad,
                             k_data_page_stride=None if layout == "single" else 8192 + 48,
                             k_scale_page_stride=None if layout == "single" else 512 + 4)
    ref, bad = _oracle_pool(case)
    got, st = _gpu_pool(case)
    assert bad == 0 and st == 0
    _same(got, ref)


def test_writer_unaligned_rows_take_the_scalar_path():
    case = W.make_write_case("w-odd", seed=41, num_tokens=515, num_pool_pages=8, dist="wide", row_width=131)
    ref, _ = _oracle_pool(case)
    # a key tensor whose rows start 2 bytes past a 16-byte boundary
    big = torch.zeros((case.num_tokens * 131 + 1,), dtype=torch.bfloat16, device="cuda")
    k = big[1:].view(case.num_tokens, 131)
    k.copy_(case.k.cuda())
    got, st = _gpu_pool(case, k=k)
    assert st == 0
    _same(got, ref)


def test_writer_every_bf16_magnitude_and_sign():
    """All 65,536 bf16 patterns except Inf/NaN, spread over groups with
    different maxima, against the oracle."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16)
    fin = torch.isfinite(x.float())
    bits = bits[fin]
    g = torch.Generator().manual_seed(42)
    bits = bits[torch.randperm(bits.numel(), generator=g)]
    n = bits.numel() // 128
    k = bits[: n * 128].view(torch.bfloat16).view(n, 128).clone()
    case = W.WriteCase(name="all", k=k, slot_mapping=torch.randperm(n + 100, generator=g)[:n].to(torch.int64),
                       num_pool_pages=(n + 100 + 127) // 128, layout="single", k_data_page_stride=W.PAGE_BYTES,
                       k_scale_page_stride=W.PAGE_BYTES)
    ref, _ = _oracle_pool(case)
    got, st = _gpu_pool(case)
    assert st == 0
    _same(got, ref)


def test_writer_out_of_pool_slots_flagged_and_skipped():
    case = W.make_write_case("w-bad", seed=43, num_tokens=200, num_pool_pages=2, pad_every=4)
    sm = case.slot_mapping.clone()
    sm[1] = 2 * 128          # first slot past a 2-page pool
    sm[2] = (1 << 40) + 3
    case = dataclasses.replace(case, slot_mapping=sm)
    ref, bad = _oracle_pool(case, num_pool_pages=2)
    got, st = _gpu_pool(case, num_pool_pages=2)
    assert bad == 2
    assert st & mx4.MX4_DEV_BAD_PAGE
    _same(got, ref)
    assert mx4.mx4_index_get_device_status() == 0


@pytest.mark.parametrize("name", W.WRITE_CONFIG_NAMES)
def test_writer_measured_workloads(name):
    case = W.make_write_config(name)
    ref, _ = _oracle_pool(case)
    got, st = _gpu_pool(case)
    assert st == 0
    _same(got, ref)


def test_writer_then_scorer_round_trip():
    """Keys written by the GPU writer, then scored by the GPU scorer, match
    the oracle scorer on the oracle writer's pages."""
    pages = 20          # the two requests use 6 + 12 pages
    base = W.make_workload("wr", seed=44, q_lens=[5, 9], seq_lens=[700, 1500], prefix_lens=[695, 1491],
                           pool_pages=pages)
    case = W.make_write_case("wr", seed=45, num_tokens=pages * 128, num_pool_pages=pages, dist="normal")
    case = dataclasses.replace(case, slot_mapping=torch.arange(pages * 128, dtype=torch.int64))
    ref_pool, _ = _oracle_pool(case)
    got_pool, st = _gpu_pool(case)
    assert st == 0
    _same(got_pool, ref_pool)
    pool = torch.from_numpy(ref_pool[0]).view(pages, W.PAGE_BYTES)
    ids = base.page_ids
    w = dataclasses.replace(base, pages_data=pool[ids, :W.DATA_BYTES].reshape(-1, 128, 64).clone(),
                            pages_scale=pool[ids, W.DATA_BYTES:].reshape(-1, 128, 4).clone())
    c = harness.to_device(w)
    out = c.run()
    torch.cuda.synchronize()
    assert mx4.mx4_index_get_device_status() == 0
    ref, _ = oracle_run(w)
    compare(out.cpu().numpy(), ref, what="writer->scorer")
