"""GPU sparse paged-attention decode (MXFP4 K and V) against the fp64 oracle.

Tolerance, from the arithmetic: the kernel rounds the softmax weights p to
bf16 (relative 2^-9) both in sum_t p v and in the normaliser, and rounds the
output to bf16; K, V and Q values are exact.  So
    |gpu - ref| <= 2^-9 (E_p|v| + |ref|) + 2^-9 |ref|,
E_p|v| = sum_t p_t |v_t| / sum_t p_t; the test allows twice each term.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_mxfp4_gb300 as mx4
from sparse_attention_mxfp4_gb300 import workloads as W
from helpers import e4m3_values_numpy
from test_oracle_attn import _dequant_pool, _run as oracle_attn

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


def _gpu(c):
    out = mx4.mx4_sparse_pa_decode(c.q.cuda(), c.k_pool.cuda(), c.v_pool.cuda(), c.block_table.cuda(),
                                   c.context_lens.cuda(), c.softmax_scale)
    torch.cuda.synchronize()
    st = mx4.mx4_index_get_device_status()
    assert st == 0, f"device status {st:#x}"
    return out.float().cpu().numpy()


def _abs_weighted_v(c):
    """E_p|v| for every (row, head, group, d), by a numpy softmax."""
    K, V = _dequant_pool(c.k_pool), _dequant_pool(c.v_pool)
    q = e4m3_values_numpy(c.q.numpy())
    out = np.zeros(q.shape)
    for r in range(c.rows):
        for h in range(c.kv_heads):
            n = int(c.context_lens[r, h])
            if n <= 0:
                continue
            ids = [int(x) for x in c.block_table[r, h, : (n + 127) // 128]]
            k = np.concatenate([K[x, h] for x in ids])[:n]
            v = np.concatenate([V[x, h] for x in ids])[:n]
            s = c.softmax_scale * (q[r, h] @ k.T)
            w = np.exp(s - s.max(axis=1, keepdims=True))
            out[r, h] = (w / w.sum(axis=1, keepdims=True)) @ np.abs(v)
    return out


def _check(c):
    got = _gpu(c)
    ref = oracle_attn(c)
    lim = 2.0 ** -8 * (_abs_weighted_v(c) + np.abs(ref)) + 2.0 ** -8 * np.abs(ref) + 1e-30
    err = np.abs(got - ref)
    bad = err > lim
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} outside; worst err {err.max():.3e}, "
                           f"at ref {ref.reshape(-1)[np.argmax(err)]:.4f}")
    rel_l2 = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel_l2 < 4e-3, rel_l2
    return rel_l2


@pytest.mark.parametrize("rows,kvh,groups,width", [(3, 1, 16, 5), (4, 2, 16, 3), (5, 1, 4, 7), (2, 2, 1, 24)])
def test_attn_small(rows, kvh, groups, width):
    c = W.make_attn_case(f"a{rows}{kvh}{groups}{width}", seed=100 + rows, rows=rows, kv_heads=kvh, groups=groups,
                         width=width)
    _check(c)


def test_attn_wide_scales_and_ragged_contexts():
    c = W.make_attn_case("wide", seed=110, rows=6, kv_heads=1, groups=16, width=6,
                         ctx=[1, 127, 128, 129, 640, 768], scale_lo=115, scale_hi=135)
    _check(c)


def test_attn_zero_query_is_mean_of_v():
    c = W.make_attn_case("mean", seed=111, rows=3, kv_heads=1, groups=16, width=4)
    c = dataclasses.replace(c, q=torch.zeros_like(c.q))
    _check(c)


def test_attn_empty_rows_are_zero():
    c = W.make_attn_case("empty", seed=112, rows=3, kv_heads=1, groups=8, width=2, ctx=[0, 5, 0])
    got = _gpu(c)
    assert (got[0] == 0).all() and (got[2] == 0).all()
    _check(c)


@pytest.mark.parametrize("name", ["pa-decode", "pa-decode-4kvh"])
def test_attn_full_size_config(name):
    c = W.make_attn_config(name)
    print("rel_l2", _check(c))


def _abs_weighted_v_rows(c):
    """E_p|v| as _abs_weighted_v, dequantizing only each row's listed pages
    (for cases whose pool is too large to dequantize whole)."""
    q = e4m3_values_numpy(c.q.numpy())
    out = np.zeros(q.shape)
    for r in range(c.rows):
        for h in range(c.kv_heads):
            n = int(c.context_lens[r, h])
            if n <= 0:
                continue
            ids = torch.tensor([int(x) for x in c.block_table[r, h, : (n + 127) // 128]], dtype=torch.long)
            k = _dequant_pool(c.k_pool[ids][:, h:h + 1])[:, 0].reshape(-1, 128)[:n]
            v = _dequant_pool(c.v_pool[ids][:, h:h + 1])[:, 0].reshape(-1, 128)[:n]
            s = c.softmax_scale * (q[r, h] @ k.T)
            w = np.exp(s - s.max(axis=1, keepdims=True))
            out[r, h] = (w / w.sum(axis=1, keepdims=True)) @ np.abs(v)
    return out


def _check_listed(c):
    """_check for a case whose pool is too large to dequantize whole."""
    got = _gpu(c)
    ref = oracle_attn(c)
    lim = 2.0 ** -8 * (_abs_weighted_v_rows(c) + np.abs(ref)) + 2.0 ** -8 * np.abs(ref) + 1e-30
    err = np.abs(got - ref)
    assert not (err > lim).any(), f"{int((err > lim).sum())} of {err.size} outside; worst err {err.max():.3e}"
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 4e-3
    return got


def test_attn_persistent_rows_of_every_length():
    """More rows than clusters, so every cluster streams several rows back to
    back with its stage, buffer and TMEM-slot rings carried across them; the
    lengths cycle through 0, 1, 127, 128, 129, 255, 256, 1536, 3071 and 3072
    tokens (rows with no page, with one page for one PV warp only, and with
    12 pages a CTA, which wraps the 12-slot ring every row) between seeded
    random ones."""
    rows, width = 400, 24
    special = [0, 1, 127, 128, 129, 255, 256, 1536, 3071, 3072]
    g = torch.Generator().manual_seed(131)
    rand = torch.randint(0, width * 128 + 1, (rows,), generator=g).tolist()
    ctx = [special[r // 2 % len(special)] if r % 2 == 0 else rand[r] for r in range(rows)]
    c = W.make_attn_case("persist", seed=132, rows=rows, kv_heads=1, groups=16, width=width,
                         pool_pages=rows * width, ctx=ctx)
    got = _check_listed(c)
    empty = np.array(ctx) == 0
    assert (got[empty] == 0).all()


@pytest.mark.parametrize("rows", [6, 64, 96])
@pytest.mark.parametrize("pattern", ["rising", "falling", "spike", "zigzag"])
def test_attn_offsets_move_within_a_row(pattern, rows):
    """K scale bytes set by each page's position within its CTA's half of the
    row, so that the scores of later pages pass the earlier ones by far more
    than 2^8 (log2 units): the per-head weight offsets then move up mid-row
    (every page for "rising", every other page for "zigzag", once for
    "spike", only on the first page for "falling"), and each move rescales
    the weight sums and both PV accumulators in TMEM.  Garbage past the
    context stays as drawn.  On GB300 (76 two-CTA clusters, 152 SMs) the 12
    items of 6 rows x 2 KV heads run in the one-group kernel, the 128 of 64
    rows in the two-group kernel on single CTAs (whole rows) and the 192 of
    96 rows in the two-group kernel on 2-CTA clusters."""
    kvh, width = 2, 16
    ctx = [[2048, 1921, 1000, 129, 2048, 1500][r % 6] for r in range(rows)]
    c = W.make_attn_case(f"offsets-{pattern}", seed=140, rows=rows, kv_heads=kvh, groups=16, width=width,
                         ctx=ctx, scale_lo=121, scale_hi=123, pool_pages=max(rows * kvh * width, 64))
    kp = c.k_pool.clone()
    for r in range(rows):
        for h in range(kvh):
            n = int(c.context_lens[r, h])
            npg = (n + 127) // 128
            half = (npg + 1) // 2
            for i in range(npg):
                pos = i if i < half else i - half
                b = {"rising": 122 + 2 * pos, "falling": 136 - 2 * pos, "spike": 136 if pos == 3 else 122,
                     "zigzag": 122 + 2 * pos if pos % 2 == 0 else 121}[pattern]
                nt = min(128, n - 128 * i)
                pg = int(c.block_table[r, h, i])
                kp[pg, h, W.DATA_BYTES:W.DATA_BYTES + 4 * nt] = b
    c = dataclasses.replace(c, k_pool=kp)
    _check_listed(c)


def _leftover_case(name, seed, rows, kvh, width=16):
    """Seeded case whose row contexts mix 0, 1, 129, 300, 383, 1000 and full
    rows with random lengths (the same for a row's KV heads)."""
    g = torch.Generator().manual_seed(seed)
    special = [0, 1, 129, 300, 383, width * 128, 1000]
    ctx = [special[r % len(special)] if r % 3 == 0 else
           int(torch.randint(0, width * 128 + 1, (1,), generator=g)) for r in range(rows)]
    return W.make_attn_case(name, seed=seed, rows=rows, kv_heads=kvh, groups=16, width=width,
                            pool_pages=rows * kvh * width, ctx=ctx)


@pytest.mark.parametrize("rows,kvh", [(77, 1), (79, 1), (151, 1), (160, 1), (233, 1), (305, 1), (64, 4)])
def test_attn_rows_past_whole_rounds(rows, kvh):
    """More rows x KV heads than 2-CTA clusters (76 on GB300), with a last
    round that is not whole.  The host runs the two-group kernel on single
    CTAs (152 on GB300: 77, 79, 151, 233 and 64 x 4 = 256 items) or on
    clusters (160, 305), whichever gives fewer pages a CTA.  Contexts ragged:
    empty rows, rows of one to three pages, full rows."""
    c = _leftover_case(f"left{rows}x{kvh}", 150 + rows, rows, kvh)
    got = _check_listed(c)
    empty = c.context_lens.numpy() == 0
    assert (got[empty] == 0).all()
