"""Pins of the oracle's sparse paged-attention decode (MXFP4 K and V).

- uniform scores (zero query) give the plain mean of the valid V rows;
- two valid tokens give the closed form (e^a V1 + e^b V2) / (e^a + e^b);
- a numpy formulation (bit-field dequantisation, float64 softmax) agrees;
- garbage past the context and -1 entries past the list change nothing;
- attention is invariant under reordering the row's full pages.
"""
import dataclasses
import math

import numpy as np
import torch

import oracle
from sparse_attention_mxfp4_gb300 import workloads as W
from helpers import e4m3_values_numpy


def _dequant_pool(pool):
    """[pages, heads, 8704] -> values [pages, heads, 128, 128] from bit fields."""
    data = pool[:, :, :W.DATA_BYTES].numpy().reshape(pool.shape[0], pool.shape[1], 128, 64)
    scale = pool[:, :, W.DATA_BYTES:].numpy().reshape(pool.shape[0], pool.shape[1], 128, 4).astype(np.float64)
    codes = np.stack([data & 15, data >> 4], axis=-1).reshape(pool.shape[0], pool.shape[1], 128, 128)
    s, e, m = (codes >> 3) & 1, (codes >> 1) & 3, codes & 1
    mag = np.where(e > 0, np.exp2(e.astype(np.float64) - 1) * (1 + m / 2.0), m / 2.0)
    return np.where(s == 1, -mag, mag) * np.exp2(np.repeat(scale, 32, axis=-1) - 127.0)


def _run(c):
    kd, ks, kps, khs, sps, shs = c.views(c.k_pool)
    vd, vs, vps, vhs, vsps, vshs = c.views(c.v_pool)
    return oracle.pa_decode(q=c.q.numpy(), k_data=kd.numpy(), k_scale=ks.numpy(), kd_ps=kps, kd_hs=khs, ks_ps=sps,
                            ks_hs=shs, v_data=vd.numpy(), v_scale=vs.numpy(), vd_ps=vps, vd_hs=vhs, vs_ps=vsps,
                            vs_hs=vshs, block_table=c.block_table.numpy(), context_lens=c.context_lens.numpy(),
                            softmax_scale=c.softmax_scale, num_pool_pages=c.num_pool_pages)


def _numpy_attn(c):
    K = _dequant_pool(c.k_pool)
    V = _dequant_pool(c.v_pool)
    q = e4m3_values_numpy(c.q.numpy())
    out = np.zeros(q.shape)
    for r in range(c.rows):
        for h in range(c.kv_heads):
            n = int(c.context_lens[r, h])
            if n <= 0:
                continue
            ids = [int(p) for p in c.block_table[r, h, : (n + 127) // 128]]
            k = np.concatenate([K[p, h] for p in ids])[:n]
            v = np.concatenate([V[p, h] for p in ids])[:n]
            s = c.softmax_scale * (q[r, h] @ k.T)                 # [groups, n]
            s = np.exp(s - s.max(axis=1, keepdims=True))
            out[r, h] = (s / s.sum(axis=1, keepdims=True)) @ v
    return out


def test_zero_query_gives_mean_of_v():
    c = W.make_attn_case("mean", seed=90, rows=3, kv_heads=2, groups=4, width=3)
    c = dataclasses.replace(c, q=torch.zeros_like(c.q))
    got = _run(c)
    V = _dequant_pool(c.v_pool)
    for r in range(3):
        for h in range(2):
            n = int(c.context_lens[r, h])
            ids = [int(p) for p in c.block_table[r, h, : (n + 127) // 128]]
            mean = np.concatenate([V[p, h] for p in ids])[:n].mean(axis=0)
            for g in range(4):
                # summation order differs (pairwise vs sequential): bound by the terms, |v| <= 6
                np.testing.assert_allclose(got[r, h, g], mean, rtol=1e-12, atol=1e-13)


def test_two_tokens_closed_form():
    c = W.make_attn_case("two", seed=91, rows=1, kv_heads=1, groups=2, width=1, ctx=2)
    q = torch.zeros_like(c.q)
    q[0, 0, 0, 5] = 0x48        # e4m3 0x48 = 4.0
    q[0, 0, 1, 6] = 0xB8        # -1.0
    c = dataclasses.replace(c, q=q)
    got = _run(c)
    K = _dequant_pool(c.k_pool)[int(c.block_table[0, 0, 0]), 0]
    V = _dequant_pool(c.v_pool)[int(c.block_table[0, 0, 0]), 0]
    for g, (d, qv) in enumerate(((5, 4.0), (6, -1.0))):
        a, b = c.softmax_scale * qv * K[0, d], c.softmax_scale * qv * K[1, d]
        want = (math.exp(a) * V[0] + math.exp(b) * V[1]) / (math.exp(a) + math.exp(b))
        np.testing.assert_allclose(got[0, 0, g], want, rtol=1e-12, atol=1e-300)


def test_numpy_formulation():
    c = W.make_attn_case("np", seed=92, rows=4, kv_heads=2, groups=16, width=5, scale_lo=110, scale_hi=140)
    np.testing.assert_allclose(_run(c), _numpy_attn(c), rtol=1e-10, atol=1e-12)


def test_garbage_and_padding_do_not_leak():
    c = W.make_attn_case("gb", seed=93, rows=2, kv_heads=1, groups=4, width=3, ctx=[300, 257])
    a = _run(c)
    kp, vp = c.k_pool.clone(), c.v_pool.clone()
    bt = c.block_table.clone()
    for r in range(2):
        n = int(c.context_lens[r, 0])
        p = int(bt[r, 0, (n - 1) // 128])
        i0 = n % 128
        for pool in (kp, vp):
            pool[p, 0, i0 * 64:W.DATA_BYTES] = 0x77
            pool[p, 0, W.DATA_BYTES + i0 * 4:] = 255
    bt[bt < 0] = 12345678       # entries past the list are never read
    b = _run(dataclasses.replace(c, k_pool=kp, v_pool=vp, block_table=bt))
    np.testing.assert_array_equal(a, b)


def test_full_pages_reordered_give_same_output():
    c = W.make_attn_case("ord", seed=94, rows=2, kv_heads=1, groups=8, width=6)
    a = _run(c)
    bt = c.block_table.clone()
    for r in range(2):
        n = int(c.context_lens[r, 0])
        full = n // 128 if n % 128 else n // 128 - 1      # keep the last (maybe partial) page last
        perm = torch.randperm(full, generator=torch.Generator().manual_seed(r))
        bt[r, 0, :full] = c.block_table[r, 0, :full][perm]
    b = _run(dataclasses.replace(c, block_table=bt))
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_empty_context_gives_zeros():
    c = W.make_attn_case("z", seed=95, rows=2, kv_heads=1, groups=2, width=2, ctx=[0, 10])
    got = _run(c)
    assert (got[0] == 0).all() and np.isfinite(got).all() and (got[1] != 0).any()
