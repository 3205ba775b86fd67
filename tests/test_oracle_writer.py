"""Pins of the oracle's MXFP4 page writer (the OCP MX conversion reading).

Each check restates the rule independently: hand-worked groups from
tests/golden, an exhaustive nearest search over the e2m1 grid, the scale
exponent's closed form, the per-element rounding bound, exact round trips of
representable groups, byte placement by one-hot keys, and a vectorised numpy
writer written from the same definition in another formulation.
"""
import math
import os

import numpy as np
import torch

import oracle
from sparse_attention_mxfp4_gb300 import workloads as W
from helpers import dequant_numpy, scores_numpy, oracle_run

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_grid():
    """(codes 0..7, magnitudes) from the e2m1 bit fields: 1 sign, 2 exponent
    bits (bias 1), 1 mantissa bit."""
    codes = np.arange(8)
    e, m = codes >> 1, codes & 1
    mag = np.where(e > 0, np.exp2(e - 1.0) * (1 + m / 2.0), m / 2.0)
    return codes, mag


def _nearest_e2m1(x):
    """Exhaustive nearest search (ties to the even code, clamp at 6)."""
    codes, mag = _e2m1_grid()
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 6.0)
    d = np.abs(a[..., None] - mag)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    even = cand & (codes % 2 == 0)
    pick = np.where(cand.sum(-1) == 1, np.argmax(cand, -1), np.argmax(even, -1))
    return pick | (np.signbit(x).astype(np.int64) << 3)


def _parse_value(tok):
    m, e = tok.split("*2^")
    return float(m) * 2.0 ** int(e)


def _golden_groups():
    out = []
    with open(os.path.join(GOLDEN, "mxfp4_writer_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            ins, byte, codes = [s.strip() for s in line.split("|")]
            x = np.zeros(32)
            if ins != "-":
                for ent in ins.split(","):
                    i, v = ent.split(":")
                    x[int(i)] = _parse_value(v)
            c = np.zeros(32, dtype=np.uint8)
            if codes != "-":
                for ent in codes.split(","):
                    i, v = ent.split(":")
                    c[int(i)] = int(v)
            out.append((x, int(byte), c))
    return out


def test_golden_groups():
    groups = _golden_groups()
    assert len(groups) == 13
    for x, byte, codes in groups:
        b, c = oracle.quantize_group(x)
        assert b == byte, (x[np.nonzero(x)], b, byte)
        np.testing.assert_array_equal(c, codes)


def test_e2m1_rounding_exhaustive_grid():
    # every multiple of 1/64 in [-9, 9] (all ties and both saturation sides),
    # plus random reals and signed zeros
    xs = np.concatenate([np.arange(-9 * 64, 9 * 64 + 1) / 64.0,
                         np.random.default_rng(0).normal(0, 3, 4000), [0.0, -0.0]])
    got = np.array([oracle.e2m1_from_double(v) for v in xs])
    np.testing.assert_array_equal(got, _nearest_e2m1(xs))


def test_scale_byte_closed_form_and_element_bound():
    """4 * 2^(byte-127) <= amax < 8 * 2^(byte-127) whenever the clamp does not
    apply, and every element is within half an e2m1 step (or saturated)."""
    rng = np.random.default_rng(1)
    codes, mag = _e2m1_grid()
    for _ in range(3000):
        x = rng.normal(0, 1, 32) * 2.0 ** rng.integers(-100, 100)
        b, c = oracle.quantize_group(x)
        X = 2.0 ** (b - 127)
        amax = np.abs(x).max()
        if 1 < b < 254:
            assert 4 * X <= amax < 8 * X
        deq = mag[c & 7] * np.where(c & 8, -1.0, 1.0) * X
        r = np.abs(x) / X
        step = np.where(r < 2, 0.5, np.where(r < 4, 1.0, 2.0))
        sat = r > 6
        assert np.all(np.abs(deq - x)[~sat] <= step[~sat] / 2 * X)
        assert np.all(np.abs(deq[sat]) == 6 * X)
        assert np.all(np.signbit(deq) == np.signbit(x))


def test_representable_groups_round_trip_exactly():
    rng = np.random.default_rng(2)
    for _ in range(500):
        E = int(rng.integers(-120, 120))
        c = rng.integers(0, 8, 32)
        c[rng.integers(0, 32)] = rng.choice([6, 7])          # amax code 4 or 6 fixes E
        sign = rng.integers(0, 2, 32) * (c > 0)              # no negative zero here
        _, mag = _e2m1_grid()
        x = mag[c] * np.where(sign, -1.0, 1.0) * 2.0 ** E
        b, got = oracle.quantize_group(x)
        assert b == E + 127
        np.testing.assert_array_equal(got, c | (sign << 3))


def _write(case, **kw):
    bufs, (dbuf, doff), (sbuf, soff) = W.write_pool(case)
    kd = dbuf.numpy()
    ks = sbuf.numpy()
    before = [b.numpy().copy() for b in bufs]
    kbits = case.k.view(torch.int16).numpy().view(np.uint16)
    # the scale view of a single-region pool starts 8192 bytes into the buffer
    if case.layout == "single":
        ks_view = kd[doff + W.DATA_BYTES:]
        bad = oracle.write_index_k(k_bits=kbits, slot_mapping=case.slot_mapping.numpy(), k_data=kd[doff:],
                                   k_scale=ks_view, k_data_page_stride=case.k_data_page_stride,
                                   k_scale_page_stride=case.k_scale_page_stride, **kw)
    else:
        bad = oracle.write_index_k(k_bits=kbits, slot_mapping=case.slot_mapping.numpy(), k_data=kd[doff:],
                                   k_scale=ks[soff:], k_data_page_stride=case.k_data_page_stride,
                                   k_scale_page_stride=case.k_scale_page_stride, **kw)
    return bufs, before, bad


def test_one_hot_byte_placement():
    """Element d of a key lands in nibble d%2 of byte slot*64 + d//2 (low
    nibble for even d), its group's scale at byte slot*4 + d//32."""
    for d in (0, 1, 31, 32, 63, 64, 97, 126, 127):
        for slot in (0, 5, 128 + 77, 3 * 128 + 127):
            k = torch.zeros((1, 128), dtype=torch.bfloat16)
            k[0, d] = 1.0                 # amax 1 -> byte 125, code 6
            case = W.WriteCase(name="onehot", k=k, slot_mapping=torch.tensor([slot]), num_pool_pages=4,
                               layout="split", k_data_page_stride=8192 + 64, k_scale_page_stride=512 + 32)
            bufs, before, bad = _write(case)
            assert bad == 0
            dbuf, sbuf = bufs[0].numpy(), bufs[1].numpy()
            p, i = divmod(slot, 128)
            tok = dbuf[p * case.k_data_page_stride + i * 64:][:64]
            exp = np.zeros(64, dtype=np.uint8)
            exp[d // 2] = 6 << (4 * (d % 2))
            np.testing.assert_array_equal(tok, exp)
            sc = sbuf[p * case.k_scale_page_stride + i * 4:][:4]
            exp_s = np.full(4, 127, dtype=np.uint8)
            exp_s[d // 32] = 125
            np.testing.assert_array_equal(sc, exp_s)
            # nothing else changed
            dmask = np.ones_like(dbuf, dtype=bool)
            dmask[p * case.k_data_page_stride + i * 64:][:64] = False
            smask = np.ones_like(sbuf, dtype=bool)
            smask[p * case.k_scale_page_stride + i * 4:][:4] = False
            np.testing.assert_array_equal(dbuf[dmask], before[0][dmask])
            np.testing.assert_array_equal(sbuf[smask], before[1][smask])


def _numpy_writer(kbits):
    """Vectorised restatement: byte from the bf16 exponent field of the group
    maximum, codes by exhaustive nearest search of x / 2^(byte-127)."""
    x = (kbits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)[:, :128]
    g = x.reshape(-1, 4, 32)
    amax = np.abs(g).max(-1)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(amax > 0, amax, 1.0)))
    byte = np.where(amax > 0, np.clip(e - 2 + 127, 1, 254), 127).astype(np.int64)
    codes = _nearest_e2m1(g / np.exp2(byte - 127.0)[..., None])
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).reshape(-1, 64).astype(np.uint8)
    return packed, byte.astype(np.uint8)


def test_random_keys_against_numpy_writer():
    for dist, layout in (("normal", "single"), ("wide", "split")):
        case = W.make_write_case("rnd", seed=3, num_tokens=700, num_pool_pages=8, dist=dist, layout=layout,
                                 row_width=136, pad_every=9,
                                 k_data_page_stride=None if layout == "single" else 8192 + 96,
                                 k_scale_page_stride=None if layout == "single" else 512 + 16)
        bufs, before, bad = _write(case)
        assert bad == 0
        kbits = case.k.view(torch.int16).numpy().view(np.uint16)
        packed, byte = _numpy_writer(kbits)
        dbuf = bufs[0].numpy()
        sbuf = bufs[-1].numpy()
        soff = W.DATA_BYTES if layout == "single" else 0
        for t, s in enumerate(case.slot_mapping.tolist()):
            if s < 0:
                continue
            p, i = divmod(s, 128)
            np.testing.assert_array_equal(dbuf[p * case.k_data_page_stride + i * 64:][:64], packed[t])
            np.testing.assert_array_equal(sbuf[soff + p * case.k_scale_page_stride + i * 4:][:4], byte[t])


def test_padding_and_out_of_pool_slots_write_nothing():
    case = W.make_write_case("pad", seed=4, num_tokens=40, num_pool_pages=2, pad_every=3)
    sm = case.slot_mapping.clone()
    sm[1] = 2 * 128 + 5           # page 2 of a 2-page pool
    sm[2] = 1 << 40
    case.slot_mapping = sm
    bufs, before, bad = _write(case, num_pool_pages=2)
    assert bad == 2
    kbits = case.k.view(torch.int16).numpy().view(np.uint16)
    packed, _ = _numpy_writer(kbits)
    buf = bufs[0].numpy()
    touched = np.zeros_like(buf, dtype=bool)
    for t, s in enumerate(sm.tolist()):
        if 0 <= s < 2 * 128:
            p, i = divmod(s, 128)
            touched[p * W.PAGE_BYTES + i * 64:][:64] = True
            touched[p * W.PAGE_BYTES + W.DATA_BYTES + i * 4:][:4] = True
    np.testing.assert_array_equal(buf[~touched], before[0][~touched])


def test_written_pages_score_like_their_dequantised_values():
    """Writer then scorer (both oracle) against the numpy dequantisation of
    the written pages: the writer lays tokens out where the scorer reads."""
    pages = 3
    case = W.make_write_case("ws", seed=5, num_tokens=pages * 128, num_pool_pages=pages)
    case.slot_mapping = torch.arange(pages * 128, dtype=torch.int64)
    bufs, _, _ = _write(case)
    buf = bufs[0].view(pages, W.PAGE_BYTES)
    pd = buf[:, :W.DATA_BYTES].reshape(pages, 128, 64).clone()
    ps = buf[:, W.DATA_BYTES:].reshape(pages, 128, 4).clone()
    base = W.make_workload("ws", seed=6, q_lens=[3], seq_lens=[300], prefix_lens=[297], pool_pages=pages)
    ids = base.page_ids
    import dataclasses
    w = dataclasses.replace(base, pages_data=pd[ids], pages_scale=ps[ids])
    ref, _ = oracle_run(w)
    alt, _ = scores_numpy(w)
    np.testing.assert_allclose(ref, alt, rtol=1e-12, atol=1e-12)
    # and the dequantised keys are the bf16 keys within the rounding bound
    deq = dequant_numpy(w).reshape(-1, 128)
    kx = case.k.float().numpy().astype(np.float64)[np.concatenate([
        np.arange(int(p) * 128, int(p) * 128 + 128) for p in ids.tolist()])]
    sc = np.abs(kx).reshape(-1, 4, 32).max(-1).repeat(32, -1).reshape(kx.shape)
    assert np.all(np.abs(deq - kx) <= sc / 4 + 1e-300)
