"""The C-ABI library loads and exports every symbol include/mx4_index.h
declares; host-side argument checks reject bad calls before any CUDA call.
CPU only: no call here reaches a kernel launch."""
import ctypes
import os
import re

import pytest

import sparse_attention_mxfp4_gb300 as mx4
from sparse_attention_mxfp4_gb300.buildlib import LIB_PATH, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mx4_index.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return mx4.load_library()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"\b(mx4_[a-z0-9_]+)\s*\(", src)


def test_header_declarations_match_exports(lib):
    declared = _declared()
    assert declared, "no declarations parsed"
    assert sorted(declared) == sorted(mx4.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.mx4_abi_version() == 2
    names = [lib.mx4_status_string(i).decode() for i in range(5)]
    assert names == ["MX4_OK", "MX4_ERR_INVALID_ARG", "MX4_ERR_MISALIGNED", "MX4_ERR_UNSUPPORTED",
                     "MX4_ERR_CUDA"]
    assert lib.mx4_status_string(99).decode() == "MX4_ERR_UNKNOWN"


# Fake, never dereferenced device addresses: every call below fails host
# validation before the library touches CUDA.
A = 1 << 20          # 1 MiB: aligned to everything
GOOD = dict(q=A, e4=0, kd=A, ks=A + 8192, sd=8704, ss=8704, bt=A, cu=A, sl=A, pl=A,
            mq=4, ms=1024, sm=0.088, out=A, stream=None, B=1, bts=8, npool=16)


def _prefill(lib, **kw):
    a = dict(GOOD)
    a.update(kw)
    return lib.mx4_index_score_prefill(a["q"], a["e4"], a["kd"], a["ks"], a["sd"], a["ss"], a["bt"], a["cu"],
                                       a["sl"], a["pl"], a["mq"], a["ms"], a["sm"], a["out"], a["stream"],
                                       a["B"], a["bts"], a["npool"])


def _decode(lib, **kw):
    a = dict(GOOD)
    a.update(kw)
    return lib.mx4_index_score_decode(a["q"], a["e4"], a["kd"], a["ks"], a["sd"], a["ss"], a["bt"], a["sl"],
                                      a["ms"], a["sm"], a["out"], a["stream"], a["B"], a["bts"], a["npool"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(kd=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(out=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(cu=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(e4=2), mx4.MX4_ERR_INVALID_ARG),
    (dict(sd=8191 + 1 - 32), mx4.MX4_ERR_INVALID_ARG),          # narrow data view
    (dict(ss=8704, sd=8704, ks=A + 8192, npool=0), mx4.MX4_ERR_INVALID_ARG),
    (dict(ss=496), mx4.MX4_ERR_INVALID_ARG),                   # narrow scale view
    (dict(bts=7), mx4.MX4_ERR_INVALID_ARG),                    # narrow block table
    (dict(ms=-1), mx4.MX4_ERR_INVALID_ARG),
    (dict(mq=-1), mx4.MX4_ERR_INVALID_ARG),
    (dict(B=-1), mx4.MX4_ERR_INVALID_ARG),
    (dict(sm=0.0), mx4.MX4_ERR_INVALID_ARG),
    (dict(sm=-1.0), mx4.MX4_ERR_INVALID_ARG),
    (dict(sm=float("inf")), mx4.MX4_ERR_INVALID_ARG),
    (dict(sm=float("nan")), mx4.MX4_ERR_INVALID_ARG),
    (dict(npool=1 << 31), mx4.MX4_ERR_UNSUPPORTED),
    (dict(kd=A + 16), mx4.MX4_ERR_MISALIGNED),                 # 4-bit TMA wants 32 B
    (dict(sd=8704 + 16, ss=8704 + 16), mx4.MX4_ERR_MISALIGNED),
    (dict(ks=A + 8), mx4.MX4_ERR_MISALIGNED),
    (dict(q=A + 8), mx4.MX4_ERR_MISALIGNED),
    (dict(out=A + 4), mx4.MX4_ERR_MISALIGNED),
])
def test_prefill_rejections(lib, kw, status):
    assert _prefill(lib, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(sl=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(bt=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(bts=3), mx4.MX4_ERR_INVALID_ARG),
    (dict(sd=4096), mx4.MX4_ERR_INVALID_ARG),
    (dict(kd=A + 48), mx4.MX4_ERR_MISALIGNED),
])
def test_decode_rejections(lib, kw, status):
    # decode does not need cu_seqlens / prefix_lens
    assert _decode(lib, cu=None, pl=None, **kw) == status


def test_quantize_rejections(lib):
    assert lib.mx4_quantize_q_e4m3(A, A, -1, None) == mx4.MX4_ERR_INVALID_ARG
    assert lib.mx4_quantize_q_e4m3(None, A, 16, None) == mx4.MX4_ERR_INVALID_ARG
    assert lib.mx4_quantize_q_e4m3(A, A, 0, None) == mx4.MX4_OK       # nothing to do
    assert lib.mx4_quantize_q_e4m3(A + 1, A, 16, None) == mx4.MX4_ERR_MISALIGNED


@pytest.mark.parametrize("kw,status", [
    (dict(n=-1), mx4.MX4_ERR_INVALID_ARG),
    (dict(n=0, k=None, slots=None), mx4.MX4_OK),                  # nothing to do
    (dict(k=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(slots=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(kd=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(ks=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(row=127), mx4.MX4_ERR_INVALID_ARG),                     # narrow key rows
    (dict(sd=8176), mx4.MX4_ERR_INVALID_ARG),                     # narrow data view
    (dict(ss=508), mx4.MX4_ERR_INVALID_ARG),                      # narrow scale view
    (dict(k=A + 1), mx4.MX4_ERR_MISALIGNED),
    (dict(slots=A + 4), mx4.MX4_ERR_MISALIGNED),
    (dict(kd=A + 8), mx4.MX4_ERR_MISALIGNED),
    (dict(sd=8192 + 8), mx4.MX4_ERR_MISALIGNED),
    (dict(ks=A + 2), mx4.MX4_ERR_MISALIGNED),
    (dict(ss=514), mx4.MX4_ERR_MISALIGNED),
])
def test_writer_rejections(lib, kw, status):
    a = dict(k=A, n=16, row=128, slots=A, kd=A, ks=A, sd=8704, ss=8704, pages=4)
    a.update(kw)
    assert lib.mx4_index_k_write(a["k"], a["n"], a["row"], a["slots"], a["kd"], a["ks"], a["sd"], a["ss"],
                                 a["pages"], None) == status


@pytest.mark.parametrize("kw,status", [
    (dict(k=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(sd=16384 - 16), mx4.MX4_ERR_INVALID_ARG),             # narrow fp8 page
    (dict(k=A + 8), mx4.MX4_ERR_MISALIGNED),
    (dict(sd=16384 + 8), mx4.MX4_ERR_MISALIGNED),
    (dict(pages=0), mx4.MX4_ERR_INVALID_ARG),
    (dict(B=0, k=None), mx4.MX4_OK),                             # nothing to do
])
def test_fp8_rejections(lib, kw, status):
    a = dict(q=A, k=A, sd=16384, bt=A, cu=A, sl=A, pl=A, mq=4, ms=512, out=A, B=1, bts=4, pages=8)
    a.update(kw)
    got = lib.mx4_index_score_prefill_fp8(a["q"], 0, a["k"], a["sd"], a["bt"], a["cu"], a["sl"], a["pl"], a["mq"],
                                          a["ms"], 0.088, a["out"], None, a["B"], a["bts"], a["pages"])
    assert got == status
    got_d = lib.mx4_index_score_decode_fp8(a["q"], 0, a["k"], a["sd"], a["bt"], a["sl"], a["ms"], 0.088, a["out"],
                                           None, a["B"], a["bts"], a["pages"])
    assert got_d == status


@pytest.mark.parametrize("kw,status", [
    (dict(k=0), mx4.MX4_ERR_INVALID_ARG),
    (dict(local=5, k=4), mx4.MX4_ERR_INVALID_ARG),
    (dict(local=-1), mx4.MX4_ERR_INVALID_ARG),
    (dict(groups=3), mx4.MX4_ERR_INVALID_ARG),
    (dict(groups=128), mx4.MX4_ERR_INVALID_ARG),
    (dict(sc=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(sel=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(ms=16384 * 128 + 1, bts=16385), mx4.MX4_ERR_UNSUPPORTED),
    (dict(bts=3), mx4.MX4_ERR_INVALID_ARG),                     # narrow block table
    (dict(sc=A + 2), mx4.MX4_ERR_MISALIGNED),
    (dict(tok=A + 2), mx4.MX4_ERR_MISALIGNED),                   # the optional token count output
    (dict(B=0, sc=None), mx4.MX4_OK),                            # no row
])
def test_topk_rejections(lib, kw, status):
    a = dict(sc=A, bt=A, sl=A, ms=512, k=4, local=1, groups=1, sel=A, cnt=A, tok=None, B=1, bts=4)
    a.update(kw)
    assert lib.mx4_index_topk_decode(a["sc"], a["bt"], a["sl"], a["ms"], a["k"], a["local"], a["groups"],
                                     a["sel"], a["cnt"], a["tok"], None, a["B"], a["bts"]) == status


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    missing = str(tmp_path / "nope.so")
    saved = mx4._lib
    try:
        mx4._lib = None
        with pytest.raises(RuntimeError, match="not built"):
            mx4.load_library(missing)
    finally:
        mx4._lib = saved


@pytest.mark.parametrize("kw,status", [
    (dict(rows=-1), mx4.MX4_ERR_INVALID_ARG),
    (dict(kvh=0), mx4.MX4_ERR_INVALID_ARG),
    (dict(groups=0), mx4.MX4_ERR_INVALID_ARG),
    (dict(width=-1), mx4.MX4_ERR_INVALID_ARG),
    (dict(scale=0.0), mx4.MX4_ERR_INVALID_ARG),
    (dict(scale=-0.5), mx4.MX4_ERR_INVALID_ARG),
    (dict(scale=float("nan")), mx4.MX4_ERR_INVALID_ARG),
    (dict(scale=float("inf")), mx4.MX4_ERR_INVALID_ARG),
    (dict(rows=0, q=None), mx4.MX4_OK),                            # nothing to do
    (dict(groups=17), mx4.MX4_ERR_UNSUPPORTED),                     # more than 16 query heads a KV head
    (dict(width=25), mx4.MX4_ERR_UNSUPPORTED),                      # more than 24 listed pages
    (dict(rows=1 << 30), mx4.MX4_ERR_UNSUPPORTED),                  # rows x KV heads x 2 CTAs past grid.x's limit
    (dict(rows=1 << 29, kvh=2, kd_ps=17408, ks_ps=17408, vd_ps=17408, vs_ps=17408), mx4.MX4_ERR_UNSUPPORTED),
    (dict(q=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(vs=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(bt=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(ctx=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(out=None), mx4.MX4_ERR_INVALID_ARG),
    (dict(pages=0), mx4.MX4_ERR_INVALID_ARG),
    (dict(kd_hs=8192 - 32), mx4.MX4_ERR_INVALID_ARG),              # narrow code view
    (dict(vs_hs=512 - 16), mx4.MX4_ERR_INVALID_ARG),               # narrow scale view
    (dict(kvh=2), mx4.MX4_ERR_INVALID_ARG),                         # page stride below 2 heads
    (dict(kd_ps=-8704), mx4.MX4_ERR_INVALID_ARG),
    (dict(kd=A + 16), mx4.MX4_ERR_MISALIGNED),                     # 4-bit TMA view: 32-byte rule
    (dict(kd_ps=8704 + 16), mx4.MX4_ERR_MISALIGNED),
    (dict(ks=A + 8192 + 8), mx4.MX4_ERR_MISALIGNED),
    (dict(vd=A + 8), mx4.MX4_ERR_MISALIGNED),
    (dict(vs_ps=8704 + 8), mx4.MX4_ERR_MISALIGNED),
    (dict(q=A + 8), mx4.MX4_ERR_MISALIGNED),
    (dict(out=A + 1), mx4.MX4_ERR_MISALIGNED),
    (dict(bt=A + 2), mx4.MX4_ERR_MISALIGNED),
    (dict(ctx=A + 2), mx4.MX4_ERR_MISALIGNED),
])
def test_sparse_attention_rejections(lib, kw, status):
    """Single-head pools ([pages, 1, 8704]: codes at byte 0, scales at 8192)
    with one argument broken at a time; every case returns before any CUDA
    call."""
    a = dict(q=A, rows=4, kvh=1, groups=16, kd=A, ks=A + 8192, kd_ps=8704, kd_hs=8704, ks_ps=8704, ks_hs=8704,
             vd=A, vs=A + 8192, vd_ps=8704, vd_hs=8704, vs_ps=8704, vs_hs=8704, bt=A, width=16, ctx=A,
             scale=0.088388, out=A, pages=64)
    a.update(kw)
    assert lib.mx4_sparse_pa_decode(a["q"], a["rows"], a["kvh"], a["groups"], a["kd"], a["ks"], a["kd_ps"],
                                    a["kd_hs"], a["ks_ps"], a["ks_hs"], a["vd"], a["vs"], a["vd_ps"], a["vd_hs"],
                                    a["vs_ps"], a["vs_hs"], a["bt"], a["width"], a["ctx"], a["scale"], a["out"],
                                    a["pages"], None) == status
