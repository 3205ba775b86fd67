"""Seeded synthetic inputs for the paged MXFP4 index-K scorer.

This module only draws random inputs and lays them out in memory; it holds
none of the scorer's arithmetic and imports neither the CUDA binding nor the
oracle.  Tests, ``bench.py`` and ``__graft_entry__`` use it to feed both sides
the same bytes.

Distributions follow the workloads the pages measure on (aiter #7061,
"Performance": random K data, e8m0 bytes in [122, 127]; the wide-scale check
of the same page, "Format", uses bytes 100..150):

* Q bf16: N(0, 1) per element, rounded to bf16 by torch.
* Q e4m3 (MTP workload only): N(0, 1) cast to float8_e4m3fn by torch (round to
  nearest even; |x| < 448 always holds for these draws).  This is input
  synthesis, not the scorer's query rounding.
* K data: uniform random bytes, i.e. all 16 e2m1 codes in both nibbles.
* K scales: uniform integers in [lo, hi] per (token, 32-element group).
* Bytes of tokens past a request's ``seq_len`` inside its last page are random
  garbage, scale bytes 0 and 255 included.
* Block-table entries past a request's last page are filled with -1.
* sm_scale = fp32(1/sqrt(128)).
* fp8 index cache (cache="fp8"): keys N(0, 1) cast to float8_e4m3fn by torch;
  garbage tails are random bytes with the e4m3 NaN codes planted.
* Index-K writes: bf16 keys N(0, 1), or a wide-range mix (see _keys), into
  slots from seeded block tables or seeded distinct pool slots.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

HEADS = 64
DIM = 128
PAGE = 128
DATA_BYTES = PAGE * DIM // 2      # 8192: 128 tokens x 64 B of e2m1 codes
SCALE_BYTES = PAGE * DIM // 32    # 512: 128 tokens x 4 e8m0 bytes
PAGE_BYTES = DATA_BYTES + SCALE_BYTES  # 8704

SM_SCALE = float(np.float32(1.0 / math.sqrt(DIM)))
FP8_PAGE_BYTES = PAGE * DIM       # 16384: 128 tokens x 128 e4m3 bytes (fp8 index cache)


@dataclasses.dataclass
class Workload:
    name: str
    decode: bool
    q: torch.Tensor                 # [rows, 64, 128] bfloat16, or uint8 e4m3 bytes
    q_is_e4m3: bool
    pages_data: torch.Tensor        # [U, 128, 64] uint8: contents of the used pages
    pages_scale: torch.Tensor       # [U, 128, 4] uint8
    page_ids: torch.Tensor          # [U] int64: physical id of each used page
    num_pool_pages: int
    layout: str                     # "single" (8704 B pages) or "split"
    k_data_page_stride: int         # bytes
    k_scale_page_stride: int        # bytes
    block_table: torch.Tensor       # [B, width] int32 physical ids (-1 padded)
    seq_lens: torch.Tensor          # [B] int32
    cu_seqlens_q: Optional[torch.Tensor]   # [B+1] int32 (prefill)
    prefix_lens: Optional[torch.Tensor]    # [B] int32 (prefill)
    max_query_len: int
    max_seq_len: int
    sm_scale: float = SM_SCALE
    description: str = ""
    cache: str = "mxfp4"            # "mxfp4", or "fp8": pages_fp8 holds the cache
    pages_fp8: Optional[torch.Tensor] = None   # [U, 128, 128] uint8 e4m3 bytes

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_out_pages(self) -> int:
        return (self.max_seq_len + PAGE - 1) // PAGE

    @property
    def block_table_stride(self) -> int:
        return int(self.block_table.shape[1])


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _q_bf16(g, rows):
    return torch.randn((rows, HEADS, DIM), generator=g, dtype=torch.float32).to(torch.bfloat16)


def _q_e4m3(g, rows):
    x = torch.randn((rows, HEADS, DIM), generator=g, dtype=torch.float32).clamp_(-448.0, 448.0)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def _page_contents(g, n_pages, scale_lo, scale_hi):
    data = torch.randint(0, 256, (n_pages, PAGE, DIM // 2), generator=g, dtype=torch.uint8)
    scale = torch.randint(scale_lo, scale_hi + 1, (n_pages, PAGE, DIM // 32),
                          generator=g, dtype=torch.uint8)
    return data, scale


def _garbage_tails(g, bt, seq_lens, page_index, pages_data, pages_scale):
    """Fill bytes of tokens past each request's end (inside its last page)
    with random garbage, including e8m0 bytes 0 and 255."""
    for b in range(bt.shape[0]):
        s = int(seq_lens[b])
        if s % PAGE == 0 or s == 0:
            continue
        pid = int(bt[b, s // PAGE])
        u = page_index[pid]
        tail = PAGE - s % PAGE
        pages_data[u, PAGE - tail:] = torch.randint(0, 256, (tail, DIM // 2), generator=g,
                                                    dtype=torch.uint8)
        sc = torch.randint(0, 256, (tail, DIM // 32), generator=g, dtype=torch.uint8)
        sc[0, 0] = 0
        sc[-1, -1] = 255
        pages_scale[u, PAGE - tail:] = sc


def _fp8_pages(g, n_pages):
    """fp8 index-cache pages: N(0, 1) keys cast to float8_e4m3fn by torch
    (input synthesis; |x| < 448 for these draws)."""
    x = torch.randn((n_pages, PAGE, DIM), generator=g, dtype=torch.float32)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def _fp8_garbage_tails(g, bt, seq_lens, page_index, pages_fp8):
    """Random bytes past each request's end inside its last page, the e4m3
    NaN codes 0x7F and 0xFF included."""
    for b in range(bt.shape[0]):
        s = int(seq_lens[b])
        if s % PAGE == 0 or s == 0:
            continue
        u = page_index[int(bt[b, s // PAGE])]
        tail = PAGE - s % PAGE
        t = torch.randint(0, 256, (tail, DIM), generator=g, dtype=torch.uint8)
        t[0, 0] = 0x7F
        t[-1, -1] = 0xFF
        pages_fp8[u, PAGE - tail:] = t


def make_workload(name, *, seed, q_lens, seq_lens, prefix_lens=None, decode=False,
                  pool_pages, q_e4m3=False, scale_lo=122, scale_hi=127,
                  layout="single", k_data_page_stride=None, k_scale_page_stride=None,
                  page_id_range=None, forced_page_ids=(), bt_width=None,
                  description="", cache="mxfp4") -> Workload:
    """Generic seeded workload.

    ``q_lens`` (prefill) / one row per request (decode), ``seq_lens`` and
    ``prefix_lens`` per request.  Physical pages are distinct and drawn from
    ``page_id_range`` (default the whole pool) by a seeded permutation.
    """
    g = _gen(seed)
    B = len(seq_lens)
    seq_lens_t = torch.tensor(seq_lens, dtype=torch.int32)
    if decode:
        q_lens = [1] * B
    rows = int(sum(q_lens))
    q = _q_e4m3(g, rows) if q_e4m3 else _q_bf16(g, rows)
    max_seq_len = int(max(seq_lens)) if B else 0
    pages_per_req = [(s + PAGE - 1) // PAGE for s in seq_lens]
    width = bt_width if bt_width is not None else max(1, (max_seq_len + PAGE - 1) // PAGE)
    n_used = int(sum(pages_per_req))
    lo, hi = page_id_range if page_id_range is not None else (0, pool_pages)
    assert hi - lo >= n_used and hi <= pool_pages
    forced = [int(p) for p in forced_page_ids]
    perm = (torch.randperm(hi - lo, generator=g) + lo).tolist()
    ids = forced + [p for p in perm if p not in set(forced)]
    ids = ids[:n_used]
    # shuffle so forced ids do not always land on request 0's first page
    order = torch.randperm(n_used, generator=g).tolist()
    ids = [ids[i] for i in order]
    bt = torch.full((B, width), -1, dtype=torch.int32)
    k = 0
    for b in range(B):
        for j in range(pages_per_req[b]):
            bt[b, j] = ids[k]
            k += 1
    page_ids = torch.tensor(ids, dtype=torch.int64)
    pages_data, pages_scale = _page_contents(g, n_used, scale_lo, scale_hi)
    page_index = {int(p): u for u, p in enumerate(ids)}
    _garbage_tails(g, bt, seq_lens, page_index, pages_data, pages_scale)
    pages_fp8 = None
    if cache == "fp8":
        # drawn after everything else, so the MXFP4 fields match the same
        # seed's MXFP4 workload
        pages_fp8 = _fp8_pages(g, n_used)
        _fp8_garbage_tails(g, bt, seq_lens, page_index, pages_fp8)
        layout = "fp8"
        sd = k_data_page_stride or FP8_PAGE_BYTES
        ss = 0
    elif layout == "single":
        sd = ss = k_data_page_stride or PAGE_BYTES
    else:
        sd = k_data_page_stride or DATA_BYTES
        ss = k_scale_page_stride or SCALE_BYTES
    if decode:
        cu = None
        pl = None
        max_q = 1
    else:
        cu = torch.zeros(B + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
        if prefix_lens is None:
            prefix_lens = [s - ql for s, ql in zip(seq_lens, q_lens)]
        pl = torch.tensor(prefix_lens, dtype=torch.int32)
        max_q = int(max(q_lens)) if B else 0
    return Workload(name=name, decode=decode, q=q, q_is_e4m3=q_e4m3,
                    pages_data=pages_data, pages_scale=pages_scale, page_ids=page_ids,
                    num_pool_pages=pool_pages, layout=layout, k_data_page_stride=sd,
                    k_scale_page_stride=ss, block_table=bt, seq_lens=seq_lens_t,
                    cu_seqlens_q=cu, prefix_lens=pl, max_query_len=max_q,
                    max_seq_len=max_seq_len, description=description, cache=cache, pages_fp8=pages_fp8)


# ---------------------------------------------------------------- configs --
CONFIG_NAMES = ("prefill-tiny", "decode", "prefill-long", "mtp", "chunked")
# the same workloads over an fp8 index cache (128 B per token), the format the
# MXFP4 cache replaces
FP8_CONFIG_NAMES = ("decode-fp8", "prefill-long-fp8")

# 2^32 lies inside page 493447 of an 8704 B-page pool (it starts at byte
# 4,294,962,688), so forcing that page in exercises the 64-bit page rebase.
STRADDLE_2_32_PAGE = 493447


def make_config(name: str, seed: Optional[int] = None) -> Workload:
    """The five measured configurations (H=64, D=128, 128-token pages), and
    the decode and prefill-long shapes over an fp8 index cache."""
    if name == "decode-fp8":
        return make_workload(name, seed=5 if seed is None else seed, q_lens=None, seq_lens=[131072] * 64,
                             decode=True, pool_pages=70000, cache="fp8",
                             description="B=64 x 1 row, seq 131072, fp8 cache (16384 B pages) in a 70000-page pool")
    if name == "prefill-long-fp8":
        return make_workload(name, seed=6 if seed is None else seed, q_lens=[4096], seq_lens=[131072],
                             prefix_lens=[126976], pool_pages=2048, cache="fp8",
                             description="B=1, 4096 rows, prefix 126976, seq 131072, fp8 cache, 2048-page pool")
    idx = CONFIG_NAMES.index(name)
    seed = idx if seed is None else seed
    if name == "prefill-tiny":
        return make_workload(name, seed=seed, q_lens=[32], seq_lens=[1024], prefix_lens=[992],
                             pool_pages=16, layout="single",
                             description="B=1, 32 rows, prefix 992, seq 1024, 16-page pool")
    if name == "decode":
        return make_workload(name, seed=seed, q_lens=None, seq_lens=[131072] * 64, decode=True,
                             pool_pages=70000, layout="split", k_data_page_stride=8320,
                             k_scale_page_stride=576,
                             description="B=64 x 1 row, seq 131072, split views in a 70000-page pool")
    if name == "prefill-long":
        return make_workload(name, seed=seed, q_lens=[4096], seq_lens=[131072],
                             prefix_lens=[126976], pool_pages=2048, layout="single",
                             description="B=1, 4096 rows, prefix 126976, seq 131072, 2048-page pool")
    if name == "mtp":
        return make_workload(name, seed=seed, q_lens=[8] * 32, seq_lens=[32768] * 32,
                             prefix_lens=[32760] * 32, pool_pages=600000, q_e4m3=True,
                             scale_lo=100, scale_hi=150, layout="single",
                             page_id_range=(480000, 600000),
                             forced_page_ids=(STRADDLE_2_32_PAGE,),
                             description="B=32 x 8 rows, seq 32768, e4m3 Q, e8m0 100..150, "
                                         "600000-page pool (5.2 GB, pages past 2^32 B)")
    if name == "chunked":
        return make_workload(name, seed=seed, q_lens=[32768], seq_lens=[132768],
                             prefix_lens=[100000], pool_pages=1200, layout="single",
                             description="B=1, 32768 rows, prefix 100000, seq 132768, 1200-page pool")
    raise KeyError(name)


# ---------------------------------------------------------------- layouts --
def relayout(w: Workload, layout: str, k_data_page_stride=None, k_scale_page_stride=None,
             num_pool_pages=None) -> Workload:
    """Same logical cache, other memory layout (single-region or split views)."""
    if layout == "single":
        sd = ss = k_data_page_stride or PAGE_BYTES
    else:
        sd = k_data_page_stride or DATA_BYTES
        ss = k_scale_page_stride or SCALE_BYTES
    return dataclasses.replace(w, layout=layout, k_data_page_stride=sd, k_scale_page_stride=ss,
                               num_pool_pages=num_pool_pages or w.num_pool_pages)


def permute_pages(w: Workload, seed: int) -> Workload:
    """Move every used page to another physical id and rewrite the block table."""
    g = _gen(seed)
    new_ids = torch.randperm(w.num_pool_pages, generator=g)[: w.page_ids.shape[0]].to(torch.int64)
    mapping = {int(o): int(n) for o, n in zip(w.page_ids.tolist(), new_ids.tolist())}
    bt = w.block_table.clone()
    flat = bt.view(-1)
    for i in range(flat.shape[0]):
        v = int(flat[i])
        if v >= 0:
            flat[i] = mapping[v]
    return dataclasses.replace(w, page_ids=new_ids, block_table=bt)


def _fill_pool(data_buf, scale_buf, w, ids, pages_data, pages_scale):
    sd, ss = w.k_data_page_stride, w.k_scale_page_stride
    n = ids.shape[0]
    if n == 0:
        return
    d_idx = (ids.view(-1, 1) * sd + torch.arange(DATA_BYTES, device=ids.device)).view(-1)
    s_idx = (ids.view(-1, 1) * ss + torch.arange(SCALE_BYTES, device=ids.device)).view(-1)
    data_buf.index_copy_(0, d_idx, pages_data.reshape(-1))
    scale_buf.index_copy_(0, s_idx, pages_scale.reshape(-1))


def pool_nbytes(w: Workload):
    """Bytes of the pool buffers: (data_buffer, scale_buffer or 0 when single)."""
    if w.cache == "fp8":
        return (w.num_pool_pages - 1) * w.k_data_page_stride + FP8_PAGE_BYTES, 0
    if w.layout == "single":
        return (w.num_pool_pages - 1) * w.k_data_page_stride + PAGE_BYTES, 0
    return ((w.num_pool_pages - 1) * w.k_data_page_stride + DATA_BYTES,
            (w.num_pool_pages - 1) * w.k_scale_page_stride + SCALE_BYTES)


def build_pool(w: Workload, device="cpu", fill_seed: Optional[int] = 1234,
               pin_memory: bool = False):
    """Materialise the pool.  Returns (buffers, k_data_view, k_scale_view) where
    the views are (tensor, byte offset) pairs into the buffers; unused pages
    hold seeded random bytes (or zeros when ``fill_seed`` is None)."""
    nd, ns = pool_nbytes(w)
    # 256-byte slack so the views can be placed on any alignment on request
    def alloc(n):
        if fill_seed is None or device != "cpu":
            t = torch.zeros(n, dtype=torch.uint8, device=device)
        else:
            t = torch.randint(0, 256, (n,), generator=_gen(fill_seed), dtype=torch.uint8)
        if pin_memory:
            t = t.pin_memory()
        return t
    ids = w.page_ids.to(device)
    if w.cache == "fp8":
        buf = alloc(nd)
        d_idx = (ids.view(-1, 1) * w.k_data_page_stride
                 + torch.arange(FP8_PAGE_BYTES, device=device)).view(-1)
        buf.index_copy_(0, d_idx, w.pages_fp8.to(device).reshape(-1))
        return [buf], (buf, 0), (buf, 0)
    pd = w.pages_data.to(device)
    ps = w.pages_scale.to(device)
    if w.layout == "single":
        buf = alloc(nd)
        # data of page p at p*stride, scales at p*stride + 8192
        d_idx = (ids.view(-1, 1) * w.k_data_page_stride
                 + torch.arange(DATA_BYTES, device=device)).view(-1)
        s_idx = (ids.view(-1, 1) * w.k_data_page_stride + DATA_BYTES
                 + torch.arange(SCALE_BYTES, device=device)).view(-1)
        buf.index_copy_(0, d_idx, pd.reshape(-1))
        buf.index_copy_(0, s_idx, ps.reshape(-1))
        return [buf], (buf, 0), (buf, DATA_BYTES)
    dbuf = alloc(nd)
    sbuf = alloc(ns)
    _fill_pool(dbuf, sbuf, w, ids, pd, ps)
    return [dbuf, sbuf], (dbuf, 0), (sbuf, 0)


def compact_host(w: Workload):
    """Host arrays for the oracle holding only the used pages: returns
    (k_data, k_scale, sd, ss, block_table, num_pool_pages) with the block
    table rewritten to compact page indices.  Physical placement does not
    enter the arithmetic; the layout and 64-bit placement invariances are
    checked separately on the real pools."""
    ids = w.page_ids.tolist()
    index = {p: u for u, p in enumerate(ids)}
    bt = w.block_table.clone()
    flat = bt.view(-1)
    for i in range(flat.shape[0]):
        v = int(flat[i])
        flat[i] = index[v] if v >= 0 else -1
    if w.cache == "fp8":
        kd = w.pages_fp8.numpy().reshape(-1)
        return kd, None, FP8_PAGE_BYTES, 0, bt.numpy(), len(ids)
    kd = w.pages_data.numpy().reshape(-1)
    ks = w.pages_scale.numpy().reshape(-1)
    return kd, ks, DATA_BYTES, SCALE_BYTES, bt.numpy(), len(ids)


def q_numpy(w: Workload) -> np.ndarray:
    """Q as raw bits for the oracle: uint16 (bf16) or uint8 (e4m3)."""
    if w.q_is_e4m3:
        return w.q.numpy()
    return w.q.view(torch.int16).numpy().view(np.uint16)


def sample_rows(w: Workload, n: int, seed: int = 0) -> np.ndarray:
    """Seeded sample of query rows (sorted), always including the first and
    last row."""
    total = w.total_rows
    if n >= total:
        return np.arange(total, dtype=np.int64)
    g = _gen(seed + 77)
    pick = torch.randperm(total, generator=g)[: max(0, n - 2)].tolist()
    s = sorted(set(pick) | {0, total - 1})
    return np.array(s[:n] if len(s) > n else s, dtype=np.int64)


# ------------------------------------------------------------ index-K writes --
@dataclasses.dataclass
class WriteCase:
    """Keys to quantise into pool page slots.

    ``k`` is [num_tokens, row_width] bfloat16; the key of token t is
    ``k[t, :128]`` (``row_width`` > 128 models a key that is a slice of a wider
    projection output).  ``slot_mapping[t]`` = page * 128 + token-in-page, or
    -1 for a padding token that is not written."""
    name: str
    k: torch.Tensor
    slot_mapping: torch.Tensor      # [num_tokens] int64
    num_pool_pages: int
    layout: str                     # "single" or "split"
    k_data_page_stride: int
    k_scale_page_stride: int
    description: str = ""

    @property
    def num_tokens(self) -> int:
        return int(self.k.shape[0])

    @property
    def k_row_stride(self) -> int:
        return int(self.k.stride(0))

    def pool_view(self) -> Workload:
        """A Workload shell carrying only the pool geometry (for pool_nbytes)."""
        return Workload(name=self.name, decode=True, q=torch.empty(0, HEADS, DIM, dtype=torch.bfloat16),
                        q_is_e4m3=False, pages_data=torch.empty(0, PAGE, DIM // 2, dtype=torch.uint8),
                        pages_scale=torch.empty(0, PAGE, DIM // 32, dtype=torch.uint8),
                        page_ids=torch.empty(0, dtype=torch.int64), num_pool_pages=self.num_pool_pages,
                        layout=self.layout, k_data_page_stride=self.k_data_page_stride,
                        k_scale_page_stride=self.k_scale_page_stride,
                        block_table=torch.empty(0, 1, dtype=torch.int32),
                        seq_lens=torch.empty(0, dtype=torch.int32), cu_seqlens_q=None, prefix_lens=None,
                        max_query_len=0, max_seq_len=0)


def _keys(g, n, width, dist):
    """bf16 keys.  "normal": N(0, 1).  "wide": N(0, 1) times 2^u per 32-element
    group with u uniform in [-60, 60], plus all-zero groups, signed zeros,
    groups near the bottom of the bf16 range (subnormals included) and near the
    top, so every scale byte branch and rounding tie occurs."""
    x = torch.randn((n, width), generator=g, dtype=torch.float32)
    if dist == "wide":
        grp = x[:, :DIM].view(n, DIM // 32, 32)
        u = torch.randint(-60, 61, (n, DIM // 32, 1), generator=g).to(torch.float32)
        grp.mul_(torch.exp2(u))
        sel = torch.rand((n, DIM // 32), generator=g)
        grp[sel < 0.03] = 0.0
        tiny = (sel >= 0.03) & (sel < 0.06)
        grp[tiny] = torch.randn((int(tiny.sum()), 32), generator=g) * 2.0 ** -128
        huge = (sel >= 0.06) & (sel < 0.08)
        grp[huge] = torch.randn((int(huge.sum()), 32), generator=g) * 2.0 ** 120
        z = torch.rand((n, DIM), generator=g) < 0.01
        x[:, :DIM][z] = 0.0
        negz = torch.rand((n, DIM), generator=g) < 0.005
        x[:, :DIM][negz] = -0.0
    elif dist != "normal":
        raise ValueError(dist)
    return x.to(torch.bfloat16)


def make_write_case(name, *, seed, num_tokens, num_pool_pages, row_width=DIM, layout="single",
                    k_data_page_stride=None, k_scale_page_stride=None, dist="normal",
                    pad_every=0, block_table=None, positions=None, description="") -> WriteCase:
    """Seeded write case.  Slots come from ``block_table`` [B, width] and
    ``positions`` (pairs (b, pos): slot = block_table[b, pos // 128] * 128 +
    pos % 128) when given, else from a seeded draw of distinct slots of the
    pool.  Every ``pad_every``-th token (when > 0) is padding (slot -1)."""
    g = _gen(seed)
    k = _keys(g, num_tokens, row_width, dist)
    if block_table is not None:
        b, pos = positions
        slot = block_table[b, pos // PAGE].to(torch.int64) * PAGE + pos % PAGE
    else:
        slot = torch.randperm(num_pool_pages * PAGE, generator=g)[:num_tokens].to(torch.int64)
    slot = slot.clone()
    if pad_every > 0:
        slot[::pad_every] = -1
    if layout == "single":
        sd = ss = k_data_page_stride or PAGE_BYTES
    else:
        sd = k_data_page_stride or DATA_BYTES
        ss = k_scale_page_stride or SCALE_BYTES
    return WriteCase(name=name, k=k, slot_mapping=slot, num_pool_pages=num_pool_pages, layout=layout,
                     k_data_page_stride=sd, k_scale_page_stride=ss, description=description)


def write_pool(c: WriteCase, device="cpu", fill_seed: Optional[int] = 4321):
    """Pool buffers for a write case, filled with seeded random bytes (so a
    test can see which bytes a write touched).  Returns (buffers, (data_buf,
    data_offset), (scale_buf, scale_offset)) like ``build_pool``."""
    nd, ns = pool_nbytes(c.pool_view())

    def alloc(n):
        t = torch.randint(0, 256, (n,), generator=_gen(fill_seed), dtype=torch.uint8)
        return t.to(device)
    if c.layout == "single":
        buf = alloc(nd)
        return [buf], (buf, 0), (buf, DATA_BYTES)
    dbuf = alloc(nd)
    sbuf = alloc(ns)
    return [dbuf, sbuf], (dbuf, 0), (sbuf, 0)


WRITE_CONFIG_NAMES = ("write-decode", "write-chunk")


def make_write_config(name: str, seed: Optional[int] = None) -> WriteCase:
    """Index-K writes of the measured workloads: one new key per request of
    the decode workload (64 tokens), and the 32768 new keys of the chunked
    prefill (positions 100000..132767 of its request)."""
    if name == "write-decode":
        seed = 10 if seed is None else seed
        g = _gen(seed + 1000)
        bt = torch.randperm(70000, generator=g)[: 64 * 1025].view(64, 1025).to(torch.int32)
        pos = torch.full((64,), 131072, dtype=torch.int64)
        return make_write_case(name, seed=seed, num_tokens=64, num_pool_pages=70000, layout="split",
                               k_data_page_stride=8320, k_scale_page_stride=576, block_table=bt,
                               positions=(torch.arange(64), pos),
                               description="64 requests x 1 new key at position 131072, split views, "
                                           "70000-page pool")
    if name == "write-chunk":
        seed = 11 if seed is None else seed
        g = _gen(seed + 1000)
        bt = torch.randperm(1200, generator=g)[:1038].view(1, 1038).to(torch.int32)
        pos = torch.arange(100000, 132768, dtype=torch.int64)
        return make_write_case(name, seed=seed, num_tokens=32768, num_pool_pages=1200, layout="single",
                               block_table=bt, positions=(torch.zeros_like(pos), pos),
                               description="32768 keys at positions 100000..132767 of one request, "
                                           "1200-page pool")
    raise KeyError(name)


# ----------------------------------------------- sparse paged attention --
@dataclasses.dataclass
class AttnCase:
    """Decode attention over each row's selected pages.

    K and V pools are [pool_pages, kv_heads, 8704] uint8: one MXFP4 page per
    (page, kv head), codes at byte 0 and scales at byte 8192 of each page
    (ATOM #2770 "How it works", item "Pool").  ``block_table`` [rows,
    kv_heads, width] lists each row's pages in order (-1 padded);
    ``context_lens`` [rows, kv_heads] counts its valid tokens (a prefix of the
    list); ``q`` is e4m3 bytes [rows, kv_heads, groups, 128]."""
    name: str
    q: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_table: torch.Tensor
    context_lens: torch.Tensor
    softmax_scale: float = SM_SCALE
    description: str = ""

    @property
    def rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def kv_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def groups(self) -> int:
        return int(self.q.shape[2])

    @property
    def num_pool_pages(self) -> int:
        return int(self.k_pool.shape[0])

    def views(self, pool):
        """(data, scale, data page stride, data head stride, scale page
        stride, scale head stride) of a [pages, kv_heads, 8704] pool (flat
        uint8 views starting at page 0 of each)."""
        flat = pool.reshape(-1)
        ps = self.kv_heads * PAGE_BYTES
        return flat, flat[DATA_BYTES:], ps, PAGE_BYTES, ps, PAGE_BYTES


def make_attn_case(name, *, seed, rows, kv_heads=1, groups=16, width=16, pool_pages=None, ctx=None,
                   scale_lo=122, scale_hi=127, description="") -> AttnCase:
    """Seeded attention case: each (row, kv head) selects ``width`` distinct
    pool pages (a seeded draw); ``ctx`` gives each row's valid tokens (default:
    a seeded length in ((width-1)*128, width*128], so the last page is partial
    most of the time); bytes past a row's context in its last page are garbage
    (e8m0 0 and 255 included).  Q: N(0, 1) cast to float8_e4m3fn by torch."""
    g = _gen(seed)
    pool_pages = pool_pages or max(2 * width * rows * kv_heads, 64)
    q = torch.randn((rows, kv_heads, groups, DIM), generator=g).clamp_(-448, 448)
    q = q.to(torch.float8_e4m3fn).view(torch.uint8)
    pools = []
    for _ in range(2):
        data = torch.randint(0, 256, (pool_pages, kv_heads, DATA_BYTES), generator=g, dtype=torch.uint8)
        scale = torch.randint(scale_lo, scale_hi + 1, (pool_pages, kv_heads, SCALE_BYTES), generator=g,
                              dtype=torch.uint8)
        pools.append(torch.cat([data, scale], dim=2).contiguous())
    bt = torch.full((rows, kv_heads, width), -1, dtype=torch.int32)
    cl = torch.zeros((rows, kv_heads), dtype=torch.int32)
    # distinct pages across the whole case (a page belongs to one row)
    assert pool_pages >= rows * kv_heads * width
    ids = torch.randperm(pool_pages, generator=g)[: rows * kv_heads * width].to(torch.int32)
    for r in range(rows):
        for h in range(kv_heads):
            if ctx is None:
                c = int(torch.randint((width - 1) * PAGE + 1, width * PAGE + 1, (1,), generator=g))
            else:
                c = int(ctx[r] if hasattr(ctx, "__len__") else ctx)
            npg = (c + PAGE - 1) // PAGE
            k0 = (r * kv_heads + h) * width
            bt[r, h, :npg] = ids[k0:k0 + npg]
            cl[r, h] = c
            if c % PAGE:
                # garbage past the context inside the last page, K and V
                p = int(bt[r, h, npg - 1])
                i0 = c % PAGE
                for pool in pools:
                    pool[p, h, i0 * 64:DATA_BYTES] = torch.randint(0, 256, (DATA_BYTES - i0 * 64,), generator=g,
                                                                   dtype=torch.uint8)
                    sc = torch.randint(0, 256, (SCALE_BYTES - i0 * 4,), generator=g, dtype=torch.uint8)
                    sc[0] = 0
                    sc[-1] = 255
                    pool[p, h, DATA_BYTES + i0 * 4:] = sc
    return AttnCase(name=name, q=q, k_pool=pools[0], v_pool=pools[1], block_table=bt, context_lens=cl,
                    description=description)


ATTN_CONFIG_NAMES = ("pa-decode",)


def make_attn_config(name: str, seed: Optional[int] = None) -> AttnCase:
    """Sparse decode attention of the decode workload's shape: 64 requests,
    one KV head (or four) with 16 query heads each, 16 selected pages (2,048
    tokens) per (request, KV head)."""
    if name == "pa-decode":
        return make_attn_case(name, seed=20 if seed is None else seed, rows=64, kv_heads=1, groups=16, width=16,
                              pool_pages=8192,
                              description="64 rows x 1 KV head x 16 query heads, 16 selected pages of an "
                                          "8192-page pool (K+V pools 143 MB), context 1921..2048 tokens")
    if name == "pa-decode-4kvh":
        return make_attn_case(name, seed=21 if seed is None else seed, rows=64, kv_heads=4, groups=16, width=16,
                              pool_pages=4096,
                              description="64 rows x 4 KV heads x 16 query heads, 16 selected pages per (row, KV "
                                          "head) of a 4096-page pool (K+V pools 285 MB), context 1921..2048 tokens")
    raise KeyError(name)
