"""Device-side staging of a seeded workload and one call of the scorer.

Used by the GPU tests, ``bench.py`` and ``__graft_entry__.smoke()``.  It
places the workload's pool, query and metadata in device memory and calls the
binding; it performs none of the scorer's arithmetic.
"""
from __future__ import annotations

import dataclasses

import torch

from . import (mx4_index_score_decode, mx4_index_score_decode_fp8, mx4_index_score_prefill,
               mx4_index_score_prefill_fp8)
from . import workloads as W


@dataclasses.dataclass
class DeviceCase:
    w: W.Workload
    buffers: list
    k_data: torch.Tensor       # uint8 view whose first byte is page 0's data
    k_scale: torch.Tensor      # uint8 view whose first byte is page 0's scales
    q: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    cu_seqlens_q: torch.Tensor | None
    prefix_lens: torch.Tensor | None

    @property
    def out_shape_scores(self):
        return (self.w.total_rows, W.HEADS, self.w.num_out_pages)

    @property
    def out_shape_logits(self):
        return (self.w.total_rows, W.HEADS, self.w.max_seq_len)

    def run(self, out=None, logits=False, stream=None):
        w = self.w
        if w.cache == "fp8":
            if w.decode:
                return mx4_index_score_decode_fp8(
                    self.q, self.k_data, w.k_data_page_stride, self.block_table, self.seq_lens, w.max_seq_len,
                    w.sm_scale, out, num_pool_pages=w.num_pool_pages, stream=stream, logits=logits)
            return mx4_index_score_prefill_fp8(
                self.q, self.k_data, w.k_data_page_stride, self.block_table, self.cu_seqlens_q, self.seq_lens,
                self.prefix_lens, w.max_query_len, w.max_seq_len, w.sm_scale, out,
                num_pool_pages=w.num_pool_pages, stream=stream, logits=logits)
        if w.decode:
            return mx4_index_score_decode(
                self.q, self.k_data, self.k_scale, w.k_data_page_stride, w.k_scale_page_stride,
                self.block_table, self.seq_lens, w.max_seq_len, w.sm_scale, out,
                num_pool_pages=w.num_pool_pages, stream=stream, logits=logits)
        return mx4_index_score_prefill(
            self.q, self.k_data, self.k_scale, w.k_data_page_stride, w.k_scale_page_stride,
            self.block_table, self.cu_seqlens_q, self.seq_lens, self.prefix_lens, w.max_query_len,
            w.max_seq_len, w.sm_scale, out, num_pool_pages=w.num_pool_pages, stream=stream,
            logits=logits)

    def input_nbytes(self) -> int:
        n = sum(b.numel() for b in self.buffers) + self.q.numel() * self.q.element_size()
        n += self.block_table.numel() * 4 + self.seq_lens.numel() * 4
        if self.cu_seqlens_q is not None:
            n += self.cu_seqlens_q.numel() * 4 + self.prefix_lens.numel() * 4
        return n


def to_device(w: W.Workload, device="cuda", fill_seed=None) -> DeviceCase:
    """Stage workload ``w`` on ``device`` (pool pages not used by ``w`` are
    zero unless ``fill_seed`` asks for random bytes)."""
    bufs, (dbuf, doff), (sbuf, soff) = W.build_pool(w, device if fill_seed is None else "cpu",
                                                   fill_seed=fill_seed)
    if fill_seed is not None:
        bufs = [b.to(device) for b in bufs]
        dbuf = bufs[0]
        sbuf = bufs[-1] if w.layout == "split" else bufs[0]
    q = w.q.to(device)
    bt = w.block_table.to(device)
    sl = w.seq_lens.to(device)
    cu = None if w.decode else w.cu_seqlens_q.to(device)
    pl = None if w.decode else w.prefix_lens.to(device)
    return DeviceCase(w=w, buffers=bufs, k_data=dbuf[doff:], k_scale=sbuf[soff:], q=q, block_table=bt,
                      seq_lens=sl, cu_seqlens_q=cu, prefix_lens=pl)
