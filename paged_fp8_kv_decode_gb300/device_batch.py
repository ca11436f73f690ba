"""A decode batch resident on the GPU: pool, tables, tags, query and outputs.

``DeviceBatch`` allocates every buffer of one decode step once (caller-owned
device memory, as the C ABI requires), fills the cached tokens through
``pfkv_kv_append`` and then runs steps: append the new token (when the
workload appends) and attend.  It is the path the benchmark times and the
smoke check runs; all arithmetic happens in libpfkv.so.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import binding as B
from . import workloads as W


def _i32(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(device)


class DeviceBatch:
    def __init__(self, batch: W.Batch, device="cuda", keep_rows: bool = False,
                 tags: Optional[bool] = None, fill_chunk_tokens: int = 8192, rows=None,
                 q: Optional[torch.Tensor] = None, fused_tags: bool = False,
                 max_seq_len: Optional[int] = None):
        spec = batch.spec
        self.spec, self.batch, self.device = spec, batch, device
        self.fused_tags = fused_tags  # tag check inside the attention kernel
        use_tags = spec.tags if tags is None else tags
        NP, H, D = spec.num_pages, spec.Hkv, spec.D
        if spec.kv_dtype == "bf16":
            kp = torch.empty((NP, H, W.PAGE_SIZE, D), dtype=torch.bfloat16, device=device)
            ks = vs = None
        else:
            kp = torch.empty((NP, H, W.PAGE_SIZE, D), dtype=torch.uint8, device=device)
            ks = torch.ones((NP, H), dtype=torch.float32, device=device)
            vs = torch.ones((NP, H), dtype=torch.float32, device=device)
        vp = torch.empty_like(kp)
        kp.zero_()
        vp.zero_()
        self.page_tags = _i32(batch.page_tags, device)
        self.cache = B.Cache(kp, vp, ks, vs, self.page_tags if use_tags else None)
        self.cache_untracked = B.Cache(kp, vp, ks, vs, None)
        self.block_tables = _i32(batch.block_tables, device)
        self.expected_tags = _i32(batch.expected_tags, device)
        self.seq_lens = _i32(batch.seq_lens, device)
        self.fill_lens = _i32(batch.fill_lens, device)
        self.positions = _i32(batch.positions, device)
        sb, sh = batch.len_strides
        tb, th = batch.bt_strides
        self.pages = B.Pages(spec.B, batch.max_pages, self.block_tables, tb, th, self.seq_lens,
                             sb, sh, self.expected_tags if use_tags else None)
        self.pages_untracked = B.Pages(spec.B, batch.max_pages, self.block_tables, tb, th,
                                       self.fill_lens, sb, sh, None)
        self.max_seq_len = int(batch.seq_lens.max()) if batch.seq_lens.size else 0
        if max_seq_len is not None:  # a looser host-known bound, as a caller may pass
            self.max_seq_len = max(self.max_seq_len, int(max_seq_len))
        self.q = W.draw_q(spec, device=device) if q is None else q.to(device).contiguous()
        self.out = torch.empty((spec.B, spec.Hq, D), dtype=torch.bfloat16, device=device)
        nflag = max(4, (spec.B + 3) // 4 * 4)
        self.flags = torch.zeros(nflag, dtype=torch.uint8, device=device)
        self.append_flags = torch.zeros(nflag, dtype=torch.uint8, device=device)
        self.k_new = W.draw_new_token(spec, "k", device=device) if spec.append else None
        self.v_new = W.draw_new_token(spec, "v", device=device) if spec.append else None
        self.split_tokens = spec.split_tokens
        ws = B.pfkv_decode_workspace_size(self.cache, self.pages, spec.Hq, self.split_tokens,
                                          self.max_seq_len)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=device)
        self.k_rows = self.v_rows = None
        self._fill(keep_rows, fill_chunk_tokens, rows)

    # ------------------------------------------------------------------
    def _fill(self, keep_rows: bool, chunk: int, rows=None):
        """Write the cached tokens (positions 0..fill_len-1) of every (b, h)
        with kv_append, in page-aligned chunks of tokens.  Tags are not checked
        while filling: stale tags model pages reallocated afterwards."""
        spec = self.spec
        T = int(self.batch.fill_lens.max()) if self.batch.fill_lens.size else 0
        if T == 0:
            return
        if rows is None:
            k_rows = W.draw_kv_rows(spec, T, "k", device=self.device)
            v_rows = W.draw_kv_rows(spec, T, "v", device=self.device)
        else:
            k_rows = rows[0].to(self.device).contiguous()
            v_rows = rows[1].to(self.device).contiguous()
            assert k_rows.shape == (spec.B, spec.Hkv, T, spec.D), k_rows.shape
        if keep_rows:
            self.k_rows, self.v_rows = k_rows, v_rows
        chunk = max(W.PAGE_SIZE, chunk // W.PAGE_SIZE * W.PAGE_SIZE)
        fill = self.batch.fill_lens
        for t0 in range(0, T, chunk):
            t1 = min(T, t0 + chunk)
            pos = np.full_like(fill, t0)
            cnt = np.clip(fill - t0, 0, t1 - t0).astype(np.int32)
            B.pfkv_kv_append(self.cache_untracked, self.pages_untracked, _i32(pos, self.device),
                             k_rows[:, :, t0:t1].contiguous(), v_rows[:, :, t0:t1].contiguous(),
                             new_lens=_i32(cnt, self.device), flags=self.append_flags)
        torch.cuda.synchronize()
        if int(self.append_flags.sum()) != 0:
            raise RuntimeError(f"fill flagged requests: {self.append_flags.tolist()}")

    # ------------------------------------------------------------------
    def pack_step_io(self):
        """Move the tensors a decode step takes from the host (q, the new K/V
        rows, positions, lengths, block table, expected tags) into one device
        buffer, ``io_in``, and the step's outputs (out, flags) into another,
        ``io_out``, keeping their contents; a caller then moves each direction
        with one copy.  Call before taking pointers of these tensors."""
        spec = self.spec
        names = ["q", "positions", "seq_lens", "block_tables"]
        if spec.append:
            names += ["k_new", "v_new"]
        if self.pages.expected_tags is not None:
            names.append("expected_tags")
        self.io_in = self._pack(names)
        self.io_out = self._pack(["out", "flags"])
        sb, sh = self.batch.len_strides
        tb, th = self.batch.bt_strides
        self.pages = B.Pages(spec.B, self.batch.max_pages, self.block_tables, tb, th,
                             self.seq_lens, sb, sh,
                             self.expected_tags if self.pages.expected_tags is not None else None)

    def _pack(self, names):
        sizes = [getattr(self, n).numel() * getattr(self, n).element_size() for n in names]
        offs, off = [], 0
        for n in sizes:
            offs.append(off)
            off += (n + 255) // 256 * 256
        buf = torch.empty(max(off, 256), dtype=torch.uint8, device=self.device)
        for n, o, size in zip(names, offs, sizes):
            old = getattr(self, n)
            view = buf[o:o + size].view(old.dtype).view(old.shape)
            view.copy_(old)
            setattr(self, n, view)
        return buf

    def append_step(self, stream=None):
        if self.spec.append:
            B.pfkv_kv_append(self.cache, self.pages, self.positions, self.k_new, self.v_new,
                             flags=self.append_flags, stream=stream)

    def attend(self, stream=None, split_tokens: Optional[int] = None):
        fn = B.pfkv_paged_decode_attn_fused_tags if self.fused_tags else B.pfkv_paged_decode_attn
        fn(self.cache, self.pages, self.q, self.spec.sm_scale,
           self.split_tokens if split_tokens is None else split_tokens,
           self.max_seq_len, self.workspace, self.out, self.flags, stream=stream)

    def step(self, stream=None, one_call: bool = True):
        """One decode step: append the new token (if any), then attention;
        with ``one_call`` through pfkv_decode_step, else as the two calls."""
        if not (one_call and self.spec.append):
            self.append_step(stream)
            self.attend(stream)
            return
        B.pfkv_decode_step(self.cache, self.pages, self.positions, self.k_new, self.v_new, self.q,
                           self.spec.sm_scale, self.split_tokens, self.max_seq_len, self.workspace,
                           self.out, self.flags, append_flags=self.append_flags,
                           options=B.PFKV_STAGE_FUSED_TAGS if self.fused_tags else 0, stream=stream)

    # ------------------------------------------------------------------
    def _lens(self, skip=None) -> np.ndarray:
        lens = self.batch.lens_bh("seq").astype(np.int64)
        if skip is not None:
            lens = lens * ~np.asarray(skip, dtype=bool)[:, None]
        return lens

    def kv_bytes(self, skip=None) -> int:
        """Bytes of K and V the attention must read (partial pages count only
        their tokens).  ``skip``: bool per request, True for requests whose
        pages are not read (aborted by the tag check)."""
        el = 2 if self.spec.kv_dtype == "bf16" else 1
        return int(self._lens(skip).sum()) * self.spec.D * el * 2

    def algorithmic_bytes(self, skip=None, tags: Optional[bool] = None) -> int:
        """KV bytes + per-live-page table entry, FP8 scales and tags + q, out
        and flags: what one attention call must move at minimum.  Table
        entries and tags of every live page are read whatever the outcome; a
        skipped request's KV and scales are not."""
        spec = self.spec
        tags = self.cache.page_tags is not None if tags is None else tags
        all_pages = int(((self._lens() + W.PAGE_SIZE - 1) // W.PAGE_SIZE).sum())
        read_pages = int(((self._lens(skip) + W.PAGE_SIZE - 1) // W.PAGE_SIZE).sum())
        return (self.kv_bytes(skip) + 4 * all_pages
                + (8 * read_pages if spec.kv_dtype == "fp8" else 0)
                + (8 * all_pages if tags else 0)
                + 2 * spec.B * spec.Hq * spec.D * 2 + spec.B)
