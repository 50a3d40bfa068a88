"""Host-side owner of one layer's paged OSCAR cache.

Allocates the caller-owned device buffers the library writes (INT2 pool, BF16
window, page table, sequence state) with torch, hands pages out from a free
list, and builds shared-prefix forks by aliasing page-table entries. No
arithmetic of the method happens here; all cache writes and reads are the
library's kernels.

Paged attention with prefix reuse is the serving setting of the method:
"OSCAR: Offline Spectral Covariance-Aware Rotation ..." (gist.science, it),
Riepilogo Tecnico 2.2 B and 5 (paged KV cache, prefix caching kept).
"""

from __future__ import annotations

import numpy as np
import torch

from . import abi


class PagedCache:
    def __init__(self, ctx: "abi.Context", num_pages: int, device="cuda", page_order=None,
                 bind: bool = True):
        cfg = ctx.cfg
        self.ctx = ctx
        self.cfg = cfg
        self.num_pages = int(num_pages)
        self.page = cfg.page_size
        pool_bytes, window_bytes = abi.cache_bytes(cfg, self.num_pages)
        self.pool = torch.empty(pool_bytes, dtype=torch.uint8, device=device)
        self.window = torch.zeros(window_bytes // 2, dtype=torch.bfloat16, device=device)
        self.page_table_host = np.full((cfg.max_batch, cfg.max_pages_per_seq), -1, dtype=np.int32)
        self.page_table = torch.from_numpy(self.page_table_host.copy()).to(device)
        # oscar_seq_state rows: seq_len, int2_end, window_row, reserved
        st = np.zeros((cfg.max_batch, 4), dtype=np.int32)
        st[:, 1] = cfg.sink
        st[:, 2] = np.arange(cfg.max_batch)
        self.state = torch.from_numpy(st).to(device)
        order = np.arange(self.num_pages, dtype=np.int32) if page_order is None else \
            np.asarray(page_order, dtype=np.int32)
        if sorted(order.tolist()) != list(range(self.num_pages)):
            raise ValueError("page_order must be a permutation of range(num_pages)")
        self.free = list(order[::-1])  # pop() hands pages out in `order`
        self.refcount = np.zeros(self.num_pages, dtype=np.int32)
        if bind:
            ctx.bind_cache(self.pool, self.num_pages, self.window)

    # ---------------------------------------------------------------- pages
    def pages_needed(self, n_tokens: int) -> int:
        return (n_tokens + self.page - 1) // self.page

    def reserve(self, b: int, n_tokens: int, upload: bool = True):
        """Map positions [0, n_tokens) of request b to pages (allocating as needed)."""
        need = self.pages_needed(n_tokens)
        if need > self.cfg.max_pages_per_seq:
            raise ValueError("request needs %d pages, page table holds %d" % (need, self.cfg.max_pages_per_seq))
        row = self.page_table_host[b]
        for n in range(need):
            if row[n] < 0:
                if not self.free:
                    raise MemoryError("INT2 page pool exhausted")
                pid = self.free.pop()
                row[n] = pid
                self.refcount[pid] += 1
        if upload:
            self.upload(b)

    def upload(self, b=None):
        if b is None:
            self.page_table.copy_(torch.from_numpy(self.page_table_host))
        else:
            self.page_table[b].copy_(torch.from_numpy(self.page_table_host[b]))

    def release(self, b: int):
        row = self.page_table_host[b]
        for n in range(row.shape[0]):
            pid = row[n]
            if pid >= 0:
                self.refcount[pid] -= 1
                if self.refcount[pid] == 0:
                    self.free.append(pid)
                row[n] = -1
        self.upload(b)
        self.state[b] = torch.tensor([0, self.cfg.sink, b, 0], dtype=torch.int32)

    def fork(self, src: int, dst: int, prefix_tokens: int):
        """Request dst shares the first prefix_tokens of src (page aligned, all INT2 or sink).

        Page-table entries are aliased, the BF16 sink is copied, and dst's
        state is {prefix, prefix}: every later write lands in private pages.
        """
        if prefix_tokens % self.page:
            raise ValueError("a shared prefix must be page aligned")
        st = self.state[src].cpu().numpy()
        if prefix_tokens > max(int(st[1]), self.cfg.sink) or prefix_tokens < self.cfg.sink:
            raise ValueError("the shared prefix must lie in the source's sink + INT2 region")
        if self.page_table_host[dst].max() >= 0:
            self.release(dst)
        n = prefix_tokens // self.page
        self.page_table_host[dst, :n] = self.page_table_host[src, :n]
        for pid in self.page_table_host[dst, :n]:
            self.refcount[pid] += 1
        self.upload(dst)
        w = self.window.view(self.cfg.max_batch, self.cfg.num_kv_heads, 2,
                             self.cfg.sink + self.cfg.recent, 128)
        if self.cfg.sink:
            w[dst, :, :, :self.cfg.sink].copy_(w[src, :, :, :self.cfg.sink])
        self.state[dst] = torch.tensor([prefix_tokens, prefix_tokens, dst, 0], dtype=torch.int32)

    # ------------------------------------------------------------- accounting
    def footprint_bytes(self, batch: int):
        """(INT2 bytes of the mapped pages, BF16 window bytes) for `batch` requests."""
        used = np.unique(self.page_table_host[:batch][self.page_table_host[:batch] >= 0]).size
        kv = self.cfg.num_kv_heads
        return (used * kv * abi.page_block_bytes(self.cfg.group_size),
                batch * kv * 2 * (self.cfg.sink + self.cfg.recent) * 128 * 2)
