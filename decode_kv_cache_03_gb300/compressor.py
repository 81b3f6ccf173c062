"""Convenience wrapper around the C ABI for one paged cache."""
from __future__ import annotations

import torch

from . import kara


class Compressor:
    """Periodic compression of the trailing windows of selected sequences.

    Holds the device workspace and error word; the cache, tables and fresh
    block ids stay owned by the caller.
    """

    def __init__(self, k: torch.Tensor, v: torch.Tensor, num_q_heads: int, W: int, B: int, K: int, R: int,
                 lam: float = 0.1, score_mode: int = 0, select_mode: int = 0, chunk: int = 0):
        self.k, self.v = k, v
        self.cache = kara.cache(k, v, num_q_heads)
        self.params = kara.params(W, B, K, R, lam, score_mode, select_mode, chunk)
        self.err = torch.zeros(1, dtype=torch.int32, device=k.device)
        self._ws = torch.empty(0, dtype=torch.uint8, device=k.device)
        self._dws = torch.empty(0, dtype=torch.uint8, device=k.device)

    def workspace(self, n: int) -> torch.Tensor:
        need = kara.kara_workspace_size(self.cache, self.params, n)
        if self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.k.device)
        return self._ws

    def plan(self, lengths_host: torch.Tensor, bt_stride: int):
        return kara.kara_plan(self.params, self.cache.block_size, lengths_host, bt_stride)

    def compress(self, lengths, block_table, q, fresh, freed, new_len, scores=None, cand=None, kept=None,
                 stream=None):
        """Enqueue the whole step; block_table is rewritten in place on success."""
        b = kara.batch(lengths, block_table, q)
        ws = self.workspace(b.n)
        kara.kara_compress_batch(self.cache, self.params, b, fresh, freed, new_len, ws, self.err, scores, cand,
                                 kept, stream)

    def decode(self, layer: int, lengths, block_table, q, out, stream=None):
        """Enqueue decode attention for one layer over the paged cache.  Called on
        the same stream right after compress() with its new_len and the table it
        rewrote in place, it reads the compacted cache with no host round trip."""
        n, bt_stride = block_table.shape
        need = kara.kara_decode_workspace_size(self.cache, n, bt_stride)
        if self._dws.numel() < need:
            self._dws = torch.empty(need, dtype=torch.uint8, device=self.k.device)
        kara.kara_decode_attention(self.cache, layer, lengths, block_table, q, out, self._dws, self.err, stream)

    def error(self, stream=None) -> int:
        return kara.kara_get_error(self.err, stream)
