"""Device-side session for one decode workload: upload, fill the cache, decode.

Uses only the C ABI through :mod:`.binding`; torch allocates device memory and
supplies the stream.  No arithmetic of the method happens here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from .workloads import CACHE_FP8, ROW_BYTES, Workload

# Byte pattern of cache memory before anything is appended: 0xFF makes every
# bf16 value NaN and every e4m3 byte NaN, so a read of an unwritten slot that
# is not masked out shows up in the output.
SENTINEL = 0xFF


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


class DecodeSession:
    def __init__(self, wl: Workload, device: str = "cuda", max_position: int | None = None,
                 splits: int = 0, stream=None, fp8_mma: bool | None = None, small_heads: bool | None = None):
        self.wl = wl
        self.device = torch.device(device)
        self.stream = stream
        fp8 = wl.cache_dtype == CACHE_FP8
        max_pos = int(max_position or max(64, wl.max_ctx))
        self.config = B.make_config(wl.n_h, cache_dtype=wl.cache_dtype, max_position=max_pos,
                                    rope_base=wl.rope_base, fp8_scale=wl.fp8_scale if fp8 else 0.0)
        self.w_uk = bf16_tensor(wl.w_uk, self.device)
        self.w_uv = bf16_tensor(wl.w_uv, self.device)
        self.mla = B.Mla(self.config, self.w_uk, self.w_uv, stream)
        if splits:
            self.mla.set_option(B.MLA_OPT_SPLITS, splits)
        if fp8_mma is not None:                 # None: the library's default (FP8 MMAs)
            self.mla.set_option(B.MLA_OPT_FP8_MMA, int(fp8_mma))
        if small_heads is not None:             # None: the library's default
            self.mla.set_option(B.MLA_OPT_SMALL_HEADS, int(small_heads))
        row_bytes = ROW_BYTES[wl.cache_dtype]
        self.cache = torch.full((wl.num_pages, wl.page_size, row_bytes), SENTINEL, dtype=torch.uint8,
                                device=self.device)
        self.block_table = torch.from_numpy(wl.block_table).to(self.device)
        self.ctx_len = torch.from_numpy(wl.ctx_len.astype(np.int32)).to(self.device)
        self.q = bf16_tensor(wl.q, self.device)
        self.out = torch.empty((wl.B, wl.n_h, wl.d_v), dtype=torch.bfloat16, device=self.device)
        ws = self.mla.decode_workspace_size(wl.B, wl.max_ctx)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.device)

    # -- cache fill -------------------------------------------------------------------
    def append_rows(self, idx: np.ndarray | None = None, chunk: int = 1 << 18) -> None:
        """Append workload rows ``idx`` (default: all) through mla_kv_append."""
        wl = self.wl
        idx = np.arange(wl.rows.shape[0]) if idx is None else np.asarray(idx)
        for a in range(0, len(idx), chunk):
            sel = idx[a:a + chunk]
            rows = bf16_tensor(wl.rows[sel], self.device)
            seq = torch.from_numpy(wl.row_seq[sel].astype(np.int32)).to(self.device)
            pos = torch.from_numpy(wl.row_pos[sel].astype(np.int32)).to(self.device)
            self.mla.kv_append(rows, seq, pos, self.block_table, self.cache, wl.num_pages, self.stream)

    def prefill(self) -> None:
        """Append every row except each sequence's last (the decode token's own row)."""
        self.append_rows(np.setdiff1d(np.arange(self.wl.rows.shape[0]), self.wl.last_row_index()))

    def step_inputs(self):
        """Device tensors of one decode step's new rows (each sequence's last row)."""
        wl = self.wl
        last = wl.last_row_index()
        rows = bf16_tensor(wl.rows[last], self.device)
        seq = torch.from_numpy(wl.row_seq[last].astype(np.int32)).to(self.device)
        pos = torch.from_numpy(wl.row_pos[last].astype(np.int32)).to(self.device)
        return rows, seq, pos

    # -- one step ------------------------------------------------------------------------
    def append_step(self, rows, seq, pos) -> None:
        self.mla.kv_append(rows, seq, pos, self.block_table, self.cache, self.wl.num_pages, self.stream)

    def decode(self, q=None, out=None) -> torch.Tensor:
        out = self.out if out is None else out
        self.mla.decode(self.q if q is None else q, self.ctx_len, self.wl.max_ctx, self.block_table, self.cache,
                        self.wl.num_pages, self.workspace, out, self.stream)
        return out

    def status(self) -> int:
        return self.mla.get_status(self.stream)

    def close(self) -> None:
        self.mla.close()
