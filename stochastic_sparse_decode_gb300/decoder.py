"""A convenience wrapper: owns the problem description and the workspaces.

    dec = Decoder(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
                  total_tokens=32768, max_len=32768, tile=256, S=128, dtype="bf16")
    out = dec("prop", q, k, v, kv_indptr, U)

Workspaces are allocated once per mode with torch (device memory only); each
call is one C-ABI call on the current stream.  Debug buffers can be requested
to inspect tile records, budgets and sampled indices.
"""

from __future__ import annotations

import torch

from . import (MODES, Debug, decode, k_feature_blocked_size, make_pages, make_problem, santa_decode_prop_bernoulli,
               santa_decode_prop_paged, santa_k_feature_blocked, santa_prop_pass1, santa_prop_pass2, workspace_size)


class Decoder:
    def __init__(self, batch, num_q_heads, num_kv_heads, head_dim, total_tokens, max_len, tile, S, dtype,
                 device=None):
        self.problem = make_problem(batch, num_q_heads, num_kv_heads, head_dim, total_tokens, max_len, tile, S,
                                    dtype)
        self.device = torch.device(device if device is not None else "cuda")
        self.Tmax = -(-max_len // tile) if max_len > 0 else 0
        self._ws = {}

    def workspace(self, mode: str) -> torch.Tensor:
        if mode not in self._ws:
            n = workspace_size(self.problem, MODES[mode])
            # zero-filled: a prop workspace must start zero (santa_workspace_init)
            self._ws[mode] = torch.zeros(n, dtype=torch.uint8, device=self.device)
        return self._ws[mode]

    def debug_buffers(self, mode: str, sample_stride: int = 0):
        """(Debug struct, dict of the tensors it points to)."""
        p = self.problem
        B, Hq, T = p.batch, p.num_q_heads, max(self.Tmax, 1)
        dev = self.device
        bufs = {
            "tile_m": torch.full((B, Hq, T), float("nan"), device=dev),
            "tile_z": torch.full((B, Hq, T), float("nan"), device=dev),
            "tile_count": torch.full((B, Hq, T), -1, dtype=torch.int32, device=dev),
            "error_flags": torch.zeros(1, dtype=torch.int32, device=dev),
        }
        if mode in ("prop", "prop_fused", "strat", "iid", "prop_bernoulli"):
            bufs["sample_idx"] = torch.full((B, Hq, p.S), -1, dtype=torch.int32, device=dev)
        if mode == "prop_bernoulli":
            bufs["features_read"] = torch.full((B, p.num_kv_heads), -1, dtype=torch.int32, device=dev)
        elif mode == "flash":
            bufs["sample_idx"] = torch.full((B, Hq, T, max(sample_stride, 1)), -1, dtype=torch.int32, device=dev)
        dbg = Debug()
        dbg.tile_m = bufs["tile_m"].data_ptr()
        dbg.tile_z = bufs["tile_z"].data_ptr()
        dbg.tile_count = bufs["tile_count"].data_ptr()
        dbg.sample_idx = bufs["sample_idx"].data_ptr() if "sample_idx" in bufs else None
        dbg.sample_stride = int(sample_stride) if mode == "flash" else 0
        dbg.error_flags = bufs["error_flags"].data_ptr()
        if "features_read" in bufs:
            dbg.features_read = bufs["features_read"].data_ptr()
        return dbg, bufs

    def __call__(self, mode, q, k, v, kv_indptr, U=None, out=None, debug=None, stream=None) -> torch.Tensor:
        p = self.problem
        if out is None:
            out = torch.empty((p.batch, p.num_q_heads, p.head_dim), dtype=torch.float32, device=self.device)
        decode(mode, p, q, k, v, kv_indptr, U, out, self.workspace(mode), debug, stream)
        return out

    def pass1(self, q, k, kv_indptr, debug=None, stream=None) -> None:
        """Pass 1 of prop alone, into the prop workspace (santa_prop_pass1)."""
        santa_prop_pass1(self.problem, q, k, kv_indptr, self.workspace("prop"), debug, stream)

    def pass2(self, v, kv_indptr, U, out=None, debug=None, stream=None) -> torch.Tensor:
        """Pass 2 of prop alone, on the prop workspace pass 1 filled (santa_prop_pass2)."""
        p = self.problem
        if out is None:
            out = torch.empty((p.batch, p.num_q_heads, p.head_dim), dtype=torch.float32, device=self.device)
        santa_prop_pass2(self.problem, v, kv_indptr, U, out, self.workspace("prop"), debug, stream)
        return out

    def prop_paged(self, q, k_pool, v_pool, page_table, kv_lens, page_size, U, out=None, debug=None,
                   stream=None) -> torch.Tensor:
        """S2ANTA-prop on a paged cache (santa_decode_prop_paged); the problem's
        total_tokens must be the pools' rows, num_pages * page_size."""
        p = self.problem
        if out is None:
            out = torch.empty((p.batch, p.num_q_heads, p.head_dim), dtype=torch.float32, device=self.device)
        pages = make_pages(page_table, kv_lens, page_size, p.total_tokens // page_size)
        santa_decode_prop_paged(p, pages, q, k_pool, v_pool, U, out, self.workspace("prop"), debug, stream)
        return out

    def feature_blocked(self, k, stream=None) -> torch.Tensor:
        """The feature-blocked copy of the token-major K cache k (santa_k_feature_blocked)."""
        p = self.problem
        esz = 2 if k.dtype in (torch.bfloat16, torch.int16, torch.uint16) else 4
        n = k_feature_blocked_size(p)
        kfb = torch.empty(n // esz, dtype=k.dtype, device=self.device)
        santa_k_feature_blocked(p, k, kfb, stream)
        return kfb

    def prop_bernoulli(self, q, k_fb, v, kv_indptr, U, bern_u, draws, group_mean, out=None, debug=None,
                       stream=None) -> torch.Tensor:
        """S2ANTA-prop with the Bernoulli score stage (santa_decode_prop_bernoulli)."""
        p = self.problem
        if out is None:
            out = torch.empty((p.batch, p.num_q_heads, p.head_dim), dtype=torch.float32, device=self.device)
        santa_decode_prop_bernoulli(p, q, k_fb, v, kv_indptr, U, bern_u, draws, group_mean, out,
                                    self.workspace("prop"), debug, stream)
        return out
