"""Runs the CUDA library on synthetic inputs and checks it against the oracle.

Shared by the GPU parity tests.  Device work goes through the C ABI only
(stochastic_sparse_decode_gb300); expected values come only from ``oracle``.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import compare
from stochastic_sparse_decode_gb300.decoder import Decoder
from synthetic import Inputs, max_length, to_torch


# Every parity check of the session, by test: (name, Report).  conftest.py prints
# the totals -- samples compared, excused boundary mismatches, worst output error --
# at the end of the run, so they reach the run's log even under `pytest -q`.
REPORTS: list = []


def record(name: str, rep: compare.Report) -> compare.Report:
    """Registers a finished check and enforces the excused-mismatch bound."""
    REPORTS.append((name, rep))
    assert compare.excused_within_bound(rep), (
        f"{name}: {rep.excused} of {rep.samples} samples excused (bound {compare.EXCUSED_FRACTION:.0%})")
    return rep


def decoder_for(inp: Inputs, S: int | None = None) -> Decoder:
    w = inp.workload
    return Decoder(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, inp.total_tokens,
                   max(max_length(w), 0), w.tile, S if S is not None else w.S, w.dtype)


def run(inp: Inputs, mode: str, S: int | None = None, U_index: int = 0, debug: bool = True,
        sample_stride: int | None = None, dev_inputs=None, U=None):
    """One call of `mode`; returns numpy out plus the debug buffers."""
    dec = decoder_for(inp, S)
    q, k, v, indptr, U0 = dev_inputs if dev_inputs is not None else to_torch(inp, "cuda", U_index)
    if U is None:
        U = U0
    if sample_stride is None:
        p = dec.problem
        sample_stride = max(1, -(-p.S // max(1, min(int(x) for x in _tiles(inp)))))
    dbg, bufs = dec.debug_buffers(mode, sample_stride) if debug else (None, {})
    out = dec(mode, q, k, v, indptr, U, debug=dbg)
    torch.cuda.synchronize()
    res = {"out": out.cpu().numpy()}
    for name, t in bufs.items():
        res[name] = t.cpu().numpy()
    if "error_flags" in res:  # a bounded wait that gave up, or a flagged input, fails the call
        assert int(res["error_flags"][0]) == 0, f"device error flags {int(res['error_flags'][0]):#x}"
    res["sample_stride"] = sample_stride
    return res


def _tiles(inp: Inputs):
    w = inp.workload
    T = [-(-int(L) // w.tile) for L in inp.lengths if L > 0]
    return T or [1]


def head_slices(inp: Inputs, b: int, h: int):
    w = inp.workload
    g = h // w.group
    t0, t1 = int(inp.kv_indptr[b]), int(inp.kv_indptr[b + 1])
    K = inp.k_f32(b)[:, g, :].astype(np.float64) if t1 > t0 else np.zeros((0, w.head_dim))
    V = inp.v_f32(b)[:, g, :].astype(np.float64) if t1 > t0 else np.zeros((0, w.head_dim))
    return inp.q[b, h].astype(np.float64), K, V


def pick_heads(inp: Inputs, count: int | None, seed: int = 0):
    w = inp.workload
    allh = [(b, h) for b in range(w.batch) for h in range(w.num_q_heads)]
    if count is None or count >= len(allh):
        return allh
    rng = np.random.default_rng(seed)
    sel = {allh[0], allh[-1]}
    for i in rng.choice(len(allh), size=count, replace=False):
        sel.add(allh[int(i)])
    return sorted(sel)


def check(inp: Inputs, mode: str, res: dict, S: int | None = None, U_index: int = 0, heads=None,
          U_values=None) -> compare.Report:
    w = inp.workload
    S = S if S is not None else w.S
    U = inp.U[U_index] if U_values is None else U_values
    rep = compare.Report()
    for b, h in (heads if heads is not None else pick_heads(inp, None)):
        q, K, V = head_slices(inp, b, h)
        what = f"{w.name}/{mode}/b{b}h{h}"
        if mode in ("prop", "prop_fused"):
            rep.merge(compare.check_prop_head(q, K, V, S, float(U[b, h]), w.tile, res["out"][b, h],
                                              res["sample_idx"][b, h], res["tile_count"][b, h],
                                              res["tile_m"][b, h], res["tile_z"][b, h], what=what))
        elif mode in ("strat", "iid"):
            rep.merge(compare.check_sampled_head(mode, q, K, V, U[b, h], res["out"][b, h], res["sample_idx"][b, h],
                                                 what=what))
        elif mode == "flash":
            rep.merge(compare.check_flash_head(q, K, V, S, float(U[b, h]), w.tile, res["out"][b, h],
                                               res["sample_idx"][b, h], res["tile_m"][b, h],
                                               res["tile_z"][b, h], what=what))
        else:
            rep.merge(compare.check_exact_head(q, K, V, res["out"][b, h], what=what))
    return record(f"{w.name}/{mode}/S{S}", rep)
