"""The two passes of S2ANTA-prop called one by one through the C ABI.

"Stochastic Sparse Attention for Memory-Bound Inference" (paper notes, Key
design 2) splits prop into pass 1 (read all of K; stash the exponentiated
scores and the partition records) and pass 2 (reduce, sample, gather V).
santa_prop_pass1 followed by santa_prop_pass2 must give bit for bit what
santa_decode_prop gives, on a ragged batch (empty, one-key and tail-chunk
sequences) and on the 32k Llama-3.1-8B layer; and pass 2 alone must read
only what pass 1 left, so re-running pass 2 gives the same result again.
"""

import numpy as np
import pytest
import torch

from synthetic import Workload, generate, get_workload, to_torch

from santa_harness import decoder_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session", autouse=True)
def built_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from stochastic_sparse_decode_gb300.build import build

    build()


def _both_ways(inp):
    import stochastic_sparse_decode_gb300 as sd

    dec = decoder_for(inp)
    q, k, v, indptr, U = to_torch(inp)
    dbg1, b1 = dec.debug_buffers("prop")
    whole = dec("prop", q, k, v, indptr, U, debug=dbg1).clone()
    torch.cuda.synchronize()
    dbg2, b2 = dec.debug_buffers("prop")
    ws = dec.workspace("prop")
    ws.fill_(0xA5)  # nothing of the whole call may carry over
    dec.pass1(q, k, indptr, debug=dbg2)
    split = dec.pass2(v, indptr, U, debug=dbg2).clone()
    # pass 2 sets the records back to zero; with the header cleared as well (the
    # fill above wrote it), the workspace serves the fused kernel
    sd.santa_workspace_init(dec.problem, sd.MODE_PROP, ws)
    dbg3, b3 = dec.debug_buffers("prop")
    fused_a = torch.empty_like(whole)
    sd.santa_decode_prop_fused(dec.problem, q, k, v, indptr, U, fused_a, ws, dbg3)
    # the fused kernel leaves the workspace as it found it: the two kernels, the split
    # pair and the fused kernel again follow without any initialisation
    dbg4, b4 = dec.debug_buffers("prop")
    again = dec("prop", q, k, v, indptr, U, debug=dbg4).clone()
    dec.pass1(q, k, indptr)
    split2 = dec.pass2(v, indptr, U).clone()
    fused_b = torch.empty_like(whole)
    dbg5, b5 = dec.debug_buffers("prop")
    sd.santa_decode_prop_fused(dec.problem, q, k, v, indptr, U, fused_b, ws, dbg5)
    torch.cuda.synchronize()
    for b in (b1, b2, b3, b4, b5):
        assert int(b["error_flags"][0]) == 0
    assert torch.equal(fused_a, fused_b)
    # the fused kernel adds the same V rows in another order: equal to rounding
    # wherever its samples are the two kernels' samples
    same = (b3["sample_idx"] == b1["sample_idx"]).all(dim=-1)
    assert same.float().mean() > 0.9
    assert torch.allclose(fused_a[same], whole[same], rtol=0, atol=1e-5)
    return whole, split, again, split2, b1, b2


@pytest.mark.parametrize("name", ["ragged_edges", "llama8b_32k_b1"])
def test_pass1_then_pass2_matches_whole_call(name):
    if name == "ragged_edges":
        w = Workload(name="passes_ragged", config=41, batch=5, num_q_heads=8, num_kv_heads=2, head_dim=128,
                     tile=64, S=50, dtype="bf16", lengths=(0, 1, 33, 300, 2500))
    else:
        w = get_workload(name)
    inp = generate(w)
    whole, split, again, split2, b1, b2 = _both_ways(inp)
    assert torch.equal(whole, split)
    assert torch.equal(whole, again)
    assert torch.equal(whole, split2)
    for key in ("sample_idx", "tile_count"):
        assert torch.equal(b1[key], b2[key]), key
    for key in ("tile_m", "tile_z"):
        assert torch.equal(torch.nan_to_num(b1[key], nan=-7.0), torch.nan_to_num(b2[key], nan=-7.0)), key


def test_pass2_on_a_workspace_pass1_did_not_fill_is_clamped_not_faulted():
    """santa_prop_pass2 on chunk records and a stash holding NaN, +-inf, negative and
    huge values: every index it derives stays in range (counts clamped to be
    non-negative, sample numbers to [0, S)), the output is finite, and a clamp
    that fired raises SANTA_ERR_WORKSPACE."""
    import stochastic_sparse_decode_gb300 as sd

    w = Workload(name="passes_garbage", config=42, batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128,
                 tile=64, S=50, dtype="bf16", lengths=(2500, 0, 700))
    inp = generate(w)
    dec = decoder_for(inp)
    q, k, v, indptr, U = to_torch(inp)
    ws = dec.workspace("prop").view(torch.float32)
    # the stash (and anything else): NaN, +-inf, huge, negative and tiny values
    g = torch.Generator(device="cpu").manual_seed(7)
    vals = torch.tensor([float("nan"), float("inf"), -float("inf"), -1.0e30, 3.0e38, -7.0, 0.0, 1.0, 1e-30])
    ws[:] = vals[torch.randint(0, vals.numel(), (ws.numel(),), generator=g)].cuda()
    # the chunk records, 64-bit words (m, z) after the 256-byte header and the
    # [B][Hq] counters: m = 0 everywhere and z alternating +20 / -19, so the masses'
    # running sum goes up and down and the threshold counts cannot all be
    # non-negative -- a clamp must fire
    nrec = w.batch * w.num_q_heads * (-(-max(w.lengths) // 32))
    rec0 = (256 + -(-w.batch * w.num_q_heads * 4 // 256) * 256) // 8
    z = torch.where(torch.arange(nrec, device="cuda") % 2 == 0, 20.0, -19.0).view(torch.int32).to(torch.int64)
    ws.view(torch.int64)[rec0 : rec0 + nrec] = (z & 0xFFFFFFFF) << 32
    dbg, bufs = dec.debug_buffers("prop")
    out = dec.pass2(v, indptr, U, debug=dbg)
    flags = sd.santa_read_device_error(bufs["error_flags"])
    assert torch.isfinite(out).all()
    assert flags & sd.ERR_WORKSPACE, f"flags {flags:#x}"
    idx = bufs["sample_idx"].cpu().numpy()
    for b, L in enumerate(inp.lengths):
        sel = idx[b][idx[b] >= 0]
        assert sel.size == 0 or (sel.min() >= 0 and sel.max() < max(int(L), 1))


def test_a_sampler_wait_that_runs_out_flags_and_returns():
    """The fused prop kernel's samplers wait, bounded, for their head's chunk records.
    With santa_debug.wait_cycles = -2000 on the 32k layer each sampler waits ~1 us
    for a publication that never comes (one chunk more than its head has) and gives
    up: the call returns with SANTA_ERR_TIMEOUT raised and zeros in out, the context
    stays usable, the workspace is marked poisoned (the next call writes zeros and
    raises SANTA_ERR_WORKSPACE), and santa_workspace_init makes it whole again."""
    import stochastic_sparse_decode_gb300 as sd

    inp = generate(get_workload("llama8b_32k_b1"))
    dec = decoder_for(inp)
    q, k, v, indptr, U = to_torch(inp)
    ref = decoder_for(inp)("prop_fused", q, k, v, indptr, U).clone()  # a separate workspace

    dbg, bufs = dec.debug_buffers("prop_fused")
    dbg.wait_cycles = -2000
    out = dec("prop_fused", q, k, v, indptr, U, debug=dbg)
    flags = sd.santa_read_device_error(bufs["error_flags"])
    assert flags & sd.ERR_TIMEOUT, f"flags {flags:#x}"
    assert (flags >> 8) & 0xF == 3  # the location code of a sampler's wait
    assert torch.isfinite(out).all()

    dbg, bufs = dec.debug_buffers("prop_fused")
    out = dec("prop_fused", q, k, v, indptr, U, debug=dbg)
    assert sd.santa_read_device_error(bufs["error_flags"]) == sd.ERR_WORKSPACE
    assert torch.count_nonzero(out) == 0

    sd.santa_workspace_init(dec.problem, sd.MODE_PROP, dec.workspace("prop_fused"))
    dbg, bufs = dec.debug_buffers("prop_fused")
    out = dec("prop_fused", q, k, v, indptr, U, debug=dbg)
    assert sd.santa_read_device_error(bufs["error_flags"]) == 0
    assert torch.equal(out, ref)
