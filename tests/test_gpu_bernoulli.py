"""S2ANTA-prop with the Bernoulli ternary score stage against the oracle.

"Stochastic Sparse Attention for Memory-Bound Inference" (paper notes), Key
design 4 (Bernoulli q K^T) and the ablation table (mean group query).  Given the
same uniforms, the GPU's kept-feature counts equal the oracle's exactly (both
take the draw decisions in single precision), and the sampled indices, budgets
and outputs match the oracle's prop head run on the oracle's effective queries,
under the same rule as plain prop.  The feature-blocked K copy is checked
element by element against the token-major cache.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from santa_harness import decoder_for, head_slices, pick_heads, record
from synthetic import generate, get_workload, to_torch
from synthetic.workloads import Workload, draw_uniforms

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from stochastic_sparse_decode_gb300.build import build

    build()


def _uniforms(inp, draws: int, group_mean: bool, seed: int) -> np.ndarray:
    w = inp.workload
    heads = w.num_kv_heads if group_mean else w.num_q_heads
    return draw_uniforms((w.batch, heads, draws, w.head_dim), np.random.default_rng(seed)).astype(np.float32)


def _run(inp, draws: int, group_mean: bool, seed: int = 0):
    dec = decoder_for(inp)
    q, k, v, indptr, U = to_torch(inp)
    kfb = dec.feature_blocked(k)
    bu = _uniforms(inp, draws, group_mean, seed)
    dbg, bufs = dec.debug_buffers("prop_bernoulli")
    out = dec.prop_bernoulli(q, kfb, v, indptr, U, torch.from_numpy(bu).cuda(), draws, group_mean, debug=dbg)
    torch.cuda.synchronize()
    res = {"out": out.cpu().numpy()}
    for name, t in bufs.items():
        res[name] = t.cpu().numpy()
    assert int(res["error_flags"][0]) == 0, f"device error flags {int(res['error_flags'][0]):#x}"
    return res, bu


def _check(inp, res, bu, draws: int, group_mean: bool, heads=None, tag: str = "") -> compare.Report:
    w = inp.workload
    G = w.group
    rep = compare.Report()
    heads = heads if heads is not None else pick_heads(inp, None)
    groups = sorted({(b, h // G) for b, h in heads})
    eff = {}
    for b, kvh in groups:
        qg = inp.q[b, kvh * G:(kvh + 1) * G].astype(np.float64)
        ug = bu[b, kvh:kvh + 1] if group_mean else bu[b, kvh * G:(kvh + 1) * G]
        c, read = oracle.bernoulli_query(qg, ug.astype(np.float64), group_mean)
        assert int(res["features_read"][b, kvh]) == int(read.sum()), (b, kvh)
        eff[(b, kvh)] = c
    for b, h in heads:
        _, K, V = head_slices(inp, b, h)
        c = eff[(b, h // G)][h % G]
        rep.merge(compare.check_prop_head(c, K, V, w.S, float(inp.U[0][b, h]), w.tile, res["out"][b, h],
                                          res["sample_idx"][b, h], res["tile_count"][b, h], res["tile_m"][b, h],
                                          res["tile_z"][b, h], what=f"{w.name}/bernoulli/b{b}h{h}"))
    return record(f"{w.name}/bernoulli{'_group' if group_mean else ''}/draws{draws}{tag}", rep)


SMALL = [
    Workload(name="bern_ragged_bf16", config=61, batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128, tile=128,
             S=64, dtype="bf16", lengths=(2500, 0, 733)),
    Workload(name="bern_fp32_d64", config=62, batch=2, num_q_heads=4, num_kv_heads=1, head_dim=64, tile=64, S=16,
             dtype="f32", lengths=(1000, 37)),
    Workload(name="bern_bf16_g8", config=63, batch=2, num_q_heads=16, num_kv_heads=2, head_dim=128, tile=256,
             S=128, dtype="bf16", lengths=(4096, 1500)),
]


@pytest.mark.parametrize("draws", [1, 4])
@pytest.mark.parametrize("group_mean", [False, True])
@pytest.mark.parametrize("case", range(len(SMALL)))
def test_bernoulli_matches_oracle(case, group_mean, draws):
    inp = generate(SMALL[case])
    res, bu = _run(inp, draws, group_mean, seed=case * 10 + draws)
    _check(inp, res, bu, draws, group_mean)


@pytest.mark.parametrize("group_mean", [False, True])
def test_bernoulli_llama8b_32k_sampled_heads(group_mean):
    """The 32k Llama-3.1-8B-shaped layer, four draws (the pages' B = 4), sampled
    heads; every group's kept-feature count is compared."""
    inp = generate(get_workload("llama8b_32k_b1"))
    res, bu = _run(inp, 4, group_mean, seed=5)
    _check(inp, res, bu, 4, group_mean, heads=pick_heads(inp, 8, seed=1))
    w = inp.workload
    for b in range(w.batch):
        for kvh in range(w.num_kv_heads):
            G = w.group
            qg = inp.q[b, kvh * G:(kvh + 1) * G].astype(np.float64)
            ug = bu[b, kvh:kvh + 1] if group_mean else bu[b, kvh * G:(kvh + 1) * G]
            _, read = oracle.bernoulli_query(qg, ug.astype(np.float64), group_mean)
            assert int(res["features_read"][b, kvh]) == int(read.sum())


def test_all_probabilities_one_is_plain_prop():
    """Queries whose entries all have one magnitude: every draw keeps every
    feature, the effective query is q itself, and the call draws the samples of
    santa_decode_prop on the same inputs (its logits differ from the tensor-core
    pass 1's only in the order of the additions)."""
    w = Workload(name="bern_pm1", config=64, batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, tile=128, S=64,
                 dtype="bf16", lengths=(3000, 900))
    inp = generate(w)
    sign = np.where(inp.q >= 0, 1.0, -1.0).astype(np.float32) * 0.125
    inp.q[...] = sign
    inp.q_native[...] = (sign.view(np.uint32) >> 16).astype(np.uint16)
    res, bu = _run(inp, 2, False, seed=3)
    assert np.all(res["features_read"] == w.head_dim)
    dec = decoder_for(inp)
    q, k, v, indptr, U = to_torch(inp)
    dbg, bufs = dec.debug_buffers("prop")
    ref = dec("prop", q, k, v, indptr, U, debug=dbg).cpu().numpy()
    np.testing.assert_array_equal(bufs["sample_idx"].cpu().numpy(), res["sample_idx"])
    np.testing.assert_allclose(res["out"], ref, rtol=0, atol=1e-6)


def test_feature_blocked_copy_is_exact():
    """K_fb[r / 64][h][f][r % 64] = K[r][h][f]; rows past the end are zero."""
    inp = generate(SMALL[0])
    dec = decoder_for(inp)
    _, k, _, _, _ = to_torch(inp)
    kfb = dec.feature_blocked(k)
    rows, hkv, d = k.shape
    nb = -(-rows // 64)
    pad = torch.zeros((nb * 64 - rows, hkv, d), dtype=k.dtype, device=k.device)
    expect = torch.cat([k, pad]).view(nb, 64, hkv, d).permute(0, 2, 3, 1).contiguous().view(-1)
    assert torch.equal(kfb.view(torch.int16), expect.view(torch.int16)) if k.dtype == torch.bfloat16 else \
        torch.equal(kfb, expect)
