"""GPU parity of the prop pipeline with the stratified and i.i.d. samplers.

"Stochastic Sparse Attention for Memory-Bound Inference" (paper notes, Key
design 1) gives three samplers of the same estimator: SANTA (i.i.d. draws),
S2ANTA-strat (one draw per stratum) and S2ANTA-sys.  Through the C ABI
(santa_decode_prop_strat / santa_decode_prop_iid) with seeded caller uniforms,
against the float64 oracle's own strat / iid samplers on the same uniforms:
indices bit-exact except within 1e-5 of a CDF boundary, out within 2e-3.
"""

import numpy as np
import pytest
import torch

from synthetic import Workload, generate, get_workload, to_torch
from synthetic.workloads import draw_uniforms

from santa_harness import check, pick_heads, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session", autouse=True)
def built_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from stochastic_sparse_decode_gb300.build import build

    build()


def _uniforms(inp, S, seed):
    w = inp.workload
    return draw_uniforms((w.batch, w.num_q_heads, S), np.random.default_rng(seed))


def _run_check(inp, mode, S, seed, heads=None):
    dev = to_torch(inp)
    u = _uniforms(inp, S, seed)
    res = run(inp, mode, S=S, dev_inputs=dev[:4] + (torch.from_numpy(u).cuda(),))
    rep = check(inp, mode, res, S=S, heads=heads, U_values=u)
    plain = run(inp, mode, S=S, dev_inputs=dev[:4] + (torch.from_numpy(u).cuda(),), debug=False)
    assert np.array_equal(plain["out"], res["out"]), "debug outputs changed the result"
    print(f"[parity] {inp.workload.name}/{mode} S={S}: heads={rep.heads} samples={rep.samples} "
          f"excused={rep.excused} max_out_err={rep.max_out_err:.2e}")
    return rep


@pytest.mark.parametrize("mode", ["strat", "iid"])
def test_tiny_fp32_eight_draws(mode):
    inp = generate(get_workload("tiny_fp32"))
    for seed in range(8):
        _run_check(inp, mode, inp.workload.S, seed)


EDGE = [
    # (dtype, d, Hq, Hkv, tile, S, lengths)
    ("bf16", 128, 8, 2, 32, 7, (0, 1, 33, 300, 2500)),
    ("f32", 64, 4, 4, 64, 1, (5, 64, 65, 700)),
    ("bf16", 64, 16, 2, 1024, 300, (1, 2049, 4096)),
    ("bf16", 128, 64, 8, 256, 128, (4096, 0, 777)),
    ("bf16", 64, 16, 2, 128, 64, (3000, 31)),
]


@pytest.mark.parametrize("case", range(len(EDGE)))
@pytest.mark.parametrize("mode", ["strat", "iid"])
def test_edge_shapes(case, mode):
    dtype, d, Hq, Hkv, tile, S, lengths = EDGE[case]
    w = Workload(name=f"sampler_edge{case}", config=90 + case, batch=len(lengths), num_q_heads=Hq, num_kv_heads=Hkv,
                 head_dim=d, tile=tile, S=S, dtype=dtype, lengths=lengths, planted_per_head=2, sinks=2)
    _run_check(generate(w), mode, S, 100 + case)


@pytest.mark.parametrize("mode", ["strat", "iid"])
def test_llama8b_32k_batch1_sampled_heads(mode):
    inp = generate(get_workload("llama8b_32k_b1"))
    _run_check(inp, mode, 128, 7, heads=pick_heads(inp, 8, seed=3))


def test_largest_supported_sample_count():
    """S = 16384 uniforms per head (the on-chip limit), more samples than keys."""
    w = Workload(name="sampler_bigS", config=95, batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64, tile=128,
                 S=16384, dtype="f32", length=3000, planted_per_head=4)
    inp = generate(w)
    for mode in ("strat", "iid"):
        _run_check(inp, mode, 16384, 5)


def test_uniforms_outside_the_unit_interval_are_flagged():
    import stochastic_sparse_decode_gb300 as sd
    from stochastic_sparse_decode_gb300.decoder import Decoder

    inp = generate(get_workload("tiny_fp32"))
    w = inp.workload
    q, k, v, ind, _ = to_torch(inp)
    u = torch.from_numpy(_uniforms(inp, w.S, 1)).cuda()
    u[0, 1, 3] = 1.5
    u[0, 2, 0] = -0.25
    dec = Decoder(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, inp.total_tokens, w.length, w.tile, w.S, w.dtype)
    for mode in ("strat", "iid"):
        dbg, bufs = dec.debug_buffers(mode)
        out = dec(mode, q, k, v, ind, u, debug=dbg)
        flags = sd.santa_read_device_error(bufs["error_flags"])
        assert flags & sd.ERR_OFFSET
        assert torch.isfinite(out).all()
