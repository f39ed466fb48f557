"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Same seeded inputs and the same offsets U on both sides.  Indices and tile
budgets must match exactly except where a threshold sits within 1e-5 of a CDF
boundary (counted); tile masses within 1e-3 relative; out within 2e-3.
"""

import numpy as np
import pytest
import torch

from synthetic import Workload, float32_to_bf16_bits, generate, get_workload, to_torch
from synthetic.workloads import draw_offsets

from santa_harness import check, pick_heads, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session", autouse=True)
def built_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from stochastic_sparse_decode_gb300.build import build

    build()


def _report(name, rep):
    print(f"[parity] {name}: heads={rep.heads} samples={rep.samples} excused={rep.excused} "
          f"max_out_err={rep.max_out_err:.2e} max_mass_rel={rep.max_mass_rel:.2e}")


# ------------------------------------------------------------ tiny fp32 case


@pytest.mark.parametrize("mode", ["prop", "prop_fused", "flash", "exact"])
def test_tiny_fp32_all_offsets(mode):
    """batch 1, 4 q heads on 1 KV head, d=64, n_k=1024, tile 128, S=16: all 64 offsets."""
    inp = generate(get_workload("tiny_fp32"))
    dev = to_torch(inp)
    total = None
    n_u = 1 if mode == "exact" else inp.U.shape[0]
    for ui in range(n_u):
        U = torch.from_numpy(inp.U[ui]).cuda()
        res = run(inp, mode, dev_inputs=dev[:4] + (U,))
        rep = check(inp, mode, res, U_index=ui)
        total = rep if total is None else total.merge(rep)
    _report(f"tiny_fp32/{mode}", total)


# ------------------------------------------------------------ edge cases


EDGE = [
    # (dtype, d, Hq, Hkv, tile, S, lengths)
    ("bf16", 128, 8, 2, 32, 7, (0, 1, 33, 300, 2500)),
    ("bf16", 128, 32, 8, 256, 128, (257, 1000, 0, 4096)),
    ("f32", 64, 4, 4, 64, 1, (5, 64, 65, 700)),
    ("f32", 128, 16, 2, 128, 33, (1, 129, 1111)),
    ("bf16", 64, 8, 8, 1024, 2048, (3000, 1024, 1)),
    ("bf16", 128, 2, 1, 512, 5000, (600, 40)),
    ("f32", 64, 8, 4, 32, 16, (31, 32, 33)),
    # bf16 with G = 8: all eight tensor-core B columns and all four t lanes carry live heads
    ("bf16", 128, 64, 8, 256, 128, (4096, 1000, 0, 777)),
    ("bf16", 64, 16, 2, 128, 64, (3000, 31, 2049)),
]


@pytest.mark.parametrize("case", range(len(EDGE)))
@pytest.mark.parametrize("mode", ["prop", "prop_fused", "flash", "exact"])
def test_edge_shapes(case, mode):
    """Empty, one-key, sub-tile and ragged-tail sequences; every GQA group size;
    tiles 32..1024; S from 1 to more than n_k; fp32 and bf16; d = 64 and 128."""
    dtype, d, Hq, Hkv, tile, S, lengths = EDGE[case]
    w = Workload(name=f"edge{case}", config=90 + case, batch=len(lengths), num_q_heads=Hq, num_kv_heads=Hkv,
                 head_dim=d, tile=tile, S=S, dtype=dtype, lengths=lengths, planted_per_head=3, sinks=2,
                 n_offsets=3)
    inp = generate(w)
    dev = to_torch(inp)
    for ui in range(1 if mode == "exact" else 3):
        U = torch.from_numpy(inp.U[ui]).cuda()
        res = run(inp, mode, dev_inputs=dev[:4] + (U,))
        _report(f"edge{case}/{mode}/U{ui}", check(inp, mode, res, U_index=ui))
        # the call without debug outputs (the configuration the benchmark times)
        plain = run(inp, mode, dev_inputs=dev[:4] + (U,), debug=False)
        assert np.array_equal(plain["out"], res["out"]), "debug outputs changed the result"


def test_one_hot_returns_the_row_exactly():
    """A key with a logit far above the rest takes every sample: out == V_j bit for bit."""
    w = Workload(name="onehot", config=80, batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, tile=256, S=64,
                 dtype="bf16", lengths=(5000, 777))
    inp = generate(w)
    j = [4321, 700]
    for b in range(2):
        t0 = int(inp.kv_indptr[b])
        for g in range(2):
            qs = inp.q[b, 4 * g : 4 * g + 4]  # the group's 4 heads
            u, *_ = np.linalg.lstsq(qs.astype(np.float64), np.full(4, 400.0 * np.sqrt(128)), rcond=None)
            inp.k[t0 + j[b], g] = float32_to_bf16_bits(u.astype(np.float32))
    for mode in ("prop", "flash"):
        res = run(inp, mode)
        for b in range(2):
            V = inp.v_f32(b)
            for h in range(8):
                row = V[j[b], h // 4]
                assert np.array_equal(res["out"][b, h], row), (mode, b, h)
        check(inp, mode, res)


# ------------------------------------------------------------ the Llama-3.1-8B layer


@pytest.fixture(scope="module")
def llama8b_layer():
    inp = generate(get_workload("llama8b_32k_b1"))
    return inp, to_torch(inp)


@pytest.mark.parametrize("mode,S", [("prop", 128), ("prop", 256), ("prop_fused", 128), ("flash", 2048),
                                    ("flash", 128), ("exact", 0)])
def test_llama8b_32k_batch1(llama8b_layer, mode, S):
    """batch 1, 32 q / 8 KV heads, d=128, n_k=32768, tile 256: every head against the oracle."""
    inp, dev = llama8b_layer
    if S and S != inp.workload.S:
        U = draw_offsets(S, (1, 1, 32), np.random.default_rng(S))[0]
        res = run(inp, mode, S=S, dev_inputs=dev[:4] + (torch.from_numpy(U).cuda(),))
        rep = check(inp, mode, res, S=S, U_values=U)
    else:
        U = inp.U[0]
        res = run(inp, mode, dev_inputs=dev)
        rep = check(inp, mode, res)
    _report(f"llama8b_32k_b1/{mode}/S{S}", rep)
    # the call the benchmark times passes no debug struct: it must give the very
    # same bits as the checked call
    plain = run(inp, mode, S=S or None, dev_inputs=dev[:4] + (torch.from_numpy(np.ascontiguousarray(U)).cuda(),),
                debug=False)
    assert np.array_equal(plain["out"], res["out"]), "debug outputs changed the result"


@pytest.mark.parametrize("mode", ["prop", "prop_fused"])
def test_prop_is_deterministic(llama8b_layer, mode):
    """Two calls give bit-identical outputs (fixed-order combine, no float atomics)."""
    inp, dev = llama8b_layer
    a = run(inp, mode, dev_inputs=dev, debug=False)["out"]
    b = run(inp, mode, dev_inputs=dev, debug=False)["out"]
    assert np.array_equal(a, b)


# ------------------------------------------------------------ full-size configurations, sampled heads


@pytest.fixture(scope="module")
def batch16():
    inp = generate(get_workload("llama8b_32k_b16"))
    return inp, to_torch(inp)


@pytest.mark.parametrize("mode,S", [("prop", 64), ("prop", 128), ("prop", 256), ("prop_fused", 128), ("flash", 2048),
                                    ("exact", 0)])
def test_llama8b_32k_batch16_sampled(batch16, mode, S):
    inp, dev = batch16
    U = draw_offsets(max(S, 1), (16, 32), np.random.default_rng(1000 + S))
    res = run(inp, mode, S=S if S else None, dev_inputs=dev[:4] + (torch.from_numpy(U).cuda(),))
    heads = pick_heads(inp, 24, seed=S)
    _report(f"llama8b_32k_b16/{mode}/S{S}", check(inp, mode, res, S=S if S else None, U_values=U, heads=heads))


@pytest.mark.parametrize("mode,S", [("prop", 128), ("prop_fused", 128), ("flash", 2048), ("exact", 0)])
def test_ragged_batch64_sampled(mode, S):
    """64 sequences, n_k ~ UniformInt[4096, 32768], temperatures 0.5/1/2 per head."""
    w = get_workload("ragged_b64")
    inp = generate(w.with_(S=S) if S else w)
    res = run(inp, mode)
    _report(f"ragged_b64/{mode}/S{S}", check(inp, mode, res, heads=pick_heads(inp, 32, seed=5)))


@pytest.mark.parametrize("n", [4096, 131072])
@pytest.mark.parametrize("mode", ["prop", "exact"])
def test_context_sweep_sampled(n, mode):
    """batch 8, 32q/8kv, d=128, S=128, tile 256 at the shortest and longest context."""
    inp = generate(get_workload(f"sweep_b8_n{n}"))
    res = run(inp, mode)
    _report(f"sweep_b8_n{n}/{mode}", check(inp, mode, res, heads=pick_heads(inp, 12, seed=n)))


# ------------------------------------------------------------ device-side input checks


def test_bad_indptr_and_offsets_are_flagged_not_faulted():
    """An inconsistent kv_indptr entry gives zeros for that sequence and sets
    SANTA_ERR_INDPTR; an offset outside [0, 1/S) is clamped and sets SANTA_ERR_OFFSET."""
    import stochastic_sparse_decode_gb300 as sd

    w = Workload(name="badin", config=81, batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128, tile=128, S=16,
                 dtype="bf16", lengths=(300, 300, 300), planted_per_head=2)
    inp = generate(w)
    q, k, v, indptr, U = to_torch(inp)
    bad = indptr.clone()
    bad[2] = 100  # sequence 1 would run backwards; sequence 2 gets 800 > max_len keys
    from santa_harness import decoder_for

    dec = decoder_for(inp)
    dbg, bufs = dec.debug_buffers("prop")
    out = dec("prop", q, k, v, bad, U, debug=dbg)
    flags = sd.santa_read_device_error(bufs["error_flags"])
    assert flags & sd.ERR_INDPTR
    o = out.cpu().numpy()
    assert np.all(o[1] == 0) and np.all(o[2] == 0)
    # offsets out of range
    U2 = U.clone()
    U2[0, 0] = 1.0
    U2[0, 1] = float("nan")
    U2[0, 2] = -0.5
    dbg, bufs = dec.debug_buffers("prop")
    dec("prop", q, k, v, indptr, U2, debug=dbg)
    flags = sd.santa_read_device_error(bufs["error_flags"])
    assert flags == sd.ERR_OFFSET
    assert sd.santa_read_device_error(bufs["error_flags"]) == 0  # cleared by the read
