"""The prop entry point that allocates nothing (santa_decode_prop_static_scratch).

It is for callers that cannot allocate device memory -- for instance a plugin in
a host program that owns all device memory through its own pool and gives
plugins no allocator.  Its scratch is the library's built-in 16 MiB device
array, so it must give what santa_decode_prop gives with a caller workspace,
call after call, even though every call reuses (and leaves behind) the same
scratch.  This file is collected last, so a run that stops at the first failure
has already run every other test.
"""

import pytest
import torch

from synthetic import Workload, generate, get_workload, max_length, to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from stochastic_sparse_decode_gb300.build import build

    build()
    import stochastic_sparse_decode_gb300 as sd

    return sd


def _problem(sd, inp):
    w = inp.workload
    return sd.make_problem(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, inp.total_tokens, max_length(w),
                           w.tile, w.S, w.dtype)


def test_static_scratch_matches_the_workspace_entry_point(sd):
    """Two calls in a row on the built-in scratch -- the 32k Llama-3.1-8B layer, then
    a smaller ragged batch that runs on the first call's leftovers -- each against
    santa_decode_prop with a fresh caller workspace."""
    cases = [
        generate(get_workload("llama8b_32k_b1")),
        generate(Workload(name="noalloc_ragged", config=70, batch=3, num_q_heads=16, num_kv_heads=4, head_dim=128,
                          tile=128, S=64, dtype="bf16", lengths=(5000, 0, 1234), planted_per_head=4, sinks=4)),
    ]
    dev = [to_torch(inp) for inp in cases]
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    dbg = sd.Debug()
    dbg.error_flags = flags.data_ptr()
    outs = []
    for inp, (q, k, v, ind, U) in zip(cases, dev):  # the two static-scratch calls, back to back
        w = inp.workload
        out = torch.full((w.batch, w.num_q_heads, w.head_dim), float("nan"), device="cuda")
        sd.santa_decode_prop_static_scratch(_problem(sd, inp), q, k, v, ind, U, out, debug=dbg)
        outs.append(out)
    assert sd.santa_read_device_error(flags) == 0
    for inp, (q, k, v, ind, U), got in zip(cases, dev, outs):
        p = _problem(sd, inp)
        ws = torch.empty(sd.workspace_size(p, sd.MODE_PROP), dtype=torch.uint8, device="cuda")
        sd.santa_workspace_init(p, sd.MODE_PROP, ws)  # a fresh prop workspace starts zero-filled
        ref = torch.full_like(got, float("nan"))
        sd.santa_decode_prop(p, q, k, v, ind, U, ref, ws)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        # the same kernels on the same inputs: bit for bit, whatever the scratch held
        assert torch.equal(got, ref)


def test_static_scratch_rejects_problems_beyond_its_size(sd):
    """Batch 16 at 32k needs a 64 MiB score stash: refused before anything runs."""
    w = get_workload("llama8b_32k_b16")
    p = sd.make_problem(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.batch * w.length, w.length, w.tile,
                        w.S, w.dtype)
    assert sd.workspace_size(p, sd.MODE_PROP) > sd.STATIC_SCRATCH_BYTES
    t = torch.empty(16, device="cuda")
    with pytest.raises(sd.SantaError) as e:
        sd.santa_decode_prop_static_scratch(p, t, t, t, t, t, t)
    assert e.value.status == sd.WORKSPACE_TOO_SMALL
