"""S2ANTA-prop on a paged K/V cache (page-table indirection), through the C ABI.

"Stochastic Sparse Attention for Memory-Bound Inference" (paper notes,
Overall framework) claims compatibility with paged serving caches; the method
itself is unchanged.  A chunk of 32 keys never straddles a page (page sizes are
multiples of 32), so santa_decode_prop_paged must give, bit for bit, what
santa_decode_prop gives on the same keys laid out contiguously: outputs, the
sampled indices and the tile records.  The pools are filled around the live
pages with values that would wreck any result read from the wrong row, the
page-table entries past a sequence's pages with invalid ids that would be
flagged if read, and one paged result is also checked against the float64
oracle directly.  A bad page id must be flagged, not fault.
"""

import numpy as np
import pytest
import torch

from synthetic import Workload, generate, get_workload, to_torch

from santa_harness import check, decoder_for
from stochastic_sparse_decode_gb300.decoder import Decoder
from synthetic.workloads import max_length

pytestmark = pytest.mark.gpu

ERR_INDPTR = 1  # SANTA_ERR_INDPTR


@pytest.fixture(scope="session", autouse=True)
def built_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from stochastic_sparse_decode_gb300.build import build

    build()


def _paginate(inp, k, v, page_size, seed, spare=3):
    """Pools [num_pages * page_size][Hkv][d] holding every sequence's keys in a
    shuffled set of pages, the page table [B][max_pages] and kv_lens [B]."""
    w = inp.workload
    rng = np.random.default_rng(seed)
    L = inp.lengths.astype(np.int64)
    npg = -(-L // page_size)
    max_pages = max(1, int(-(-max_length(w) // page_size)))
    num_pages = int(npg.sum()) + spare
    ids = rng.permutation(num_pages)
    rows = num_pages * page_size
    poison = torch.full((rows, w.num_kv_heads, w.head_dim), 40.0, device="cuda").to(k.dtype)
    kp, vp = poison.clone(), poison.clone()
    table = np.full((w.batch, max_pages), -7, dtype=np.int32)
    nxt = 0
    for b in range(w.batch):
        t0 = int(inp.kv_indptr[b])
        for j in range(int(npg[b])):
            pid = int(ids[nxt])
            nxt += 1
            table[b, j] = pid
            n = min(page_size, int(L[b]) - j * page_size)
            kp[pid * page_size: pid * page_size + n] = k[t0 + j * page_size: t0 + j * page_size + n]
            vp[pid * page_size: pid * page_size + n] = v[t0 + j * page_size: t0 + j * page_size + n]
    return (kp, vp, torch.from_numpy(table).cuda(), torch.from_numpy(L.astype(np.int32)).cuda(), num_pages)


def _run_both(inp, page_size, seed=0, break_page=False):
    w = inp.workload
    q, k, v, indptr, U = to_torch(inp)
    dec = decoder_for(inp)
    dbg1, b1 = dec.debug_buffers("prop")
    whole = dec("prop", q, k, v, indptr, U, debug=dbg1).clone()
    kp, vp, table, lens, num_pages = _paginate(inp, k, v, page_size, seed)
    if break_page:
        b = int(np.argmax(inp.lengths))
        table[b, 0] = num_pages + 5
    decp = Decoder(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, num_pages * page_size, max_length(w),
                   w.tile, w.S, w.dtype)
    dbg2, b2 = decp.debug_buffers("prop")
    paged = decp.prop_paged(q, kp, vp, table, lens, page_size, U, debug=dbg2).clone()
    torch.cuda.synchronize()
    return whole, paged, b1, b2


RAGGED = Workload(name="paged_ragged", config=43, batch=6, num_q_heads=8, num_kv_heads=2, head_dim=128, tile=64,
                  S=50, dtype="bf16", lengths=(0, 1, 33, 300, 2500, 4096))


@pytest.mark.parametrize("page_size", [32, 96, 256])
def test_paged_equals_contiguous_on_a_ragged_batch(page_size):
    inp = generate(RAGGED)
    whole, paged, b1, b2 = _run_both(inp, page_size, seed=page_size)
    assert int(b1["error_flags"][0]) == 0 and int(b2["error_flags"][0]) == 0
    assert torch.equal(whole, paged)
    for key in ("sample_idx", "tile_count"):
        assert torch.equal(b1[key], b2[key]), key
    for key in ("tile_m", "tile_z"):
        assert torch.equal(torch.nan_to_num(b1[key], nan=-7.0), torch.nan_to_num(b2[key], nan=-7.0)), key
    if page_size == 96:  # and against the float64 oracle directly
        res = {"out": paged.cpu().numpy()}
        for key, t in b2.items():
            res[key] = t.cpu().numpy()
        rep = check(inp, "prop", res)
        print(f"[parity] paged ragged ps={page_size}: heads={rep.heads} samples={rep.samples} "
              f"excused={rep.excused} max_out_err={rep.max_out_err:.2e}")


def test_paged_equals_contiguous_on_the_32k_layer():
    inp = generate(get_workload("llama8b_32k_b1"))
    whole, paged, b1, b2 = _run_both(inp, 64, seed=5)
    assert int(b2["error_flags"][0]) == 0
    assert torch.equal(whole, paged)
    assert torch.equal(b1["sample_idx"], b2["sample_idx"])


def test_a_bad_page_id_is_flagged_not_a_fault():
    inp = generate(RAGGED)
    _, paged, _, b2 = _run_both(inp, 32, seed=1, break_page=True)
    assert int(b2["error_flags"][0]) & ERR_INDPTR
    assert torch.isfinite(paged).all()
