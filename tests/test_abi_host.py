"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host before enqueuing anything.

No call here reaches a kernel launch: every argument set fails host validation
(the device pointers are never dereferenced on the host).
"""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "santa_decode.h")


@pytest.fixture(scope="module")
def sd():
    from stochastic_sparse_decode_gb300.build import build

    build()
    import stochastic_sparse_decode_gb300 as sd

    return sd


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("santa_decode_prop", "santa_decode_flash", "exact_decode", "santa_workspace_size",
              "santa_read_device_error", "santa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(sd):
    names = _declared_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", sd.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    lib = sd.lib()
    for n in names:
        assert getattr(lib, n) is not None
        # every argument typed: an untyped pointer argument would be passed as a 32-bit int
        assert getattr(lib, n).argtypes is not None, n
    assert set(sd.EXPORTS) == set(names)


def test_split_passes_validate_only_what_they_read(sd):
    p = _llama8b_problem(sd)
    need = sd.workspace_size(p, sd.MODE_PROP)
    L = sd.lib()
    dev = 0x10000000  # never dereferenced: every call below is rejected before any launch
    Q = K = V = U = OUT = IND = dev

    def p1(q=Q, k=K, ind=IND, ws=dev, nbytes=need):
        return L.santa_prop_pass1(ctypes.byref(p), q, k, ind, ws, nbytes, None, None)

    def p2(v=V, ind=IND, u=U, out=OUT, ws=dev, nbytes=need):
        return L.santa_prop_pass2(ctypes.byref(p), v, ind, u, out, ws, nbytes, None, None)

    assert p1(q=None) == sd.INVALID_ARG
    assert p1(k=None) == sd.INVALID_ARG
    assert p1(ind=None) == sd.INVALID_ARG
    assert p1(k=dev + 8) == sd.INVALID_ARG
    assert p1(nbytes=need - 1) == sd.WORKSPACE_TOO_SMALL
    assert p2(v=None) == sd.INVALID_ARG
    assert p2(u=None) == sd.INVALID_ARG
    assert p2(out=None) == sd.INVALID_ARG
    assert p2(ws=dev + 128) == sd.INVALID_ARG
    assert p2(nbytes=need - 1) == sd.WORKSPACE_TOO_SMALL
    # batch 0 is a no-op for either pass
    p0 = _llama8b_problem(sd, batch=0)
    assert L.santa_prop_pass1(ctypes.byref(p0), None, None, None, None, 0, None, None) == sd.OK
    assert L.santa_prop_pass2(ctypes.byref(p0), None, None, None, None, None, 0, None, None) == sd.OK


def _llama8b_problem(sd, **kw):
    args = dict(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128, total_tokens=32768, max_len=32768,
                tile=256, S=128, dtype="bf16")
    args.update(kw)
    return sd.make_problem(**args)


def test_workspace_layout_matches_the_byte_model(sd):
    """prop: a 256-byte header, a published-chunk counter per (sequence, query head),
    the chunk records [B][Hq][ceil(max_len/32)] as 64-bit words, a finished-split
    counter per head, the fp32 score stash [B][Hq][32 ceil(max_len/32)], a
    largest-key byte per chunk (rows rounded up to 4), the splits' d-float sums,
    min(8, 256 // (B Hq)) splits per head, and the Bernoulli score stage's effective
    queries [B][Hq][d] float, kept features [B][Hkv][d] bytes and their counts
    [B][Hkv]; flash: prop's regions up to the chunk offsets (its pass 1 is prop's
    streaming pass), then 2 tile-record arrays [B][Hq][T] and the tile estimates
    [B][Hq][T][d]; exact: the streaming
    warps' partial states; each rounded up to 256 B."""
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    p = _llama8b_problem(sd)
    T, nch = 32768 // 256, 32768 // 32
    tq = lambda B: r(B * 32 * 128 * 4) + r(B * 8 * 128) + r(B * 8 * 4)  # noqa: E731
    prop = (256 + r(1 * 32 * 4) + r(1 * 32 * nch * 8) + r(1 * 32 * 4) + r(32 * nch * 32 * 4) + r(32 * nch)
            + r(32 * 8 * 128 * 4) + tq(1))
    assert sd.workspace_size(p, sd.MODE_PROP) == prop
    stream = lambda B, nch: (256 + r(B * 32 * 4) + r(B * 32 * nch * 8) + r(B * 32 * 4)  # noqa: E731
                             + r(B * 32 * nch * 32 * 4) + r(B * 32 * ((nch + 3) // 4 * 4)))
    flash = stream(1, nch) + 2 * r(1 * 32 * T * 4) + r(1 * 32 * T * 128 * 4)
    assert sd.workspace_size(p, sd.MODE_FLASH) == flash
    # exact: (M, Z) and O per (sequence, streaming warp, head of the group); the
    # streaming grid is at most 160 CTAs of 12 warps for bf16 at d = 128
    n = 1 * 160 * 12 * 4
    assert sd.workspace_size(p, sd.MODE_EXACT) == r(n * 8) + r(n * 128 * 4)
    # ragged tail: T = ceil(max_len / tile), chunks = ceil(max_len / 32)
    p = _llama8b_problem(sd, batch=3, max_len=1000, total_tokens=2000, tile=128)
    T, nch = 8, 32
    assert sd.workspace_size(p, sd.MODE_FLASH) == stream(3, nch) + 2 * r(3 * 32 * T * 4) + r(3 * 32 * T * 128 * 4)
    assert sd.workspace_size(p, sd.MODE_PROP) == (256 + r(3 * 32 * 4) + r(3 * 32 * nch * 8) + r(3 * 32 * 4)
                                                  + r(3 * 32 * nch * 32 * 4) + r(3 * 32 * nch) + r(96 * 2 * 128 * 4)
                                                  + tq(3))
    # a batch of 16 (512 heads): one split per head
    p = _llama8b_problem(sd, batch=16, max_len=1000, total_tokens=16000, tile=128)
    assert sd.workspace_size(p, sd.MODE_PROP) == (256 + r(16 * 32 * 4) + r(16 * 32 * nch * 8) + r(16 * 32 * 4)
                                                  + r(16 * 32 * nch * 32 * 4) + r(16 * 32 * nch)
                                                  + r(16 * 32 * 1 * 128 * 4) + tq(16))


def test_very_long_prop_contexts_are_unsupported_not_wrong(sd):
    """The sampler sums a head's chunk masses as 64-bit fixed-point integers, exact
    for up to 2^17 chunks (2^22 keys): a longer max_len is refused on the host,
    before anything is enqueued (flash and exact still take it)."""
    p = _llama8b_problem(sd, max_len=32 * 1024 * 1024, total_tokens=32 * 1024 * 1024, tile=1024)
    n = ctypes.c_size_t(0)
    assert sd.lib().santa_workspace_size(ctypes.byref(p), sd.MODE_PROP, ctypes.byref(n)) == sd.UNSUPPORTED
    assert sd.lib().santa_workspace_size(ctypes.byref(p), sd.MODE_FLASH, ctypes.byref(n)) == sd.OK
    assert _call_prop(sd, p, ws_bytes=1 << 40) == sd.UNSUPPORTED
    p = _llama8b_problem(sd, max_len=1 << 22, total_tokens=1 << 22, tile=1024)
    assert sd.lib().santa_workspace_size(ctypes.byref(p), sd.MODE_PROP, ctypes.byref(n)) == sd.OK


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 96, "UNSUPPORTED"),
    ("dtype", 7, "UNSUPPORTED"),
    ("num_q_heads", 24, "UNSUPPORTED"),   # group of 3
    ("num_q_heads", 30, "INVALID_ARG"),   # not a multiple of Hkv
    ("tile", 48, "INVALID_ARG"),
    ("tile", 2048, "INVALID_ARG"),
    ("tile", 16, "INVALID_ARG"),
    ("S", 0, "INVALID_ARG"),
    ("S", (1 << 20) + 1, "INVALID_ARG"),
    ("batch", -1, "INVALID_ARG"),
    ("max_len", -5, "INVALID_ARG"),
    ("total_tokens", 1 << 40, "INVALID_ARG"),
])
def test_bad_problems_are_rejected(sd, field, value, status):
    p = _llama8b_problem(sd)
    setattr(p, field, value)
    n = ctypes.c_size_t(0)
    st = sd.lib().santa_workspace_size(ctypes.byref(p), sd.MODE_PROP, ctypes.byref(n))
    assert st == getattr(sd, status)


def test_exact_ignores_S(sd):
    p = _llama8b_problem(sd, S=0)
    assert sd.workspace_size(p, sd.MODE_EXACT) > 0
    with pytest.raises(sd.SantaError):
        sd.workspace_size(p, sd.MODE_PROP)


class _FakeTensor:
    """A device address that is never dereferenced (validation fails first)."""

    def __init__(self, addr, nbytes=0):
        self.addr, self.nbytes = addr, nbytes

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.nbytes

    def element_size(self):
        return 1


def _call_prop(sd, p, q=0x10000, k=0x20000, v=0x30000, ind=0x40000, U=0x50000, out=0x60000, ws=0x100000,
               ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = sd.workspace_size(p, sd.MODE_PROP)
    t = lambda a: None if a is None else _FakeTensor(a)  # noqa: E731
    try:
        sd.santa_decode_prop(p, t(q), t(k), t(v), t(ind), t(U), t(out), _FakeTensor(ws, ws_bytes), stream=0)
    except sd.SantaError as e:
        return e.status
    return sd.OK


def test_null_misaligned_and_small_workspace_are_rejected(sd):
    p = _llama8b_problem(sd)
    assert _call_prop(sd, p, q=None) == sd.INVALID_ARG
    assert _call_prop(sd, p, U=None) == sd.INVALID_ARG
    assert _call_prop(sd, p, out=None) == sd.INVALID_ARG
    assert _call_prop(sd, p, k=0x20008) == sd.INVALID_ARG      # K not 16-byte aligned
    assert _call_prop(sd, p, ind=0x40004) == sd.INVALID_ARG    # kv_indptr not 8-byte aligned
    assert _call_prop(sd, p, ws=0x100080) == sd.INVALID_ARG    # workspace not 256-byte aligned
    need = sd.workspace_size(p, sd.MODE_PROP)
    assert _call_prop(sd, p, ws_bytes=need - 1) == sd.WORKSPACE_TOO_SMALL
    # batch 0 is a no-op that touches nothing
    assert _call_prop(sd, _llama8b_problem(sd, batch=0), q=None, k=None) == sd.OK


@pytest.mark.parametrize("name", ["santa_decode_prop_strat", "santa_decode_prop_iid"])
def test_sampler_modes_refuse_more_uniforms_than_shared_memory_holds(sd, name):
    """The stratified and i.i.d. samplers keep a head's S uniforms on chip: S <= 16384."""
    t = _FakeTensor
    for S, status in ((16385, sd.UNSUPPORTED), (1 << 20, sd.UNSUPPORTED)):
        p = _llama8b_problem(sd, S=S)
        ws = sd.workspace_size(p, sd.MODE_PROP)
        with pytest.raises(sd.SantaError) as e:
            getattr(sd, name)(p, t(0x10000), t(0x20000), t(0x30000), t(0x40000), t(0x50000), t(0x60000),
                              t(0x100000, ws), stream=0)
        assert e.value.status == status
    p = _llama8b_problem(sd, S=64)
    with pytest.raises(sd.SantaError) as e:  # null uniforms
        getattr(sd, name)(p, t(0x10000), t(0x20000), t(0x30000), t(0x40000), None, t(0x60000),
                          t(0x100000, sd.workspace_size(p, sd.MODE_PROP)), stream=0)
    assert e.value.status == sd.INVALID_ARG


def test_exact_needs_no_offsets(sd):
    p = _llama8b_problem(sd)
    ws = sd.workspace_size(p, sd.MODE_EXACT)
    with pytest.raises(sd.SantaError) as e:
        sd.exact_decode(p, _FakeTensor(0x10000), _FakeTensor(0x20000), _FakeTensor(0x30000), None,
                        _FakeTensor(0x60000), _FakeTensor(0x100000, ws), stream=0)
    assert e.value.status == sd.INVALID_ARG  # kv_indptr is required


def test_status_strings(sd):
    for s in range(6):
        assert sd.status_string(s) and sd.status_string(s) != "unknown status"
    assert sd.status_string(99) == "unknown status"


def test_missing_library_fails_loudly(monkeypatch, sd):
    monkeypatch.setattr(sd, "_lib", None)
    monkeypatch.setattr(sd, "LIB_PATH", "/nonexistent/libsanta_decode.so")
    with pytest.raises(RuntimeError, match="missing"):
        sd.lib()


def test_paged_problems_are_validated_before_any_launch(sd):
    L = sd.lib()
    dev = 0x10000000  # never dereferenced: every call below is rejected before any launch
    p = _llama8b_problem(sd, total_tokens=512 * 64)
    need = sd.workspace_size(p, sd.MODE_PROP)

    def call(page_size=64, max_pages=512, num_pages=512, table=dev, lens=dev, prob=p, nbytes=need):
        pg = sd.Pages(table, lens, page_size, max_pages, num_pages)
        return L.santa_decode_prop_paged(ctypes.byref(prob), ctypes.byref(pg), dev, dev, dev, dev, dev, dev, nbytes,
                                         None, None)

    assert call(page_size=48) == sd.INVALID_ARG                    # not a multiple of 32
    assert call(page_size=0) == sd.INVALID_ARG
    assert call(num_pages=511) == sd.INVALID_ARG                   # pools disagree with total_tokens
    assert call(max_pages=511) == sd.INVALID_ARG                   # max_len beyond a page-table row
    assert call(table=None) == sd.INVALID_ARG
    assert call(lens=dev + 2) == sd.INVALID_ARG                    # kv_lens not 4-byte aligned
    assert call(nbytes=need - 1) == sd.WORKSPACE_TOO_SMALL
    assert L.santa_decode_prop_paged(ctypes.byref(p), None, dev, dev, dev, dev, dev, dev, need, None,
                                     None) == sd.INVALID_ARG


def test_fused_prop_validates_like_prop(sd):
    """santa_decode_prop_fused takes santa_decode_prop's arguments and checks them the same way."""
    p = _llama8b_problem(sd)
    t = _FakeTensor
    ws = sd.workspace_size(p, sd.MODE_PROP)
    for args, status in (((t(0x10000), t(0x20000), t(0x30000), t(0x40000), None, t(0x60000)), sd.INVALID_ARG),
                         ((t(0x10000), t(0x20008), t(0x30000), t(0x40000), t(0x50000), t(0x60000)), sd.INVALID_ARG)):
        with pytest.raises(sd.SantaError) as e:
            sd.santa_decode_prop_fused(p, *args, t(0x100000, ws), stream=0)
        assert e.value.status == status
    with pytest.raises(sd.SantaError) as e:
        sd.santa_decode_prop_fused(p, t(0x10000), t(0x20000), t(0x30000), t(0x40000), t(0x50000), t(0x60000),
                                   t(0x100000, ws - 1), stream=0)
    assert e.value.status == sd.WORKSPACE_TOO_SMALL


def _call_bern(sd, p, u=0x70000, draws=4, group_mean=0, kfb=0x20000):
    t = lambda a: None if a is None else _FakeTensor(a)  # noqa: E731
    ws = sd.workspace_size(p, sd.MODE_PROP)
    try:
        sd.santa_decode_prop_bernoulli(p, t(0x10000), t(kfb), t(0x30000), t(0x40000), t(0x50000), t(u), draws,
                                       group_mean, t(0x60000), _FakeTensor(0x100000, ws), stream=0)
    except sd.SantaError as e:
        return e.status
    return sd.OK


def test_bernoulli_arguments_are_checked(sd):
    """1 <= draws <= 64, uniforms present and 4-byte aligned, K 16-byte aligned."""
    p = _llama8b_problem(sd)
    assert _call_bern(sd, p, draws=0) == sd.INVALID_ARG
    assert _call_bern(sd, p, draws=65) == sd.INVALID_ARG
    assert _call_bern(sd, p, u=None) == sd.INVALID_ARG
    assert _call_bern(sd, p, u=0x70002) == sd.INVALID_ARG
    assert _call_bern(sd, p, kfb=0x20008, group_mean=1) == sd.INVALID_ARG
    # batch 0 is a no-op after the argument checks
    assert _call_bern(sd, _llama8b_problem(sd, batch=0)) == sd.OK


def test_feature_blocked_size_and_checks(sd):
    """K_fb holds ceil(total_tokens / 64) blocks of Hkv x d x 64 elements; a buffer
    too small or misaligned is refused before anything is enqueued."""
    p = _llama8b_problem(sd, total_tokens=1000, max_len=1000)
    n = sd.k_feature_blocked_size(p)
    assert n == 16 * 8 * 128 * 64 * 2  # ceil(1000 / 64) = 16 blocks, bf16
    t = _FakeTensor
    with pytest.raises(sd.SantaError) as e:
        sd.santa_k_feature_blocked(p, t(0x10000), t(0x200000, n - 1), stream=0)
    assert e.value.status == sd.WORKSPACE_TOO_SMALL
    with pytest.raises(sd.SantaError) as e:
        sd.santa_k_feature_blocked(p, t(0x10008), t(0x200000, n), stream=0)
    assert e.value.status == sd.INVALID_ARG
