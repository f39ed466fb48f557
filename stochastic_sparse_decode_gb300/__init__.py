"""Python binding of libsanta_decode.so -- GB300 stochastic sparse decode attention.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/santa_decode.h``.  Tensors are
torch CUDA tensors (PyTorch provides device memory and streams); the functions
take the same names and arguments as the C entry points.

If the library has not been built (``python -m stochastic_sparse_decode_gb300.build``)
every call raises -- there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libsanta_decode.so")

# status codes, dtypes, modes and device error bits of santa_decode.h
OK, INVALID_ARG, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA_ERROR, DEVICE_CHECK = range(6)
F32, BF16 = 0, 1
MODE_PROP, MODE_FLASH, MODE_EXACT = 0, 1, 2
ERR_INDPTR, ERR_OFFSET, ERR_TIMEOUT, ERR_WORKSPACE = 1, 2, 4, 8

EXPORTS = (
    "santa_workspace_size",
    "santa_workspace_init",
    "santa_decode_prop",
    "santa_decode_prop_fused",
    "santa_decode_prop_bernoulli",
    "santa_k_feature_blocked_size",
    "santa_k_feature_blocked",
    "santa_prop_pass1",
    "santa_prop_pass2",
    "santa_decode_prop_paged",
    "santa_decode_prop_strat",
    "santa_decode_prop_iid",
    "santa_decode_flash",
    "exact_decode",
    "santa_read_device_error",
    "santa_decode_prop_static_scratch",
    "santa_status_string",
)


class SantaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class Problem(ctypes.Structure):
    """santa_problem"""

    _fields_ = [
        ("batch", ctypes.c_int),
        ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("total_tokens", ctypes.c_longlong),
        ("max_len", ctypes.c_int),
        ("tile", ctypes.c_int),
        ("S", ctypes.c_int),
        ("dtype", ctypes.c_int),
    ]


class Debug(ctypes.Structure):
    """santa_debug"""

    _fields_ = [
        ("tile_m", ctypes.c_void_p),
        ("tile_z", ctypes.c_void_p),
        ("tile_count", ctypes.c_void_p),
        ("sample_idx", ctypes.c_void_p),
        ("sample_stride", ctypes.c_int),
        ("error_flags", ctypes.c_void_p),
        ("main_begin", ctypes.c_void_p),
        ("main_end", ctypes.c_void_p),
        ("wait_cycles", ctypes.c_longlong),
        ("features_read", ctypes.c_void_p),
    ]


class Pages(ctypes.Structure):
    """santa_pages"""

    _fields_ = [
        ("page_table", ctypes.c_void_p),
        ("kv_lens", ctypes.c_void_p),
        ("page_size", ctypes.c_int),
        ("max_pages", ctypes.c_int),
        ("num_pages", ctypes.c_longlong),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m stochastic_sparse_decode_gb300.build`"
            )
        L = ctypes.CDLL(LIB_PATH)
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        P, Dp = ctypes.POINTER(Problem), ctypes.POINTER(Debug)
        L.santa_workspace_size.argtypes = [P, ctypes.c_int, ctypes.POINTER(sz)]
        L.santa_workspace_init.argtypes = [P, ctypes.c_int, vp, sz, vp]
        for name in ("santa_decode_prop", "santa_decode_prop_fused", "santa_decode_prop_strat", "santa_decode_prop_iid",
                     "santa_decode_flash"):
            getattr(L, name).argtypes = [P, vp, vp, vp, vp, vp, vp, vp, sz, Dp, vp]
        L.santa_prop_pass1.argtypes = [P, vp, vp, vp, vp, sz, Dp, vp]
        L.santa_decode_prop_bernoulli.argtypes = [P, vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp, sz,
                                                  Dp, vp]
        L.santa_k_feature_blocked_size.argtypes = [P, ctypes.POINTER(sz)]
        L.santa_k_feature_blocked.argtypes = [P, vp, vp, sz, vp]
        L.santa_prop_pass2.argtypes = [P, vp, vp, vp, vp, vp, sz, Dp, vp]
        L.santa_decode_prop_paged.argtypes = [P, ctypes.POINTER(Pages), vp, vp, vp, vp, vp, vp, sz, Dp, vp]
        L.exact_decode.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, Dp, vp]
        L.santa_decode_prop_static_scratch.argtypes = [P, vp, vp, vp, vp, vp, vp, Dp, vp]
        L.santa_read_device_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint)]
        L.santa_status_string.argtypes = [ctypes.c_int]
        L.santa_status_string.restype = ctypes.c_char_p
        for name in EXPORTS[:-1]:
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().santa_status_string(int(status)).decode()


def make_problem(batch, num_q_heads, num_kv_heads, head_dim, total_tokens, max_len, tile, S, dtype) -> Problem:
    if isinstance(dtype, str):
        dtype = {"f32": F32, "bf16": BF16}[dtype]
    return Problem(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim), int(total_tokens),
                   int(max_len), int(tile), int(S), int(dtype))


def workspace_size(problem: Problem, mode: int) -> int:
    n = ctypes.c_size_t(0)
    st = lib().santa_workspace_size(ctypes.byref(problem), int(mode), ctypes.byref(n))
    if st != OK:
        raise SantaError(st, "santa_workspace_size")
    return n.value


def santa_workspace_init(problem: Problem, mode: int, workspace, stream=None) -> None:
    """Enqueues the zero fill a workspace needs before its first call (and after a
    SANTA_ERR_TIMEOUT): see santa_decode.h."""
    st = lib().santa_workspace_init(ctypes.byref(problem), int(mode), _ptr(workspace), _nbytes(workspace),
                                    _stream(stream))
    if st != OK:
        raise SantaError(st, "santa_workspace_init")


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _call(name, problem, args, workspace, debug, stream):
    dbg = ctypes.byref(debug) if debug is not None else None
    st = getattr(lib(), name)(ctypes.byref(problem), *args, _ptr(workspace), _nbytes(workspace), dbg, _stream(stream))
    if st != OK:
        raise SantaError(st, name)


def santa_decode_prop(problem, q, k, v, kv_indptr, U, out, workspace, debug=None, stream=None):
    """S2ANTA-prop decode: see santa_decode.h.  All tensors on the current CUDA device."""
    _call("santa_decode_prop", problem, [_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr), _ptr(U), _ptr(out)],
          workspace, debug, stream)


def santa_decode_prop_fused(problem, q, k, v, kv_indptr, U, out, workspace, debug=None, stream=None):
    """S2ANTA-prop decode in one persistent kernel: see santa_decode.h."""
    _call("santa_decode_prop_fused", problem, [_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr), _ptr(U), _ptr(out)],
          workspace, debug, stream)


def santa_decode_prop_bernoulli(problem, q, k_fb, v, kv_indptr, U, bern_u, draws, group_mean, out, workspace,
                                debug=None, stream=None):
    """S2ANTA-prop with the Bernoulli ternary score stage on a feature-blocked K: see santa_decode.h."""
    dbg = ctypes.byref(debug) if debug is not None else None
    st = lib().santa_decode_prop_bernoulli(ctypes.byref(problem), _ptr(q), _ptr(k_fb), _ptr(v), _ptr(kv_indptr),
                                           _ptr(U), _ptr(bern_u), int(draws), int(bool(group_mean)), _ptr(out),
                                           _ptr(workspace), _nbytes(workspace), dbg, _stream(stream))
    if st != OK:
        raise SantaError(st, "santa_decode_prop_bernoulli")


def k_feature_blocked_size(problem) -> int:
    n = ctypes.c_size_t(0)
    st = lib().santa_k_feature_blocked_size(ctypes.byref(problem), ctypes.byref(n))
    if st != OK:
        raise SantaError(st, "santa_k_feature_blocked_size")
    return n.value


def santa_k_feature_blocked(problem, k, k_fb, stream=None):
    """The feature-blocked copy of the token-major K cache (santa_k_feature_blocked)."""
    st = lib().santa_k_feature_blocked(ctypes.byref(problem), _ptr(k), _ptr(k_fb), _nbytes(k_fb), _stream(stream))
    if st != OK:
        raise SantaError(st, "santa_k_feature_blocked")


def santa_prop_pass1(problem, q, k, kv_indptr, workspace, debug=None, stream=None):
    """Pass 1 of S2ANTA-prop alone: chunk records and score stash into the workspace."""
    _call("santa_prop_pass1", problem, [_ptr(q), _ptr(k), _ptr(kv_indptr)], workspace, debug, stream)


def santa_prop_pass2(problem, v, kv_indptr, U, out, workspace, debug=None, stream=None):
    """Pass 2 of S2ANTA-prop alone, on a workspace that santa_prop_pass1 filled."""
    _call("santa_prop_pass2", problem, [_ptr(v), _ptr(kv_indptr), _ptr(U), _ptr(out)], workspace, debug, stream)


def make_pages(page_table, kv_lens, page_size, num_pages) -> Pages:
    """santa_pages for device tensors page_table [B][max_pages] and kv_lens [B] (int32)."""
    return Pages(int(page_table.data_ptr()), int(kv_lens.data_ptr()), int(page_size), int(page_table.shape[-1]),
                 int(num_pages))


def santa_decode_prop_paged(problem, pages, q, k_pool, v_pool, U, out, workspace, debug=None, stream=None):
    """S2ANTA-prop decode on a paged cache: see santa_decode.h."""
    dbg = ctypes.byref(debug) if debug is not None else None
    st = lib().santa_decode_prop_paged(ctypes.byref(problem), ctypes.byref(pages), _ptr(q), _ptr(k_pool),
                                       _ptr(v_pool), _ptr(U), _ptr(out), _ptr(workspace), _nbytes(workspace), dbg,
                                       _stream(stream))
    if st != OK:
        raise SantaError(st, "santa_decode_prop_paged")


def santa_decode_prop_strat(problem, q, k, v, kv_indptr, u, out, workspace, debug=None, stream=None):
    """S2ANTA-strat through the prop pipeline: u is [B][Hq][S] float32 in [0, 1)."""
    _call("santa_decode_prop_strat", problem, [_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr), _ptr(u), _ptr(out)],
          workspace, debug, stream)


def santa_decode_prop_iid(problem, q, k, v, kv_indptr, u, out, workspace, debug=None, stream=None):
    """SANTA (i.i.d. draws) through the prop pipeline: u is [B][Hq][S] float32 in [0, 1)."""
    _call("santa_decode_prop_iid", problem, [_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr), _ptr(u), _ptr(out)],
          workspace, debug, stream)


def santa_decode_flash(problem, q, k, v, kv_indptr, U, out, workspace, debug=None, stream=None):
    """S2ANTA-flash decode: see santa_decode.h."""
    _call("santa_decode_flash", problem, [_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr), _ptr(U), _ptr(out)],
          workspace, debug, stream)


def exact_decode(problem, q, k, v, kv_indptr, out, workspace, debug=None, stream=None):
    """Exact split-KV decode: see santa_decode.h."""
    _call("exact_decode", problem, [_ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr), _ptr(out)],
          workspace, debug, stream)


STATIC_SCRATCH_BYTES = 16 << 20  # SANTA_STATIC_SCRATCH_BYTES


def santa_decode_prop_static_scratch(problem, q, k, v, kv_indptr, U, out, debug=None, stream=None):
    """S2ANTA-prop decode with the library's built-in 16 MiB scratch array instead of a
    caller workspace, for callers that cannot allocate device memory (see santa_decode.h)."""
    dbg = ctypes.byref(debug) if debug is not None else None
    st = lib().santa_decode_prop_static_scratch(ctypes.byref(problem), _ptr(q), _ptr(k), _ptr(v), _ptr(kv_indptr),
                                                _ptr(U), _ptr(out), dbg, _stream(stream))
    if st != OK:
        raise SantaError(st, "santa_decode_prop_static_scratch")


def santa_read_device_error(error_flags, stream=None) -> int:
    """Waits for the stream, returns and clears the device error word."""
    h = ctypes.c_uint(0)
    st = lib().santa_read_device_error(_ptr(error_flags), _stream(stream), ctypes.byref(h))
    if st not in (OK, DEVICE_CHECK):
        raise SantaError(st, "santa_read_device_error")
    return h.value


MODES = {"prop": MODE_PROP, "prop_fused": MODE_PROP, "strat": MODE_PROP, "iid": MODE_PROP, "flash": MODE_FLASH,
         "exact": MODE_EXACT}


def decode(mode: str, problem, q, k, v, kv_indptr, U, out, workspace, debug=None, stream=None):
    """Dispatch by mode name ('prop', 'prop_fused', 'strat', 'iid', 'flash', 'exact'); U is the
    offsets [B][Hq] for prop and flash, the uniforms [B][Hq][S] for strat and iid, ignored by exact."""
    if mode == "prop":
        santa_decode_prop(problem, q, k, v, kv_indptr, U, out, workspace, debug, stream)
    elif mode == "prop_fused":
        santa_decode_prop_fused(problem, q, k, v, kv_indptr, U, out, workspace, debug, stream)
    elif mode == "strat":
        santa_decode_prop_strat(problem, q, k, v, kv_indptr, U, out, workspace, debug, stream)
    elif mode == "iid":
        santa_decode_prop_iid(problem, q, k, v, kv_indptr, U, out, workspace, debug, stream)
    elif mode == "flash":
        santa_decode_flash(problem, q, k, v, kv_indptr, U, out, workspace, debug, stream)
    elif mode == "exact":
        exact_decode(problem, q, k, v, kv_indptr, out, workspace, debug, stream)
    else:
        raise ValueError(mode)
