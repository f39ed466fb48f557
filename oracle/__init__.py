"""CPU oracle for stochastic sparse decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never does, and this package imports nothing from it.

The arithmetic lives in ``santa_oracle.c`` (plain C, float64, single threaded),
compiled with gcc into ``libsanta_oracle.so`` next to it; this module only
marshals numpy arrays into it and loops over (sequence, query head).

Parity status of each function (pins live in ``tests/test_oracle_pins.py``):

* logits / softmax / exact A V ....... pinned (closed forms, torch SDPA in float64)
* systematic sampler (prop) .......... pinned (hand-derived example, one-hot,
  uniform with S = n_k, count bounds, exact integration over U, Monte Carlo)
* tile budgets S_tile ................ pinned (sum = S, |S_tile - S Z_tile/Z| < 1)
* flash (per-tile sampling + merge) .. pinned (exact integration over U,
  one-hot, uniform, S_loc = S/T closed form)
* i.i.d. / stratified samplers ....... pinned (exact integration over u)
* Bernoulli q K^T, per head and mean
  group query ........................ pinned (exact enumeration of the draws:
  E[c] = q, read probability 1 - prod (1-p)^draws; ternary entries; all p = 1
  reduces to the exact query)
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "santa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libsanta_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no -ffast-math: IEEE double semantics)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        L, I, D = ctypes.c_long, ctypes.c_int, ctypes.c_double
        lib.oracle_logits.argtypes = [L, I, _dp, _dp, L, _dp]
        lib.oracle_softmax.argtypes = [L, _dp, _dp]
        lib.oracle_cdf.argtypes = [L, _dp, _dp]
        lib.oracle_inverse_cdf.argtypes = [L, _dp, D]
        lib.oracle_inverse_cdf.restype = L
        lib.oracle_gather_mean.argtypes = [I, _lp, I, _dp, L, _dp]
        lib.oracle_exact_head.argtypes = [L, I, _dp, _dp, L, _dp, L, _dp]
        lib.oracle_prop_head.argtypes = [L, I, I, I, D, _dp, _dp, L, _dp, L, _dp, _lp, _ip, _dp, _dp]
        lib.oracle_sampled_head.argtypes = [I, L, I, I, _dp, _dp, _dp, L, _dp, L, _dp, _lp]
        lib.oracle_flash_head.argtypes = [L, I, I, I, D, _dp, _dp, L, _dp, L, _dp, _lp, _dp, _dp, _dp]
        lib.oracle_bernoulli_query.argtypes = [I, I, I, I, _dp, _dp, _dp, _ip]
        for f in ("oracle_exact_head", "oracle_prop_head", "oracle_sampled_head", "oracle_flash_head",
                  "oracle_bernoulli_query"):
            getattr(lib, f).restype = I
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray, typ=_dp):
    return a.ctypes.data_as(typ) if a is not None else None


# --------------------------------------------------------------------- one head


def logits(q, K) -> np.ndarray:
    """x_i = q . k_i / sqrt(d) for one query head; K is [n][d]."""
    q, K = _f64(q), _f64(K)
    n, d = K.shape
    x = np.empty(n)
    _load().oracle_logits(n, d, _ptr(q), _ptr(K), d, _ptr(x))
    return x


def softmax(x) -> np.ndarray:
    x = _f64(x)
    A = np.empty_like(x)
    _load().oracle_softmax(x.size, _ptr(x), _ptr(A))
    return A


def cdf(A) -> np.ndarray:
    A = _f64(A)
    F = np.empty_like(A)
    _load().oracle_cdf(A.size, _ptr(A), _ptr(F))
    return F


def inverse_cdf(F, t: float) -> int:
    F = _f64(F)
    return int(_load().oracle_inverse_cdf(F.size, _ptr(F), float(t)))


def gather_mean(J, V) -> np.ndarray:
    """(1/S) sum_s V[J_s] for the given indices."""
    J = np.ascontiguousarray(J, dtype=np.int64)
    V = _f64(V)
    out = np.empty(V.shape[1])
    _load().oracle_gather_mean(J.size, _ptr(J, _lp), V.shape[1], _ptr(V), V.shape[1], _ptr(out))
    return out


def exact_head(q, K, V) -> np.ndarray:
    q, K, V = _f64(q), _f64(K), _f64(V)
    n, d = K.shape
    out = np.empty(d)
    if _load().oracle_exact_head(n, d, _ptr(q), _ptr(K), d, _ptr(V), d, _ptr(out)) != 0:
        raise MemoryError("oracle_exact_head")
    return out


@dataclass
class PropHead:
    out: np.ndarray  # [d]
    J: np.ndarray  # [S] int64, index within the sequence
    counts: np.ndarray  # [T] int32, S_tile
    mass: np.ndarray  # [T] Z_tile / Z
    F: np.ndarray | None  # [n] global CDF


def prop_head(q, K, V, S: int, U: float, tile: int, want_F: bool = True) -> PropHead:
    q, K, V = _f64(q), _f64(K), _f64(V)
    n, d = K.shape
    T = -(-n // tile) if n > 0 else 0
    out = np.empty(d)
    J = np.zeros(S, dtype=np.int64)
    counts = np.zeros(max(T, 1), dtype=np.int32)
    mass = np.zeros(max(T, 1))
    F = np.empty(max(n, 1)) if want_F else None
    rc = _load().oracle_prop_head(
        n, d, tile, S, float(U), _ptr(q), _ptr(K), d, _ptr(V), d, _ptr(out),
        _ptr(J, _lp), _ptr(counts, _ip), _ptr(mass), _ptr(F) if want_F else None,
    )
    if rc != 0:
        raise MemoryError("oracle_prop_head")
    return PropHead(out, J if n > 0 else J[:0], counts[:T], mass[:T], F[:n] if want_F else None)


def bernoulli_query(q, u, group_mean: bool) -> tuple[np.ndarray, np.ndarray]:
    """Bernoulli q K^T for one KV group (oracle_bernoulli_query): q [G][d], u
    [G or 1][draws][d] uniforms in [0, 1).  Returns the effective queries c [G][d]
    (c_g . k estimates q_g . k) and the read mask [d] of the features selected."""
    q, u = _f64(q), _f64(u)
    G, d = q.shape
    draws = u.shape[1]
    assert u.shape == ((1 if group_mean else G), draws, d)
    c = np.empty((G, d))
    read = np.zeros(d, dtype=np.int32)
    rc = _load().oracle_bernoulli_query(G, d, draws, int(bool(group_mean)), _ptr(q), _ptr(u), _ptr(c),
                                         _ptr(read, _ip))
    if rc < 0:
        raise MemoryError("oracle_bernoulli_query")
    return c, read.astype(bool)


def sampled_head(mode: str, q, K, V, u) -> tuple[np.ndarray, np.ndarray]:
    """mode 'iid' (SANTA) or 'strat' (S2ANTA-strat) with caller uniforms u[S] in [0,1)."""
    q, K, V, u = _f64(q), _f64(K), _f64(V), _f64(u)
    n, d = K.shape
    out = np.empty(d)
    J = np.zeros(u.size, dtype=np.int64)
    m = {"iid": 0, "strat": 1}[mode]
    if _load().oracle_sampled_head(m, n, d, u.size, _ptr(u), _ptr(q), _ptr(K), d, _ptr(V), d,
                                   _ptr(out), _ptr(J, _lp)) != 0:
        raise MemoryError("oracle_sampled_head")
    return out, J


@dataclass
class FlashHead:
    out: np.ndarray  # [d]
    S_loc: int
    J: np.ndarray  # [T][S_loc] int64
    tile_m: np.ndarray  # [T]
    tile_z: np.ndarray  # [T]
    weight: np.ndarray  # [T] w_t / Z


def flash_head(q, K, V, S: int, U: float, tile: int) -> FlashHead:
    q, K, V = _f64(q), _f64(K), _f64(V)
    n, d = K.shape
    T = -(-n // tile) if n > 0 else 0
    S_loc = -(-S // T) if T > 0 else 0
    out = np.empty(d)
    J = np.zeros(max(T * S_loc, 1), dtype=np.int64)
    tm, tz, w = (np.zeros(max(T, 1)) for _ in range(3))
    rc = _load().oracle_flash_head(n, d, tile, S, float(U), _ptr(q), _ptr(K), d, _ptr(V), d,
                                   _ptr(out), _ptr(J, _lp), _ptr(tm), _ptr(tz), _ptr(w))
    if rc < 0:
        raise MemoryError("oracle_flash_head")
    assert rc == S_loc
    return FlashHead(out, S_loc, J[: T * S_loc].reshape(T, S_loc), tm[:T], tz[:T], w[:T])


# ------------------------------------------------------------- whole problems


def _heads(B: int, Hq: int, heads):
    return [(b, h) for b in range(B) for h in range(Hq)] if heads is None else list(heads)


def _group_slices(k, v, kv_indptr, b: int, g: int):
    t0, t1 = int(kv_indptr[b]), int(kv_indptr[b + 1])
    return _f64(k[t0:t1, g, :]), _f64(v[t0:t1, g, :])


def run_problem(mode: str, q, k, v, kv_indptr, *, S: int = 0, U=None, tile: int = 256,
                heads=None, want_F: bool = False) -> dict:
    """Run one mode over (sequence, query head) pairs.

    q [B][Hq][d], k/v [tokens][Hkv][d] (any float dtype), kv_indptr [B+1],
    U [B][Hq].  Query head h reads KV head h // (Hq / Hkv).  Returns a dict
    keyed by (b, h) of PropHead / FlashHead / exact output vectors.
    """
    B, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    res = {}
    cache = {}
    for b, h in _heads(B, Hq, heads):
        key = (b, h // G)
        if key not in cache:
            cache.clear()
            cache[key] = _group_slices(k, v, kv_indptr, b, h // G)
        Kb, Vb = cache[key]
        if mode == "exact":
            res[(b, h)] = exact_head(q[b, h], Kb, Vb)
        elif mode == "prop":
            res[(b, h)] = prop_head(q[b, h], Kb, Vb, S, float(U[b, h]), tile, want_F=want_F)
        elif mode == "flash":
            res[(b, h)] = flash_head(q[b, h], Kb, Vb, S, float(U[b, h]), tile)
        else:
            raise ValueError(mode)
    return res
