"""Seeded synthetic workloads shaped like one Llama-3.1-8B decode attention layer.

The pages measure on RULER-32k, GSM8K and MMLU with Llama-3.1-8B weights
(Stochastic Sparse Attention for Memory-Bound Inference, Main experiments,
Tables 1-3).  Neither the datasets nor the weights are available, so these
generators stand in for them with the layer's shapes (32 query heads sharing 8
KV heads, head dim 128, 32k context) and a score distribution with heavy hitters:

* q, K, V ~ N(0, 1) in float32 (PCG64, seed = 1000 * config + instance);
* "planted" keys: k += 3 * sqrt(d) * q_h / |q_h| for the query head h that the
  key is assigned to (round-robin over the heads of its GQA group), which lifts
  that head's logit by about 3 * |q_h| (~34 at d = 128);
* attention sinks: the first ``sinks`` tokens of a sequence get the minimum-norm
  vector delta with Q delta = 2 * sqrt(d) * 1 over the group's queries Q, so
  every head of the group sees its logit raised by exactly +2 (before rounding);
* optional per-head temperature tau_h, folded into q as q / tau_h;
* finally everything is rounded to the workload dtype (bf16: round to nearest
  even), and the rounded values are what both the GPU path and the oracle read.

Offsets U ~ Unif[0, 1/S) are drawn per (sequence, query head) as float32 values
that are exactly what both sides consume.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

__all__ = [
    "Workload",
    "Inputs",
    "WORKLOADS",
    "get_workload",
    "generate",
    "float32_to_bf16_bits",
    "bf16_bits_to_float32",
    "to_torch",
]


@dataclass(frozen=True)
class Workload:
    """Shape and structure of one synthetic decode-attention problem."""

    name: str
    config: int  # seed base: seed = 1000 * config + instance
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    tile: int
    S: int
    dtype: str  # "f32" or "bf16"
    length: int = 0  # fixed length of every sequence (ignored if length_range set)
    length_range: tuple[int, int] | None = None  # ragged: UniformInt[lo, hi]
    lengths: tuple[int, ...] = ()  # explicit per-sequence lengths (edge cases)
    planted_per_head: int = 0  # fixed count of planted keys per query head
    planted_fraction: float = 0.0  # or a fraction of each sequence per KV head
    sinks: int = 0
    temperatures: tuple[float, ...] = ()  # tau_h = temperatures[h % len]
    n_offsets: int = 1  # number of independent U draws per (sequence, head)
    description: str = ""

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


@dataclass
class Inputs:
    """One seeded instance.  K/V are token-major [total_tokens][Hkv][d]."""

    workload: Workload
    seed: int
    lengths: np.ndarray  # int64 [B]
    kv_indptr: np.ndarray  # int64 [B + 1]
    q: np.ndarray  # float32 [B][Hq][d]; values exactly representable in dtype
    k: np.ndarray  # bf16 bits (uint16) or float32, [tok][Hkv][d]
    v: np.ndarray  # same layout as k
    U: np.ndarray  # float32 [n_offsets][B][Hq], each in [0, 1/S)
    q_native: np.ndarray = field(repr=False, default=None)  # uint16 bits or float32

    @property
    def total_tokens(self) -> int:
        return int(self.kv_indptr[-1])

    def k_f32(self, b: int | None = None) -> np.ndarray:
        """K as float32 (all tokens, or the tokens of sequence b)."""
        return _as_f32(self._slice(self.k, b), self.workload.dtype)

    def v_f32(self, b: int | None = None) -> np.ndarray:
        return _as_f32(self._slice(self.v, b), self.workload.dtype)

    def _slice(self, a: np.ndarray, b: int | None) -> np.ndarray:
        if b is None:
            return a
        return a[int(self.kv_indptr[b]) : int(self.kv_indptr[b + 1])]


def float32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_float32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _as_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_float32(a) if dtype == "bf16" else np.asarray(a, dtype=np.float32)


def _round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return float32_to_bf16_bits(x)
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


_LLAMA8B = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16")

WORKLOADS: dict[str, Workload] = {
    # Parity-only case: one GQA group, d = 64, 8 tiles of 128 keys.
    "tiny_fp32": Workload(
        name="tiny_fp32", config=1, batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64,
        length=1024, tile=128, S=16, dtype="f32", planted_per_head=8, n_offsets=64,
        description="batch 1, 4 q heads / 1 KV head, d=64, n_k=1024, tile 128, S=16, fp32",
    ),
    # One Llama-3.1-8B decode layer at 32k context.
    "llama8b_32k_b1": Workload(
        name="llama8b_32k_b1", config=2, batch=1, length=32768, tile=256, S=128,
        planted_fraction=0.01, sinks=4, **_LLAMA8B,
        description="batch 1, 32 q / 8 KV heads, d=128, n_k=32768, tile 256, S=128, bf16",
    ),
    # The same layer at batch 16 (S is varied per run: 64/128/256 prop, 2048 flash).
    "llama8b_32k_b16": Workload(
        name="llama8b_32k_b16", config=3, batch=16, length=32768, tile=256, S=128,
        planted_fraction=0.01, sinks=4, **_LLAMA8B,
        description="batch 16, 32 q / 8 KV heads, d=128, n_k=32768, tile 256, bf16",
    ),
    # Ragged serving batch with per-head temperatures.
    "ragged_b64": Workload(
        name="ragged_b64", config=5, batch=64, length_range=(4096, 32768), tile=256, S=128,
        planted_fraction=0.01, sinks=4, temperatures=(0.5, 1.0, 2.0), **_LLAMA8B,
        description="64 sequences, n_k ~ UniformInt[4096, 32768], 32q/8kv, d=128, S=128, "
        "tau_h in {0.5, 1, 2}, bf16",
    ),
}
# Context sweep at batch 8.
for _n in (4096, 8192, 16384, 32768, 65536, 131072):
    WORKLOADS[f"sweep_b8_n{_n}"] = Workload(
        name=f"sweep_b8_n{_n}", config=4, batch=8, length=_n, tile=256, S=128,
        planted_fraction=0.01, **_LLAMA8B,
        description=f"batch 8, 32q/8kv, d=128, n_k={_n}, tile 256, S=128, bf16",
    )


def max_length(w: Workload) -> int:
    if w.lengths:
        return max(w.lengths)
    if w.length_range is not None:
        return w.length_range[1]
    return w.length


def get_workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return w.with_(**overrides) if overrides else w


def _lengths(w: Workload, rng: np.random.Generator) -> np.ndarray:
    if w.lengths:
        assert len(w.lengths) == w.batch
        return np.asarray(w.lengths, dtype=np.int64)
    if w.length_range is not None:
        lo, hi = w.length_range
        return rng.integers(lo, hi + 1, size=w.batch, dtype=np.int64)
    return np.full(w.batch, w.length, dtype=np.int64)


def draw_offsets(S: int, shape, rng: np.random.Generator) -> np.ndarray:
    """U ~ Unif[0, 1/S) as float32 values strictly below 1/S."""
    u = rng.random(size=shape, dtype=np.float64) / S
    U = u.astype(np.float32)
    top = np.float32(1.0 / S)
    # float32 rounding may land exactly on 1/S: step back below it.
    bad = U >= top
    if np.any(bad):
        U[bad] = np.nextafter(top, np.float32(0.0), dtype=np.float32)
    return U


def draw_uniforms(shape, rng: np.random.Generator) -> np.ndarray:
    """Uniforms in [0, 1) as float32 values strictly below 1 (the stratified and
    i.i.d. samplers' draws, passed to both sides as inputs)."""
    u = rng.random(size=shape, dtype=np.float64).astype(np.float32)
    u[u >= np.float32(1.0)] = np.nextafter(np.float32(1.0), np.float32(0.0), dtype=np.float32)
    return u


def generate(w: Workload, instance: int = 0, n_offsets: int | None = None) -> Inputs:
    """Draw one seeded instance of workload ``w``."""
    seed = 1000 * w.config + instance
    root = np.random.SeedSequence(seed)
    s_len, s_q, s_u, s_seq = root.spawn(4)
    B, Hq, Hkv, d, G = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group
    if Hq % Hkv != 0:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")

    lengths = _lengths(w, np.random.Generator(np.random.PCG64(s_len)))
    indptr = np.zeros(B + 1, dtype=np.int64)
    np.cumsum(lengths, out=indptr[1:])
    total = int(indptr[-1])

    q = np.random.Generator(np.random.PCG64(s_q)).standard_normal((B, Hq, d), dtype=np.float32)
    native_dtype = np.uint16 if w.dtype == "bf16" else np.float32
    k = np.empty((total, Hkv, d), dtype=native_dtype)
    v = np.empty((total, Hkv, d), dtype=native_dtype)
    root_d = math.sqrt(d)

    for b, s in enumerate(s_seq.spawn(B)):
        rng = np.random.Generator(np.random.PCG64(s))
        L = int(lengths[b])
        kb = rng.standard_normal((L, Hkv, d), dtype=np.float32)
        vb = rng.standard_normal((L, Hkv, d), dtype=np.float32)
        for g in range(Hkv):
            Q = q[b, g * G : (g + 1) * G, :].astype(np.float64)  # [G][d], before temperature
            n_sink = min(w.sinks, L)
            if w.planted_per_head:
                n_plant = w.planted_per_head * G
            else:
                n_plant = int(round(w.planted_fraction * L))
            n_plant = min(n_plant, L - n_sink)
            if n_plant > 0:
                pos = n_sink + rng.choice(L - n_sink, size=n_plant, replace=False)
                heads = np.arange(n_plant) % G
                dirs = Q / np.linalg.norm(Q, axis=1, keepdims=True)
                kb[pos, g, :] += (3.0 * root_d * dirs[heads]).astype(np.float32)
            if n_sink > 0:
                # minimum-norm delta with Q @ delta = 2 sqrt(d) for every head of the group
                delta = Q.T @ np.linalg.solve(Q @ Q.T, np.full(G, 2.0 * root_d))
                kb[:n_sink, g, :] += delta.astype(np.float32)
        t0 = int(indptr[b])
        k[t0 : t0 + L] = _round_to(kb, w.dtype)
        v[t0 : t0 + L] = _round_to(vb, w.dtype)

    if w.temperatures:
        tau = np.array([w.temperatures[h % len(w.temperatures)] for h in range(Hq)], dtype=np.float32)
        q = q / tau[None, :, None]
    q_native = _round_to(q, w.dtype)
    q = _as_f32(q_native, w.dtype).reshape(B, Hq, d)

    n_off = w.n_offsets if n_offsets is None else n_offsets
    U = draw_offsets(w.S, (n_off, B, Hq), np.random.Generator(np.random.PCG64(s_u)))
    return Inputs(workload=w, seed=seed, lengths=lengths, kv_indptr=indptr, q=q, k=k, v=v, U=U,
                  q_native=q_native.reshape(B, Hq, d))


def to_torch(inp: Inputs, device="cuda", U_index: int = 0):
    """Device tensors (q, k, v, kv_indptr, U) of an instance, in the workload dtype."""
    import torch

    def native(a):
        if inp.workload.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))

    return (
        native(inp.q_native).to(device),
        native(inp.k).to(device),
        native(inp.v).to(device),
        torch.from_numpy(inp.kv_indptr).to(device),
        torch.from_numpy(np.ascontiguousarray(inp.U[U_index])).to(device),
    )
