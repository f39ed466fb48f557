"""Parity checks of GPU results against the oracle -- TEST INFRASTRUCTURE ONLY.

Numpy only.  Acceptance rules (same U on both sides):

* sampled indices and tile budgets bit-exact, except where the threshold lies
  within 1e-5 (relative) of EVERY CDF boundary separating the two answers,
  measured in the oracle's float64 CDF -- such mismatches are excused and
  counted (``Report.excused``); any other mismatch fails;
* tile mass Z_tile / Z within 1e-3 relative (both below 1e-6 where the
  oracle's mass is under 1e-30);
* out within 2e-3 absolute; where excused mismatches occurred, against the
  oracle's gather-average over the GPU's own indices.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import cdf, exact_head, flash_head, gather_mean, logits, prop_head, sampled_head, softmax

IDX_REL = 1e-5
MASS_REL = 1e-3
OUT_ABS = 2e-3
# Excused mismatches are rare by construction (a threshold must fall within
# rounding of a boundary); a run that excuses more than this fraction of its
# samples points at a kernel whose CDF drifts, not at rounding.
EXCUSED_FRACTION = 0.01


@dataclass
class Report:
    heads: int = 0
    samples: int = 0
    excused: int = 0
    max_out_err: float = 0.0
    max_mass_rel: float = 0.0
    notes: list = field(default_factory=list)

    def merge(self, o: "Report") -> "Report":
        self.heads += o.heads
        self.samples += o.samples
        self.excused += o.excused
        self.max_out_err = max(self.max_out_err, o.max_out_err)
        self.max_mass_rel = max(self.max_mass_rel, o.max_mass_rel)
        self.notes += o.notes
        return self


def excused_within_bound(rep: "Report") -> bool:
    """At most EXCUSED_FRACTION of the samples excused (two allowed in any run)."""
    return rep.excused <= max(2, EXCUSED_FRACTION * rep.samples)


def excused(F: np.ndarray, t: float, a: int, b: int) -> bool:
    """May a sampler return key a where the float64 inverse CDF returns key b?

    Only if float rounding of the CDF can explain it: the two answers differ by
    crossing the boundaries F(i), i in [min(a, b), max(a, b)), and every one of
    them must lie within IDX_REL (relative) of the threshold t.  F is
    non-decreasing, so the farthest boundary is the one at min(a, b) when a < b
    and at max(a, b) - 1 when a > b; checking all of them covers both."""
    lo, hi = min(a, b), max(a, b)
    if lo == hi:
        return True
    return bool(np.max(np.abs(F[lo:hi] - t)) <= IDX_REL * t)


def _check_masses(gpu_m, gpu_z, ref_mass, what, rep):
    """GPU tile records (m_t, z_t) -> Z_tile / Z in float64, against the oracle's masses."""
    m = np.asarray(gpu_m, dtype=np.float64)
    z = np.asarray(gpu_z, dtype=np.float64)
    w = z * np.exp(m - m.max())
    mass = w / w.sum()
    big = ref_mass > 1e-30
    if big.any():
        rel = np.abs(mass[big] - ref_mass[big]) / ref_mass[big]
        rep.max_mass_rel = max(rep.max_mass_rel, float(rel.max()))
        assert rel.max() <= MASS_REL, f"{what}: tile mass rel err {rel.max():.3e}"
    if (~big).any():
        assert np.all(mass[~big] < 1e-6) and np.all(ref_mass[~big] < 1e-6), f"{what}: tiny tile masses"


def check_prop_head(q, K, V, S, U, tile, gpu_out, gpu_idx, gpu_count=None, gpu_m=None, gpu_z=None,
                    what="prop") -> Report:
    """One (sequence, query head) of S2ANTA-prop.  K, V are that head's [n][d] rows."""
    rep = Report(heads=1, samples=S)
    n = K.shape[0]
    gpu_out = np.asarray(gpu_out, dtype=np.float64)
    if n == 0:
        assert np.all(gpu_out == 0.0), f"{what}: empty sequence must give zeros"
        return rep
    ref = prop_head(q, K, V, S, U, tile, want_F=True)
    T = ref.counts.size
    idx = None if gpu_idx is None else np.asarray(gpu_idx, dtype=np.int64)
    if idx is not None:
        assert idx.min() >= 0 and idx.max() < n, f"{what}: index out of range"
        t = float(U) + np.arange(S, dtype=np.float64) / S
        bad = np.nonzero(idx != ref.J)[0]
        for m in bad:
            assert excused(ref.F, t[m], int(idx[m]), int(ref.J[m])), (
                f"{what}: sample {m} picked {idx[m]}, oracle {ref.J[m]}, threshold {t[m]!r}")
        rep.excused += bad.size
        if gpu_count is not None:
            cnt = np.asarray(gpu_count, dtype=np.int64)[:T]
            assert cnt.sum() == S, f"{what}: budgets sum to {cnt.sum()}, not S={S}"
            assert np.array_equal(cnt, np.bincount(idx // tile, minlength=T)), f"{what}: budgets vs indices"
            if bad.size == 0:
                assert np.array_equal(cnt, ref.counts), f"{what}: budgets differ without index mismatches"
        expect = ref.out if bad.size == 0 else gather_mean(idx, V)
    else:
        expect = ref.out
    err = float(np.max(np.abs(gpu_out - expect)))
    rep.max_out_err = err
    assert err <= OUT_ABS, f"{what}: out err {err:.3e}"
    if gpu_m is not None:
        _check_masses(np.asarray(gpu_m)[:T], np.asarray(gpu_z)[:T], ref.mass, what, rep)
    return rep


def check_flash_head(q, K, V, S, U, tile, gpu_out, gpu_idx=None, gpu_m=None, gpu_z=None, what="flash") -> Report:
    """One (sequence, query head) of S2ANTA-flash.  gpu_idx is [T][>= S_loc]."""
    rep = Report(heads=1)
    n = K.shape[0]
    gpu_out = np.asarray(gpu_out, dtype=np.float64)
    if n == 0:
        assert np.all(gpu_out == 0.0), f"{what}: empty sequence must give zeros"
        return rep
    ref = flash_head(q, K, V, S, U, tile)
    T, S_loc = ref.J.shape
    rep.samples = T * S_loc
    expect = ref.out
    if gpu_idx is not None:
        idx = np.asarray(gpu_idx, dtype=np.int64)[:T, :S_loc]
        x = logits(q, K)
        Ut = float(U) * S / S_loc
        tt = Ut + np.arange(S_loc, dtype=np.float64) / S_loc
        any_bad = False
        tile_est = np.empty((T, K.shape[1]))
        for ti in range(T):
            k0, k1 = ti * tile, min(n, (ti + 1) * tile)
            assert idx[ti].min() >= k0 and idx[ti].max() < k1, f"{what}: tile {ti} index out of tile"
            bad = np.nonzero(idx[ti] != ref.J[ti])[0]
            if bad.size:
                any_bad = True
                e = np.exp(x[k0:k1] - x[k0:k1].max())
                Ft = cdf(e / e.sum())
                for s in bad:
                    assert excused(Ft, tt[s], int(idx[ti, s]) - k0, int(ref.J[ti, s]) - k0), (
                        f"{what}: tile {ti} sample {s} picked {idx[ti, s]}, oracle {ref.J[ti, s]}")
                rep.excused += bad.size
            tile_est[ti] = gather_mean(idx[ti], V)
        if any_bad:
            expect = ref.weight @ tile_est
    err = float(np.max(np.abs(gpu_out - expect)))
    rep.max_out_err = err
    assert err <= OUT_ABS, f"{what}: out err {err:.3e}"
    if gpu_m is not None:
        _check_masses(np.asarray(gpu_m)[:T], np.asarray(gpu_z)[:T], ref.weight, what, rep)
    return rep


def check_exact_head(q, K, V, gpu_out, what="exact") -> Report:
    rep = Report(heads=1)
    expect = exact_head(q, K, V)
    err = float(np.max(np.abs(np.asarray(gpu_out, dtype=np.float64) - expect)))
    rep.max_out_err = err
    assert err <= OUT_ABS, f"{what}: out err {err:.3e}"
    return rep


def check_sampled_head(mode, q, K, V, u, gpu_out, gpu_idx, what=None) -> Report:
    """One (sequence, query head) of the prop pipeline with the stratified ('strat') or
    i.i.d. ('iid') sampler and caller uniforms u[S].  strat: gpu_idx[m] is the key of
    threshold (m + u_m)/S; iid: gpu_idx[m] is the key of the m-th smallest u."""
    what = what or mode
    S = int(np.asarray(u).size)
    rep = Report(heads=1, samples=S)
    n = K.shape[0]
    gpu_out = np.asarray(gpu_out, dtype=np.float64)
    if n == 0:
        assert np.all(gpu_out == 0.0), f"{what}: empty sequence must give zeros"
        return rep
    u = np.asarray(u, dtype=np.float64)
    ref_out, ref_J = sampled_head(mode, q, K, V, u)
    if mode == "strat":
        t = (np.arange(S, dtype=np.float64) + u) / S
        J = ref_J
    else:  # threshold order: increasing u (F^-1 is monotone, so J follows)
        order = np.argsort(u, kind="stable")
        t, J = u[order], ref_J[order]
    idx = np.asarray(gpu_idx, dtype=np.int64)
    assert idx.min() >= 0 and idx.max() < n, f"{what}: index out of range"
    F = cdf(softmax(logits(q, K)))
    bad = np.nonzero(idx != J)[0]
    for m in bad:
        assert excused(F, t[m], int(idx[m]), int(J[m])), (
            f"{what}: sample {m} picked {idx[m]}, oracle {J[m]}, threshold {t[m]!r}")
    rep.excused += bad.size
    expect = ref_out if bad.size == 0 else gather_mean(idx, V)
    err = float(np.max(np.abs(gpu_out - expect)))
    rep.max_out_err = err
    assert err <= OUT_ABS, f"{what}: out err {err:.3e}"
    return rep
