#!/usr/bin/env python3
"""Benchmark: decode-attention microseconds per layer-step and HBM GB/s vs roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--mode prop|flash|exact] [--workload NAME] [--S S]

One step is one decode-attention layer-step of the workload (all kernels of one
C-ABI call) over seeded synthetic inputs already resident in HBM.  Steps are
replayed from CUDA graphs of --graph-steps consecutive calls; successive calls
rotate through copies of the K/V cache whose total size exceeds 4x the L2 cache,
so no call finds its cache in L2.  Timing uses CUDA events on the launching
stream with a barrier and a synchronize on both sides; with N GPUs (torchrun,
one process per GPU) every rank runs its own replica of the workload and the
time is the maximum over ranks.  Rank 0 prints one JSON line.

--impl reference times the CPU oracle on the host cores instead (each step one
query head of the same layer-step; the value is scaled to a whole layer-step).
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/layer-step and HBM GB/s vs roofline, n_k=32k, S=128"
UNIT = "us/layer-step"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------- setup


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=15000)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["prop", "strat", "iid", "flash", "exact"], default="prop")
    ap.add_argument("--workload", default="llama8b_32k_b1")
    ap.add_argument("--S", type=int, default=0, help="override the workload's sample count")
    ap.add_argument("--graph-steps", type=int, default=100)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample length")
    ap.add_argument("--no-extras", action="store_true", help="skip the exact/flash comparison timings")
    ap.add_argument("--profile", action="store_true",
                    help="no benchmark: two rounds of one call of each path on the workload, for profiler "
                         "captures (round 1 warms up; skip its " + str(PROFILE_ROUND_LAUNCHES) + " matched launches)")
    return ap.parse_args(argv)


# The launches of one --profile round that the profiler filter
# regex:"prop_stream|prop_pass2|fb_pass1|exact_stream|merge_kernel|flash_sample|prop_fused" matches:
# prop (stream, pass 2), Bernoulli with the mean group query (feature-blocked pass 1,
# pass 2), exact (stream, merge), flash at S = 2048 (stream, tile sampler, merge),
# the fused kernel.
PROFILE_ROUND_LAUNCHES = 10


def run_profile(args) -> dict:
    """Two rounds of one call of each path (prop, Bernoulli mean group query, exact,
    flash at S = 2048, fused prop) on the workload: a short, fixed launch sequence
    for profiler captures of every kernel on the same inputs."""
    import torch

    from stochastic_sparse_decode_gb300.build import build
    from stochastic_sparse_decode_gb300.decoder import Decoder
    from synthetic import generate, get_workload, max_length, to_torch
    from synthetic.workloads import draw_offsets, draw_uniforms

    build()
    dev = torch.device("cuda", 0)
    w = get_workload(args.workload)
    inp = generate(w)
    q, k, v, indptr, U = to_torch(inp, dev)
    dec = Decoder(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, inp.total_tokens, max_length(w), w.tile,
                  w.S, w.dtype, device=dev)
    decf = Decoder(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, inp.total_tokens, max_length(w), w.tile,
                   2048, w.dtype, device=dev)
    Uf = torch.from_numpy(draw_offsets(2048, (w.batch, w.num_q_heads), np.random.default_rng(7))).to(dev)
    bu = torch.from_numpy(draw_uniforms((w.batch, w.num_kv_heads, 4, w.head_dim), np.random.default_rng(17))
                          .astype(np.float32)).to(dev)
    kfb = dec.feature_blocked(k)
    out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device=dev)
    for _ in range(2):
        dec("prop", q, k, v, indptr, U, out=out)
        dec.prop_bernoulli(q, kfb, v, indptr, U, bu, 4, True, out=out)
        dec("exact", q, k, v, indptr, U, out=out)
        decf("flash", q, k, v, indptr, Uf, out=out)
        dec("prop_fused", q, k, v, indptr, U, out=out)
        torch.cuda.synchronize()
    return {"profile": w.name, "launches_per_round": PROFILE_ROUND_LAUNCHES}


class Dist:
    """Rank bookkeeping; a process group only when launched by torchrun with N > 1."""

    def __init__(self, backend: str | None = None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist

            if backend is None:
                import torch

                backend = "nccl" if torch.cuda.is_available() else "gloo"
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            if self.pg.get_backend() == "nccl":
                import torch

                self.pg.barrier(device_ids=[torch.cuda.current_device()])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        """Maximum of a float over ranks."""
        if self.pg is None:
            return float(x)
        import torch

        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate_value(max_elapsed_ms: float, steps: int, world: int) -> float:
    """Whole-job microseconds per layer-step: every rank ran `steps` layer-steps of
    its own replica within max_elapsed_ms, so the job did world * steps of them."""
    return max_elapsed_ms * 1000.0 / (steps * world)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest() -> str:
    """Digest of the device code (the kernels live in the .cuh headers and .cu files)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "stochastic_sparse_decode_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "*.cuh")) + glob.glob(os.path.join(csrc, "*.cu"))):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel sources (the summary records their digest)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_digest") != source_digest():
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu, self.period, self.proc, self.path = gpu_index, period_ms, None, None

    def start(self):
        try:
            out_dir = os.environ.get("SANTA_CLOCKS_DIR") or tempfile.gettempdir()
            os.makedirs(out_dir, exist_ok=True)
            self.path = os.path.join(out_dir, f"clocks_rank{self.gpu}.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={self.period}"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- byte model


def byte_model(inp, mode: str, S: int, sample_idx=None):
    """Algorithmic HBM bytes of one call and of its dominant kernel.

    prop:  K (Hkv * sum L * d * e) + q + stash write (Hq * sum L * 4) + the
           partition records, one (m, z) per 32-key chunk (written by pass 1,
           read by pass 2: 2 * 8 * Hq * sum ceil(L / 32)) + the stash of the
           chunks that received samples (4 * len per chunk) + the distinct V
           rows the samples touch (d * e each, per KV head) + out.
    flash: prop's pass 1 (K + q + stash write + chunk records) + the whole stash and
           the chunk records read back by the tiles' sampler + distinct V rows +
           tile partials and records (written and read) + out.
    exact: K + V + q + out (its split-KV partials are overhead, not counted).
    Pass 1: K + q + its writes.
    """
    w = inp.workload
    e = 2 if w.dtype == "bf16" else 4
    L = inp.lengths.astype(np.int64)
    T = -(-L // w.tile)
    NC = -(-L // 32)
    sumL, sumT, sumC = int(L.sum()), int(T.sum()), int(NC.sum())
    B, Hq, Hkv, d = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    K = Hkv * sumL * d * e
    q = B * Hq * d * e
    out = B * Hq * d * 4
    vrows = 0
    stash_read = 0
    if sample_idx is not None and mode in ("prop", "flash"):
        G = w.group
        for b in range(B):
            for g in range(Hkv):
                heads = sample_idx[b, g * G : (g + 1) * G]
                rows = np.unique(heads[heads >= 0])
                vrows += rows.size
                if mode == "prop":
                    for h in range(G):
                        for c in np.unique(sample_idx[b, g * G + h] // 32):
                            stash_read += 4 * int(min(32, L[b] - c * 32))
    if mode == "prop":
        rec = 8 * Hq * sumC  # (m_c, z_c) per (b, h, chunk)
        main = K + q + Hq * sumL * 4 + rec
        total = main + rec + stash_read + vrows * d * e + out
    elif mode == "flash":
        crec = 8 * Hq * sumC  # (m_c, z_c) per (b, h, chunk)
        rec = 8 * Hq * sumT  # (m_t, z_t) per (b, h, t)
        part = 4 * Hq * sumT * d
        main = K + q + Hq * sumL * 4 + crec
        total = main + Hq * sumL * 4 + crec + vrows * d * e + 2 * (rec + part) + out
    else:
        # the dense method's own bytes; the split-KV partials of the streaming
        # kernel (one (M, Z, O) per warp and head) are overhead, not counted
        main = 2 * K + q
        total = main + out
    return {"total": int(total), "main": int(main), "v_rows": int(vrows), "stash_read": int(stash_read),
            "k_bytes": int(K)}


# ----------------------------------------------------------------------------- our arm


def run_ours(args, dist: Dist):
    import torch

    import stochastic_sparse_decode_gb300 as sd
    from stochastic_sparse_decode_gb300.build import build
    from stochastic_sparse_decode_gb300.decoder import Decoder
    from synthetic import generate, get_workload, max_length, to_torch

    build()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    w = get_workload(args.workload)
    if args.S:
        w = w.with_(S=args.S)
    elif args.mode == "flash" and args.workload.startswith("llama8b"):
        w = w.with_(S=2048)  # the flash mode's configuration (6.25% of n_k)
    inp = generate(w)
    q, k, v, indptr, U = to_torch(inp, dev)
    if args.mode in ("strat", "iid"):  # the samplers' uniforms [B][Hq][S]
        from synthetic.workloads import draw_uniforms

        U = torch.from_numpy(draw_uniforms((w.batch, w.num_q_heads, w.S), np.random.default_rng(11))).to(dev)
    dec = Decoder(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, inp.total_tokens, max_length(w), w.tile,
                  w.S, w.dtype, device=dev)
    out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device=dev)

    # one debug call: sample indices for the byte model, and (rank 0, one GPU) the
    # outputs the CPU-baseline leg checks against the oracle
    dbg, bufs = dec.debug_buffers(args.mode, sample_stride=max(1, -(-w.S // max(1, int((-(-inp.lengths // w.tile)).min())))))
    dec(args.mode, q, k, v, indptr, U, out=out, debug=dbg)
    torch.cuda.synchronize()
    checked = {"out": out.cpu().numpy().copy(), "U": U.cpu().numpy().copy(),
               **{name: t.cpu().numpy().copy() for name, t in bufs.items()}}
    sidx = bufs.get("sample_idx")
    sidx = sidx.cpu().numpy().reshape(w.batch, w.num_q_heads, -1) if sidx is not None else None
    bm = byte_model(inp, "prop" if args.mode in ("strat", "iid") else args.mode, w.S, sidx)

    # L2-safe rotation of the K/V cache
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_copy = k.numel() * k.element_size() + v.numel() * v.element_size()
    nrot = max(2, math.ceil(4 * l2 / per_copy) + 1)
    ks, vs = [k], [v]
    for _ in range(nrot - 1):
        ks.append(k.clone())
        vs.append(v.clone())
    for i in range(nrot):  # warm every descriptor / attribute before capture
        dec(args.mode, q, ks[i], vs[i], indptr, U, out=out)
    torch.cuda.synchronize()

    def capture(nsteps, mode=args.mode, decoder=dec, Uarg=U):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for i in range(min(nsteps, nrot)):
                decoder(mode, q, ks[i % nrot], vs[i % nrot], indptr, Uarg, out=out)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for i in range(nsteps):
                decoder(mode, q, ks[i % nrot], vs[i % nrot], indptr, Uarg, out=out)
        return g

    def timed(nsteps, warm, mode=args.mode, decoder=dec, Uarg=U, sampler=None):
        """Device time of exactly `nsteps` calls, replayed from graphs of up to
        --graph-steps calls.  Every graph that is timed has been replayed once before
        (its first replay uploads it), after `warm` untimed calls; the GPU is kept
        busy by a sleep kernel while the host enqueues the timed replays, so the host
        launch latency stays outside the events."""
        R = max(1, min(args.graph_steps, nsteps))
        full, rem = divmod(nsteps, R)
        g = capture(R, mode, decoder, Uarg)
        gr = capture(rem, mode, decoder, Uarg) if rem else None
        g.replay()
        if gr is not None:
            gr.replay()
        wf, wr = divmod(warm, R)
        for _ in range(wf):
            g.replay()
        if wr:
            capture(wr, mode, decoder, Uarg).replay()
        torch.cuda.synchronize()
        if sampler:
            sampler.start()
        dist.barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(2e6))  # ~1 ms: the replays below queue up behind it
        a.record()
        for _ in range(full):
            g.replay()
        if gr is not None:
            gr.replay()
        b.record()
        b.synchronize()
        torch.cuda.synchronize()
        dist.barrier()
        clocks = sampler.stop() if sampler else None
        return a.elapsed_time(b), clocks

    sampler = ClockSampler(dist.local_rank)
    elapsed_ms, clocks = timed(args.steps, args.warmup, sampler=sampler)
    max_ms = dist.max(elapsed_ms)
    value = aggregate_value(max_ms, args.steps, dist.world)
    per_step_us = elapsed_ms * 1000.0 / args.steps

    # dominant kernel alone: events around it inside each call, GPU kept ahead of the host
    nmain = 200
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nmain)]
    dbgs = []
    for a_, b_ in evs:
        a_.record()  # torch creates the CUDA event on its first record
        b_.record()
        d_ = sd.Debug()
        d_.main_begin = a_.cuda_event
        d_.main_end = b_.cuda_event
        dbgs.append(d_)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(50e6))  # ~25 ms of spinning so all launches below queue up
    for i in range(nmain):
        dec(args.mode, q, ks[i % nrot], vs[i % nrot], indptr, U, out=out, debug=dbgs[i])
    torch.cuda.synchronize()
    main_us_eager = statistics.mean(a_.elapsed_time(b_) * 1000.0 for a_, b_ in evs[10:])
    main_us_in_call = main_us_eager
    peak, peak_kind = measured_peaks()
    pass1 = None
    if args.mode in ("prop", "strat", "iid"):
        # the whole call (pass 1 and pass 2) against its algorithmic bytes: the timed
        # region's per-step time; pass 1, the dominant kernel, is reported beside it
        kernel_name = "prop_call"
        main_us = per_step_us
        main_bytes = bm["total"]
        main_timing = ("the whole call: the timed region's CUDA graphs of back-to-back santa_decode_prop calls "
                       "(pass 1 + pass 2 each); CUDA events on the launching stream")
        # pass 1 alone (santa_prop_pass1, on a workspace of its own), for context: a
        # graph of nmain back-to-back launches over the rotating K copies
        dec1 = Decoder(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, inp.total_tokens, max_length(w),
                       w.tile, w.S, w.dtype, device=dev)
        gm = torch.cuda.CUDAGraph()
        sm_ = torch.cuda.Stream(device=dev)
        sm_.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(sm_):
            for i in range(nrot):
                dec1.pass1(q, ks[i], indptr)
        torch.cuda.current_stream().wait_stream(sm_)
        torch.cuda.synchronize()
        with torch.cuda.graph(gm):
            for i in range(nmain):
                dec1.pass1(q, ks[i % nrot], indptr)
        for _ in range(3):
            gm.replay()
        torch.cuda.synchronize()
        reps = []
        for _ in range(5):
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(int(2e6))
            a_.record()
            gm.replay()
            b_.record()
            b_.synchronize()
            reps.append(a_.elapsed_time(b_) * 1000.0 / nmain)
        p1_us = statistics.median(reps)
        p1_gbs = bm["main"] / (p1_us * 1e-6) / 1e9
        pass1 = {"kernel": "prop_stream (santa_prop_pass1 alone)", "us": round(p1_us, 3),
                 "us_in_call": round(main_us_eager, 3),
                 "algorithmic_bytes": bm["main"], "achieved": round(p1_gbs, 1), "frac": round(p1_gbs / peak, 4),
                 "traffic": profiled_traffic("prop_pass1", w.name),
                 "timing": f"CUDA events around replays of a graph of {nmain} back-to-back launches over the "
                           "rotating K copies (median of 5 replays)"}
        del gm, dec1
    else:
        kernel_name = {"flash": "prop_pass1", "exact": "exact_stream"}[args.mode]
        main_us = main_us_eager
        main_bytes = bm["main"]
        main_timing = "CUDA events around the kernel inside each call, eager launches"
    achieved = main_bytes / (main_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": profiled_traffic(kernel_name, w.name),
                "kernel": kernel_name, "kernel_us": round(main_us, 3), "kernel_us_in_call": round(main_us_in_call, 3),
                "kernel_timing": main_timing, "algorithmic_bytes": main_bytes,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else
                f"{peak_kind} (no MEASURED_PEAKS.json)"}
    if pass1 is not None:
        roofline["pass1"] = pass1

    # end to end through the public API with pinned host buffers
    hq_, hk, hv, hind, hU = (t.cpu().pin_memory() for t in (q, k, v, indptr, U))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dq, dk, dv, dind, dU = (torch.empty_like(t, device=dev) for t in (q, k, v, indptr, U))
    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk, hv, hind, hU))
    d2h = hout.numel() * hout.element_size()

    # V comes over a second stream (a second copy engine) while q, K and the small
    # inputs come over the launching stream; for prop, pass 1 (which reads no V) runs
    # meanwhile through santa_prop_pass1, and santa_prop_pass2 waits for V.
    s_copy = torch.cuda.Stream(device=dev)
    split = args.mode == "prop"

    def e2e_step():
        cur = torch.cuda.current_stream()
        s_copy.wait_stream(cur)  # the previous step is done reading dv
        with torch.cuda.stream(s_copy):
            dv.copy_(hv, non_blocking=True)
        for dst, src in ((dq, hq_), (dk, hk), (dind, hind), (dU, hU)):
            dst.copy_(src, non_blocking=True)
        if split:
            dec.pass1(dq, dk, dind)
            cur.wait_stream(s_copy)
            dec.pass2(dv, dind, dU, out=out)
        else:
            cur.wait_stream(s_copy)
            dec(args.mode, dq, dk, dv, dind, dU, out=out)
        hout.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.e2e_steps):
        e2e_step()
    b.record()
    b.synchronize()
    e2e_ms = dist.max(a.elapsed_time(b))
    e2e = {"value": round(aggregate_value(e2e_ms, args.e2e_steps, dist.world), 3), "unit": UNIT,
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": args.e2e_steps,
           "pipeline": ("V copied on a second stream while K's copy and santa_prop_pass1 run; "
                        "santa_prop_pass2 waits for it" if split else
                        "V copied on a second stream alongside q and K")}
    del dq, dk, dv, hk, hv

    extras = {}
    if not args.no_extras and args.mode == "prop":
        n_x = min(args.steps, 5000)
        ms, _ = timed(n_x, min(args.warmup, 200), mode="exact")
        exact_us = ms * 1000.0 / n_x
        extras["exact_us_per_layer_step"] = round(exact_us, 3)
        extras["speedup_vs_exact"] = round(exact_us / per_step_us, 3)
        # how close the dense comparison call is to the HBM roofline (its algorithmic
        # bytes: all of K and V, q, out)
        ex_bytes = byte_model(inp, "exact", w.S)["total"]
        ex_gbs = ex_bytes / (exact_us * 1e-6) / 1e9
        extras["exact_hbm_gbs"] = round(ex_gbs, 1)
        extras["exact_roofline_frac"] = round(ex_gbs / measured_peaks()[0], 4)
        if w.name.startswith("llama8b"):
            wf = w.with_(S=2048)
            from synthetic.workloads import draw_offsets

            Uf = torch.from_numpy(draw_offsets(2048, (w.batch, w.num_q_heads), np.random.default_rng(7))).to(dev)
            decf = Decoder(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, inp.total_tokens, max_length(w),
                           w.tile, 2048, w.dtype, device=dev)
            for i in range(nrot):
                decf("flash", q, ks[i], vs[i], indptr, Uf, out=out)
            ms, _ = timed(n_x, min(args.warmup, 200), mode="flash", decoder=decf, Uarg=Uf)
            extras["flash_S2048_us_per_layer_step"] = round(ms * 1000.0 / n_x, 3)
            del wf
        # the same call as one persistent kernel (santa_decode_prop_fused)
        for i in range(nrot):
            dec("prop_fused", q, ks[i], vs[i], indptr, U, out=out)
        ms, _ = timed(n_x, min(args.warmup, 200), mode="prop_fused")
        extras["prop_fused_us_per_layer_step"] = round(ms * 1000.0 / n_x, 3)
        # the Bernoulli ternary score stage on a feature-blocked K (four draws, as the
        # pages' B = 4): the fraction of K features read and the call's time
        extras.update(bernoulli_extras(dec, q, ks, vs, indptr, U, out, nrot, n_x, inp, bm, w))
        # the prop pipeline with the stratified and i.i.d. samplers, same S
        from synthetic.workloads import draw_uniforms

        Uu = torch.from_numpy(draw_uniforms((w.batch, w.num_q_heads, w.S), np.random.default_rng(11))).to(dev)
        for smode in ("strat", "iid"):
            for i in range(nrot):
                dec(smode, q, ks[i], vs[i], indptr, Uu, out=out)
            ms, _ = timed(n_x, min(args.warmup, 200), mode=smode, Uarg=Uu)
            extras[f"{smode}_us_per_layer_step"] = round(ms * 1000.0 / n_x, 3)

    launches_per_step = 2  # prop: pass 1 + pass 2; flash: tiles + merge; exact: stream + merge
    res = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "mode": args.mode, "batch": w.batch, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "n_k": int(inp.lengths.max()),
                   "tile": w.tile, "S": w.S, "kv_dtype": w.dtype, "accumulate": "f32",
                   "parallelism": f"replicas{dist.world}",
                   "l2": f"rotating {nrot} K/V copies, {nrot * per_copy / 2**20:.0f} MiB >= 4x L2 "
                         f"({l2 / 2**20:.0f} MiB)",
                   "timing": f"CUDA graphs of {args.graph_steps} calls, CUDA events on the launching stream"},
        "hbm_gbs": round(bm["total"] / (per_step_us * 1e-6) / 1e9, 1),
        "algorithmic_bytes_per_step": bm["total"],
        "v_row_fraction": round(bm["v_rows"] / max(1, w.num_kv_heads * int(inp.lengths.sum())), 6)
        if args.mode != "exact" else None,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "extras": extras,
    }
    if dist.rank == 0 and dist.world == 1:
        res["cpu_baseline"] = cpu_baseline(inp, args.mode, w.S, args.cpu_seconds)
        res["parity"] = oracle_parity(inp, args.mode, w.S, checked)
    return res


def bernoulli_extras(dec, q, ks, vs, indptr, U, out, nrot, nsteps, inp, bm, w) -> dict:
    """santa_decode_prop_bernoulli on the timed workload, per head and with the mean
    group query, four draws: the K-feature read fraction (the kept-feature counts
    over the sequences' keys), the bytes it saves, and the call's time (graphs of
    back-to-back calls over the rotating copies)."""
    import torch

    from synthetic.workloads import draw_uniforms

    dev = q.device
    kfbs = [dec.feature_blocked(ks[i]) for i in range(nrot)]
    lengths = inp.lengths.astype(np.int64)
    k_bytes = int(lengths.sum()) * w.num_kv_heads * w.head_dim * (2 if w.dtype == "bf16" else 4)
    res = {}
    for gm in (False, True):
        tag = "bernoulli_group_mean" if gm else "bernoulli"
        heads = w.num_kv_heads if gm else w.num_q_heads
        bu = torch.from_numpy(draw_uniforms((w.batch, heads, 4, w.head_dim), np.random.default_rng(17))
                              .astype(np.float32)).to(dev)
        dbg, bufs = dec.debug_buffers("prop_bernoulli")
        dec.prop_bernoulli(q, kfbs[0], vs[0], indptr, U, bu, 4, gm, out=out, debug=dbg)
        torch.cuda.synchronize()
        feat = bufs["features_read"].cpu().numpy().astype(np.int64)  # [B][Hkv]
        frac = float((feat * lengths[:, None]).sum()) / max(1, int(lengths.sum()) * w.num_kv_heads * w.head_dim)
        g = torch.cuda.CUDAGraph()
        s_ = torch.cuda.Stream(device=dev)
        s_.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_):
            for i in range(nrot):
                dec.prop_bernoulli(q, kfbs[i], vs[i], indptr, U, bu, 4, gm, out=out)
        torch.cuda.current_stream().wait_stream(s_)
        torch.cuda.synchronize()
        n = min(nsteps, 200)
        with torch.cuda.graph(g):
            for i in range(n):
                dec.prop_bernoulli(q, kfbs[i % nrot], vs[i % nrot], indptr, U, bu, 4, gm, out=out)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = []
        for _ in range(5):
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(int(2e6))
            a_.record()
            g.replay()
            b_.record()
            b_.synchronize()
            reps.append(a_.elapsed_time(b_) * 1000.0 / n)
        us = statistics.median(reps)
        alg = bm["total"] - (1.0 - frac) * k_bytes  # the K features not kept are not read
        res[f"{tag}_k_feature_read_fraction"] = round(frac, 4)
        res[f"{tag}_k_bytes_saved_per_step"] = int(round((1.0 - frac) * k_bytes))
        res[f"{tag}_us_per_layer_step"] = round(us, 3)
        res[f"{tag}_hbm_gbs"] = round(alg / (us * 1e-6) / 1e9, 1)
        del g
    del kfbs
    return res


# ----------------------------------------------------------------------------- the oracle on the host


def _oracle_problem(inp):
    """float64 K/V per (sequence, KV head), prepared once outside any timing."""
    w = inp.workload
    kv = {}
    for b in range(w.batch):
        Kb, Vb = inp.k_f32(b), inp.v_f32(b)
        for g in range(w.num_kv_heads):
            kv[(b, g)] = (np.ascontiguousarray(Kb[:, g, :], dtype=np.float64),
                          np.ascontiguousarray(Vb[:, g, :], dtype=np.float64))
    return kv


def _oracle_head(oracle, inp, kv, mode, S, b, h):
    w = inp.workload
    K, V = kv[(b, h // w.group)]
    qh = np.ascontiguousarray(inp.q[b, h], dtype=np.float64)
    U = float(inp.U[0, b, h])
    if mode in ("strat", "iid"):
        from synthetic.workloads import draw_uniforms

        oracle.sampled_head(mode, qh, K, V, draw_uniforms(S, np.random.default_rng(11 + h)))
    elif mode == "prop":
        oracle.prop_head(qh, K, V, S, U, w.tile, want_F=False)
    elif mode == "flash":
        oracle.flash_head(qh, K, V, S, U, w.tile)
    else:
        oracle.exact_head(qh, K, V)


def cpu_baseline(inp, mode, S, seconds):
    """The oracle (single-threaded C, float64) on whole layer-steps until `seconds` pass."""
    import oracle

    oracle.build()
    w = inp.workload
    kv = _oracle_problem(inp)
    heads = [(b, h) for b in range(w.batch) for h in range(w.num_q_heads)]
    n = 0
    t0 = time.perf_counter()
    while True:
        for b, h in heads:
            _oracle_head(oracle, inp, kv, mode, S, b, h)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    return {"value": round(el * 1e6 / n, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} whole layer-steps of {w.name} ({len(heads)} query heads), {mode}, "
                      f"single-threaded C float64 oracle, {el:.1f} s", "cpu": _cpu_name()}


def oracle_parity(inp, mode, S, got, max_heads=64):
    """The benchmark's own debug call against the oracle (part of the CPU-baseline
    leg, outside every timed region): the acceptance rule of oracle/compare.py on up
    to `max_heads` (sequence, query head) pairs of the timed workload -- samples
    compared, boundary mismatches excused, worst output error, and whether every
    head passed."""
    from oracle import compare

    w = inp.workload
    heads = [(b, h) for b in range(w.batch) for h in range(w.num_q_heads)]
    if len(heads) > max_heads:
        pick = np.random.default_rng(0).choice(len(heads), size=max_heads, replace=False)
        heads = [heads[i] for i in sorted(pick)]
    kv = {}
    rep, failures = compare.Report(), []
    for b, h in heads:
        g = h // w.group
        if (b, g) not in kv:
            kv[(b, g)] = (inp.k_f32(b)[:, g, :].astype(np.float64), inp.v_f32(b)[:, g, :].astype(np.float64))
        K, V = kv[(b, g)]
        qh = inp.q[b, h].astype(np.float64)
        try:
            if mode == "prop":
                r = compare.check_prop_head(qh, K, V, S, float(got["U"][b, h]), w.tile, got["out"][b, h],
                                            got["sample_idx"][b, h], got["tile_count"][b, h],
                                            got["tile_m"][b, h], got["tile_z"][b, h])
            elif mode in ("strat", "iid"):
                r = compare.check_sampled_head(mode, qh, K, V, got["U"][b, h], got["out"][b, h],
                                               got["sample_idx"][b, h])
            elif mode == "flash":
                r = compare.check_flash_head(qh, K, V, S, float(got["U"][b, h]), w.tile, got["out"][b, h],
                                             got["sample_idx"][b, h], got["tile_m"][b, h], got["tile_z"][b, h])
            else:
                r = compare.check_exact_head(qh, K, V, got["out"][b, h])
            rep.merge(r)
        except AssertionError as e:
            failures.append(f"b{b}h{h}: {e}")
    return {"heads": len(heads), "samples": rep.samples, "excused": rep.excused,
            "max_out_err": float(f"{rep.max_out_err:.3e}"), "max_mass_rel": float(f"{rep.max_mass_rel:.3e}"),
            "ok": not failures and compare.excused_within_bound(rep), "failures": failures[:3],
            "rule": "indices bit-exact unless every CDF boundary between the answers is within 1e-5 "
                    "of the threshold; tile mass 1e-3 rel; out 2e-3 abs"}


# Arm CPU part numbers (implementer 0x41) of the cores this runs on, for a readable name.
_ARM_PARTS = {0xD0C: "Arm Neoverse-N1", 0xD40: "Arm Neoverse-V1", 0xD49: "Arm Neoverse-N2",
              0xD4F: "Arm Neoverse-V2", 0xD8E: "Arm Neoverse-N3", 0xD84: "Arm Neoverse-V3"}


def _cpu_name():
    """Model name of the host CPU: /proc/cpuinfo's "model name" on x86; on Arm, where
    cpuinfo only lists part numbers, the part's name with its number."""
    try:
        part = impl = None
        for line in open("/proc/cpuinfo"):
            key, _, val = line.partition(":")
            key, val = key.strip().lower(), val.strip()
            if key == "model name":
                return val
            if key == "cpu part" and part is None:
                part = val
            if key == "cpu implementer" and impl is None:
                impl = val
        if part is not None:
            name = _ARM_PARTS.get(int(part, 16)) if impl in (None, "0x41") else None
            return f"{name} (part {part})" if name else f"cpu part {part}"
    except (OSError, ValueError):
        pass
    return os.uname().machine


def run_reference(args):
    """Reference arm: the oracle on the host cores; one step = one query head."""
    import oracle
    from synthetic import generate, get_workload

    w = get_workload(args.workload)
    if args.S:
        w = w.with_(S=args.S)
    elif args.mode == "flash" and args.workload.startswith("llama8b"):
        w = w.with_(S=2048)
    inp = generate(w)
    oracle.build()
    kv = _oracle_problem(inp)
    heads = [(b, h) for b in range(w.batch) for h in range(w.num_q_heads)]
    for i in range(args.warmup):
        _oracle_head(oracle, inp, kv, args.mode, w.S, *heads[i % len(heads)])
    t0 = time.perf_counter()
    for i in range(args.steps):
        _oracle_head(oracle, inp, kv, args.mode, w.S, *heads[i % len(heads)])
    el = time.perf_counter() - t0
    per_head_us = el * 1e6 / args.steps
    value = per_head_us * len(heads)
    return {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el * 1000 / args.steps, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "mode": args.mode, "batch": w.batch, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "n_k": int(inp.lengths.max()),
                   "tile": w.tile, "S": w.S, "kv_dtype": w.dtype},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"each step one query head of {w.name} ({args.mode}); value scaled by the "
                                   f"{len(heads)} heads of a layer-step", "cpu": _cpu_name()},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    if args.profile:
        print(json.dumps(run_profile(args)), flush=True)
        return 0
    dist = Dist()
    if args.gpus != dist.world and dist.world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {dist.world}")
    res = run_ours(args, dist)
    if dist.rank == 0:
        print(json.dumps(res), flush=True)
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
