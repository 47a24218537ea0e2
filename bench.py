"""Benchmark: the W4A16 decode round on one GB300 (or N independent replicas).

A step is one decode round: 64 layers x the four linears of a 27B-class
decode layer (qkv 5120->8192, o 6144->5120, gate+up 5120->34816, down
17408->5120), group 128, M = 4 tokens (1 + 3 drafted tokens of a speculative
verify pass), back to back on one stream.  Weights are ~11.4 GB per round, far
larger than L2, so every step streams them from HBM.

Printed (one JSON line on rank 0):
  value         algorithmic GB/s of the round (packed nibbles + fp16 scales +
                4-bit zeros + x + y, GB = 1e9 B), whole job (sum over ranks)
  ms_per_step   milliseconds per round
  roofline      the dominant kernel: algorithmic bytes per launch / its mean
                CUDA-event duration, against the measured HBM copy bandwidth
  e2e           the same round through the C ABI with host buffers, each step:
                x copied in from pinned memory, and every y written by the
                kernels straight into pinned host memory (one captured round)
  cpu_baseline  the oracle on the host cores, on a bounded sample of the round
  extra         single-linear numbers for the M = 1 / 4 / 8 shapes and the
                M sweep (L2 flushed between timed launches)

--impl reference times the oracle itself (the reference arm) on a bounded
sample of the same round, on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("W4A16 linear HBM GB/s (% of GB300 peak) at M=1/4/8; 64-layer decode-round ms")
ROUND_SHAPES = [("qkv", 5120, 8192), ("o", 6144, 5120), ("gate_up", 5120, 34816),
                ("down", 17408, 5120)]  # (name, K, N)
N_LAYERS = 64
M_ROUND = 4
GROUP = 128
WORKLOAD = ("decode round: 64 layers x {qkv 5120x8192, o 6144x5120, gate+up 5120x34816, "
            "down 17408x5120} (KxN), M=4, group 128, int4 weights + fp16 scales + u4 zeros, "
            "fp16 activations")


def linear_bytes(M: int, N: int, K: int) -> int:
    """Algorithmic bytes of one linear: what the method must move, once."""
    G = K // GROUP
    return N * K // 2 + 2 * N * G + N * G // 2 + 2 * M * K + 2 * M * N


def round_bytes(M: int | None = None, layers: int = N_LAYERS) -> int:
    M = M_ROUND if M is None else M
    return layers * sum(linear_bytes(M, N, K) for _, K, N in ROUND_SHAPES)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, log_dir: str | None = None):
        """Samples go to clocks_rank<index>.csv in log_dir (default: the
        system's temporary directory)."""
        import tempfile
        self.index = index
        self.proc = None
        self.path = os.path.join(log_dir or tempfile.gettempdir(), f"clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# workload construction
# ---------------------------------------------------------------------------
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the fused 64-layer round kernel, from one ncu capture of the current kernel;
# None once the kernel changes.
ROUND_KERNEL_TRAFFIC = 11_405_690_112


def build_round(dev, M=None, layers=N_LAYERS):
    """The round's linears.  The four inputs are views of one device buffer and
    the 256 outputs views of another (one copy each way per end-to-end step);
    each linear's x and y stay separate tensors to the library."""
    import synthetic_inputs as si
    M = M_ROUND if M is None else M
    xs = [si.x(si.config_seed(3, 0, 8 + j), M, K) for j, (_, K, _) in enumerate(ROUND_SHAPES)]
    x_all = torch.cat([x.reshape(-1) for x in xs]).to(dev)
    xs_dev, off = [], 0
    for x in xs:
        xs_dev.append(x_all[off:off + x.numel()].view(x.shape))
        off += x.numel()
    y_all = torch.empty(layers * sum(M * N for _, _, N in ROUND_SHAPES), dtype=torch.float16,
                        device=dev)
    lin, off = [], 0
    for l in range(layers):
        for j, (name, K, N) in enumerate(ROUND_SHAPES):
            qw, s, zw = si.layer(si.config_seed(3, l, j), N, K, device=dev)
            y = y_all[off:off + M * N].view(M, N)
            off += M * N
            lin.append(dict(name=name, x=xs_dev[j], qweight=qw, scales=s, zeros=zw, y=y, N=N, K=K,
                            j=j, x_all=x_all, y_all=y_all))
    return lin, xs, xs_dev


def time_round(w4, descs, steps, warmup, stream, M=None):
    M = M_ROUND if M is None else M
    for _ in range(warmup):
        w4.w4a16_decode_round(descs, M, stream=stream)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        w4.w4a16_decode_round(descs, M, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1) / 1e3


def round_at(w4, lin, M, dev):
    """The same round's weights with x [M, K] and y [M, N] buffers of their own
    (x drawn from the same seeds as the M = 4 round's)."""
    import synthetic_inputs as si
    xs = {j: si.x(si.config_seed(3, 0, 8 + j), M, K).to(dev)
          for j, (_, K, _) in enumerate(ROUND_SHAPES)}
    out = []
    for L in lin:
        out.append(dict(x=xs[L["j"]], qweight=L["qweight"], scales=L["scales"], zeros=L["zeros"],
                        y=torch.empty((M, L["N"]), dtype=torch.float16, device=dev)))
    return out


def time_rounds_at(w4, lin, dev, stream, steps, warmup, peak, layers, Ms=(1, 8)):
    """The decode round at other token counts (the ends of the verify range):
    ms per round over `steps` back-to-back rounds, GB/s of the round's
    algorithmic bytes at that M, the fraction of the measured HBM copy rate,
    and the mean per-launch CUDA-event time of the fused kernel."""
    out = {}
    for M in Ms:
        rl = round_at(w4, lin, M, dev)
        d = w4.make_descs(rl)
        w4.w4a16_probe_reset()
        t = time_round(w4, d, steps, warmup, stream, M=M)
        launches = w4.w4a16_kernel_launches() // (steps + warmup)
        evs = []
        for _ in range(4):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            w4.w4a16_decode_round(d, M, stream=stream)
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        t_l = float(np.mean([a.elapsed_time(b) for a, b in evs])) / 1e3
        by = round_bytes(M, layers)
        out[f"M{M}"] = {"ms_per_round": t / steps * 1e3, "GBps": by / (t / steps) / 1e9,
                        "frac_of_peak": by / (t / steps) / 1e9 / peak,
                        "mean_launch_us": t_l * 1e6,
                        "launch_frac_of_peak": by / t_l / 1e9 / peak,
                        "launches_per_round": int(launches), "round_bytes": by}
        del rl, d
    return out


def per_kernel_durations(w4, lin, steps, stream):
    """Each linear launched alone with CUDA events around it, on the launching
    stream; returns {rung: (launches, seconds, algorithmic bytes)}."""
    stats = {}
    evs = []
    for _ in range(steps):
        for L in lin:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            w4.w4a16_linear(L["x"], L["qweight"], L["scales"], L["zeros"], y=L["y"], stream=stream)
            b.record(stream)
            evs.append((L, a, b))
    torch.cuda.synchronize()
    for L, a, b in evs:
        rung = w4.w4a16_select_rung(M_ROUND, L["N"], L["K"])
        n, t, by = stats.get(rung, (0, 0.0, 0))
        stats[rung] = (n + 1, t + a.elapsed_time(b) / 1e3, by + linear_bytes(M_ROUND, L["N"], L["K"]))
    return stats


def time_e2e(w4, lin, xs, steps, warmup, stream, parts=1, host_y=True):
    """x from pinned host memory in, decode round, every y on the host, waited
    for every step.  host_y: the round's descriptors point y at pinned host
    memory, so the kernels store every output there themselves (no copy
    back), and the round is one captured launch.  Otherwise each y goes back
    by copy: with parts > 1 the round runs as that many captured rounds over
    consecutive layers, and each part's outputs (final once its round ends)
    go back on a second stream while the next part runs; the step still ends
    only when every output is on the host."""
    x_all, y_all = lin[0]["x_all"], lin[0]["y_all"]
    pinned_x = torch.cat([x.reshape(-1) for x in xs]).pin_memory()
    pinned_y = torch.empty(y_all.shape, dtype=torch.float16).pin_memory()
    h2d = pinned_x.numel() * 2
    d2h = pinned_y.numel() * 2
    if host_y:
        layers = []
        for L in lin:
            off = (L["y"].data_ptr() - y_all.data_ptr()) // 2
            layers.append(dict(L, y=pinned_y[off:off + L["y"].numel()].view(L["y"].shape)))
        g = w4.RoundGraph(w4.make_descs(layers), M_ROUND)

        def step():
            x_all.copy_(pinned_x, non_blocking=True)
            g.launch(stream)
            stream.synchronize()
    else:
        # the linears of each part, and the span of y_all their outputs fill
        # (several parts: each a captured round with descriptors of its own,
        # so that no call re-uploads descriptors the previous part replaced)
        per = (len(lin) + parts - 1) // parts
        chunks = []
        for i in range(0, len(lin), per):
            group = lin[i:i + per]
            lo = group[0]["y"].data_ptr() - y_all.data_ptr()
            hi = group[-1]["y"].data_ptr() + group[-1]["y"].numel() * 2 - y_all.data_ptr()
            descs = w4.make_descs(group)
            run = (w4.RoundGraph(descs, M_ROUND).launch if parts > 1 else
                   (lambda d=descs, st=stream: w4.w4a16_decode_round(d, M_ROUND, stream=st)))
            chunks.append((run, lo // 2, hi // 2))
        copier = torch.cuda.Stream(device=y_all.device)
        done = [torch.cuda.Event() for _ in chunks]

        def step():
            x_all.copy_(pinned_x, non_blocking=True)
            for (run, lo, hi), ev in zip(chunks, done):
                run(stream) if parts > 1 else run()
                ev.record(stream)
                copier.wait_event(ev)
                with torch.cuda.stream(copier):
                    pinned_y[lo:hi].copy_(y_all[lo:hi], non_blocking=True)
            copier.synchronize()
            stream.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            step()
        t1 = time.perf_counter()
    if host_y:
        g.destroy()
        # the host copy holds what the same round writes into device memory
        # (run once more: the per-linear launches since then split K differently)
        w4.w4a16_decode_round(w4.make_descs(lin), M_ROUND, stream=stream)
        torch.cuda.synchronize()
        if not torch.equal(pinned_y.view(torch.int16), y_all.cpu().view(torch.int16)):
            raise RuntimeError("outputs written to host memory differ from the device round's")
    return (t1 - t0), h2d, d2h


def job_rate(elapsed_s: float, bytes_per_step: int, steps: int, world: int, device=None):
    """Whole-job GB/s of `world` replicas that each moved bytes_per_step * steps:
    the job's time is the slowest rank's (max over ranks, one all-reduce when
    world > 1).  Returns (GB/s, that time)."""
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_s = float(t.item())
    return bytes_per_step * steps * world / elapsed_s / 1e9, elapsed_s


def flush_l2(buf):
    # read-only sweep of a buffer larger than L2: evicts the weights without
    # leaving dirty lines whose write-back would slow the timed kernel
    buf.sum()


def epilogue_bytes(M: int, N: int, K: int, epi: int) -> int:
    """Algorithmic bytes of a linear with an epilogue: y has N/2 columns after
    SiLU-and-mul; the residual add reads M x N fp16 more."""
    if epi == 2:
        return linear_bytes(M, N, K) - M * N
    if epi == 1:
        return linear_bytes(M, N, K) + 2 * M * N
    return linear_bytes(M, N, K)


def time_single(w4, M, N, K, seed_cfg, dev, reps=50, flush=None, rungs=(-1,), epi=0, spread=None,
                warmup=10):
    """Median single-launch time of one linear (with epilogue `epi`) with L2
    flushed before each launch, per rung (-1 = the dispatch table's choice);
    None where a rung cannot run the shape.  After `warmup` launches per rung,
    the rungs take turns launch by launch (A/B alternated, not one after the
    other).  `spread`, a dict, receives each rung's (p10, p90) times."""
    import synthetic_inputs as si
    seed = si.config_seed(seed_cfg, 0, M)
    qw, s, zw = si.layer(seed, N, K, device=dev)
    x = si.x(seed, M, K).to(dev)
    y = torch.empty((M, N // 2 if epi == 2 else N), dtype=torch.float16, device=dev)
    res = si.residual(seed, M, N).to(dev) if epi == 1 else None

    def call():
        if epi:
            w4.w4a16_linear_epilogue(x, qw, s, zw, epi, residual=res, y=y)
        else:
            w4.w4a16_linear(x, qw, s, zw, y=y)
    out, runnable, events = {}, [], {}
    prev = w4.w4a16_set_forced_rung(-1)
    try:
        for rung in rungs:
            w4.w4a16_set_forced_rung(rung)
            try:
                for _ in range(warmup):
                    call()
            except w4.W4A16Error:
                out[rung] = None
                continue
            runnable.append(rung)
            events[rung] = []
        for _ in range(reps):
            for rung in runnable:
                w4.w4a16_set_forced_rung(rung)
                flush_l2(flush)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record()
                call()
                b.record()
                events[rung].append((a, b))
        torch.cuda.synchronize()
    finally:
        w4.w4a16_set_forced_rung(prev)
    for rung in runnable:
        times = np.array([a.elapsed_time(b) for a, b in events[rung]]) / 1e3
        out[rung] = float(np.median(times))
        if spread is not None:
            spread[rung] = (float(np.percentile(times, 10)), float(np.percentile(times, 90)))
    del qw, s, zw
    return out


def time_repack(w4, dev, flush, peak, reps=10):
    """Load-time repack of a gate+up checkpoint stored transposed (qweight
    [5120, 34816/8] packed along N): median time with L2 evicted, and GB/s
    of bytes read + written."""
    import synthetic_inputs as si
    K, N = 5120, 34816
    src = si.qweight(si.config_seed(6), K, N, device=dev)
    dst = torch.empty((N, K // 8), dtype=torch.int32, device=dev)
    for _ in range(3):
        w4.w4a16_repack_transpose(src, K, N, dst=dst)
    ts = []
    for _ in range(reps):
        flush_l2(flush)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        w4.w4a16_repack_transpose(src, K, N, dst=dst)
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    t = float(np.median([a.elapsed_time(b) for a, b in ts])) / 1e3
    by = 2 * src.numel() * 4
    return {"rows": K, "cols": N, "us": t * 1e6, "GBps": by / t / 1e9,
            "frac_of_peak": by / t / 1e9 / peak}


def time_dense(w4, dev, flush, peak, reps=20):
    """The dense 16-bit linear on the pages' shape (N 8192, K 5120, M 2/4/8) and
    on a gate+up-sized layer (N 34816): median single launch, L2 evicted."""
    import synthetic_inputs as si
    out = {}
    for N, K in ((8192, 5120), (34816, 5120)):
        qw, s, zw = si.layer(si.config_seed(7), N, K, device=dev)
        _, w16 = w4.w4a16_dequant(qw, s, zw, K, f32=False)  # seeded weights made on the device
        del qw, s, zw
        for dt in (torch.float16, torch.bfloat16):
            w = w16 if dt == torch.float16 else w16.to(dt)
            for M in (1, 2, 4, 8):
                x = si.x(si.config_seed(7, 0, M), M, K).to(dev).to(dt)
                y = torch.empty((M, N), dtype=dt, device=dev)
                for _ in range(3):
                    w4.w4a16_dense_linear(x, w, y=y)
                ts = []
                for _ in range(reps):
                    flush_l2(flush)
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record()
                    w4.w4a16_dense_linear(x, w, y=y)
                    b.record()
                    ts.append((a, b))
                torch.cuda.synchronize()
                t = float(np.median([a.elapsed_time(b) for a, b in ts])) / 1e3
                by = 2 * N * K + 2 * M * K + 2 * M * N
                out[f"{'bf16' if dt == torch.bfloat16 else 'f16'}_M{M}_K{K}_N{N}"] = {
                    "us": t * 1e6, "GBps": by / t / 1e9, "frac_of_peak": by / t / 1e9 / peak}
            del w
        del w16
    return out


def time_moe(w4, dev, peak, reps=20):
    """A decode-time expert MLP of a Qwen3-MoE-like shape (E 128, top 8,
    hidden 2048, intermediate 768) with L2 evicted: w4a16_moe_mlp on its
    decode path (one launch: routing, gate+up with SiLU-and-mul, down, the
    weighted sum), on its chain path (align, prepare, one expert-MMA launch for
    both linears, the weighted sum), and the chain call by call; GB/s counts
    the weights of the experts in use."""
    import synthetic_inputs as si
    E, k, H, I = 128, 8, 2048, 768
    parts_g = [si.layer(si.config_seed(8, e, 0), 2 * I, H, device=dev) for e in range(E)]
    parts_d = [si.layer(si.config_seed(8, e, 1), H, I, device=dev) for e in range(E)]
    g = [torch.stack([p[i] for p in parts_g]) for i in range(3)]
    d = [torch.stack([p[i] for p in parts_d]) for i in range(3)]
    del parts_g, parts_d
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)
    out = {}
    for T in (1, 4, 8):
        rng = np.random.default_rng(T)
        ids = torch.from_numpy(np.stack([rng.permutation(E)[:k] for _ in range(T)])
                               .astype(np.int32)).to(dev)
        wts = torch.full((T, k), 1.0 / k, dtype=torch.float32, device=dev)
        x = si.x(si.config_seed(8, 0, 9), T, H).to(dev)
        gu = w4.MoeExperts(*g, epilogue=w4.EPILOGUE_SILU_MUL, max_slots=T * k)
        dn = w4.MoeExperts(*d, max_slots=T * k)
        mlp = w4.MoeMlp(gu, dn, T, k)
        y = torch.empty((T, H), dtype=torch.float16, device=dev)

        def chain():
            srt, pos, off = w4.w4a16_moe_align(ids, E)
            h = gu.linear(x, srt, off, T * k, gather_k=k)
            o = dn.linear(h, srt, off, T * k, gather_k=0)
            return w4.w4a16_moe_sum(o, pos, wts)

        def one():
            return mlp(x, ids, wts, out=y)

        def one_chain():
            mlp.set_path(w4.MOE_PATH_CHAIN)
            r = mlp(x, ids, wts, out=y)
            mlp.set_path(w4.MOE_PATH_AUTO)
            return r

        def timed(step):
            for _ in range(3):
                step()
            ts = []
            for _ in range(reps):
                flush_l2(flush)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record()
                step()
                b.record()
                ts.append((a, b))
            torch.cuda.synchronize()
            return float(np.median([a.elapsed_time(b) for a, b in ts])) / 1e3
        t = timed(one)
        t_mlp_chain = timed(one_chain)
        t_chain = timed(chain)
        used = len(set(ids.cpu().numpy().reshape(-1).tolist()))
        by = used * (linear_bytes(0, 2 * I, H) + linear_bytes(0, H, I))
        out[f"T{T}"] = {"experts_used": used, "path": "decode" if mlp.path(T) == w4.MOE_PATH_DECODE
                        else "chain", "us": t * 1e6, "GBps": by / t / 1e9,
                        "frac_of_peak": by / t / 1e9 / peak, "us_chain_path": t_mlp_chain * 1e6,
                        "us_call_by_call": t_chain * 1e6}
        mlp.destroy()
        gu.destroy()
        dn.destroy()
    return out


_LAYER0 = None


def _layer0_host():
    """Layer 0 of the decode round on the host (oracle arrays), built once."""
    global _LAYER0
    if _LAYER0 is None:
        import synthetic_inputs as si
        out = []
        for j, (_, K, N) in enumerate(ROUND_SHAPES):
            qw, s, zw = si.layer(si.config_seed(3, 0, j), N, K)
            x = si.x(si.config_seed(3, 0, 8 + j), M_ROUND, K)
            out.append((si.as_u16(x), si.as_u32(qw), si.as_u16(s), si.as_u32(zw),
                        linear_bytes(M_ROUND, N, K)))
        _LAYER0 = out
    return _LAYER0


def cpu_model() -> str:
    """The host CPU's model name (or its implementer / part on Arm)."""
    try:
        fields = {}
        for line in open("/proc/cpuinfo"):
            if ":" in line:
                k, v = line.split(":", 1)
                fields.setdefault(k.strip(), v.strip())
        for k in ("model name", "Model"):
            if k in fields:
                return fields[k]
        return f"implementer {fields.get('CPU implementer', '?')} part {fields.get('CPU part', '?')}"
    except OSError:
        return "unknown"


def cpu_baseline(seconds_target: float = 12.0):
    """The oracle, as it stands, on all host cores, over a bounded sample of the
    decode round: layer 0's four linears (all rows, M = 4), passed over
    repeatedly until about `seconds_target` seconds have elapsed."""
    import oracle
    cores = os.cpu_count() or 1
    layer = _layer0_host()
    t_total, by_total, passes = 0.0, 0, 0
    while t_total < seconds_target or passes == 0:
        for x, qw, s, zw, nbytes in layer:
            t0 = time.perf_counter()
            oracle.linear(x, qw, s, zw, nthreads=cores)
            t_total += time.perf_counter() - t0
            by_total += nbytes
        passes += 1
    gbs = by_total / t_total / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"layer 0 of the decode round (qkv, o, gate+up, down; "
                      f"{by_total / passes / 1e6:.0f} MB) at M=4, {passes} passes, "
                      f"{t_total:.1f} s on {cores} threads; a full 64-layer round would take "
                      f"{round_bytes() / (gbs * 1e9):.0f} s",
            "seconds": t_total}


ORACLE_CONFIGS = ([("cfg0_M1_K512_N1024", 1, 1024, 512, 0), ("cfg1_M1_K5120_N34816", 1, 34816, 5120, 1),
                   ("cfg2_M4_K17408_N5120", 4, 5120, 17408, 2),
                   ("cfg2_M8_K17408_N5120", 8, 5120, 17408, 2)] +
                  [(f"cfg4_M{m}_K5120_N27648", m, 27648, 5120, 4) for m in (1, 2, 4, 8, 16, 32, 64)])


def oracle_legs(cores: int):
    """The oracle, as it stands, on every single-linear workload in full (all
    outputs), on `cores` host threads, and once more on one thread for the
    M = 1 gate+up shape: milliseconds and GB/s of the linear's algorithmic
    bytes."""
    import oracle
    import synthetic_inputs as si
    out = {}
    cache = {}
    for label, M, N, K, cfg in ORACLE_CONFIGS:
        if (N, K, cfg) not in cache:
            cache.clear()
            qw, sc, zw = si.layer(si.config_seed(cfg, 0, M), N, K)
            cache[(N, K, cfg)] = (si.as_u32(qw), si.as_u16(sc), si.as_u32(zw))
        qw, sc, zw = cache[(N, K, cfg)]
        x = si.as_u16(si.x(si.config_seed(cfg, 0, M), M, K))
        by = linear_bytes(M, N, K)
        runs = [(label, cores)] + ([(label + "_1thread", 1)] if cfg == 1 else [])
        for name, nt in runs:
            t0 = time.perf_counter()
            oracle.linear(x, qw, sc, zw, nthreads=nt)
            t = time.perf_counter() - t0
            out[name] = {"ms": t * 1e3, "GBps": by / t / 1e9, "threads": nt}
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    secs = []
    vals = []
    base = None
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(seconds_target=6.0 if i >= args.warmup else 1.0)
        if i >= args.warmup:
            vals.append(cb["value"])
            secs.append(cb["seconds"])
            base = cb
    value = float(np.median(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            # a full round on the host cores would take minutes: each step
            # times a sample (layer 0's four linears, passed over for about
            # 6 s), and ms_per_step is a full round's bytes at that rate
            "ms_per_step": round_bytes() / (value * 1e9) * 1e3,
            "ms_per_step_extrapolated_from_sample": True,
            "sample_seconds_per_step": float(np.median(secs)), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": base["sample"]},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": base["cores"],
                             "kind": "oracle", "sample": base["sample"]},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_case(M: int, N: int, K: int, rung: int, reps: int):
    """One seeded linear launched `reps` times (the target of ncu captures)."""
    import __graft_entry__
    __graft_entry__.build()
    import synthetic_inputs as si
    import weight_only_int4_w4a16_gb300 as w4
    dev = torch.device("cuda:0")
    w4.w4a16_init(0, 512 << 20)
    qw, s, zw = si.layer(si.config_seed(1), N, K, device=dev)
    x = si.x(si.config_seed(1), M, K).to(dev)
    y = torch.empty((M, N), dtype=torch.float16, device=dev)
    w4.w4a16_set_forced_rung(rung)
    for _ in range(reps):
        w4.w4a16_linear(x, qw, s, zw, y=y)
    torch.cuda.synchronize()
    status = w4.w4a16_device_status()
    print(f"case M={M} N={N} K={K} rung={w4.rung_name(w4.w4a16_select_rung(M, N, K))} "
          f"reps={reps} device_status={status}")
    if status:
        raise SystemExit(1)


def run_dense_case(M: int, N: int, K: int, reps: int):
    """One dense 16-bit linear (fp16 weights made on the device from a seeded
    4-bit layer) launched `reps` times: the target of ncu captures."""
    import __graft_entry__
    __graft_entry__.build()
    import synthetic_inputs as si
    import weight_only_int4_w4a16_gb300 as w4
    dev = torch.device("cuda:0")
    w4.w4a16_init(0, 512 << 20)
    qw, s, zw = si.layer(si.config_seed(1), N, K, device=dev)
    _, w = w4.w4a16_dequant(qw, s, zw, K, f32=False)
    del qw, s, zw
    x = si.x(si.config_seed(1), M, K).to(dev)
    y = torch.empty((M, N), dtype=torch.float16, device=dev)
    for _ in range(reps):
        w4.w4a16_dense_linear(x, w, y=y)
    torch.cuda.synchronize()
    status = w4.w4a16_device_status()
    print(f"dense case M={M} N={N} K={K} reps={reps} device_status={status}")
    if status:
        raise SystemExit(1)


def run_round_case(dtype: str, layers: int, reps: int, M: int):
    """The bench's decode round (its shapes, `layers` layers, M tokens) with
    fp16 or bf16 activations and scales, `reps` rounds on one stream: the
    target of ncu captures."""
    import __graft_entry__
    __graft_entry__.build()
    import weight_only_int4_w4a16_gb300 as w4
    dev = torch.device("cuda:0")
    w4.w4a16_init(0, 512 << 20)
    lin, _, _ = build_round(dev, M=M, layers=layers)
    if dtype == "bf16":
        bxs = {id(L["x"]): L["x"].to(torch.bfloat16) for L in lin}
        lin = [dict(x=bxs[id(L["x"])], qweight=L["qweight"], zeros=L["zeros"],
                    scales=L["scales"].to(torch.bfloat16),
                    y=torch.empty_like(L["y"], dtype=torch.bfloat16)) for L in lin]
    descs = w4.make_descs(lin)
    for _ in range(reps):
        w4.w4a16_decode_round(descs, M)
    torch.cuda.synchronize()
    status = w4.w4a16_device_status()
    print(f"round case dtype={dtype} layers={layers} M={M} reps={reps} device_status={status}")
    if status:
        raise SystemExit(1)


def run_moe_case(T: int, reps: int):
    """The expert MLP of the bench's MoE entry (E 128, top 8, hidden 2048,
    intermediate 768) for T tokens on its default path, `reps` calls: the
    target of ncu captures."""
    import __graft_entry__
    __graft_entry__.build()
    import synthetic_inputs as si
    import weight_only_int4_w4a16_gb300 as w4
    dev = torch.device("cuda:0")
    w4.w4a16_init(0, 512 << 20)
    E, k, H, I = 128, 8, 2048, 768
    parts_g = [si.layer(si.config_seed(8, e, 0), 2 * I, H, device=dev) for e in range(E)]
    parts_d = [si.layer(si.config_seed(8, e, 1), H, I, device=dev) for e in range(E)]
    g = [torch.stack([p[i] for p in parts_g]) for i in range(3)]
    d = [torch.stack([p[i] for p in parts_d]) for i in range(3)]
    del parts_g, parts_d
    rng = np.random.default_rng(T)
    ids = torch.from_numpy(np.stack([rng.permutation(E)[:k] for _ in range(T)])
                           .astype(np.int32)).to(dev)
    wts = torch.full((T, k), 1.0 / k, dtype=torch.float32, device=dev)
    x = si.x(si.config_seed(8, 0, 9), T, H).to(dev)
    gu = w4.MoeExperts(*g, epilogue=w4.EPILOGUE_SILU_MUL, max_slots=T * k)
    dn = w4.MoeExperts(*d, max_slots=T * k)
    mlp = w4.MoeMlp(gu, dn, T, k)
    y = torch.empty((T, H), dtype=torch.float16, device=dev)
    for _ in range(reps):
        mlp(x, ids, wts, out=y)
    torch.cuda.synchronize()
    status = w4.w4a16_device_status()
    path = "decode" if mlp.path(T) == w4.MOE_PATH_DECODE else "chain"
    mlp.destroy()
    gu.destroy()
    dn.destroy()
    print(f"moe case T={T} path={path} reps={reps} device_status={status}")
    if status:
        raise SystemExit(1)


def main():
    global M_ROUND
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=N_LAYERS)
    ap.add_argument("--round-m", type=int, default=M_ROUND,
                    help="tokens of the timed round (the benchmark's workload is M=4; other values "
                         "are for profiling)")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--case", type=int, nargs=5, metavar=("M", "N", "K", "RUNG", "REPS"),
                    help="profiling helper: run one seeded linear REPS times on a forced rung "
                         "(-1 = dispatch table) and exit; prints no benchmark line")
    ap.add_argument("--clocks-dir", default=None,
                    help="where to keep the nvidia-smi samples of the timed region")
    ap.add_argument("--moe-case", type=int, nargs=2, metavar=("T", "REPS"),
                    help="run the expert MLP for T tokens REPS times and exit (for ncu)")
    ap.add_argument("--dense-case", type=int, nargs=4, metavar=("M", "N", "K", "REPS"),
                    help="profiling helper: run one dense fp16 linear REPS times and exit")
    ap.add_argument("--round-case", nargs=3, metavar=("DTYPE", "LAYERS", "REPS"),
                    help="profiling helper: run the decode round (f16 or bf16, at --round-m "
                         "tokens) REPS times and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.case:
        run_case(*args.case)
        return
    if args.moe_case:
        run_moe_case(*args.moe_case)
        return
    if args.dense_case:
        run_dense_case(*args.dense_case)
        return
    if args.round_case:
        dt, nl, reps = args.round_case
        if dt not in ("f16", "bf16"):
            raise SystemExit("--round-case DTYPE is f16 or bf16")
        run_round_case(dt, int(nl), int(reps), args.round_m)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    M_ROUND = args.round_m

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import weight_only_int4_w4a16_gb300 as w4
    w4.w4a16_init(local, 512 << 20)

    stream = torch.cuda.Stream(device=dev)
    lin, xs, _ = build_round(dev, layers=args.layers)
    descs = w4.make_descs(lin)
    torch.cuda.synchronize()

    # ---- timed region: K decode rounds --------------------------------------
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local, args.clocks_dir)
    clocks.start()
    w4.w4a16_probe_reset()
    for _ in range(args.warmup):
        w4.w4a16_decode_round(descs, M_ROUND, stream=stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches0 = w4.w4a16_kernel_launches()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        w4.w4a16_decode_round(descs, M_ROUND, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    launches1 = w4.w4a16_kernel_launches()
    elapsed = ev0.elapsed_time(ev1) / 1e3
    clk = clocks.stop()
    launches = int(launches1 - launches0)
    # the rungs that ran (the library's per-rung counters) must be the ones
    # the dispatch table names for the round's shapes
    expect = [0] * w4.NUM_RUNGS
    for L in lin:
        expect[w4.w4a16_select_rung(M_ROUND, L["N"], L["K"])] += args.warmup + args.steps
    ran = w4.w4a16_probe_counts()
    if ran != expect:
        raise SystemExit(f"the round ran rungs {ran}, the dispatch table names {expect}")
    rungs_ran = {w4.rung_name(r): n for r, n in enumerate(ran) if n}

    rb = round_bytes(layers=args.layers)
    value, elapsed = job_rate(elapsed, rb, args.steps, world, dev)
    ms = elapsed / args.steps * 1e3
    peak, peak_kind = load_peaks()

    # ---- dominant kernel, timed launch by launch on the same stream ---------
    # A round of mma-rung linears is one launch of the fused round kernel:
    # CUDA events around each launch on the launching stream.
    per_round = launches // max(1, args.steps)
    n_l = max(3, min(args.steps, 8))
    evs = []
    for _ in range(n_l):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        w4.w4a16_decode_round(descs, M_ROUND, stream=stream)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    t_l = sum(a.elapsed_time(b) for a, b in evs) / 1e3
    achieved = rb / (t_l / n_l) / 1e9
    roofline = {"bound": "hbm",
                "kernel": ("mma_kernel (fused decode round, one launch per round)"
                           if per_round == 1 else f"decode round ({per_round} launches)"),
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy)",
                "traffic": (ROUND_KERNEL_TRAFFIC if per_round == 1 and args.layers == N_LAYERS
                            and M_ROUND == 4
                            else None), "launches_timed": n_l,
                "mean_launch_us": t_l / n_l * 1e6,
                "mean_algorithmic_bytes_per_launch": rb}
    # each linear launched alone (its own kernel), for the per-shape picture
    stats = per_kernel_durations(w4, lin, 2, stream)
    per_linear = {w4.rung_name(r): {"launches": n, "mean_us": t / n * 1e6,
                                    "GBps": by / t / 1e9}
                  for r, (n, t, by) in stats.items()}

    # ---- end to end through the C ABI with host buffers ----------------------
    # the kernels write every y into pinned host memory (measured: 1.97 ms
    # against 2.12 ms for the best copy-back schedule, two parts with the
    # first half's outputs copied back while the second half runs)
    e2e_steps = max(3, args.steps // 2)
    e2e_s, h2d, d2h = time_e2e(w4, lin, xs, e2e_steps, 2, stream)
    e2e_value, e2e_s = job_rate(e2e_s, rb, e2e_steps, world, dev)
    e2e = {"value": e2e_value, "unit": "GB/s",
           "ms_per_step": e2e_s / e2e_steps * 1e3, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h,
           "d2h_by": "the round's kernels store every y into pinned host memory"}
    cb_s, _, _ = time_e2e(w4, lin, xs, e2e_steps, 2, stream, parts=2, host_y=False)
    e2e["copy_back_ms_per_step"] = cb_s / e2e_steps * 1e3

    # ---- graph replay of the same round --------------------------------------
    g = w4.RoundGraph(descs, M_ROUND)
    for _ in range(2):
        g.launch(stream)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        g.launch(stream)
    b.record(stream)
    torch.cuda.synchronize()
    graph_ms = a.elapsed_time(b) / args.steps
    g.destroy()

    # the same round as 256 launches back to back (one w4a16_linear per
    # linear, as a caller without the fused round would run it)
    for L in lin:
        w4.w4a16_linear(L["x"], L["qweight"], L["scales"], L["zeros"], y=L["y"], stream=stream)
    torch.cuda.synchronize()
    n_sep = 3
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n_sep):
        for L in lin:
            w4.w4a16_linear(L["x"], L["qweight"], L["scales"], L["zeros"], y=L["y"], stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    sep_ms = a.elapsed_time(b) / n_sep
    # and those 256 launches captured into one CUDA graph (no host cost per
    # launch; consecutive kernels overlap by programmatic dependent launch)
    sep_graph_ms = None
    try:
        sg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(sg, stream=stream):
            for L in lin:
                w4.w4a16_linear(L["x"], L["qweight"], L["scales"], L["zeros"], y=L["y"],
                                stream=stream)
        with torch.cuda.stream(stream):  # a replay runs on the current stream
            for _ in range(2):
                sg.replay()
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(n_sep):
                sg.replay()
            b.record(stream)
        torch.cuda.synchronize()
        sep_graph_ms = a.elapsed_time(b) / n_sep
        sg.reset()
    except RuntimeError as exc:  # reported, not fatal: the timed round is above
        print(f"[bench] separate-launch graph not measured: {exc}", file=sys.stderr)

    extra = {"round_graph_ms": graph_ms, "round_graph_GBps": rb / (graph_ms / 1e3) / 1e9,
             "round_as_separate_launches_ms": sep_ms,
             "round_as_separate_launches_GBps": rb / (sep_ms / 1e3) / 1e9,
             "round_as_separate_launches_graph_ms": sep_graph_ms,
             "round_bytes": rb, "launches_per_round": per_round,
             "linears_launched_alone": per_linear,
             "rung_per_shape": {n: w4.rung_name(w4.w4a16_select_rung(M_ROUND, N, K))
                                for n, K, N in ROUND_SHAPES},
             "linears_per_rung_in_timed_and_warmup_rounds": rungs_ran}
    if not args.no_extra and rank == 0:
        # the same round with bf16 activations and scales (the same packed
        # weights and zeros; bf16 copies of x and the scales, bf16 outputs)
        bxs = {id(L["x"]): L["x"].to(torch.bfloat16) for L in lin}
        blin = [dict(x=bxs[id(L["x"])], qweight=L["qweight"], zeros=L["zeros"],
                     scales=L["scales"].to(torch.bfloat16),
                     y=torch.empty_like(L["y"], dtype=torch.bfloat16)) for L in lin]
        bdescs = w4.make_descs(blin)
        t = time_round(w4, bdescs, args.steps, args.warmup, stream)
        bms = t / args.steps * 1e3
        extra["round_bf16_ms"] = bms
        extra["round_bf16_GBps"] = rb / (bms / 1e3) / 1e9
        extra["round_bf16_frac_of_peak"] = rb / (bms / 1e3) / 1e9 / peak
        del blin, bdescs, bxs
    rounds = None
    if not args.no_extra and rank == 0:
        # M = 1 and 8 (the mma rungs), 16 and 64 (one tcgen05 launch per round)
        rounds = time_rounds_at(w4, lin, dev, stream, max(10, args.steps // 2), args.warmup, peak,
                                args.layers, Ms=(1, 8, 16, 64))
        rounds["M4"] = {"ms_per_round": ms, "GBps": value / world, "frac_of_peak": value / world / peak,
                        "mean_launch_us": roofline["mean_launch_us"],
                        "launch_frac_of_peak": roofline["frac"], "launches_per_round": per_round,
                        "round_bytes": rb}
    del lin, descs
    torch.cuda.empty_cache()

    if not args.no_extra and rank == 0:
        flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)  # 256 MB > L2
        singles = {}
        for label, M, N, K, cfg in [("cfg0_M1_K512_N1024", 1, 1024, 512, 0),
                                    ("cfg1_M1_K5120_N34816", 1, 34816, 5120, 1),
                                    ("cfg2_M4_K17408_N5120", 4, 5120, 17408, 2),
                                    ("cfg2_M8_K17408_N5120", 8, 5120, 17408, 2)] + \
                [(f"cfg4_M{m}_K5120_N27648", m, 27648, 5120, 4) for m in (1, 2, 4, 8, 16, 32, 64)]:
            spread = {}
            ts = time_single(w4, M, N, K, cfg, dev, flush=flush, rungs=(-1, 0, 1, 2, 3, 4, 5),
                             spread=spread)
            by = linear_bytes(M, N, K)
            t = ts[-1]
            singles[label] = {"us": t * 1e6, "us_p10": spread[-1][0] * 1e6,
                              "us_p90": spread[-1][1] * 1e6,
                              "GBps": by / t / 1e9, "frac_of_peak": by / t / 1e9 / peak,
                              "rung": w4.rung_name(w4.w4a16_select_rung(M, N, K)),
                              "us_per_rung": {w4.rung_name(r): (None if v is None else v * 1e6)
                                              for r, v in ts.items() if r >= 0}}
        extra["single_linear_l2_flushed"] = singles
        # the fused epilogues against the same linear without one
        epis = {}
        for label, M, N, K, epi in [("gate_up_silu_M1_K5120_N34816", 1, 34816, 5120, 2),
                                    ("gate_up_silu_M4_K5120_N34816", 4, 34816, 5120, 2),
                                    ("gate_up_silu_M8_K5120_N34816", 8, 34816, 5120, 2),
                                    ("gate_up_silu_M16_K5120_N34816", 16, 34816, 5120, 2),
                                    ("gate_up_silu_M64_K5120_N34816", 64, 34816, 5120, 2),
                                    ("down_residual_M4_K17408_N5120", 4, 5120, 17408, 1),
                                    ("down_residual_M16_K17408_N5120", 16, 5120, 17408, 1),
                                    ("down_residual_M64_K17408_N5120", 64, 5120, 17408, 1),
                                    ("o_residual_M4_K6144_N5120", 4, 5120, 6144, 1)]:
            t = time_single(w4, M, N, K, 5, dev, flush=flush, epi=epi)[-1]
            t0 = time_single(w4, M, N, K, 5, dev, flush=flush)[-1]
            by = epilogue_bytes(M, N, K, epi)
            epis[label] = {"us": t * 1e6, "GBps": by / t / 1e9, "frac_of_peak": by / t / 1e9 / peak,
                           "us_without_epilogue": t0 * 1e6}
        extra["epilogue_l2_flushed"] = epis
        extra["repack_transpose"] = time_repack(w4, dev, flush, peak)
        extra["dense_linear_l2_flushed"] = time_dense(w4, dev, flush, peak)
        extra["moe_expert_mlp_l2_flushed"] = time_moe(w4, dev, peak)
        del flush

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cb = cpu_baseline()
        cpu = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
        cpu["cpu_model"] = cpu_model()
        cpu["per_config"] = oracle_legs(cb["cores"])

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic",
                "config": {"workload": WORKLOAD, "layers": args.layers, "M": M_ROUND,
                           "l2": "inputs larger than L2: 11.4 GB of weights per step",
                           "percent_of_hbm_peak": 100.0 * value / world / peak,
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
                "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
                "clocks": clk, "cpu_baseline": cpu}
        # the metric's other parts: the round at M = 1, 4, 8 and the lone
        # single linears (L2 evicted) at M = 1 / 4 / 8
        if rounds is not None:
            line["rounds"] = rounds
        if "single_linear_l2_flushed" in extra:
            line["singles"] = {k: {f: v[f] for f in ("us", "GBps", "frac_of_peak", "rung")}
                               for k, v in extra["single_linear_l2_flushed"].items()
                               if k.startswith(("cfg0", "cfg1", "cfg2"))}
        line["extra"] = extra
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
