#!/usr/bin/env python3
"""Benchmark of the fused mHC post+pre step (mhc_shifted_post_pre) on GB300.

One step = one call of the whole op (post, RMS + projection, heads + Sinkhorn,
combine + RMSNorm) over the prefill-chunk workload: T=8192 tokens, H=7168,
hc_mult=4, seeded synthetic inputs already resident in HBM.  Prints one JSON
line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain fp64 C implementation used by
the tests) on the host cores over a bounded token sample of the same workload.
Under torchrun with N > 1 every rank runs an independent replica on its own GPU
(the op has no exchange step: tokens are independent), and value is the total
over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from manifold_constrained_hyper_mhc_gb300 import synth  # noqa: E402

WORKLOAD = "prefill_chunk"
METRIC = "tokens/s and HBM GB/s (% of GB300 peak) for fused mHC post+pre vs T, H"
FALLBACK_HBM_GBS = 6800.0


def algorithmic_bytes(T: int, H: int, mxfp8: bool = False, no_bf16: bool = False) -> int:
    """Bytes the op must move per call: per token R 8H + Y 2H + prev mixes 80 B in,
    R' 8H + layer input 2H + mixes 96 B out; per call phi (fp32 [4H, 24]) 384H + gamma 2H
    + bias and mix scales 108 B.  With the MXFP8 layer input: + H E4M3 bytes and H/32 scale
    bytes per token."""
    b = T * (20 * H + 176) + 384 * H + 2 * H + 108
    if mxfp8:
        b += T * (H + H // 32)
    if no_bf16:
        b -= T * 2 * H
    return b


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def wait_first(self, timeout=3.0):
        """Blocks until the sampler has delivered a row (nvidia-smi takes a moment to start)."""
        t0 = time.time()
        while self.proc is not None and not self.rows and time.time() - t0 < timeout:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        rows = [r for r in self.rows if len(r) >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[0]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.lower() == "active"})
        return {"sm_mhz": float(np.nanmedian(sm)), "sm_max_mhz": num(rows[0][1]), "reasons": reasons,
                "samples": len(rows), "power_w_max": float(np.nanmax([num(r[2]) for r in rows]))}


def measured_traffic(schedule, workload, T, H):
    """DRAM bytes (read + write) per launch of the dominant kernel from the committed ncu
    capture in profiles/, or None when there is none for this schedule and workload or the
    kernel source has changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{schedule.replace('+', '_')}_{workload}_{T}x{H}.traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    # one kernel, or the kernels of the call's main span (ws with the token-tile kernel beside it),
    # each captured alone: the call's traffic is their sum
    total = 0
    for k in rec.get("kernels", [rec]):
        with open(os.path.join(ROOT, k["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != k["sha256"]:
                return None
        total += k["dram_bytes_read"] + k["dram_bytes_write"]
    return total


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0, None
    import torch
    import torch.distributed as dist
    rank, lr = int(os.environ["RANK"]), int(os.environ.get("LOCAL_RANK", "0"))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(lr)
    dist.init_process_group(backend)
    return rank, ws, lr, dist


def max_over_ranks(value, dist, device=None):
    """The largest of the ranks' values (the job's time is its slowest rank's); the value itself
    when there is one process."""
    if dist is None:
        return value
    import torch
    on_dev = device is not None and dist.get_backend() == "nccl"
    t = torch.tensor([value], dtype=torch.float64, device=device if on_dev else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_oracle(w, phi, bias, ms, gamma, n_tokens, min_seconds, t_offset=0):
    """Times the CPU oracle over n_tokens tokens of the workload, repeated until
    min_seconds have passed.  Returns (tokens/s, threads, seconds, tokens)."""
    import oracle
    oracle.build()
    t0 = t_offset % max(1, w.T - n_tokens + 1)
    R, Y, pp, pc = synth.tokens(w, t0, t0 + n_tokens)
    nt = oracle.default_threads()
    done, start = 0, time.perf_counter()
    while True:
        oracle.shifted_post_pre(R, Y, pp, pc, phi, bias, ms, gamma, **synth.scalars(), nthreads=nt)
        done += n_tokens
        el = time.perf_counter() - start
        if el >= min_seconds:
            return done / el, nt, el, done


def run_reference(args, rank, world, dist):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    phi, bias, ms, gamma = synth.weights(w)
    n = min(512, w.T)
    times = []
    for s in range(args.warmup + args.steps):
        tps, nt, el, done = time_oracle(w, phi, bias, ms, gamma, n, 0.0, t_offset=s * n)
        if s >= args.warmup:
            times.append(el)
    ms_step = 1e3 * float(np.mean(times))
    value = n / (ms_step / 1e3)
    sample = f"{n} consecutive tokens of the {w.name} workload (T={w.T}, H={w.H}) per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name} T={w.T} H={w.H} hc_mult=4", "T": w.T, "H": w.H,
                   "tokens_per_step": n},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nt, "kind": "oracle", "sample": sample,
                         "machine": platform.machine()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, lr, dist):
    import torch
    import manifold_constrained_hyper_mhc_gb300 as mhc
    from manifold_constrained_hyper_mhc_gb300 import _build
    _build.build()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    dev = torch.device("cuda", lr if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    if args.tokens:
        w = synth.Workload(f"{w.name}[:{args.tokens}]", args.tokens, w.H, w.seed, w.token_scale, w.special_tokens)
    T, H = w.T, w.H
    if args.schedule != "auto":
        mhc.set_schedule(args.schedule)
    phi, bias, msc, gamma = synth.weights(w)
    R, Y, pp, pc = synth.tokens(w)

    def d_bf16(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    Rd, Yd = d_bf16(R), d_bf16(Y)
    ppd, pcd = torch.from_numpy(pp).to(dev), torch.from_numpy(pc).to(dev)
    wd = (torch.from_numpy(phi).to(dev), torch.from_numpy(bias).to(dev), torch.from_numpy(msc).to(dev),
          d_bf16(gamma))
    sc = synth.scalars()
    ws = mhc.new_workspace(T, H, dev)
    # phi is a weight: packed once (mhc_pack_phi), as at model load, and the fused call and the pre
    # take the packed form (mhc_*_prepacked, bit-identical to the plain calls); --pack-per-call
    # times the plain calls, which pack phi in their workspace on every call
    packed = mhc.pack_phi(wd[0]) if args.op in ("fused", "pre") and not args.pack_per_call else None
    out = {"residual_out": torch.empty((T, 4, H), dtype=torch.bfloat16, device=dev),
           "layer_in": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
           "pre_mix": torch.empty((T, 4), device=dev), "post_mix": torch.empty((T, 4), device=dev),
           "comb_res_mix": torch.empty((T, 4, 4), device=dev)}
    stream = torch.cuda.current_stream(dev)

    mx_mode = {"none": None, "floor": mhc.MX_SCALE_FLOOR, "ceil": mhc.MX_SCALE_CEIL}[args.mxfp8]
    if mx_mode is not None:
        out["layer_in_fp8"] = torch.empty((T, H), dtype=torch.uint8, device=dev)
        out["layer_in_scales"] = torch.empty(mhc.mxfp8_scale_bytes(T, H), dtype=torch.uint8, device=dev)
        if args.no_bf16:  # the MXFP8 layer input only
            del out["layer_in"]

    xsd = None
    if args.op in ("post", "post_sqrsum", "post_int8"):
        # the post variants: outputs R' (and the square sum); post_int8 takes the layer output as
        # int8 codes with one scale per token (a symmetric per-token quantization of Y)
        out = {"residual_out": out["residual_out"]}
        if args.op != "post":
            out["sqrsum"] = torch.empty(T, dtype=torch.float32, device=dev)
        if args.op == "post_int8":
            yf = synth.bf16_bits_to_f32(Y).astype(np.float64)
            amax = np.abs(yf).max(axis=1)
            xs = np.where(amax > 0, amax / 127.0, 1.0).astype(np.float32)
            Y = np.clip(np.rint(yf / xs[:, None]), -127, 127).astype(np.int8)
            Yd = torch.from_numpy(Y).to(dev)
            xsd = torch.from_numpy(xs).to(dev)

    if args.op == "pre_broadcast":
        out = {"residual_out": out["residual_out"], "layer_in": out["layer_in"], "pre_mix": out["pre_mix"],
               "post_mix": out["post_mix"], "comb_res_mix": out["comb_res_mix"]}
    if args.op == "pre":  # the pre alone (non-shift order): R plays the post-updated streams
        out = {"layer_in": out["layer_in"], "pre_mix": out["pre_mix"], "post_mix": out["post_mix"],
               "comb_res_mix": out["comb_res_mix"]}

    if args.op == "split":
        # two workspaces and event pairs: call i waits on the join of call i-2, so the side
        # kernel of call i (post and residual mixes) overlaps the main kernel of call i+1
        side = torch.cuda.Stream(dev)
        wss = [ws, mhc.new_workspace(T, H, dev)]
        sevs = []
        ncall = [0]

    def fresh_split_events():
        """New event pairs (an event recorded inside a stream capture cannot be waited on
        outside it, so each capture and the eager phase get their own)."""
        if args.op != "split":
            return
        torch.cuda.synchronize(dev)
        sevs[:] = [(torch.cuda.Event(), torch.cuda.Event()) for _ in range(2)]
        for f_, j_ in sevs:
            f_.record(stream)
            j_.record(stream)
        torch.cuda.synchronize(dev)
        ncall[0] = 0
    fresh_split_events()

    def call(R_, Y_, pp_, pc_, st=stream, o=None):
        o = out if o is None else o
        if args.op == "split":
            i = ncall[0]
            ncall[0] += 1
            f_, j_ = sevs[i % 2]
            if i >= 2:
                st.wait_event(j_)
            mhc.shifted_post_pre_split(R_, Y_, pp_, pc_, *wd, **sc, side_stream=side, fork_event=f_, join_event=j_,
                                       out=o, workspace=wss[i % 2], stream=st)
        elif args.op == "pre":
            mhc.pre(R_, *wd, **sc, out=o, workspace=ws, stream=st, packed_phi=packed)
        elif args.op == "pre_broadcast":  # the first layer: Y plays the (T, H) input  # the first layer: Y plays the (T, H) input
            mhc.pre_broadcast(Y_, *wd, **sc, out=o, workspace=ws, stream=st)
        elif args.op == "post":
            mhc.post(R_, Y_, pp_, pc_, out=o["residual_out"], stream=st)
        elif args.op == "post_sqrsum":
            mhc.lib().mhc_post_sqrsum(*[mhc._ptr(x) for x in (R_, Y_, pp_, pc_)], T, H,
                                      mhc._ptr(o["residual_out"]), mhc._ptr(o["sqrsum"]), mhc._stream(st, dev))
        elif args.op == "post_int8":
            mhc.lib().mhc_post_int8(*[mhc._ptr(x) for x in (R_, Y_, xsd, pp_, pc_)], T, H,
                                    mhc._ptr(o["residual_out"]), mhc._ptr(o["sqrsum"]), mhc._stream(st, dev))
        elif mx_mode is None:
            mhc.shifted_post_pre(R_, Y_, pp_, pc_, *wd, **sc, out=o, workspace=ws, stream=st, packed_phi=packed)
        else:
            mhc.shifted_post_pre_mxfp8(R_, Y_, pp_, pc_, *wd, **sc, scale_mode=mx_mode,
                                       out=dict(o, layer_in=None) if args.no_bf16 else o, workspace=ws,
                                       want_bf16=not args.no_bf16, stream=st, packed_phi=packed)

    def step():
        call(Rd, Yd, ppd, pcd)

    for _ in range(max(3, args.warmup)):
        step()
    launches = mhc.last_launch_count()
    torch.cuda.synchronize(dev)
    mhc.check_status(ws)
    run_steps, n_replay = step, args.steps
    if args.graph > 0:
        # launch-bound sizes: capture `graph` calls into one CUDA graph and replay it, so the
        # timed region measures the device, not the host's per-call launch overhead
        gstream = torch.cuda.Stream(dev)
        gstream.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        fresh_split_events()
        with torch.cuda.graph(g, stream=gstream):
            for _ in range(args.graph):
                call(Rd, Yd, ppd, pcd, gstream)
            if args.op == "split":  # join the side stream back
                for f_, j_ in sevs:
                    gstream.wait_event(j_)
        n_replay = max(1, args.steps // args.graph)
        args.steps = n_replay * args.graph

        def run_steps():
            g.replay()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    # clocks: the sampler runs through an untimed pre-roll of the same steps (about 0.3 s, so that
    # it has samples under this load however short the timed region is) and the timed region
    with ClockSampler(dev.index) as clk:
        clk.wait_first()
        t_roll = time.perf_counter()
        while time.perf_counter() - t_roll < 0.3:
            run_steps()
            torch.cuda.synchronize(dev)
        barrier()
        ev0.record(stream)
        for _ in range(n_replay):
            run_steps()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    el_ms = ev0.elapsed_time(ev1)
    mhc.check_status(ws)
    # the main kernel alone (for the roofline): events recorded by the library right around
    # its launch, one pair per call, over a separate run of calls
    nk = max(3, min(args.steps, 200))
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nk)]
    for a_, b_ in kev:  # torch creates the CUDA event on its first record
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize(dev)
    if args.graph > 0:  # the event pairs recorded inside a captured graph, replayed once
        kg = torch.cuda.CUDAGraph()
        gstream2 = torch.cuda.Stream(dev)
        gstream2.wait_stream(stream)
        fresh_split_events()
        with torch.cuda.graph(kg, stream=gstream2):
            for a_, b_ in kev:
                mhc.set_main_kernel_events(a_, b_)
                call(Rd, Yd, ppd, pcd, gstream2)
            mhc.set_main_kernel_events(None, None)
            if args.op == "split":
                for f_, j_ in sevs:
                    gstream2.wait_event(j_)
        kg.replay()
    else:
        for a_, b_ in kev:
            mhc.set_main_kernel_events(a_, b_)
            step()
        mhc.set_main_kernel_events(None, None)
    torch.cuda.synchronize(dev)
    span_each = np.array([a_.elapsed_time(b_) for a_, b_ in kev]) * 1e3  # us, one per call
    kernel_ms = float(np.mean(span_each)) / 1e3
    el_ms = max_over_ranks(el_ms, dist, dev)
    ms_step = el_ms / args.steps
    value = world * T / (ms_step / 1e3)

    fresh_split_events()
    # e2e through the public API with host buffers: every step copies its inputs in from pinned
    # host memory, runs the call and copies all its outputs back.  The steps are pipelined over
    # two buffer sets: host-to-device copies on one copy stream, the calls on the compute
    # stream, device-to-host copies on another copy stream, ordered by events, so the copies of
    # one step overlap the call of its neighbour; the timed region spans the first copy in to
    # the last copy out.
    hR = torch.from_numpy(R.view(np.int16)).pin_memory()
    hY = torch.from_numpy(Y if Y.dtype == np.int8 else Y.view(np.int16)).pin_memory()
    hpp, hpc = torch.from_numpy(pp).pin_memory(), torch.from_numpy(pc).pin_memory()
    # the inputs this op reads: the pre alone takes the residual only, the broadcast pre the
    # (T, H) input only (Y plays it), the rest the residual, the layer output and the mixes
    need_R, need_Y, need_mix = args.op != "pre_broadcast", args.op != "pre", args.op not in ("pre", "pre_broadcast")
    h2d = sum(t.numel() * t.element_size() for t, n in ((hR, need_R), (hY, need_Y), (hpp, need_mix), (hpc, need_mix)) if n)
    sets = []
    for _ in range(2):
        o2 = {k: torch.empty_like(v) for k, v in out.items()}
        sets.append({"R": torch.empty_like(Rd), "Y": torch.empty_like(Yd), "pp": torch.empty_like(ppd),
                     "pc": torch.empty_like(pcd), "out": o2,
                     "host": {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in o2.items()},
                     "ev_in": torch.cuda.Event(), "ev_done": torch.cuda.Event(), "ev_free": torch.cuda.Event()})
    d2h = sum(t.numel() * t.element_size() for t in sets[0]["host"].values())
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    for b_ in sets:
        b_["ev_free"].record(s_out)
    torch.cuda.synchronize(dev)

    def e2e_step(i, capturing=False):
        b_ = sets[i % 2]
        if not (capturing and i < 2):  # inside a capture, only events recorded in it can be waited on
            s_in.wait_event(b_["ev_free"])        # step i-2 is done with this set
        with torch.cuda.stream(s_in):
            if need_R:
                b_["R"].view(torch.int16).copy_(hR, non_blocking=True)
            if need_Y:
                b_["Y"].view(hY.dtype).copy_(hY, non_blocking=True)
            if need_mix:
                b_["pp"].copy_(hpp, non_blocking=True)
                b_["pc"].copy_(hpc, non_blocking=True)
        b_["ev_in"].record(s_in)
        stream.wait_event(b_["ev_in"])
        call(b_["R"], b_["Y"], b_["pp"], b_["pc"], stream, b_["out"])
        b_["ev_done"].record(stream)
        s_out.wait_event(b_["ev_done"])
        with torch.cuda.stream(s_out):
            for k, v in b_["out"].items():
                b_["host"][k].copy_(v, non_blocking=True)
        b_["ev_free"].record(s_out)

    e2e_steps = max(4, min(args.steps, 20))
    for i in range(2):
        e2e_step(i)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.graph > 0:
        # launch-bound sizes: the same pipelined steps captured into one CUDA graph (forked onto
        # the copy streams and joined back inside the capture), replayed
        fresh_split_events()
        cs0 = torch.cuda.Stream(dev)
        cs0.wait_stream(stream)
        eg = torch.cuda.CUDAGraph()
        stream_saved = stream
        with torch.cuda.graph(eg, stream=cs0):
            stream = cs0
            fork = torch.cuda.Event()
            fork.record(cs0)
            s_in.wait_event(fork)
            s_out.wait_event(fork)
            for i in range(args.graph):
                e2e_step(i, capturing=True)
            for st_ in (s_in, s_out):
                jn = torch.cuda.Event()
                jn.record(st_)
                cs0.wait_event(jn)
            if args.op == "split":  # the side stream of the last calls
                for f_, j_ in sevs:
                    cs0.wait_event(j_)
        stream = stream_saved
        eg.replay()
        torch.cuda.synchronize(dev)
        n_rep = max(1, e2e_steps // args.graph)
        e0.record(stream)
        for _ in range(n_rep):
            eg.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / (n_rep * args.graph)
    else:
        e0.record(s_in)
        for i in range(e2e_steps):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)

    if rank != 0:
        return
    peak, peak_src = peaks()
    abytes = algorithmic_bytes(T, H, mx_mode is not None, mx_mode is not None and args.no_bf16) \
        if args.op in ("fused", "split") else \
        {"post": T * (18 * H + 80), "post_sqrsum": T * (18 * H + 84), "post_int8": T * (17 * H + 88),
         "pre": T * (10 * H + 96) + 384 * H + 2 * H + 108,
         "pre_broadcast": T * (12 * H + 96) + 384 * H + 2 * H + 108}[args.op]
    # calls whose bytes are split over several kernels (the MXFP8 output written by a second
    # pass, the broadcast pre): the roofline uses the whole call's time
    whole_call = (mx_mode is not None and not args.no_bf16) or args.op == "pre_broadcast"
    # a step whose launches are all the main span (phi packed before the timed region, no separate
    # quantize pass): the main span's duration is the timed region's time per call.  Consecutive
    # calls overlap there (each ws launch sets up while the previous call drains), which the
    # per-call event pair, recorded between the calls, prevents; it is reported beside.
    # Both bound the span's duration from above (the events add the calls' serialisation, the
    # timed region the host's launch gaps of launch-bound calls), so the smaller one is taken.
    main_only = not whole_call and packed is not None and args.op in ("fused", "pre") and args.graph == 0
    span_ms = ms_step if whole_call else (min(ms_step, kernel_ms) if main_only else kernel_ms)
    achieved = abytes / (span_ms / 1e3) / 1e9
    auto_name = {v: k for k, v in mhc.SCHEDULES.items()}.get(mhc.auto_schedule(T, H), "?")
    side_tokens = 0
    if args.schedule != "auto":
        sched = args.schedule
    elif args.op in ("fused", "split", "pre"):
        sched = auto_name
        if args.op in ("fused", "pre") and auto_name == "ws":
            side_tokens = mhc.auto_side_tokens(T, H, args.op == "fused")
            if side_tokens > 0:  # the token-tile kernel beside ws on the SMs its clusters leave idle
                sched = "ws+tile"
    elif args.op == "pre_broadcast":  # the fused kernel from x alone above 32 tokens, else residual + pre
        sched = "bcast" if T > 32 and H % 64 == 0 else f"broadcast + {auto_name} pre"
    else:
        sched = args.op
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name} T={T} H={H} hc_mult=4", "T": T, "H": H,
                   "op": {"fused": "mhc_shifted_post_pre", "post": "mhc_post", "post_sqrsum": "mhc_post_sqrsum",
                          "post_int8": "mhc_post_int8", "pre": "mhc_pre", "pre_broadcast": "mhc_pre_broadcast",
                          "split": "mhc_shifted_post_pre_split (mixes on a side stream)"}[args.op],
                   "io": "bf16 streams, fp32 mixes" + ("" if mx_mode is None else f", + MXFP8 layer input ({args.mxfp8} scales)"
                                                         + (", no bf16 layer input" if args.no_bf16 else ""))
                         + (", int8 layer output with per-token scales" if args.op == "post_int8" else ""),
                   "schedule": sched if side_tokens <= 0 else
                   f"ws+tile (ws on the first {T - side_tokens} tokens, the token-tile kernel beside it on "
                   f"the last {side_tokens})", "l2": f"inputs larger than L2 ({abytes / 1e9:.2f} GB moved per call)",
                   "phi": "packed once before the timed region (mhc_pack_phi), the call takes the packed form"
                          if packed is not None else "packed by every call in its workspace",
                   "call_gbs": abytes / (ms_step / 1e3) / 1e9},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None if whole_call else
                     measured_traffic((sched if args.op != "pre" else "pre_" + sched)
                                      + ("" if mx_mode is None else "_mxfp8_only"), w.name, T, H),
                     "peak_source": peak_src,
                     "kernel": (f"whole call ({launches} launches), {ms_step * 1e3:.1f} us; main kernel "
                                f"{kernel_ms * 1e3:.1f} us" if whole_call else
                                f"main span of the call ({launches} launches per call, all of them the main "
                                f"span): {ms_step * 1e3:.1f} us per call over the timed region, "
                                f"{kernel_ms * 1e3:.1f} us between CUDA events around each call's main span "
                                f"({nk} calls, no overlap between calls); the smaller is used"
                                if main_only else
                                f"main kernel of the call ({launches} launches per call), "
                                f"{kernel_ms * 1e3:.1f} us per launch (CUDA events around it, {nk} launches)")
                               + f", algorithmic bytes {abytes} per call"},
        "gpu_launches": launches * args.steps,
        "launch_mode": f"CUDA graph of {args.graph} calls, replayed" if args.graph > 0 else "eager",
        "main_span_us": {"calls": int(span_each.size), "p10": float(np.percentile(span_each, 10)),
                         "p50": float(np.percentile(span_each, 50)), "p90": float(np.percentile(span_each, 90))},
        "e2e": {"value": world * T / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipelining": "two buffer sets; copies in, calls and copies out on three streams"},
        "clocks": dict(clk.summary(), window="an untimed pre-roll of the same steps (~0.3 s) and the timed region"),
    }
    if world == 1 and not args.no_cpu_baseline:
        tps, nt, el, done = time_oracle(w, phi, bias, msc, gamma, min(1024, T), 10.0)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": nt, "kind": "oracle",
                                "sample": f"first {min(1024, T)} tokens of {w.name} (T={T}, H={H}), repeated for "
                                          f"{el:.1f} s ({done} tokens)", "machine": platform.machine()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--schedule", default="auto", choices=["auto", "split", "ws", "small", "bcast", "tile"])
    ap.add_argument("--tokens", type=int, default=0, help="override T (smaller cases for profiling)")
    ap.add_argument("--op", default="fused",
                    choices=["fused", "split", "post", "post_sqrsum", "post_int8", "pre", "pre_broadcast"],
                    help="the fused step (default) or one of the post-only entry points")
    ap.add_argument("--graph", type=int, default=0,
                    help="capture this many calls into a CUDA graph and time its replays (launch-bound sizes)")
    ap.add_argument("--mxfp8", default="none", choices=["none", "floor", "ceil"],
                    help="also emit the layer input as MXFP8 (E4M3 + UE8M0 block scales)")
    ap.add_argument("--no-bf16", action="store_true", help="with --mxfp8: the MXFP8 layer input only")
    ap.add_argument("--pack-per-call", action="store_true",
                    help="time the plain calls, which pack phi on every call, instead of the prepacked ones")
    args = ap.parse_args()
    rank, world, lr, dist = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, rank, world, dist)
        else:
            run_ours(args, rank, world, lr, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
