"""Benchmark of the USP attention hot path on GB300.

One step = one pass of every built row of the hot path over one batch of
synthetic input of the named workload (default: the largest one, Wan 720p
81 frames, bf16, B1 H40 N75600 D128, ulysses 8 x ring 2, with the backward):
  * usp_attention_fwd, materialised: tok2head(q,k,v) -> per-(rank, ring step)
    chunk attention -> LSE merge -> head2tok(out, lse)
  * usp_attention_fwd, fused: one kernel over the token-sharded stacks
  * usp_attention_bwd (when the workload has a backward)
``value`` is algorithmic attention FLOP of the step (4*B*H*N^2*D per forward,
10*B*H*N^2*D per backward) / device time, in TFLOP/s, summed over ranks.
L2 is flushed (a 256 MB buffer is written) before every timed step, outside
the timed events (the Wan inputs, 774 MB each, are larger than L2 anyway;
the Qwen-Image 1024^2 ones, 25 MB, are not).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun every rank runs its own replica (weak scaling, no data-path
collective); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from diffusion_transformer_sequence_gb300 import workloads as wl  # noqa: E402

METRIC = "USP attention fwd(+bwd) TFLOP/s and % of GB300 bf16 peak; re-layout GB/s vs HBM"
L2_FLUSH_BYTES = 256 << 20
# After the L2 flush and before a start event, the device waits ~100 us
# (torch.cuda._sleep, in clock cycles) so that the host has enqueued the
# timed launches by the time the event fires: the events then time device
# work, not host launch latency.  Not used inside the end-to-end loop.
HOLD_CYCLES = 200_000


def flush_l2(buf, hold=True):
    buf.fill_(1)
    if hold:
        torch.cuda._sleep(HOLD_CYCLES)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        t0, t1 = getattr(self, "start", 0.0), getattr(self, "end", float("inf"))
        window = [ln for (t, ln) in self.lines if t0 <= t <= t1 + 0.05]
        in_window = len(window)
        if not window:  # timed region shorter than the sampling period: use the whole run
            window = [ln for (_, ln) in self.lines]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in window:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "samples_in_timed_region": in_window}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


# ---------------------------------------------------------------- reference arm
def oracle_sample_flop(w, heads):
    n = w.N + w.Nt
    return 4.0 * w.B * heads * n * n * w.D


def run_oracle_sample(w, heads: int):
    """Time the CPU oracle's USP forward (joint when the workload has text
    tokens) on `heads` heads of the workload.  Returns (seconds, parity):
    the same sub-problem also runs through the fused call on the GPU, and
    parity holds the largest |out| and relative lse differences between
    the two (image queries)."""
    import oracle
    import diffusion_transformer_sequence_gb300 as usp
    sub = wl.custom(w.name, w.dtype, w.B, heads, w.N, w.D, w.ulysses, w.ring, seed=w.seed, Nt=w.Nt)
    inp = wl.make_inputs(sub, with_dout=False)
    st = [wl.to_token_stack(inp[n], w.ulysses, w.ring) for n in ("q", "k", "v")]
    stacks = [t.double().numpy() for t in st]
    t0 = time.perf_counter()
    if w.Nt:
        txt_t = wl.make_text_inputs(sub)
        txt = {n: t.double().numpy() for n, t in txt_t.items()}
        ro, rl = oracle.usp_forward_joint(*stacks, txt["k_txt"], txt["v_txt"], w.ulysses, w.ring, w.scale,
                                          q_txt=txt["q_txt"])[:2]
    else:
        ro, rl = oracle.usp_forward(*stacks, w.ulysses, w.ring, w.scale)
    dt = time.perf_counter() - t0
    dev = [t.cuda() for t in st]
    if w.Nt:
        go, gl = usp.attention_fwd_joint(*dev, txt_t["k_txt"].cuda(), txt_t["v_txt"].cuda(), w.ulysses, w.ring,
                                         w.scale, mode="fused")
    else:
        go, gl = usp.attention_fwd(*dev, w.ulysses, w.ring, w.scale, mode="fused")
    import numpy as np
    go, gl = go.double().cpu().numpy(), gl.double().cpu().numpy()
    parity = {"max_abs_out": float(np.abs(go - ro).max()),
              "max_rel_lse": float((np.abs(gl - rl) / np.maximum(np.abs(rl), 1e-30)).max()),
              "vs": "oracle (numpy fp64) on the same sub-problem, fused call",
              "bound": {"out_abs": 2e-2 if w.dtype == "bf16" else 1e-5, "lse_rel": 1e-3 if w.dtype == "bf16" else None}}
    return dt, parity


def oracle_rows_baseline(w, step, heads, nrows, cores):
    """CPU-baseline leg for workloads too large for a full-head oracle run.

    The oracle's attention of ``nrows`` seeded query rows (always including
    shard and tile boundaries) of each listed head against all N keys -- the
    rows of unsharded attention that the USP path must equal -- timed on
    ``cores`` single-threaded spawn workers (rows split evenly), and once
    more on one worker for a single-thread figure.  Parity: the same rows of
    the step's fused output, already on the device."""
    import numpy as np
    from oracle import pool
    glob = {n: wl.from_token_stack(step.host[n])[0, heads].float().numpy() for n in ("q", "k", "v")}
    rows = wl.sample_rows(w, nrows).numpy()
    jobs = pool.split_row_jobs(glob["q"], glob["k"], glob["v"], rows, w.scale, cores)
    with pool.rows_executor(min(cores, len(jobs))) as ex:
        t0 = time.perf_counter()
        res = list(ex.map(pool.rows_job, jobs))
        dt = time.perf_counter() - t0
    ro, rl = pool.join_row_results(res, len(heads))
    flop = 4.0 * len(heads) * len(rows) * w.N * w.D
    # single thread: one worker, the first 2048 rows of the first head
    one = pool.split_row_jobs(glob["q"][:1], glob["k"][:1], glob["v"][:1], rows[:2048], w.scale, 1)
    with pool.rows_executor(1) as ex:
        t1 = time.perf_counter()
        list(ex.map(pool.rows_job, one))
        dt1 = time.perf_counter() - t1
    flop1 = 4.0 * min(2048, len(rows)) * w.N * w.D
    sel = step.out_f[:, :, :, heads]
    go = wl.from_token_stack(sel)[0][:, torch.as_tensor(rows, device=sel.device)].double().cpu().numpy()
    gl = wl.from_token_stack(step.lse_f[:, :, :, heads])[0][:, torch.as_tensor(rows, device=sel.device)]
    gl = gl.double().cpu().numpy()
    parity = {"max_abs_out": float(np.abs(go - ro).max()),
              "max_rel_lse": float((np.abs(gl - rl) / np.maximum(np.abs(rl), 1e-30)).max()),
              "vs": f"oracle (numpy fp64) at the same {len(rows)} rows x {len(heads)} heads, the step's fused call",
              "bound": {"out_abs": 2e-2, "lse_rel": 1e-3}}
    return {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": min(cores, len(jobs)), "kind": "oracle",
            "sample": (f"oracle attention (numpy fp64) of {len(rows)} seeded query rows of heads {list(heads)} of "
                       f"{w.name} against all {w.N} keys, {dt:.1f} s (a rate over a bounded sample: nothing is "
                       f"extrapolated)"),
            "single_thread": {"value": flop1 / dt1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                              "sample": f"{min(2048, len(rows))} rows of head {heads[0]} on one worker, {dt1:.1f} s"},
            "parity": parity}


def oracle_single_thread(w, heads):
    """The single-thread figure of the full-head CPU-baseline leg: one head
    of the same sub-problem's attention on one single-threaded worker."""
    import numpy as np
    from oracle import pool
    sub = wl.custom(w.name, w.dtype, w.B, w.ulysses, w.N, w.D, w.ulysses, w.ring, seed=w.seed, Nt=w.Nt)
    inp = wl.make_inputs(sub, with_dout=False)
    q, k, v = (inp[n][0, :1].float().numpy() for n in ("q", "k", "v"))
    rows = np.arange(min(w.N, 1024))
    one = pool.split_row_jobs(q, k, v, rows, w.scale, 1)
    with pool.rows_executor(1) as ex:
        t0 = time.perf_counter()
        list(ex.map(pool.rows_job, one))
        dt = time.perf_counter() - t0
    return {"value": 4.0 * len(rows) * w.N * w.D / dt / 1e12, "unit": "TFLOP/s", "cores": 1,
            "sample": f"{len(rows)} query rows of one head against all {w.N} keys on one worker, {dt:.2f} s"}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def sample_heads(w):
    """Heads of the workload the CPU-baseline leg runs (a multiple of ulysses):
    the whole workload when it is small, else about a quarter of its heads."""
    if oracle_sample_flop(w, w.H) <= 0.25e12:
        return w.H
    return min(w.H, max(w.ulysses, (w.H // 4) // w.ulysses * w.ulysses))


def reference_arm(args, w, ws, rank):
    """The oracle, as it stands, timed on the host cores (rank 0 only).

    Each step is a bounded sample of the workload: the oracle's attention of
    `rows` query rows of one head against all N keys (the unsharded result the
    USP path must equal), with `rows` sized so the whole run stays within about
    two minutes."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    sub = wl.custom(w.name, w.dtype, w.B, w.ulysses, w.N, w.D, w.ulysses, w.ring, seed=w.seed, Nt=w.Nt)
    inp = wl.make_inputs(sub, with_dout=False)
    q, k, v = (inp[n][0, 0].double().numpy() for n in ("q", "k", "v"))
    if w.Nt:   # joint: the image queries against the text + image keys of the head
        txt = wl.make_text_inputs(sub)
        k = np.concatenate([txt["k_txt"][0, 0].double().numpy(), k])
        v = np.concatenate([txt["v_txt"][0, 0].double().numpy(), v])
    nk = k.shape[0]
    ncal = min(256, w.N)
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, np.arange(ncal), w.scale)
    rate = ncal / (time.perf_counter() - t0)              # rows per second
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(16, min(w.N, rate * budget)))
    g = torch.Generator().manual_seed(w.row_seed)
    times = []
    for i in range(args.warmup + args.steps):
        sel = torch.randint(0, w.N, (rows,), generator=g).numpy()
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, sel, w.scale)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    flop = 4.0 * rows * nk * w.D
    tflops = flop / statistics.mean(times) / 1e12
    sample = (f"oracle attention (numpy fp64) of {rows} seeded query rows of one head against all {nk} keys "
              f"of {w.name}, per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "desc": w.description, "global_batch": w.B, "seq_len": w.N,
                   "text_len": w.Nt, "ulysses": w.ulysses, "ring": w.ring,
                   "parallelism": "virtual ranks on one device"},
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
class Step:
    """Device buffers and the calls of one step, with per-call CUDA events."""

    def __init__(self, w, backward: bool):
        import diffusion_transformer_sequence_gb300 as usp
        self.usp = usp
        self.w = w
        inp = wl.make_inputs(w, with_dout=backward)
        self.host = {n: wl.to_token_stack(t, w.ulysses, w.ring).pin_memory() for n, t in inp.items()}
        self.dev = {n: t.cuda() for n, t in self.host.items()}
        self.out_m = torch.empty_like(self.dev["q"])
        self.lse_m = torch.empty(w.lse_stack_shape, dtype=torch.float32, device="cuda")
        self.out_f = torch.empty_like(self.dev["q"])
        self.lse_f = torch.empty(w.lse_stack_shape, dtype=torch.float32, device="cuda")
        nws = usp.workspace_bytes(w.B, w.H, w.N, w.D, w.ulysses, w.ring, w.torch_dtype, "materialised")
        self.ws = torch.empty(max(nws, 1), dtype=torch.uint8, device="cuda")
        self.backward = backward
        self.bwd_phases = False   # record the library's phase events around the backward (timed loop only)
        if backward:
            nb = usp.workspace_bytes(w.B, w.H, w.N, w.D, w.ulysses, w.ring, w.torch_dtype, backward=True)
            self.ws_b = torch.empty(nb, dtype=torch.uint8, device="cuda")
            self.grads = [torch.empty_like(self.dev["q"]) for _ in range(3)]
            # the backward consumes the fused forward's out / lse: make them valid once up front
            usp.attention_fwd(self.dev["q"], self.dev["k"], self.dev["v"], w.ulysses, w.ring, w.scale,
                              mode="fused", out=self.out_f, lse=self.lse_f)
        self.flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        # materialised: tok2head (q, k, v in one launch), chunk attention, then the merge into the
        # token-sharded out and lse (ring > 1, one launch) or head2tok of out and lse (ring = 1: one launch
        # when both move in 16-byte vectors, else two); fused: one; backward: prep + dK/dV + dQ
        elt = 2 if w.dtype == "bf16" else 4
        h2t = 1 if (w.Ns * 4) % 16 == 0 and (w.Ns * w.D * elt) % 16 == 0 else 2
        self.launches_per_step = 2 + (1 if w.ring > 1 else h2t) + 1 + (3 if backward else 0)
        self.joint = w.Nt > 0
        if self.joint:
            # text tokens replicated on every virtual rank: q_txt, k_txt, v_txt [B, H, Nt, D]
            self.host.update({n: t.pin_memory() for n, t in wl.make_text_inputs(w).items()})
            for n in ("q_txt", "k_txt", "v_txt"):
                self.dev[n] = self.host[n].cuda()
            tshape, lshape = (w.B, w.H, w.Nt, w.D), (w.B, w.H, w.Nt)
            self.txt_out = {m: (torch.empty(tshape, dtype=w.torch_dtype, device="cuda"),
                                torch.empty(lshape, dtype=torch.float32, device="cuda")) for m in ("m", "f")}
            nws = usp.joint_workspace_bytes(w.B, w.H, w.N, w.Nt, w.D, w.ulysses, w.ring, w.torch_dtype,
                                            "materialised", True)
            self.ws = torch.empty(max(nws, 1), dtype=torch.uint8, device="cuda")
            # materialised: tok2head, partials against the image chunks, partials against the text,
            # merge into the token-sharded out and lse, text merge; fused: one launch (image and text queries)
            self.launches_per_step = 5 + 1

    def flop(self):
        if self.joint:
            return 2 * self.w.joint_flop(True)
        f = 2 * self.w.fwd_flop
        if self.backward:
            f += self.w.bwd_flop
        return f

    def fwd(self, mode):
        """One forward call of the step (joint when the workload has text tokens)."""
        usp, w, d = self.usp, self.w, self.dev
        out, lse = (self.out_m, self.lse_m) if mode == "materialised" else (self.out_f, self.lse_f)
        ws = self.ws if mode == "materialised" else None
        if not self.joint:
            usp.attention_fwd(d["q"], d["k"], d["v"], w.ulysses, w.ring, w.scale, mode=mode, out=out, lse=lse,
                              workspace=ws)
            return
        from diffusion_transformer_sequence_gb300 import _lib
        ot, lt = self.txt_out[mode[0]]
        rc = usp.lib().usp_attention_fwd_joint(
            d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["q_txt"].data_ptr(), d["k_txt"].data_ptr(),
            d["v_txt"].data_ptr(), out.data_ptr(), lse.data_ptr(), ot.data_ptr(), lt.data_ptr(), w.B, w.H, w.N,
            w.Nt, w.D, w.ulysses, w.ring, w.scale, _lib.USP_BF16 if w.dtype == "bf16" else _lib.USP_F32,
            _lib.USP_MATERIALISED if mode == "materialised" else _lib.USP_FUSED,
            ws.data_ptr() if ws is not None else None, ws.numel() if ws is not None else 0,
            torch.cuda.current_stream().cuda_stream)
        _lib.check("usp_attention_fwd_joint", rc)

    def flush(self, hold=True):
        flush_l2(self.flush_buf, hold)

    def run(self, ev=None, only=None):
        usp, w = self.usp, self.w
        if ev:
            ev[0].record()
        if only in (None, "materialised"):
            self.fwd("materialised")
        if ev and ev[1] is not None:
            ev[1].record()
        if only in (None, "fused"):
            self.fwd("fused")
        if ev and ev[2] is not None:
            ev[2].record()
        if self.backward and only in (None, "backward"):
            # phase events only around the backward: events between the
            # forward's kernels would stop each from starting under the
            # previous one's tail (programmatic dependent launch)
            if self.bwd_phases:
                self.usp.lib().usp_profile_phases(1)
            self.bwd()
            if self.bwd_phases:
                self.usp.lib().usp_profile_phases(0)
        if ev:
            ev[3].record()

    def bwd(self):
        usp, w = self.usp, self.w
        L = usp.lib()
        from diffusion_transformer_sequence_gb300 import _lib
        d = self.dev
        rc = L.usp_attention_bwd(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), self.out_f.data_ptr(),
                                 self.lse_f.data_ptr(), d["dout"].data_ptr(), self.grads[0].data_ptr(),
                                 self.grads[1].data_ptr(), self.grads[2].data_ptr(), w.B, w.H, w.N, w.D, w.ulysses,
                                 w.ring, w.scale, _lib.USP_BF16 if w.dtype == "bf16" else _lib.USP_F32,
                                 self.ws_b.data_ptr(), self.ws_b.numel(), torch.cuda.current_stream().cuda_stream)
        _lib.check("usp_attention_bwd", rc)

    def _out_names(self):
        names = ["out_m", "lse_m", "out_f", "lse_f"]
        return names + (["grads"] if self.backward else [])

    def _swap_set(self, k):
        """Point the step at buffer set k (0 or 1) of the pipelined end-to-end loop."""
        if not hasattr(self, "_sets"):
            own = {"dev": self.dev, **{n: getattr(self, n) for n in self._out_names()}}
            if self.joint:
                own["txt_out"] = self.txt_out
            clone = lambda t: [x.clone() for x in t] if isinstance(t, list) else t.clone()
            other = {"dev": {n: t.clone() for n, t in self.dev.items()},
                     **{n: clone(getattr(self, n)) for n in self._out_names()}}
            if self.joint:
                other["txt_out"] = {m: tuple(x.clone() for x in v) for m, v in self.txt_out.items()}
            self._sets = [own, other]
        for n, v in self._sets[k].items():
            setattr(self, n, v)

    def _outputs(self):
        outs = [("out_m", self.out_m), ("lse_m", self.lse_m), ("out_f", self.out_f), ("lse_f", self.lse_f)]
        if self.joint:
            outs += [("ot_m", self.txt_out["m"][0]), ("lt_m", self.txt_out["m"][1]),
                     ("ot_f", self.txt_out["f"][0]), ("lt_f", self.txt_out["f"][1])]
        if self.backward:
            outs += [("dq", self.grads[0]), ("dk", self.grads[1]), ("dv", self.grads[2])]
        return outs

    def run_e2e_pipelined(self, steps):
        """End to end with host buffers, software-pipelined over three streams:
        step i's host->device copy of its inputs (pinned) followed by the L2
        flush (so the inputs are evicted before step i starts, as in the
        device-timed loop), its compute, and the device->host copy of its
        results run on separate streams with two device buffer sets, so step
        i+1's inputs arrive and step i-1's results leave while step i
        computes.  Every step still moves its own inputs in and results out.
        Returns the elapsed seconds from before the first copy to after the
        last result has landed in host memory."""
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        s_cmp = torch.cuda.current_stream()
        ev = lambda: torch.cuda.Event()
        in_ready, done, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(s_cmp)
        s_in.wait_event(start)
        s_out.wait_event(start)
        host_out = {}
        for i in range(steps):
            k = i % 2
            self._swap_set(k)
            if i >= 2:
                s_in.wait_event(done[k])              # step i-2 has finished reading set k
            with torch.cuda.stream(s_in):
                for n in self.inputs():
                    self.dev[n].copy_(self.host[n], non_blocking=True)
                self.flush(hold=False)                # evicts the inputs just copied
                in_ready[k].record(s_in)
            s_cmp.wait_event(in_ready[k])
            if i >= 2:
                s_cmp.wait_event(out_free[k])         # step i-2's results have left set k
            self.fwd("materialised")
            self.fwd("fused")
            if self.backward:
                self.bwd()
            done[k].record(s_cmp)
            s_out.wait_event(done[k])
            with torch.cuda.stream(s_out):
                for name, t in self._outputs():
                    dst = host_out.get(name)
                    if dst is None:
                        dst = host_out[name] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                    dst.copy_(t, non_blocking=True)
                out_free[k].record(s_out)
        end.record(s_out)
        end.synchronize()
        s_cmp.wait_stream(s_out)
        self._swap_set(0)
        return start.elapsed_time(end) * 1e-3

    def inputs(self):
        names = ["q", "k", "v"] + (["dout"] if self.backward else [])
        return names + (["q_txt", "k_txt", "v_txt"] if self.joint else [])

    def io_bytes(self):
        h2d = sum(self.host[n].numel() * self.host[n].element_size() for n in self.inputs())
        d2h = 2 * (self.out_m.numel() * self.out_m.element_size() + self.lse_m.numel() * 4)
        if self.joint:
            d2h += 2 * sum(t.numel() * t.element_size() for t in self.txt_out["m"])
        if self.backward:
            d2h += sum(g.numel() * g.element_size() for g in self.grads)
        return h2d, d2h


def kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary (profiles/traffic.json), or None when the kernel's source changed
    since the counters were taken.  `a+b` sums the launches of kernels a and b."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    table = json.load(open(p))
    total = 0
    for k in kernel.split("+"):
        d = table.get(k, {}).get(workload)
        if not d:
            return None
        src = os.path.join(ROOT, "diffusion_transformer_sequence_gb300", "csrc", d["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if h != d["source_sha256_16"]:
            return None
        total += d["dram_bytes_per_launch"]
    return total


def time_rows(w, reps=10):
    """Per-row GB/s of the bandwidth-bound entry points on this workload (L2 flushed)."""
    import diffusion_transformer_sequence_gb300 as usp
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    q = torch.randn(w.stack_shape, device="cuda").to(w.torch_dtype)
    res = {}

    def timed(fn):
        ts = []
        for _ in range(reps + 2):
            flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e-3)
        return statistics.median(ts[2:])

    X = usp.relayout_tok2head(q, w.ulysses, w.ring)
    t = timed(lambda: usp.relayout_tok2head(q, w.ulysses, w.ring, out=X))
    res["tok2head"] = {"GB/s": 2 * w.t_bytes / t / 1e9, "us": t * 1e6, "bytes": 2 * w.t_bytes}
    T = torch.empty_like(q)
    t = timed(lambda: usp.relayout_head2tok(X, w.ulysses, w.ring, out=T))
    res["head2tok"] = {"GB/s": 2 * w.t_bytes / t / 1e9, "us": t * 1e6, "bytes": 2 * w.t_bytes}
    if w.dtype == "bf16":
        # the bandwidth-bound launches inside the materialised forward, as the step runs them:
        # tok2head of q, k, v in one launch, then the ring merge written straight to the token-sharded
        # out and lse (ring > 1) or head2tok of out and lse (ring = 1) (phase events)
        import ctypes
        L = usp.lib()
        kk, vv = torch.randn_like(q), torch.randn_like(q)
        om, lm = torch.empty_like(q), torch.empty(w.lse_stack_shape, device="cuda")
        wsm = torch.empty(usp.workspace_bytes(w.B, w.H, w.N, w.D, w.ulysses, w.ring, w.torch_dtype, "materialised"),
                          dtype=torch.uint8, device="cuda")
        ms = (ctypes.c_float * 8)()
        L.usp_profile_phases(1)
        ph = []
        for _ in range(reps + 2):
            flush_l2(flush)
            usp.attention_fwd(q, kk, vv, w.ulysses, w.ring, w.scale, mode="materialised", out=om, lse=lm,
                              workspace=wsm)
            n = L.usp_profile_read(ms, 8)
            ph.append([ms[i] * 1e-3 for i in range(n)])
        L.usp_profile_phases(0)
        ph = ph[2:]
        lse_b = w.B * w.H * w.N * 4
        t_in = statistics.median(p_[0] for p_ in ph)
        res["tok2head_qkv_in_step"] = {"GB/s": 6 * w.t_bytes / t_in / 1e9, "us": t_in * 1e6, "bytes": 6 * w.t_bytes}
        t_out = statistics.median(p_[2] for p_ in ph)
        if w.ring > 1:
            # the ring merge writes the token-sharded out and lse directly (merge + head2tok, one launch):
            # reads ring partial planes and their lse, writes one plane and one lse
            byt = (w.ring + 1) * (w.t_bytes + lse_b)
            res["merge_head2tok_in_step"] = {"GB/s": byt / t_out / 1e9, "us": t_out * 1e6, "bytes": byt}
        else:
            byt = 2 * (w.t_bytes + lse_b)
            res["head2tok_out_lse_in_step"] = {"GB/s": byt / t_out / 1e9, "us": t_out * 1e6, "bytes": byt}
    if w.dtype == "bf16" and not w.Nt:
        # the backward through the materialised Ulysses path (tok2head of q, k, v, O, dO and lse,
        # the per-rank chunk backward over the head-sharded stacks, head2tok of dq, dk, dv),
        # timed whole and by phase
        import ctypes
        L = usp.lib()
        k_ = torch.randn(w.stack_shape, device="cuda").to(w.torch_dtype)
        v_ = torch.randn(w.stack_shape, device="cuda").to(w.torch_dtype)
        do = torch.randn(w.stack_shape, device="cuda").to(w.torch_dtype)
        o, l = usp.attention_fwd(q, k_, v_, w.ulysses, w.ring, w.scale, mode="fused")
        wsb = torch.empty(usp.workspace_bytes(w.B, w.H, w.N, w.D, w.ulysses, w.ring, w.torch_dtype, "materialised",
                                              backward=True), dtype=torch.uint8, device="cuda")
        t = timed(lambda: usp.attention_bwd(q, k_, v_, o, l, do, w.ulysses, w.ring, w.scale, workspace=wsb,
                                            mode="materialised"))
        ms = (ctypes.c_float * 8)()
        L.usp_profile_phases(1)
        ph = []
        for _ in range(reps):
            flush_l2(flush)
            usp.attention_bwd(q, k_, v_, o, l, do, w.ulysses, w.ring, w.scale, workspace=wsb, mode="materialised")
            n = L.usp_profile_read(ms, 8)
            ph.append([ms[i] * 1e-3 for i in range(n)])
        L.usp_profile_phases(0)
        lse_b = w.B * w.H * w.N * 4
        t_in = statistics.median(p_[0] for p_ in ph)
        t_out = statistics.median(p_[-1] for p_ in ph)
        res["bwd_materialised"] = {"us": t * 1e6, "TFLOP/s": w.bwd_flop / t / 1e12}
        byt = 2 * (5 * w.t_bytes + lse_b)
        res["bwd_tok2head_qkvodo_lse_in_step"] = {"GB/s": byt / t_in / 1e9, "us": t_in * 1e6, "bytes": byt}
        byt = 2 * 3 * w.t_bytes
        res["bwd_head2tok_grads_in_step"] = {"GB/s": byt / t_out / 1e9, "us": t_out * 1e6, "bytes": byt}
        del k_, v_, do, o, l, wsb
    if w.Nt:
        # cross-attention of the sharded image queries to the replicated text K/V (tensor-bound:
        # reported as TFLOP/s beside its bytes)
        kt = torch.randn((w.B, w.H, w.Nt, w.D), device="cuda").to(w.torch_dtype)
        vt = torch.randn((w.B, w.H, w.Nt, w.D), device="cuda").to(w.torch_dtype)
        o = torch.empty_like(q)
        l = torch.empty(w.lse_stack_shape, device="cuda")
        t = timed(lambda: usp.cross_attention_fwd(q, kt, vt, w.ulysses, w.ring, w.scale, out=o, lse=l))
        flop = 4.0 * w.B * w.H * w.N * w.Nt * w.D
        byt = 2 * w.t_bytes + w.B * w.H * w.N * 4 + 2 * kt.numel() * kt.element_size()
        res["cross_attention"] = {"GB/s": byt / t / 1e9, "us": t * 1e6, "bytes": byt, "TFLOP/s": flop / t / 1e12}
    if w.dtype == "bf16" and not w.Nt:
        # FP8 (E4M3) fused forward of the same stacks: quantise q, k, v + FP8 attention (bf16-equivalent
        # FLOP rate), with the two phases timed separately
        import ctypes
        L = usp.lib()
        k_ = torch.randn(w.stack_shape, device="cuda").to(w.torch_dtype)
        v_ = torch.randn(w.stack_shape, device="cuda").to(w.torch_dtype)
        o = torch.empty_like(q)
        l = torch.empty(w.lse_stack_shape, device="cuda")
        ws8 = torch.empty(int(L.usp_attention_fp8_workspace_bytes(w.B, w.H, w.N, w.D, w.ulysses, w.ring)),
                          dtype=torch.uint8, device="cuda")
        t = timed(lambda: usp.attention_fwd_fp8(q, k_, v_, w.ulysses, w.ring, w.scale, out=o, lse=l, workspace=ws8))
        ms = (ctypes.c_float * 8)()
        L.usp_profile_phases(1)
        ph = []
        for _ in range(reps):
            flush_l2(flush)
            usp.attention_fwd_fp8(q, k_, v_, w.ulysses, w.ring, w.scale, out=o, lse=l, workspace=ws8)
            n = L.usp_profile_read(ms, 8)
            ph.append([ms[i] * 1e-3 for i in range(n)])
        L.usp_profile_phases(0)
        tq = statistics.median(p_[0] for p_ in ph)
        ta = statistics.median(p_[1] for p_ in ph)
        qbytes = 3 * 2 * w.t_bytes + 3 * w.t_bytes // 2          # amax pass + quantise pass read, codes written
        res["fp8_quantise"] = {"GB/s": qbytes / tq / 1e9, "us": tq * 1e6, "bytes": qbytes}
        res["fp8_fwd"] = {"us": t * 1e6, "TFLOP/s": w.fwd_flop / t / 1e12, "attention_us": ta * 1e6,
                          "attention_TFLOP/s": w.fwd_flop / ta / 1e12}
    if w.ring > 1:
        R = w.ring
        outs = torch.randn((R, w.B, w.H, w.N, w.D), device="cuda").to(w.torch_dtype)
        lses = torch.randn((R, w.B, w.H, w.N), device="cuda")
        o = torch.empty(outs.shape[1:], dtype=outs.dtype, device="cuda")
        l = torch.empty(lses.shape[1:], device="cuda")
        t = timed(lambda: usp.lse_merge(outs, lses, out=o, lse=l))
        byt = (R + 1) * w.t_bytes + (R + 1) * w.B * w.H * w.N * 4
        res["lse_merge"] = {"GB/s": byt / t / 1e9, "us": t * 1e6, "bytes": byt}
    return res


def our_arm(args, w, ws, rank, local):
    torch.cuda.set_device(local)
    import diffusion_transformer_sequence_gb300 as usp
    usp.lib()
    peaks = load_peaks()
    step = Step(w, backward=not args.no_backward and not w.Nt)   # the joint path is forward-only
    # The headline steps carry events at their boundaries only: an event
    # between two calls would stop the next call's first kernel from starting
    # under the previous call's tail.  The per-call rows and the per-kernel
    # roofline come from a separate pass with events between the calls and
    # the library's phase events around the backward.
    mk = lambda: torch.cuda.Event(enable_timing=True)
    evs = [[mk(), None, None, mk()] for _ in range(args.steps)]
    nb = min(args.steps, 50)
    evb = [[mk(), mk(), mk(), mk()] for _ in range(nb)]
    L = usp.lib()
    import ctypes
    phase_ms = (ctypes.c_float * 8)()
    bwd_phases = []                      # per step: [prep, dK/dV kernel, dQ kernel] ms
    with ClockSampler(local) as clocks:
        for _ in range(args.warmup):
            step.flush()
            step.run(only=args.only)
        torch.cuda.synchronize()
        if usp.device_status() != 0:
            raise RuntimeError("device error status during warm-up")
        barrier(ws)
        torch.cuda.synchronize()
        clocks.mark("start")
        for i in range(args.steps):
            step.flush()
            step.run(evs[i], only=args.only)
        torch.cuda.synchronize()
        clocks.mark("end")
    step.bwd_phases = step.backward
    for i in range(nb):                    # per-call breakdown
        step.flush()
        step.run(evb[i], only=args.only)
        if step.backward and args.only in (None, "backward"):
            n = L.usp_profile_read(phase_ms, 8)   # waits for this step's last kernel
            bwd_phases.append([phase_ms[k] * 1e-3 for k in range(n)])
    torch.cuda.synchronize()
    step.bwd_phases = False
    _lib_check(L.usp_profile_phases(0))
    barrier(ws)
    if usp.device_status() != 0:
        raise RuntimeError("device error status during the timed steps")
    mat = [e[0].elapsed_time(e[1]) * 1e-3 for e in evb]
    fus = [e[1].elapsed_time(e[2]) * 1e-3 for e in evb]
    bwd = [e[2].elapsed_time(e[3]) * 1e-3 for e in evb]
    step_s = sum(e[0].elapsed_time(e[3]) * 1e-3 for e in evs) / args.steps
    step_s = max_over_ranks(step_s, ws)
    value = ws * step.flop() / step_s / 1e12

    # end to end through the public call with host buffers
    e2e = None
    if not args.no_e2e and args.only is None:
        step.run_e2e_pipelined(max(3, args.warmup))      # warm-up, also allocates the second buffer set
        barrier(ws)
        e2e_s = max_over_ranks(step.run_e2e_pipelined(args.steps) / args.steps, ws)
        h2d, d2h = step.io_bytes()
        e2e = {"value": ws * step.flop() / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
               "how": "pinned host buffers; per step H2D of the inputs then the L2 flush (on the copy stream, "
                      "before the step starts), the step, and D2H of every result, on three streams with two "
                      "device buffer sets (steps overlap)"}

    rows = time_rows(w) if (rank == 0 and not args.no_rows) else {}
    if rank != 0:
        return
    fused_s = statistics.mean(fus)
    mat_s = statistics.mean(mat)
    fwd_flop = w.joint_flop(True) if step.joint else w.fwd_flop
    fused_tflops = fwd_flop / fused_s / 1e12
    # The roofline denominator: the burst GEMM figure for work timed in short
    # runs, the sustained one (a seconds-long GEMM loop under the power cap)
    # once the timed region itself runs for seconds, since the kernel then
    # runs under the same cap (the fraction against the burst figure is
    # reported beside it).
    timed_s = step_s * args.steps
    long_run = timed_s >= 1.0
    peak = peaks["bf16_tflops_sustained"] if long_run else peaks["bf16_tflops"]
    # the dominant kernel of the step: the one with the largest device time per step
    kernels = {"attn_tc_fwd_kernel": (fused_s, w.fwd_flop, "fused USP forward (one launch per call)")}
    if step.joint:
        kernels = {"attn_tc_fwd_kernel": (fused_s, fwd_flop,
                                          "fused joint forward (image and text queries, one launch per call)")}
    overlapped = {}
    if bwd_phases and len(bwd_phases[0]) == 3:
        dkdv_s = statistics.mean(p[1] for p in bwd_phases)
        dq_s = statistics.mean(p[2] for p in bwd_phases)
        # The backward's two kernels run concurrently (dQ on the side stream, its CTAs interleaved
        # with dK/dV's), so they are one roofline unit: the algorithmic 10*B*H*N^2*D (five GEMMs;
        # the dQ kernel's recomputation of S and dP is not counted) over the time from the end of
        # the prep to the end of the later kernel.  dK/dV alone (8*B*H*N^2*D of it) is reported.
        pair_s = statistics.mean(max(p[1], p[2]) for p in bwd_phases)
        kernels["usp_bwd_dkdv_kernel+usp_bwd_dq_kernel"] = (
            pair_s, w.bwd_flop, "backward: dK/dV and dQ kernels, concurrent (S^T, dP^T, dV, dK | S, dP, dQ GEMMs)")
        overlapped["usp_bwd_dkdv_kernel_ms"] = dkdv_s * 1e3
        overlapped["usp_bwd_dkdv_kernel_tflops"] = 0.8 * w.bwd_flop / dkdv_s / 1e12
        overlapped["usp_bwd_dq_kernel_overlapped_ms"] = dq_s * 1e3
    dom = max(kernels, key=lambda k: kernels[k][0])
    t_dom, f_dom, desc = kernels[dom]
    ach = f_dom / t_dom / 1e12
    roofline = {"kernel": f"{dom}: {desc}", "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "traffic": kernel_traffic(dom, w.name),
                "traffic_source": ("profiles/traffic.json: dram__bytes_read.sum + dram__bytes_write.sum per launch "
                                   "from one ncu capture, valid while the kernel source hash recorded there "
                                   "matches (null otherwise)"),
                "launch_ms": t_dom * 1e3, "algorithmic_flop_per_launch": f_dom,
                "frac_of_burst": ach / peaks["bf16_tflops"],
                "peak_kind": (f"bf16 dense {'sustained' if long_run else 'burst'}, {peaks['source']} "
                              f"(burst {peaks['bf16_tflops']}, sustained {peaks['bf16_tflops_sustained']}); "
                              f"the timed region ran {timed_s:.2f} s, "
                              f"{'at least' if long_run else 'under'} the 1 s that selects the sustained figure")}
    for k, r in rows.items():
        if "GB/s" in r:
            r["frac_of_hbm"] = r["GB/s"] / peaks["hbm_gbs"]
    cpu = None
    if not args.no_cpu_baseline and ws == 1:   # the oracle baseline is taken on rank 0 of a 1-GPU run only
        heads = sample_heads(w)
        if oracle_sample_flop(w, heads) <= 0.5e12:
            dt, parity = run_oracle_sample(w, heads)
            cpu = {"value": oracle_sample_flop(w, heads) / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(),
                   "kind": "oracle", "sample": f"oracle USP forward (numpy fp64) on {heads} of {w.H} heads, full N, "
                                               f"{dt:.1f} s", "parity": parity,
                   "single_thread": oracle_single_thread(w, heads)}
        elif not step.joint:
            # heads on either side of a Ulysses head-group boundary, and the last head
            hs = sorted({0, w.Hu - 1, w.Hu, w.H - 1})
            cpu = oracle_rows_baseline(w, step, hs, 28672, cpu_cores())
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "desc": w.description, "global_batch": w.B * ws, "seq_len": w.N,
                   "heads": w.H, "head_dim": w.D, "ulysses": w.ulysses, "ring": w.ring,
                   "parallelism": f"{ws} independent replicas; u x r virtual ranks per device",
                   **({"text_len": w.Nt} if step.joint else {}),
                   "step": ("usp_attention_fwd_joint materialised + usp_attention_fwd_joint fused (with text queries)"
                            if step.joint else
                            "usp_attention_fwd materialised + usp_attention_fwd fused"
                            + (" + usp_attention_bwd" if step.backward else "")),
                   "l2": "flushed (256 MB write) before every timed step, outside the events; the device then "
                         "idles ~100 us so the step is enqueued before its start event",
                   "timing": "CUDA events at each step's boundaries; the per-call rows and the kernel roofline "
                             "from a separate pass of min(steps, 50) steps with events between the calls"},
        "rows": {"materialised_fwd_ms": mat_s * 1e3, "fused_fwd_ms": fused_s * 1e3,
                 "materialised_fwd_tflops": fwd_flop / mat_s / 1e12, "fused_fwd_tflops": fused_tflops,
                 **({"bwd_ms": statistics.mean(bwd) * 1e3,
                     "bwd_tflops": w.bwd_flop / statistics.mean(bwd) / 1e12} if step.backward else {}),
                 **({k + "_ms": v[0] * 1e3 for k, v in kernels.items()}),
                 **({k + "_tflops": v[1] / v[0] / 1e12 for k, v in kernels.items()}),
                 **overlapped,
                 **{k + "_GBps": v["GB/s"] for k, v in rows.items() if "GB/s" in v},
                 **{k + "_tflops": v["TFLOP/s"] for k, v in rows.items() if "TFLOP/s" in v},
                 **({"fp8_attention_kernel_tflops": rows["fp8_fwd"]["attention_TFLOP/s"]} if "fp8_fwd" in rows else {}),
                 **{k + "_frac_hbm": v["frac_of_hbm"] for k, v in rows.items() if "frac_of_hbm" in v}},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": step.launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "peaks": peaks,
    }
    print(json.dumps(line), flush=True)


def _lib_check(rc):
    from diffusion_transformer_sequence_gb300 import _lib
    _lib.check("usp_profile", rc)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about ten seconds of work: 400 for the 1024^2 workloads, 20 for Wan 720p)")
    ap.add_argument("--warmup", type=int, default=None, help="untimed warm-up steps (default 10, 3 for the Wan workloads)")
    ap.add_argument("--impl", default="usp", choices=["usp", "reference"])
    ap.add_argument("--workload", default="wan720p", choices=wl.ORDER + wl.JOINT)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row GB/s timings")
    ap.add_argument("--no-backward", action="store_true", help="leave usp_attention_bwd out of the step")
    ap.add_argument("--heads", type=int, default=None,
                    help="run the workload with this many heads (a multiple of its ulysses degree): a head-reduced "
                         "case of the same per-head shape for profiling captures; not a bench line")
    ap.add_argument("--only", choices=["materialised", "fused", "backward"], default=None,
                    help="run one of the two forward calls per step (profiling)")
    args = ap.parse_args()
    ws, rank, local = dist_env()
    w = wl.WORKLOADS[args.workload]
    if args.heads is not None:
        if args.heads < w.ulysses or args.heads % w.ulysses:
            raise SystemExit(f"--heads must be a positive multiple of {w.ulysses}")
        import dataclasses
        w = dataclasses.replace(w, H=args.heads, name=f"{w.name}_h{args.heads}",
                                description=f"{w.description}, {args.heads} of its {w.H} heads (profiling case)")
    big = w.N * w.N * w.H > 1e11
    if args.steps is None:
        args.steps = 20 if big else 400
    if args.warmup is None:
        args.warmup = 3 if big else 10
    if args.impl == "reference":
        reference_arm(args, w, ws, rank)
        return
    if ws > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        our_arm(args, w, ws, rank, local)
    finally:
        if ws > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
