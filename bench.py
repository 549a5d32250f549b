"""Benchmark of the HYPIC linear-attention state path on GB300s.

One step = one pass of the whole hot path over the long cold request
(30 GDN layers x 32 heads, d=128, bf16, 100,000 tokens in ~78 segments of
512-2048 tokens, 8-token seam windows):
  1. hypic_segment_build over every cached body (segment 0 whole, the
     others without their seam window) -- all layers x heads in one call;
  2. the reuse chain (hypic_reuse_chain, one launch): state = pair(segment
     0); for each internal segment, its 8 seam tokens (emitting
     o_t = S_t^T q_t), then the segment's body pair.
Inputs are drawn on the device (seeded) and stay resident; they total
~50 GB, far above the 129 MB L2, so no L2 flush is needed between steps.

On N GPUs (torchrun) the default is segment parallelism over one request:
each rank builds its longest-body-first share of the segments in batches and
streams every finished batch of pairs to rank 0, which then runs the reuse
chain (strong scaling).  ``--mode replicas`` runs one independent request
per GPU instead (weak scaling).  At N = 1 both are the single-GPU step.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on a fixed bounded sample of the same workload instead (the same
sample as the ``cpu_baseline`` leg).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "segment-build tokens/s (all layers×heads) + composes/s; % tensor/HBM roofline"
WORKLOAD = dict(n_layers=30, H=32, d=128, n_tokens=100_000, seam_w=8)
FLOP_PER_TOKEN_HEAD = 180_224      # chunk-64 low-rank GDN build (gram, W, U, two state GEMMs)
COMPOSE_BYTES = 131_072            # T_p + S_p (fp32, d=128) streamed per head-compose
SEAM_TOKEN_BYTES = 3 * 256 + 8 + 512  # per seam token-head: q, k, v bf16 in, a, b fp32 in, o fp32 out
# DRAM bytes per algorithmic byte of the build kernel, from an ncu capture of
# the 32-segment x 32-head ragged batch (820.2 MB of traffic: 719.1 MB read,
# 101.1 MB written, for 837.9 MB of inputs and outputs; output still in L2
# when the kernel ends is not counted as written); the full launch is too
# large to capture, and its traffic scales with the same units (token-heads
# in, (segment, head) out).
BUILD_TRAFFIC_RATIO = 819.81 / 837.89
BUILD_IN_BYTES_PER_TOKEN_HEAD = 520   # k, v bf16 (2 x 256 B) + alpha, beta fp32
COMPOSE_TABLE_DRAM_RATIO = 8.042 / 17.381  # DRAM / algorithmic bytes of the shared compose table (ncu)
BUILD_OUT_BYTES_PER_ITEM = 131_076    # T_C and S(C|0) fp32 (2 x 64 KB) + exponent


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 50 ms while running;
    summary() keeps the samples received inside the timed region (mark it with
    begin() and end())."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index  # CUDA ordinal; nvidia-smi is given the device's UUID when torch knows it
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def _smi_id(self):
        try:
            import torch
            u = str(torch.cuda.get_device_properties(self.index).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return str(self.index)

    def begin(self):
        self.t0 = time.time()

    def end(self):
        self.t1 = time.time()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self._smi_id()}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = self.rows
        if self.t0 is not None:  # (a sample is received up to one period after it is taken)
            t1 = self.t1 if self.t1 is not None else float("inf")
            rows = [r for r in rows if self.t0 <= r[0] <= t1 + 0.06]
        rows = [r[1] for r in rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ our arm ----

class LongRequest:
    """Device-resident inputs, outputs and argument blocks of one request."""

    def __init__(self, B, seed, device):
        import torch
        from linear_attn_state_hypic_gb300 import synth
        W = WORKLOAD
        self.B, self.torch = B, torch
        r = synth.long_request_device(seed=seed, n_layers=W["n_layers"], H=W["H"], d=W["d"],
                                      n_tokens=W["n_tokens"], seam_w=W["seam_w"], device=device)
        self.r = r
        self.cu = r["cu_seqlens"]
        self.skip = r["seam_skip"]
        self.n_seg = len(self.cu) - 1
        self.L, self.H, self.d = W["n_layers"], W["H"], W["d"]
        seam_tok = torch.from_numpy(r["seam_tok"]).to(device)
        # Seam-token inputs packed per internal segment (fresh tokens at reuse time).
        self.k_seam = r["k"][:, seam_tok].contiguous()
        self.v_seam = r["v"][:, seam_tok].contiguous()
        self.a_seam = r["alpha"][:, seam_tok].contiguous()
        self.b_seam = r["beta"][:, seam_tok].contiguous()
        self.q_seam = r["q_seam"]
        self.seam_off = np.concatenate([[0], np.cumsum(self.skip[1:])]).astype(np.int64)
        self.body_tokens = int(np.sum(np.diff(self.cu) - self.skip))
        self.T, self.T_exp, self.S = B.alloc_build_outputs("gdn", self.n_seg, self.L, self.H, self.d, self.d, device)
        self.state = torch.empty((1, self.L, self.H, self.d, self.d), dtype=torch.float32, device=device)
        self.state2 = torch.empty_like(self.state)
        self.o = torch.empty((self.L, len(r["seam_tok"]), self.H, self.d), dtype=torch.float32, device=device)
        self._make_args(device)

    def _make_args(self, device):
        B, torch = self.B, self.torch
        r = self.r
        self.keep = []
        self.bargs, k1 = B.build_args("gdn", r["k"], r["v"], self.cu, alpha=r["alpha"], beta=r["beta"],
                                      seam_skip=self.skip, T_out=self.T, T_exp_out=self.T_exp, S_out=self.S)
        self.keep.append(k1)
        self.ws_bytes = B.hypic_build_workspace_size(self.bargs)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        # The reuse chain: step 0 composes the first segment's pair onto a zero
        # state; step i >= 1 advances over the seam tokens of segment i and then
        # composes its body's pair (hypic_reuse_chain, one launch).
        cu_step = np.concatenate([[0, 0], np.cumsum(self.skip[1:])]).astype(np.int32)
        self.chain_args, k2 = B.chain_args("gdn", self.S, np.array([0, self.n_seg], np.int32),
                                           np.arange(self.n_seg, dtype=np.int32), cu_step,
                                           self.q_seam, self.k_seam, self.v_seam, T_tab=self.T, T_exp_tab=self.T_exp,
                                           alpha=self.a_seam, beta=self.b_seam, S_out=self.state, o_out=self.o)
        self.keep.append(k2)
        assert B.hypic_chain_workspace_size(self.chain_args) == 0, "the fused chain path needs no workspace"
        self.final = self.state

    def run_step(self, stream, ev=None):
        """One pass of the hot path; ev = (b0, b1, c0, c1) events around the build and the chain."""
        B = self.B
        if ev:
            ev[0].record()
        st = B.hypic_segment_build(self.bargs, self.ws.data_ptr(), self.ws_bytes, stream)
        if ev:
            ev[1].record()
        st |= B.hypic_reuse_chain(self.chain_args, None, 0, stream)
        if ev:
            ev[2].record()
        if st != 0:
            raise RuntimeError("a library call failed in the step")

    def launches_per_step(self):
        return 3   # build plan + build, reuse chain


class SegmentParallelRequest:
    """The long request over `world` ranks by segment parallelism: the
    longest-body-first partition of its segments; each rank's share packed
    (its own tokens only, as a scatter worker receives them) into up to
    n_batches hypic_segment_build calls whose pairs stream to rank 0 as each
    call finishes; rank 0 holds the seam tokens and runs the reuse chain over
    its table through the table's segment index (no placement copy)."""

    def __init__(self, B, seed, device, rank, world, n_batches=4):
        import torch
        from linear_attn_state_hypic_gb300 import shard, synth
        W = WORKLOAD
        self.B, self.torch, self.rank, self.world, self.n_batches = B, torch, rank, world, n_batches
        r = synth.long_request_device(seed=seed, n_layers=W["n_layers"], H=W["H"], d=W["d"],
                                      n_tokens=W["n_tokens"], seam_w=W["seam_w"], device=device)
        cu, skip = r["cu_seqlens"], r["seam_skip"]
        self.n_seg = len(cu) - 1
        self.L, self.H, self.d = W["n_layers"], W["H"], W["d"]
        self.parts = shard.lpt_partition(np.diff(cu) - skip, world)
        offsets, self.row_of = shard.combine_rows(self.parts)
        segs = self.parts[rank]
        rows = self.n_seg if rank == 0 else len(segs)
        self.tables = list(B.alloc_build_outputs("gdn", rows, self.L, self.H, self.d, self.d, device))
        base = int(offsets[rank]) if rank == 0 else 0
        self.batches, self.host_in = [], []
        for lo, hi in shard.batch_bounds(len(segs), n_batches):
            sub_cu, sub_skip, tok = shard.local_inputs(cu, skip, segs[lo:hi])
            t = torch.from_numpy(tok).to(device)
            ins = [r[key].index_select(1, t).contiguous() for key in ("k", "v", "alpha", "beta")]
            views = [x[base + lo:base + hi] for x in self.tables]
            args, keep = B.build_args("gdn", ins[0], ins[1], sub_cu, alpha=ins[2], beta=ins[3], seam_skip=sub_skip,
                                      T_out=views[0], T_exp_out=views[1], S_out=views[2])
            ws_bytes = B.hypic_build_workspace_size(args)
            ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
            self.batches.append((args, keep, ws, ws_bytes, ins))
        self.body_tokens = int(sum(int(cu[s + 1] - cu[s] - skip[s]) for s in segs))
        self.seam_ins = []
        if rank == 0:
            seam_tok = torch.from_numpy(r["seam_tok"]).to(device)
            self.seam_ins = [r[key][:, seam_tok].contiguous() for key in ("k", "v", "alpha", "beta")] + [r["q_seam"]]
            ks, vs, a_s, b_s, qs = self.seam_ins
            self.state = torch.empty((1, self.L, self.H, self.d, self.d), dtype=torch.float32, device=device)
            self.o = torch.empty((self.L, len(r["seam_tok"]), self.H, self.d), dtype=torch.float32, device=device)
            cu_step = np.concatenate([[0, 0], np.cumsum(skip[1:])]).astype(np.int32)
            T, Te, S = self.tables
            self.chain_args, self.chain_keep = B.chain_args(
                "gdn", S, np.array([0, self.n_seg], np.int32), self.row_of.astype(np.int32), cu_step, qs, ks, vs,
                T_tab=T, T_exp_tab=Te, alpha=a_s, beta=b_s, S_out=self.state, o_out=self.o)
            self.seam_tokens = int(len(r["seam_tok"]))
        del r
        torch.cuda.empty_cache()

    def device_inputs(self):
        return [x for b in self.batches for x in b[4]] + list(self.seam_ins)

    def run_step(self, stream):
        from linear_attn_state_hypic_gb300 import shard
        B = self.B

        def build_batch(lo, hi, views):
            args, _, ws, ws_bytes, _ = next(it)
            assert args.S_out == views[2].data_ptr(), "batch order"
            if B.hypic_segment_build(args, ws.data_ptr(), ws_bytes, stream) != 0:
                raise RuntimeError("build failed")

        it = iter(self.batches)
        shard.stream_pairs(build_batch, self.tables, self.parts, self.rank, dst=0, n_batches=self.n_batches)
        if self.rank == 0 and B.hypic_reuse_chain(self.chain_args, None, 0, stream) != 0:
            raise RuntimeError("reuse chain failed")

    def launches_per_step(self):
        return 2 * len(self.batches) + (1 if self.rank == 0 else 0)


def time_segment_parallel(args, rank, world, device):
    """The segment-parallel step (see SegmentParallelRequest), timed between
    barriers on every rank; the max over ranks is the step time.  Also the
    end-to-end variant: each rank copies its share's inputs (rank 0 also the
    seam tokens) from pinned host memory inside the timed step, and rank 0
    reads the end state and seam outputs back."""
    import torch
    from linear_attn_state_hypic_gb300 import binding as B
    torch.cuda.set_device(device)
    req = SegmentParallelRequest(B, seed=0, device=device, rank=rank, world=world, n_batches=args.sp_batches)
    sp = torch.cuda.current_stream().cuda_stream
    with ClockSampler(torch.cuda.current_device()) as clk:  # (started before the warm-up: nvidia-smi needs a moment)
        for _ in range(args.warmup):
            req.run_step(sp)
        torch.cuda.synchronize()
        B.check_device(sp)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        clk.begin()
        start.record()
        for _ in range(args.steps):
            req.run_step(sp)
        stop.record()
        torch.cuda.synchronize()
        clk.end()
    barrier(world)
    B.check_device(sp)
    ms = allreduce_max(start.elapsed_time(stop), world)
    res = dict(ms=ms, clocks=clk.summary(), n_seg=req.n_seg, launches=req.launches_per_step() * args.steps,
               body_tokens=req.body_tokens, req=req)
    if args.e2e_steps > 0:
        dev_in = req.device_inputs()
        host_in = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in dev_in]
        for h, d in zip(host_in, dev_in):
            h.copy_(d)
        outs = [req.state, req.o] if rank == 0 else []
        host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs]
        barrier(world)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.e2e_steps):
            for h, d in zip(host_in, dev_in):
                d.copy_(h, non_blocking=True)
            req.run_step(sp)
            for h, d in zip(host_out, outs):
                h.copy_(d, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        barrier(world)
        res["e2e_ms"] = allreduce_max(a.elapsed_time(b), world) / args.e2e_steps
        res["h2d"] = allreduce_sum(sum(x.numel() * x.element_size() for x in host_in), world)
        res["d2h"] = sum(x.numel() * x.element_size() for x in host_out)
    return res


def time_our_arm(args, rank, world, device):
    import torch
    from linear_attn_state_hypic_gb300 import binding as B

    torch.cuda.set_device(device)
    req = LongRequest(B, seed=rank, device=device)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    with ClockSampler(torch.cuda.current_device()) as clk:  # (started before the warm-up: nvidia-smi needs a moment)
        for _ in range(args.warmup):
            req.run_step(sp)
        B.check_device(sp)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        clk.begin()
        start.record()
        for s in range(args.steps):
            req.run_step(sp, ev[s])
        stop.record()
        torch.cuda.synchronize()
        clk.end()
    barrier(world)
    B.check_device(sp)
    ms = start.elapsed_time(stop)
    build_ms = [e[0].elapsed_time(e[1]) for e in ev]
    chain_ms = [e[1].elapsed_time(e[2]) for e in ev]
    ms_max = allreduce_max(ms, world)
    res = dict(ms=ms_max, build_ms=statistics.mean(build_ms), chain_ms=statistics.mean(chain_ms),
               clocks=clk.summary(), body_tokens=req.body_tokens, n_seg=req.n_seg,
               seam_tokens=int(req.q_seam.shape[1]),
               launches=req.launches_per_step() * args.steps, req=req)
    return res


def e2e_our_arm(req, steps, seed, device):
    """Same step through the public C ABI with host inputs: every step copies
    the request's inputs from pinned host memory to the device (50 GB) and
    reads the final state and the seam outputs back.  The copy of step s + 1
    runs on its own stream while step s computes, into the other of two device
    input sets (a serving loop streaming requests): the step time is then the
    copy's, not the copy's plus the compute's."""
    import torch
    from linear_attn_state_hypic_gb300 import binding as B
    reqs = [req, LongRequest(B, seed=seed, device=device)]  # same shapes; its inputs are copied over every use
    ins = [[q.r["k"], q.r["v"], q.r["alpha"], q.r["beta"], q.q_seam, q.k_seam, q.v_seam, q.a_seam, q.b_seam]
           for q in reqs]
    t0 = time.time()
    host_in = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in ins[0]]
    for h, d in zip(host_in, ins[0]):
        h.copy_(d)
    outs = [[q.final, q.o] for q in reqs]
    host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs[0]]
    setup_s = time.time() - t0
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    copied = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    started = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]  # each in-loop copy, timed on its stream
    done = [torch.cuda.Event() for _ in range(steps)]
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    copy.wait_event(a)
    for s in range(steps):
        k = s % 2
        with torch.cuda.stream(copy):
            if s >= 2:
                copy.wait_event(done[s - 2])  # step s - 2 has finished with this input set
            started[s].record(copy)
            for h, d in zip(host_in, ins[k]):
                d.copy_(h, non_blocking=True)
            copied[s].record(copy)
        comp.wait_event(copied[s])
        reqs[k].run_step(comp.cuda_stream)
        for h, d in zip(host_out, outs[k]):
            h.copy_(d, non_blocking=True)
        done[s].record(comp)
    b.record(comp)
    torch.cuda.synchronize()
    B.check_device()
    ms = a.elapsed_time(b) / steps
    loop_copy_ms = statistics.mean(started[s].elapsed_time(copied[s]) for s in range(steps))
    # the host link on its own: one step's input copy with nothing else running
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(copy):
        c0.record(copy)
        for h, d in zip(host_in, ins[0]):
            d.copy_(h, non_blocking=True)
        c1.record(copy)
    torch.cuda.synchronize()
    copy_ms = c0.elapsed_time(c1)
    del reqs[1]
    return dict(ms=ms, h2d=h2d, d2h=d2h, setup_s=setup_s, copy_ms=copy_ms, loop_copy_ms=loop_copy_ms)


# ------------------------------------------------------- oracle (CPU) arm --

# The CPU baseline's bounded sample of the long request, the same for the
# reference arm and the cpu_baseline leg: layer 0, heads 0-15 and the first 24
# segments (their true lengths, ~30k tokens): the build of every body, then
# the chain of seam advances and composes, in fp64.
ORACLE_SAMPLE = dict(heads=16, n_seg=24)


def oracle_sample(seed=0):
    from linear_attn_state_hypic_gb300 import synth
    n_seg, heads = ORACLE_SAMPLE["n_seg"], ORACLE_SAMPLE["heads"]
    lengths = synth.long_request_lengths(seed, WORKLOAD["n_tokens"])[:n_seg]
    inp = synth.gdn_ragged(seed=seed, H=heads, d=WORKLOAD["d"], lengths=lengths, with_q=True)
    skip = np.full(n_seg, WORKLOAD["seam_w"], np.int32)
    skip[0] = 0
    return inp, skip


def run_oracle_sample(inp, skip, threads):
    """The oracle's version of the step on the sample: build the bodies, then
    seam-advance and compose along the chain."""
    from oracle import oracle as orc
    cu = inp["cu_seqlens"]
    T, S = orc.build_pairs("gdn", inp["k"], inp["v"], cu, alpha=inp["alpha"], beta=inp["beta"], skip=skip,
                           n_threads=threads)
    state = orc.compose("gdn", T, S, [0, 1], [0], n_threads=threads)
    for i in range(1, len(cu) - 1):
        sl = slice(int(cu[i]), int(cu[i]) + int(skip[i]))
        sub = {key: np.ascontiguousarray(inp[key][:, sl]) for key in ("q", "k", "v", "alpha", "beta")}
        state, _ = orc.seam("gdn", sub["q"], sub["k"], sub["v"], [0, int(skip[i])], state_in=state,
                            alpha=sub["alpha"], beta=sub["beta"], n_threads=threads)
        state = orc.compose("gdn", T, S, [0, 1], [i], S0=state, n_threads=threads)
    return state


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


def time_oracle(runs, warmup, threads):
    """Run the fixed sample warmup + runs times; returns (tokens/s scaled to
    the whole request's layers x heads, seconds per run, description)."""
    inp, skip = oracle_sample()
    for _ in range(warmup):
        run_oracle_sample(inp, skip, threads)
    t0 = time.time()
    for _ in range(runs):
        run_oracle_sample(inp, skip, threads)
    secs = (time.time() - t0) / runs
    toks = float(inp["cu_seqlens"][-1])
    heads = ORACLE_SAMPLE["heads"]
    rate = toks * heads / secs / (WORKLOAD["n_layers"] * WORKLOAD["H"])
    desc = (f"layer 0 of 30, heads 0-{heads - 1} of 32, the first {ORACLE_SAMPLE['n_seg']} segments "
            f"({int(toks)} tokens): build, seam advance and compose in fp64, {runs} runs; rate scaled to all "
            f"30x32 layer-heads")
    return rate, secs, desc


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_sum(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def allreduce_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_compose_table(steps, device, n_layers=30, shared=True):
    """hypic_compose on a compose table.  shared=True: the compose-table
    workload, 30 layers x 32 heads, a table of 128 cached pairs (fp32 T
    mantissa + exponent, S), 16 chains of 64 distinct pairs each (half from
    zero, half from a random start); chains that draw the same pair re-read
    it, mostly from L2.  shared=False: the same chains over a table of
    16 x 64 = 1,024 pairs, each read by one chain only (4 layers, 17.2 GB), so
    DRAM traffic equals the algorithmic bytes.  The T values are random with
    spectral norm ~0.7 (the kernel's time does not depend on them).  Returns
    timing and the algorithmic-byte roofline."""
    import torch
    from linear_attn_state_hypic_gb300 import binding as B
    from linear_attn_state_hypic_gb300 import synth
    H, d, n_chain, n_steps = 32, 128, 16, 64
    L = n_layers if shared else 4
    P = 128 if shared else n_chain * n_steps
    ch = synth.compose_chains(seed=0, n_pairs=P if shared else 128, n_layers=L, with_tables=False)
    seg_idx = ch["seg_idx"]
    if not shared:
        seg_idx = np.random.default_rng(2).permutation(P).astype(np.int32)
    g = torch.Generator(device=device)
    g.manual_seed(1)
    T_tab = torch.randn((P, L, H, d, d), generator=g, device=device) * (0.35 / np.sqrt(d))
    S_tab = torch.randn((P, L, H, d, d), generator=g, device=device) * (1.0 / np.sqrt(d))
    T_exp = torch.randint(-2, 2, (P, L, H), generator=g, device=device, dtype=torch.int32)
    S0 = torch.from_numpy(ch["S0"]).to(device)
    out = torch.empty_like(S0)
    a, keep = B.compose_args("gdn", S_tab, ch["cu_chain"], seg_idx, T_tab=T_tab, T_exp_tab=T_exp, S0=S0,
                             S_out=out)
    sp = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        if B.hypic_compose(a, sp) != 0:
            raise RuntimeError("compose failed")
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        B.hypic_compose(a, sp)
    e1.record()
    torch.cuda.synchronize()
    B.check_device(sp)
    ms = e0.elapsed_time(e1) / steps
    head_composes = n_chain * n_steps * L * H
    state_bytes = d * d * 4 * L * H
    algo = head_composes * COMPOSE_BYTES + n_chain * state_bytes + (n_chain // 2) * state_bytes
    del keep, T_tab, S_tab
    r = {"workload": (f"compose table: {L} layers x 32 heads, d=128, fp32 pairs ({P} cached segments), "
                      f"16 chains x 64 pairs, half from a random start state"
                      + ("" if shared else ", no pair read by two chains")),
         "ms_per_call": ms, "head_composes_per_s": head_composes / (ms / 1e3),
         "composes_per_s": n_chain * n_steps / (ms / 1e3),
         "algorithmic_bytes": algo, "gbs_algorithmic": algo / (ms / 1e3) / 1e9}
    if shared:
        # DRAM bytes per algorithmic byte from an ncu capture of the same kernel on the 4-layer table
        # (8.04 GB of DRAM traffic for 17.38 GB algorithmic): chains that share a (layer, head) pair
        # re-read it from L2
        r["dram_bytes_est"] = algo * COMPOSE_TABLE_DRAM_RATIO
        r["gbs_dram_est"] = r["dram_bytes_est"] / (ms / 1e3) / 1e9
        r["note"] = ("chains that share a pair run on neighbouring SMs and re-read it from L2: algorithmic GB/s "
                     "exceeds the DRAM traffic (gbs_dram_est, scaled from ncu)")
    else:
        r["gbs_dram_est"] = r["gbs_algorithmic"]
        r["note"] = "every pair is read by one chain only: DRAM traffic equals the algorithmic bytes"
    return r


def time_reuse_chain(steps, warmup, device, n_layers=30, H=32, d=128, n_steps=77, w=8):
    """hypic_reuse_chain over one request's chain (the long request's shape:
    n_steps cached pairs, a w-token seam before every step but the first) for
    n_layers x H heads; random pair tables (T with spectral norm ~0.7)."""
    import torch
    from linear_attn_state_hypic_gb300 import binding as B
    g = torch.Generator(device=device)
    g.manual_seed(0)
    T = torch.randn((n_steps, n_layers, H, d, d), generator=g, device=device) * (0.35 / d ** 0.5)
    S = torch.randn((n_steps, n_layers, H, d, d), generator=g, device=device) / d ** 0.5
    Te = torch.zeros((n_steps, n_layers, H), dtype=torch.int32, device=device)
    N = (n_steps - 1) * w
    q = torch.randn((n_layers, N, H, d), generator=g, device=device)
    k = torch.randn((n_layers, N, H, d), generator=g, device=device)
    q = (q / q.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    v = torch.randn((n_layers, N, H, d), generator=g, device=device).to(torch.bfloat16)
    al = torch.rand((n_layers, N, H), generator=g, device=device) * 0.15 + 0.85
    be = torch.rand((n_layers, N, H), generator=g, device=device)
    cu_step = np.concatenate([[0, 0], np.cumsum([w] * (n_steps - 1))]).astype(np.int32)
    out = torch.empty((1, n_layers, H, d, d), device=device)
    o = torch.empty((n_layers, N, H, d), device=device)
    a, keep = B.chain_args("gdn", S, np.array([0, n_steps], np.int32), np.arange(n_steps, dtype=np.int32), cu_step,
                           q, k, v, T_tab=T, T_exp_tab=Te, alpha=al, beta=be, S_out=out, o_out=o)
    sp = torch.cuda.current_stream().cuda_stream
    for _ in range(warmup):
        B._check(B.hypic_reuse_chain(a, None, 0, sp))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        B._check(B.hypic_reuse_chain(a, None, 0, sp))
    e1.record()
    torch.cuda.synchronize()
    B.check_device()
    del keep
    ms = e0.elapsed_time(e1) / steps
    LH = n_layers * H
    algo = n_steps * LH * COMPOSE_BYTES + N * LH * SEAM_TOKEN_BYTES + LH * d * d * 4
    return {"workload": f"reuse chain: {n_layers} layers x {H} heads, d={d}, {n_steps} steps, {w}-token seams",
            "ms_per_call": ms, "algorithmic_bytes": algo, "gbs_algorithmic": algo / (ms / 1e3) / 1e9}


def time_seam_advance(steps, warmup, device, n_layers=30, H=32, d=128, n_seams=76, w=8):
    """hypic_seam_advance on the long request's seams (GDN, d=128, bf16 q/k/v,
    fp32 gates): n_seams windows of w tokens for every (layer, head), each state
    advanced in place.  Algorithmic bytes: the state read and written
    (2 x 65,536 B per seam-head), q, k, v (bf16) and alpha, beta (fp32) per
    token-head in, o (fp32) out.  Returns timing and the algorithmic-byte rate."""
    import torch
    from linear_attn_state_hypic_gb300 import binding as B
    g = torch.Generator(device=device)
    g.manual_seed(5)
    N = n_seams * w
    def rows():
        x = torch.randn((n_layers, N, H, d), generator=g, device=device)
        return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    q, k = rows(), rows()
    v = torch.randn((n_layers, N, H, d), generator=g, device=device).to(torch.bfloat16)
    alpha = 0.85 + 0.15 * torch.rand((n_layers, N, H), generator=g, device=device)
    beta = torch.rand((n_layers, N, H), generator=g, device=device)
    state = torch.randn((n_seams, n_layers, H, d, d), generator=g, device=device) / d ** 0.5
    o = torch.empty((n_layers, N, H, d), dtype=torch.float32, device=device)
    cu = np.arange(0, N + 1, w, dtype=np.int32)
    cu_dev = torch.from_numpy(cu).to(device)
    sp = torch.cuda.current_stream().cuda_stream
    for _ in range(warmup):
        B.seam_advance("gdn", q, k, v, cu, alpha=alpha, beta=beta, state_in=state, state_out=state, o_out=o,
                       stream=sp, cu_seam_dev=cu_dev)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        B.seam_advance("gdn", q, k, v, cu, alpha=alpha, beta=beta, state_in=state, state_out=state, o_out=o,
                       stream=sp, cu_seam_dev=cu_dev)
    e1.record()
    torch.cuda.synchronize()
    B.check_device(sp)
    ms = e0.elapsed_time(e1) / steps
    seam_heads = n_seams * n_layers * H
    algo = seam_heads * 2 * d * d * 4 + N * n_layers * H * (3 * d * 2 + 8 + d * 4)
    return {"workload": (f"seam advance: {n_seams} windows of {w} tokens x {n_layers} layers x {H} heads, "
                         f"GDN d={d}, bf16 q/k/v, state in place"),
            "ms_per_call": ms, "seam_heads_per_s": seam_heads / (ms / 1e3), "algorithmic_bytes": algo,
            "gbs_algorithmic": algo / (ms / 1e3) / 1e9}


def time_decay_build(family, steps, warmup, device, n_layers=30, H=32, d=128, n_tokens=100_000):
    """hypic_segment_build of a decay family (retnet, mamba2, gla, vanilla) over
    the long request's segments (100k tokens, U[512,2048] lengths, no seam
    window) for n_layers x H heads, bf16 keys and values; gates as in the
    small decay workload (RetNet gamma_h = 1 - 2^(-5-h mod 8), GLA g = sigmoid(N(2,1)),
    Mamba2 a ~ U(0.9, 1)).  HBM roofline over the algorithmic bytes: keys,
    values and gates in, S (and T) out."""
    import torch
    from linear_attn_state_hypic_gb300 import binding as B
    from linear_attn_state_hypic_gb300 import synth
    lengths = synth.long_request_lengths(0, n_tokens)
    cu = synth.cu_from_lengths(lengths)
    n_seg = len(lengths)
    g = torch.Generator(device=device)
    g.manual_seed(0)
    k = torch.empty((n_layers, n_tokens, H, d), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    for layer in range(n_layers):
        x = torch.randn((n_tokens, H, d), generator=g, device=device)
        k[layer] = (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
        v[layer] = torch.randn((n_tokens, H, d), generator=g, device=device).to(torch.bfloat16)
        del x
    kw, gate_bytes = {}, 0
    if family == "retnet":
        kw["gamma"] = (1.0 - 2.0 ** (-5.0 - (torch.arange(H, device=device) % 8).float())).repeat(n_layers, 1)
        kw["gamma"] = kw["gamma"].contiguous()
    elif family == "mamba2":
        kw["alpha"] = torch.rand((n_layers, n_tokens, H), generator=g, device=device) * 0.1 + 0.9
        gate_bytes = 4
    elif family == "gla":
        kw["g"] = torch.empty((n_layers, n_tokens, H, d), dtype=torch.float32, device=device)
        for layer in range(n_layers):
            kw["g"][layer] = torch.sigmoid(torch.randn((n_tokens, H, d), generator=g, device=device) + 2.0)
        gate_bytes = 4 * d
    out = B.alloc_build_outputs(family, n_seg, n_layers, H, d, d, device)
    for _ in range(warmup):
        B.segment_build(family, k, v, cu, out=out, **kw)
    torch.cuda.synchronize()
    B.check_device()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        B.segment_build(family, k, v, cu, out=out, **kw)
    e1.record()
    torch.cuda.synchronize()
    B.check_device()
    ms = e0.elapsed_time(e1) / steps
    LH = n_layers * H
    t_bytes = {"retnet": 4, "mamba2": 4, "gla": 4 * d, "vanilla": 0}[family]
    algo = n_tokens * LH * (2 * d * 2 + gate_bytes) + n_seg * LH * (d * d * 4 + t_bytes)
    return {"workload": (f"{family} build: {n_layers} layers x {H} heads, d={d}, bf16 k/v, {n_tokens} tokens in "
                         f"{n_seg} segments of U[512,2048] tokens"),
            "ms_per_call": ms, "tokens_per_s": n_tokens / (ms / 1e3),
            "token_heads_per_s": n_tokens * LH / (ms / 1e3), "algorithmic_bytes": algo,
            "gbs_algorithmic": algo / (ms / 1e3) / 1e9,
            "tflops": n_tokens * LH * 2 * d * d * (2 if family != "vanilla" else 1) / (ms / 1e3) / 1e12}


def time_kda_build(steps, warmup, device, n_layers=1, H=32, d=128, n_tokens=100_000):
    """hypic_segment_build of KDA over the long request's segments (100k tokens,
    U[512,2048] lengths, no seam window) for n_layers x H heads, bf16 keys and
    values, per-channel gates a ~ U(0.85, 1), b ~ U(0, 1).  The tensor-core path
    (chunk pairs, then the compose of each segment's chunks) against the
    CUDA-core kernel on the same inputs (the no-alloc build runs KDA there).
    Bytes: algorithmic = keys, values, gates and b in, T and S out; path = that
    plus the chunk tables (T and S of every 64-token chunk written once, read by
    the compose's state and transition launches: 64 KB x 5 per chunk and head)."""
    import torch
    from linear_attn_state_hypic_gb300 import binding as B
    from linear_attn_state_hypic_gb300 import synth
    lengths = synth.long_request_lengths(0, n_tokens)
    cu = synth.cu_from_lengths(lengths)
    n_seg = len(lengths)
    gen = torch.Generator(device=device)
    gen.manual_seed(0)
    k = torch.empty((n_layers, n_tokens, H, d), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    g = torch.empty((n_layers, n_tokens, H, d), dtype=torch.float32, device=device)
    for layer in range(n_layers):
        x = torch.randn((n_tokens, H, d), generator=gen, device=device)
        k[layer] = (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
        v[layer] = torch.randn((n_tokens, H, d), generator=gen, device=device).to(torch.bfloat16)
        g[layer] = torch.rand((n_tokens, H, d), generator=gen, device=device) * 0.15 + 0.85
        del x
    beta = torch.rand((n_layers, n_tokens, H), generator=gen, device=device)
    out = B.alloc_build_outputs("kda", n_seg, n_layers, H, d, d, device)
    out2 = B.alloc_build_outputs("kda", n_seg, n_layers, H, d, d, device)
    a, keep = B.build_args("kda", k, v, cu, g=g, beta=beta, T_out=out[0], T_exp_out=out[1], S_out=out[2])
    a2, keep2 = B.build_args("kda", k, v, cu, g=g, beta=beta, T_out=out2[0], T_exp_out=out2[1], S_out=out2[2])
    need = B.hypic_build_workspace_size(a)
    ws = torch.empty(need, dtype=torch.uint8, device=device)

    def tc():
        B._check(B.hypic_segment_build(a, B._ptr(ws), ws.numel(), B._stream(None)))

    def cores():
        B._check(B.hypic_segment_build_noalloc(a2, B._stream(None)))

    def timed(f, n):
        for _ in range(warmup):
            f()
        torch.cuda.synchronize()
        B.check_device()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            f()
        e1.record()
        torch.cuda.synchronize()
        B.check_device()
        return e0.elapsed_time(e1) / n

    ms = timed(tc, steps)
    ms_cores = timed(cores, max(1, steps // 2))
    S1, S2 = out[2].double(), out2[2].double()
    rel_s = float((S1 - S2).norm() / S2.norm())
    LH = n_layers * H
    n_chunks = int(sum((int(x) + 63) // 64 for x in lengths))
    algo = n_tokens * LH * (2 * d * 2 + 4 * d + 4) + n_seg * LH * (2 * d * d * 4 + 4)
    path = algo + n_chunks * LH * 5 * d * d * 4
    del keep, keep2
    return {"workload": (f"kda build: {n_layers} layers x {H} heads, d={d}, bf16 k/v, fp32 gates, {n_tokens} tokens "
                         f"in {n_seg} segments of U[512,2048] tokens ({n_chunks} chunks of 64)"),
            "ms_per_call": ms, "ms_per_call_cuda_cores": ms_cores, "speedup_vs_cuda_cores": ms_cores / ms,
            "tokens_per_s": n_tokens / (ms / 1e3), "token_heads_per_s": n_tokens * LH / (ms / 1e3),
            "workspace_bytes": need, "algorithmic_bytes": algo, "path_bytes": path,
            "gbs_algorithmic": algo / (ms / 1e3) / 1e9, "gbs_path": path / (ms / 1e3) / 1e9,
            "rel_S_tc_vs_cuda_cores": rel_s}


def run_case(args, device):
    """Single-kernel cases used for profiling (one JSON line each):
    ragged_build -- the build of 32 ragged segments (U[512,2048] tokens) x 32
                    heads, d=128, bf16 (one layer);
    compose_table -- hypic_compose on the compose table with --layers layers;
    reuse_chain -- hypic_reuse_chain over the long request's chain;
    seam_advance -- hypic_seam_advance on the long request's seams (GDN);
    decay_build -- a decay family's build at serving scale (--family);
    kda_build -- KDA's build over the long request's segments (--layers), the
                 tensor-core path against the CUDA-core kernel."""
    import torch
    from linear_attn_state_hypic_gb300 import binding as B
    from linear_attn_state_hypic_gb300 import synth
    torch.cuda.set_device(device)
    peaks, peak_src = load_peaks()
    if args.case == "compose_table":
        r = time_compose_table(args.steps, device, n_layers=args.layers)
        r["frac_hbm"] = r["gbs_algorithmic"] / peaks["hbm_gbs"]
        print(json.dumps({"case": args.case, **r}))
        return
    if args.case == "kda_build":
        r = time_kda_build(args.steps, args.warmup, device, n_layers=args.layers, n_tokens=args.tokens)
        r["frac_hbm_path"] = r["gbs_path"] / peaks["hbm_gbs"]
        print(json.dumps({"case": args.case, **r}))
        return
    if args.case == "decay_build":
        r = time_decay_build(args.family, args.steps, args.warmup, device, n_layers=args.layers)
        r["frac_hbm"] = r["gbs_algorithmic"] / peaks["hbm_gbs"]
        print(json.dumps({"case": args.case, **r}))
        return
    if args.case == "seam_advance":
        r = time_seam_advance(args.steps, args.warmup, device, n_layers=args.layers)
        r["frac_hbm"] = r["gbs_algorithmic"] / peaks["hbm_gbs"]
        print(json.dumps({"case": args.case, **r}))
        return
    if args.case == "reuse_chain":
        r = time_reuse_chain(args.steps, args.warmup, device, n_layers=args.layers)
        r["frac_hbm"] = r["gbs_algorithmic"] / peaks["hbm_gbs"]
        print(json.dumps({"case": args.case, **r}))
        return
    print(json.dumps({"case": args.case, **time_ragged_build(args.steps, args.warmup, device, peaks, peak_src)}))


def time_ragged_build(steps, warmup, device, peaks, peak_src):
    """hypic_segment_build of GDN on 32 ragged segments (U[512,2048] tokens) x 32 heads, d=128,
    bf16, one layer: the build kernel alone at a small scale, against the bf16 peaks."""
    import torch
    from linear_attn_state_hypic_gb300 import binding as B
    from linear_attn_state_hypic_gb300 import synth
    inp = synth.gdn_ragged(seed=0)
    k = torch.from_numpy(inp["k"]).to(torch.bfloat16).to(device)
    v = torch.from_numpy(inp["v"]).to(torch.bfloat16).to(device)
    a = torch.from_numpy(inp["alpha"]).to(device)
    b = torch.from_numpy(inp["beta"]).to(device)
    cu = inp["cu_seqlens"]
    out = B.alloc_build_outputs("gdn", len(cu) - 1, 1, 32, 128, 128, device)
    for _ in range(warmup):
        B.segment_build("gdn", k, v, cu, alpha=a, beta=b, out=out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        B.segment_build("gdn", k, v, cu, alpha=a, beta=b, out=out)
    e1.record()
    torch.cuda.synchronize()
    B.check_device()
    ms = e0.elapsed_time(e1) / steps
    ntok = int(cu[-1])
    tf = ntok * 32 * FLOP_PER_TOKEN_HEAD / (ms / 1e3) / 1e12
    return {"workload": "GDN build: 32 segments of U[512,2048] tokens x 32 heads, d=128, bf16 k/v, one layer",
            "ms_per_call": ms, "tokens": ntok, "heads": 32, "tokens_per_s": ntok / (ms / 1e3), "tflops": tf,
            "frac_bf16_burst": tf / peaks["bf16_tflops"],
            "frac_bf16_sustained": tf / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]),
            "peak_source": peak_src}


def workload_config(n_seg=None):
    W = WORKLOAD
    return {"workload": (f"long cold request + seam: {W['n_layers']} GDN layers x {W['H']} heads, d={W['d']}, "
                         f"bf16 k/v/q, fp32 gates/state, {W['n_tokens']} tokens in "
                         f"{n_seg if n_seg else '~78'} segments of U[512,2048] tokens, "
                         f"{W['seam_w']}-token seam at each internal segment start"),
            "n_layers": W["n_layers"], "n_heads": W["H"], "d": W["d"], "n_tokens": W["n_tokens"],
            "n_segments": n_seg, "seam_w": W["seam_w"],
            "l2": "inputs ~50 GB resident, far above the 129 MB L2: no flush between steps",
            "parallelism": "one request per GPU (N = 1; --mode replicas at N > 1: independent requests, "
                           "no collective)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["auto", "segment_parallel", "replicas"], default="auto",
                    help="auto: the single-GPU step at N = 1, segment parallelism over one request at N > 1")
    ap.add_argument("--sp-batches", type=int, default=4, help="build calls per rank in segment-parallel mode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=4)
    ap.add_argument("--no-compose-table", action="store_true")
    ap.add_argument("--case", choices=["long_request", "ragged_build", "compose_table", "reuse_chain", "decay_build", "kda_build",
                                      "seam_advance"],
                    default="long_request",
                    help="long_request is the benchmark; the others time one kernel (for profiling)")
    ap.add_argument("--tokens", type=int, default=100_000, help="request tokens of the kda_build case")
    ap.add_argument("--layers", type=int, default=30, help="layers of the compose_table, reuse_chain, decay_build, kda_build cases")
    ap.add_argument("--family", choices=["retnet", "mamba2", "gla", "vanilla"], default="retnet",
                    help="family of the decay_build case")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    threads = os.cpu_count() or 1

    if args.impl == "reference":
        if rank != 0:
            return
        rate, secs, desc = time_oracle(args.steps, args.warmup, threads)
        line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload_config(),
                "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": threads, "cpu": cpu_model(),
                                 "kind": "oracle", "sample": desc},
                "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if args.case != "long_request":
        if rank == 0:
            run_case(args, int(os.environ.get("LOCAL_RANK", "0")))
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    seg_par = args.mode == "segment_parallel" or (args.mode == "auto" and world > 1)
    peaks, peak_src = load_peaks()
    W = WORKLOAD
    LH = W["n_layers"] * W["H"]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, secs, desc = time_oracle(6, 1, threads)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "cpu": cpu_model(), "kind": "oracle",
               "sample": desc, "seconds": round(6 * secs, 2)}
    if seg_par:
        res = time_segment_parallel(args, rank, world, device)
        res.pop("req")
        ms_step = res["ms"] / args.steps
        if rank != 0:
            return
        e2e = None
        if "e2e_ms" in res:
            e2e = {"value": W["n_tokens"] / (res["e2e_ms"] / 1e3), "unit": "tokens/s",
                   "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"], "ms_per_step": res["e2e_ms"],
                   "steps": args.e2e_steps,
                   "overlap": "none: each rank copies its share's inputs, then builds and streams"}
        line = {
            "metric": METRIC, "value": W["n_tokens"] * args.steps / (res["ms"] / 1e3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, drawn on the device)",
            "config": dict(workload_config(res["n_seg"]),
                           parallelism=(f"segment parallelism over {world} GPU(s): longest-body-first shares, "
                                        f"{args.sp_batches} build calls per rank streamed to rank 0 (NCCL "
                                        "point-to-point), the reuse chain on rank 0")),
            "composes_per_s": res["n_seg"] * args.steps / (res["ms"] / 1e3),
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": res["launches"], "clocks": res["clocks"],
        }
        print(json.dumps(line))
        return

    res = time_our_arm(args, rank, world, device)
    req = res.pop("req")
    ms_step = res["ms"] / args.steps
    value = world * W["n_tokens"] * args.steps / (res["ms"] / 1e3)
    build_flop = res["body_tokens"] * LH * FLOP_PER_TOKEN_HEAD
    build_tflops = build_flop / (res["build_ms"] / 1e3) / 1e12
    peak_t = peaks["bf16_tflops"]
    peak_ts = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    n_comp = res["n_seg"]
    # the fused chain keeps the running state on chip: the pair stream, the
    # seam tokens and their outputs, and the end state
    chain_bytes = (n_comp * LH * COMPOSE_BYTES + res["seam_tokens"] * LH * SEAM_TOKEN_BYTES
                   + LH * WORKLOAD["d"] ** 2 * 4)
    chain_gbs = chain_bytes / (res["chain_ms"] / 1e3) / 1e9
    e2e = None
    if args.e2e_steps > 0:
        try:
            e = e2e_our_arm(req, args.e2e_steps, rank, device)
            copy_gbs = e["h2d"] / (e["copy_ms"] / 1e3) / 1e9
            loop_gbs = e["h2d"] / (e["loop_copy_ms"] / 1e3) / 1e9
            # overlap from the loop's own copy times (a copy next to the compute runs slower than one alone)
            lo, hi = min(e["loop_copy_ms"], ms_step), max(e["loop_copy_ms"], ms_step)
            overlap = min(1.0, max(0.0, (lo + hi - e["ms"]) / lo)) if lo > 0 else None
            e2e = {"value": world * W["n_tokens"] / (e["ms"] / 1e3), "unit": "tokens/s",
                   "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"], "ms_per_step": e["ms"],
                   "steps": args.e2e_steps, "h2d_ms": e["copy_ms"], "h2d_gbs": copy_gbs,
                   "h2d_ms_in_loop": e["loop_copy_ms"], "h2d_gbs_in_loop": loop_gbs, "overlap_frac": overlap,
                   "overlap": ("the host-to-device copy of step s+1 runs during step s (two device input sets); "
                               "h2d_gbs: one copy alone; h2d_gbs_in_loop: the copies inside the timed loop; "
                               "overlap_frac = share of the shorter of in-loop copy and compute hidden under the "
                               "longer")}
        except Exception as ex:  # pinned host memory can be unavailable; report why
            e2e = {"value": None, "unit": "tokens/s", "error": f"{type(ex).__name__}: {ex}"[:200]}
    ctab = None
    if not args.no_compose_table:
        del req
        torch.cuda.empty_cache()
        ctab = time_compose_table(max(3, args.steps), device)
        ctab["frac_hbm"] = ctab["gbs_algorithmic"] / peaks["hbm_gbs"]
        ctab["frac_hbm_dram_est"] = ctab["gbs_dram_est"] / peaks["hbm_gbs"]
        torch.cuda.empty_cache()
        ns = time_compose_table(max(3, args.steps), device, shared=False)
        ns["frac_hbm"] = ns["gbs_algorithmic"] / peaks["hbm_gbs"]
        ctab["no_sharing"] = ns
    if rank != 0:
        return
    ragged = time_ragged_build(max(3, args.steps), args.warmup, device, peaks, peak_src)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "precision": "bf16/fp16 tensor-core products (tf32 / 3xtf32 where the state is an operand), fp32 "
                     "accumulation, fp32 state and T_C (with a power-of-two exponent)",
        "data": "synthetic (seeded, drawn on the device)",
        "config": workload_config(res["n_seg"]),
        "composes_per_s": world * n_comp * args.steps / (res["ms"] / 1e3),
        "head_composes_per_s": world * n_comp * LH * args.steps / (res["ms"] / 1e3),
        "phases": {"build_ms": res["build_ms"], "build_tflops": build_tflops,
                   "build_frac_bf16_burst": build_tflops / peak_t, "build_frac_bf16_sustained": build_tflops / peak_ts,
                   "chain_ms": res["chain_ms"], "chain_gbs_algorithmic": chain_gbs,
                   "chain_frac_hbm": chain_gbs / peaks["hbm_gbs"]},
        "roofline": {"kernel": "segment build (GDN)", "bound": "tensor", "achieved": build_tflops,
                     "peak": peak_t, "unit": "TFLOP/s", "frac": build_tflops / peak_t,
                     "traffic": BUILD_TRAFFIC_RATIO * (res["body_tokens"] * LH * BUILD_IN_BYTES_PER_TOKEN_HEAD
                                                       + res["n_seg"] * LH * BUILD_OUT_BYTES_PER_ITEM),
                     "traffic_note": "dram bytes per launch, scaled from an ncu capture of a 32x32 ragged batch",
                     "peak_source": f"{peak_src} bf16 burst (the kernel is timed alone, per call)",
                     "frac_of_sustained": build_tflops / peak_ts, "flop_per_token_head": FLOP_PER_TOKEN_HEAD},
        "compose_table": ctab, "ragged_build": ragged,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": res["launches"], "clocks": res["clocks"],
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
