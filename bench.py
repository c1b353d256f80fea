"""Benchmark of the UltraEP balancing hot path on B300.

One step = one microbatch of the Qwen3-235B-like workload (R=64 ranks, E=128
experts, S=1 spare slot per rank, top-8, T=131072 tokens, 94 MoE layers,
hidden 4096 bf16) through all 94 layers; every layer runs ep_balance
(ep_count -> ep_plan -> ep_reroute, chained on the device) then ep_permute
through the C ABI, on one stream.  The metric is microseconds per MoE layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ultraep|reference]

--impl reference times the CPU oracle (the plain C definition of the same
steps) on the host cores, on a bounded sample of the same workload.
With N > 1 (torchrun) every rank runs an independent replica on its own GPU
and microbatch; there is no collective on the data path.
"""
import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
import types

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_expert_load_id_b300 import workload as W  # noqa: E402
from moe_expert_load_id_b300 import quality as Q  # noqa: E402

WORKLOAD = "qwen3-235b"
METRIC = "µs per MoE layer (count+plan+reroute+permute) at EP64"
UNIT = "us/layer"
N_HIDDEN_BUFS = 2  # distinct hidden inputs (each 1.07 GB > L2): the first half of the
                   # layers reads buffer 0, the second half buffer 1

# DRAM traffic of one ep_permute launch, from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum) of the named workload at
# T_captured tokens, scaled to a full launch by T / T_captured (every token
# moves the same bytes).  Valid only for that workload and hidden size and for
# the permute source with this SHA-256; reported as null otherwise.
NCU_PERMUTE = [{"source_sha256": "329977f460e6fcc1bd4f92b8edb2598dabb7d365319f5a0f91f05ffc6d0c9b65",
                "workload": "qwen3-235b", "Hd": 4096, "k": 8, "T_captured": 16384,
                "bytes_captured": 1148404992}]


def _sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def permute_traffic(w):
    src = os.path.join(ROOT, "moe_expert_load_id_b300", "csrc", "permute.cu")
    sha = _sha(src)
    for c in NCU_PERMUTE:
        if (c["source_sha256"] == sha and c["workload"] == w.name and c["Hd"] == w.Hd
                and c["k"] == w.k):
            return int(round(c["bytes_captured"] * w.T / c["T_captured"]))
    return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) of this process's GPU during the timed region."""
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        try:
            self.uuid = str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            self.uuid = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        rows = [r.split(", ") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        mine = [r for r in rows if len(r) >= 10 and self.uuid and
                (r[1].strip().lower().endswith(self.uuid.lower().replace("gpu-", "")))]
        if not mine:
            mine = [r for r in rows if len(r) >= 10 and r[0].strip() == os.environ.get(
                "CUDA_VISIBLE_DEVICES", "0").split(",")[0]] or [r for r in rows if len(r) >= 10]
        if not mine:
            return None
        sm = [float(r[2]) for r in mine if r[2].strip().replace(".", "").isdigit()]
        mx = [float(r[3]) for r in mine if r[3].strip().replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in mine for n, v in zip(names, r[6:10]) if v.strip() == "Active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(mine)}


# ------------------------------------------------------------------ distributed plumbing
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_layer(max_ms, steps, layers, world):
    """The metric over all ranks: every rank runs `steps` steps of `layers`
    layers (its own microbatch); the slowest rank's time over all layers run."""
    return max_ms * 1000.0 / (steps * layers * world)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ the CUDA path
class LayerPipeline:
    """Per-layer launches of the path for L layers of one microbatch (device buffers)."""

    def __init__(self, U, w, device):
        self.U, self.w, self.dev = U, w, device
        i32 = dict(dtype=torch.int32, device=device)
        L, dom = w.layers, U.Domain(w.R, w.E, w.S, w.k)
        self.dom = dom
        self.counts = torch.empty((L, w.E), **i32)
        self.counts_src = torch.empty((L, w.R, w.E), **i32)
        self.quota = torch.empty((L, dom.P), **i32)
        self.slot_expert = torch.empty((L, w.R, w.S), **i32)
        self.rank_load = torch.empty((L, w.R), **i32)
        self.inst_ptr = torch.empty((L, w.E + 1), **i32)
        self.inst_id = torch.empty((L, w.E + w.R * w.S), **i32)
        self.inst_cum = torch.empty((L, w.E + w.R * w.S), **i32)
        self.n_iter = torch.empty((L,), **i32)
        self.inst_status = torch.empty((L,), **i32)
        self.dev_status = torch.zeros((1,), **i32)
        self.workspace = torch.zeros((U.ep_count_workspace_bytes(dom, w.T, 1) // 4,), **i32)
        # two dst_row buffers, even and odd layers: a layer's rows can be read
        # back to the host while the next layer computes its own
        self.dst_rows = [torch.empty((1, w.N), **i32) for _ in range(2)]
        self.dst_row = self.dst_rows[(L - 1) % 2]          # the last layer's
        self.inst_offset = torch.empty((1, dom.P + 1), **i32)
        self.grouped = torch.empty((1, w.N, w.Hd), dtype=torch.bfloat16, device=device)

        # per-layer views of the outputs, in the form ep_balance takes
        self.outs = [types.SimpleNamespace(
            counts=self.counts[l:l + 1], counts_src=self.counts_src[l:l + 1],
            quota=self.quota[l:l + 1], slot_expert=self.slot_expert[l:l + 1],
            rank_load=self.rank_load[l:l + 1], inst_ptr=self.inst_ptr[l:l + 1],
            inst_id=self.inst_id[l:l + 1], inst_cum=self.inst_cum[l:l + 1],
            n_iter=self.n_iter[l:l + 1], inst_status=self.inst_status[l:l + 1],
            dst_row=self.dst_rows[l % 2], src_slot=None, inst_offset=self.inst_offset)
            for l in range(L)]

    def layer(self, l, ids_l, hidden_l, stream, ev=None):
        """One layer as the library is meant to be called: ep_balance (count ->
        plan -> reroute, chained on the device) then ep_permute."""
        U, d = self.U, self.dom
        if ev is not None:
            ev[0].record(stream)
        U.ep_balance(d, ids_l, self.outs[l], self.dev_status, self.workspace, 0, stream)
        if ev is not None:
            ev[1].record(stream)
        U.ep_permute(hidden_l, d.k, self.outs[l].dst_row, self.grouped, self.dev_status, stream)
        if ev is not None:
            ev[2].record(stream)

    def layer_split(self, l, ids_l, hidden_l, stream, ev):
        """The same layer as four separate calls with an event between each,
        for the per-kernel breakdown."""
        U, d = self.U, self.dom
        s = slice(l, l + 1)
        ev[0].record(stream)
        U.ep_count(d, ids_l, self.counts[s], self.counts_src[s], self.dev_status, self.workspace,
                   stream)
        ev[1].record(stream)
        U.ep_plan(d, self.counts[s], self.quota[s], self.slot_expert[s], self.rank_load[s],
                  self.inst_ptr[s], self.inst_id[s], self.inst_cum[s], self.n_iter[s],
                  self.inst_status[s], 0, stream)
        ev[2].record(stream)
        dst = self.outs[l].dst_row
        U.ep_reroute(d, ids_l, self.counts_src[s], self.quota[s], self.inst_ptr[s],
                     self.inst_id[s], self.inst_cum[s], dst, None, self.inst_offset,
                     self.dev_status, stream)
        ev[3].record(stream)
        U.ep_permute(hidden_l, d.k, dst, self.grouped, self.dev_status, stream)
        ev[4].record(stream)

    def hidden_of(self, l, hiddens):
        return hiddens[l * len(hiddens) // self.w.layers]

    def step(self, ids, hiddens, stream, events=None, ready=None, done=None, before=None,
             after=None):
        """ready: optional {layer: event} the stream waits for before that layer
        (inputs still being copied in); done: {layer: event} recorded after it;
        before / after: optional callables(layer) run around each layer."""
        for l in range(self.w.layers):
            if ready is not None and l in ready:
                stream.wait_event(ready[l])
            if before is not None:
                before(l)
            self.layer(l, ids[l:l + 1], self.hidden_of(l, hiddens)[None], stream,
                       None if events is None else events[l])
            if done is not None and l in done:
                done[l].record(stream)
            if after is not None:
                after(l)

    def step_split(self, ids, hiddens, stream, events):
        for l in range(self.w.layers):
            self.layer_split(l, ids[l:l + 1], self.hidden_of(l, hiddens)[None], stream, events[l])

    def results(self):
        """The step's plan results the host reads back after the step: per-layer
        plan outcome and the status word (each layer's dst_row is read back
        separately, as soon as the layer is done)."""
        return (self.rank_load, self.n_iter, self.inst_status, self.dev_status)


def batched_report(U, w, ids, pipe, stream, device, peak, reps=5, warm=2):
    """count, plan and reroute over ALL layers of the microbatch in one launch
    each (n_inst = layers), L2 flushed before every launch.  This is the
    bandwidth view of the two streaming kernels: one layer moves only 4-13 MB,
    too little to fill HBM, while the whole microbatch moves about 400 MB."""
    L = w.layers
    b = U.Buffers(pipe.dom, w.T, L, device=device)
    # L2 flush: write 256 MB (2x L2), then read another 256 MB, so that the timed
    # launch starts with L2 holding only clean lines of neither its inputs nor
    # its outputs (a write-only flush leaves ~126 MB of dirty lines whose
    # write-back would land inside the timed launch)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    flush_r = torch.ones(64 << 20, dtype=torch.int32, device=device)
    names = ("count", "plan", "reroute")
    acc = {n: [] for n in names}
    for rep in range(warm + reps):
        for n in names:
            flush.zero_()
            flush_r.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if n == "count":
                b.count(ids, stream)
            elif n == "plan":
                b.plan(stream=stream)
            else:
                b.reroute(ids, stream)
            e1.record(stream)
            torch.cuda.synchronize(device)
            if rep >= warm:
                acc[n].append(e0.elapsed_time(e1) * 1000.0)
    # the batched launches must agree with the per-layer launches of the step
    if not (torch.equal(b.counts, pipe.counts) and torch.equal(b.quota, pipe.quota)
            and int(b.dev_status.item()) == 0):
        raise RuntimeError("batched count/plan disagree with the per-layer launches")
    us = {n: float(np.mean(v)) for n, v in acc.items()}
    count_bytes = L * (4 * w.N + 4 * w.E * (w.R + 1))
    reroute_bytes = L * 8 * w.N
    gbs = lambda by, t: by / (t * 1e-6) / 1e9
    return {"launch": f"one launch per step over all {w.layers} layers (n_inst={L}), "
                      "L2 flushed before each launch (256 MB written, then 256 MB read)",
            "count": {"us": round(us["count"], 2), "bytes": count_bytes,
                      "gbs": round(gbs(count_bytes, us["count"]), 1),
                      "frac": round(gbs(count_bytes, us["count"]) / peak, 4)},
            "plan": {"us": round(us["plan"], 2), "instances": L,
                     "us_per_instance": round(us["plan"] / L, 3)},
            "reroute": {"us": round(us["reroute"], 2), "bytes": reroute_bytes,
                        "gbs": round(gbs(reroute_bytes, us["reroute"]), 1),
                        "frac": round(gbs(reroute_bytes, us["reroute"]) / peak, 4)}}


def unpermute_report(U, w, pipe, stream, device, peak, reps=5):
    """ep_unpermute of the last layer's grouped rows back to (token, k) order,
    timed on its own (it is not part of the metric's step)."""
    y = torch.empty((1, w.T, w.k, w.Hd), dtype=torch.bfloat16, device=device)
    U.ep_unpermute(pipe.grouped, w.T, w.k, pipe.dst_row, y, pipe.dev_status, stream)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        U.ep_unpermute(pipe.grouped, w.T, w.k, pipe.dst_row, y, pipe.dev_status, stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    us = e0.elapsed_time(e1) * 1000.0 / reps
    by = w.N * (4 * w.Hd + 4)          # read a grouped row + write a y row + dst_row
    del y
    return {"us_per_launch": round(us, 2), "bytes": by,
            "gbs": round(by / (us * 1e-6) / 1e9, 1),
            "frac": round(by / (us * 1e-6) / 1e9 / peak, 4)}


def combine_report(U, w, pipe, stream, device, peak, reps=5):
    """ep_combine of the last layer's grouped rows with seeded softmax gate
    weights, timed on its own (the step after unpermute; not in the metric)."""
    gen = torch.Generator(device=device).manual_seed(7)
    wts = torch.softmax(torch.randn((1, w.T, w.k), device=device, generator=gen), -1)
    y = torch.empty((1, w.T, w.Hd), dtype=torch.bfloat16, device=device)
    U.ep_combine(pipe.grouped, w.T, w.k, pipe.dst_row, wts, y, pipe.dev_status, stream)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        U.ep_combine(pipe.grouped, w.T, w.k, pipe.dst_row, wts, y, pipe.dev_status, stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    us = e0.elapsed_time(e1) * 1000.0 / reps
    by = w.T * (2 * w.Hd * w.k + 2 * w.Hd + 8 * w.k)   # k rows read, one written, dst + weights
    del y
    return {"us_per_launch": round(us, 2), "bytes": by,
            "gbs": round(by / (us * 1e-6) / 1e9, 1),
            "frac": round(by / (us * 1e-6) / 1e9 / peak, 4)}


def stage_report(U, w, pipe, stream, device, peak, reps=3):
    """ep_stage of the last layer's plan: every filled spare slot receives its
    expert's weights (3 x hidden x 1536 bf16 = 37.7 MB per Qwen3-235B expert)
    in a slot buffer reused across layers.  One synthetic expert table stands
    in for the layer's (its contents do not change the copy)."""
    expert_bytes = 3 * w.Hd * 1536 * 2
    ew = torch.empty((w.E, expert_bytes), dtype=torch.uint8, device=device).fill_(1)
    sw = torch.empty((w.R, w.S, expert_bytes), dtype=torch.uint8, device=device)
    se = pipe.slot_expert[w.layers - 1:w.layers]
    U.ep_stage(pipe.dom, ew, se, sw, None, pipe.dev_status, stream)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        U.ep_stage(pipe.dom, ew, se, sw, None, pipe.dev_status, stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    us = e0.elapsed_time(e1) * 1000.0 / reps
    filled = int((se >= 0).sum().item())
    by = 2 * filled * expert_bytes                      # read the expert, write the slot
    del ew, sw
    return {"us_per_layer": round(us, 2), "replicas": filled, "expert_bytes": expert_bytes,
            "bytes": by, "gbs": round(by / (us * 1e-6) / 1e9, 1),
            "frac": round(by / (us * 1e-6) / 1e9 / peak, 4)}


def bruteforce_gap(U, device, n=120, seed=1):
    """The planner on the GPU (ep_plan, ep_plan_ex) against the brute-force
    optimal maximum rank load on n seeded tiny instances (R 2-4, H 1-2, S 1;
    Zipf-like or uniform counts): mean and worst of max_load / optimum, and
    how often the plan is optimal."""
    from moe_expert_load_id_b300 import bruteforce
    rng = np.random.default_rng(seed)
    groups = {}
    for _ in range(n):
        R = int(rng.integers(2, 5))
        H = int(rng.integers(1, 3))
        E = R * H
        if rng.random() < 0.5:
            c = (40.0 / (1 + rng.permutation(E)) ** rng.uniform(0.8, 1.6)).astype(np.int32)
        else:
            c = rng.integers(0, 16, size=E).astype(np.int32)
        if c.sum() == 0:
            c[0] = 1
        groups.setdefault((R, H), []).append(c)
    gaps = {"base": [], "skip": [], "skip_release": []}
    for (R, H), cs in groups.items():
        c = np.stack(cs)
        opt = np.array([bruteforce.optimum(x, R, 1) for x in c])
        b = U.Buffers(U.Domain(R, R * H, 1, 1), 1, len(cs), device=device)
        b.counts.copy_(torch.from_numpy(c))
        for name, flags in (("base", 0), ("skip", U.EP_PLAN_SKIP),
                            ("skip_release", U.EP_PLAN_SKIP | U.EP_PLAN_RELEASE)):
            b.plan(flags=flags)
            mx = b.rank_load.cpu().numpy().max(axis=1)
            gaps[name] += list(mx / opt)
    out = {"instances": n, "shapes": "R 2-4, H 1-2, S 1, seeded Zipf-like or uniform counts"}
    for name, g in gaps.items():
        g = np.array(g)
        out[name] = {"mean": round(float(g.mean()), 4), "worst": round(float(g.max()), 4),
                     "optimal": round(float(np.mean(g == 1.0)), 3)}
    return out


STRESS_POINTS = [(8, 1, 512, 0.6), (16, 2, 2048, 1.0), (32, 4, 4096, 1.6), (64, 1, 8192, 1.0),
                 (64, 2, 2048, 1.6), (64, 4, 1024, 0.6)]


def config_report(U, w, device, peak, steps=2):
    """One microbatch of workload w through all its layers, as the main step
    runs it (ep_balance + ep_permute per layer): microseconds per layer, the
    ep_balance and ep_permute launch times, the permute's roofline fraction,
    the device status and the plan quality."""
    stream = torch.cuda.current_stream(device)
    ids, hiddens = make_inputs(w, 0, device)
    pipe = LayerPipeline(U, w, device)
    L = w.layers
    for _ in range(2):
        pipe.step(ids, hiddens, stream)
    torch.cuda.synchronize(device)
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(L)]
          for _ in range(steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        pipe.step(ids, hiddens, stream, ev[k])
    e1.record(stream)
    torch.cuda.synchronize(device)
    us_layer = e0.elapsed_time(e1) * 1000.0 / (steps * L)
    bal = float(np.mean([ev[k][l][0].elapsed_time(ev[k][l][1]) * 1000.0
                         for k in range(steps) for l in range(L)]))
    perm = float(np.mean([ev[k][l][1].elapsed_time(ev[k][l][2]) * 1000.0
                          for k in range(steps) for l in range(L)]))
    perm_bytes = w.T * (2 * w.Hd + 4 * w.k + 2 * w.Hd * w.k)
    counts = pipe.counts.cpu().numpy().astype(np.int64)
    after = pipe.rank_load.cpu().numpy()
    rep = {"workload": f"{w.name}: R={w.R} E={w.E} S={w.S} k={w.k} T={w.T} layers={L} "
                       f"hidden={w.Hd}, {w.popularity_desc()}",
           "us_per_layer": round(us_layer, 2), "balance_us": round(bal, 2),
           "permute_us": round(perm, 2),
           "permute_frac": round(perm_bytes / (perm * 1e-6) / 1e9 / peak, 4),
           "dev_status": int(pipe.dev_status.item()),
           "plan_status_ok": bool((pipe.inst_status.cpu().numpy() == 0).all()),
           "moves_mean": round(float(pipe.n_iter.float().mean().item()), 1),
           "imbalance_before_median": round(float(np.median(
               [Q.imbalance(Q.home_load(counts[l], w.R)) for l in range(L)])), 4),
           "imbalance_after_median": round(float(np.median(
               [Q.imbalance(after[l]) for l in range(L)])), 4)}
    del pipe, ids, hiddens
    torch.cuda.empty_cache()
    return rep


def configs_report(U, device, peak):
    """The other workloads at one GPU: tiny, DeepSeek-V3-like, GLM-4.5-like
    (all their layers, one microbatch each) and six points of the stress grid
    (32 layers each)."""
    out = {}
    for name in ("tiny", "deepseek-v3", "glm-4.5"):
        out[name] = config_report(U, W.WORKLOADS[name], device, peak)
    out["stress"] = [config_report(U, W.stress(R, S, tpr, sk), device, peak, steps=1)
                     for R, S, tpr, sk in STRESS_POINTS]
    return out


def make_inputs(w, microbatch, device):
    ids = torch.stack([W.topk_ids(w, l, microbatch, device=device) for l in range(w.layers)])
    hiddens = [W.hidden(w.T, w.Hd, w.seed(1000 + b, microbatch), device=device)
               for b in range(N_HIDDEN_BUFS)]
    return ids, hiddens


def quality_report(U, w, ids, pipe, microbatch, device):
    """max/mean rank load over the 94 layers: before, after (GPU plan), lower bound,
    and an EPLB-style placement built from the previous microbatches' loads."""
    counts = pipe.counts.cpu().numpy().astype(np.int64)
    after = pipe.rank_load.cpu().numpy()
    dom = pipe.dom
    hist = []
    hb = U.Buffers(dom, w.T, w.layers, device=device)
    for m in range(max(0, microbatch - 3), microbatch):      # up to 3 earlier microbatches
        hids = torch.stack([W.topk_ids(w, l, m, device=device) for l in range(w.layers)])
        hb.count(hids)
        hist.append(hb.counts.cpu().numpy().astype(np.float64))
    before_r, after_r, lb_r, e1_r, ea_r = [], [], [], [], []
    for l in range(w.layers):
        c = counts[l]
        mean = c.sum() / w.R
        before_r.append(Q.imbalance(Q.home_load(c, w.R)))
        after_r.append(Q.imbalance(after[l]))
        lb_r.append(Q.lower_bound(c, w.R, w.S) / mean)
        if hist:
            e1 = Q.eval_placement(Q.eplb_global(hist[-1][l], w.R, w.H + w.S), c)
            ea = Q.eval_placement(Q.eplb_global(np.mean([h[l] for h in hist], 0), w.R,
                                                w.H + w.S), c)
            e1_r.append(Q.imbalance(e1))
            ea_r.append(Q.imbalance(ea))
    rep = {"metric": "max/mean rank load over the layers of the timed microbatch",
           "before": Q.summarize(before_r), "ultraep_rule": Q.summarize(after_r),
           "lower_bound": Q.summarize(lb_r),
           "plan_n_iter": Q.summarize(pipe.n_iter.cpu().numpy())}
    # the planner variants (ep_plan_ex) on the same counts, all layers in one launch
    vb = U.Buffers(dom, 1, w.layers, device=device)
    vb.counts.copy_(pipe.counts)
    for name, flags in (("skip", U.EP_PLAN_SKIP),
                        ("skip_release", U.EP_PLAN_SKIP | U.EP_PLAN_RELEASE)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        vb.plan(flags=flags)
        e0.record()
        vb.plan(flags=flags)
        e1.record()
        torch.cuda.synchronize(device)
        loads = vb.rank_load.cpu().numpy()
        rep[f"variant_{name}"] = Q.summarize([Q.imbalance(loads[l]) for l in range(w.layers)])
        rep[f"variant_{name}_n_iter"] = Q.summarize(vb.n_iter.cpu().numpy())
        rep[f"variant_{name}_us_batched"] = round(e0.elapsed_time(e1) * 1000.0, 2)
    if hist:
        rep["eplb_style_history_W1"] = Q.summarize(e1_r)
        rep[f"eplb_style_history_W{len(hist)}"] = Q.summarize(ea_r)
    return rep


def run_ultraep(args, rank, world, local):
    from moe_expert_load_id_b300 import ultraep as U

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w = args.w
    microbatch = 3 + rank                 # ranks process different microbatches
    ids, hiddens = make_inputs(w, microbatch, device)
    pipe = LayerPipeline(U, w, device)
    stream = torch.cuda.current_stream(device)

    for _ in range(args.warmup):
        pipe.step(ids, hiddens, stream)
    torch.cuda.synchronize(device)

    # ---- timed region: K steps, device events per step and per launch
    L = w.layers
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    kern_ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(L)]
               for _ in range(args.steps)]
    clocks = ClockSampler(device)
    barrier(world)
    torch.cuda.synchronize(device)
    clocks.start()
    step_ev[0].record(stream)
    for k in range(args.steps):
        pipe.step(ids, hiddens, stream, kern_ev[k])
        step_ev[k + 1].record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    clock_rep = clocks.stop()
    total_ms = step_ev[0].elapsed_time(step_ev[-1])
    total_ms = max_over_ranks(total_ms, world, device)
    ms_per_step = total_ms / args.steps
    value = whole_job_us_per_layer(total_ms, args.steps, L, world)

    per = {"balance": [], "permute": []}
    for k in range(args.steps):
        for l in range(L):
            e = kern_ev[k][l]
            per["balance"].append(e[0].elapsed_time(e[1]) * 1000.0)
            per["permute"].append(e[1].elapsed_time(e[2]) * 1000.0)
    avg = {n: float(np.mean(v)) for n, v in per.items()}

    # ---- per-kernel breakdown: one more (untimed) step as four separate calls
    names = ("count", "plan", "reroute", "permute")
    split_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(L)]
    pipe.step_split(ids, hiddens, stream, split_ev)
    torch.cuda.synchronize(device)
    split = {n: float(np.mean([split_ev[l][i].elapsed_time(split_ev[l][i + 1]) * 1000.0
                               for l in range(L)])) for i, n in enumerate(names)}

    status = int(pipe.dev_status.item())
    plan_status = pipe.inst_status.cpu().numpy()
    if status != 0 or (plan_status != 0).any():
        raise RuntimeError(f"device status {status}, plan status {plan_status.tolist()}")

    # ---- roofline of the dominant kernel (permute) and the bandwidth kernels
    peak, peak_kind = measured_peaks()
    perm_bytes = w.T * (2 * w.Hd + 4 * w.k + 2 * w.Hd * w.k)   # read row + k dst + k rows
    count_bytes = 4 * w.N + 4 * w.E * (w.R + 1)
    reroute_bytes = 8 * w.N      # ids read + dst_row written (no src_slot in the step)
    gbs = lambda b, us: b / (us * 1e-6) / 1e9
    roofline = {"kernel": "ep_permute", "bound": "hbm",
                "achieved": round(gbs(perm_bytes, avg["permute"]), 1), "peak": peak,
                "unit": "GB/s", "frac": round(gbs(perm_bytes, avg["permute"]) / peak, 4),
                "traffic": permute_traffic(w), "algorithmic_bytes": perm_bytes,
                "peak_source": f"{peak_kind} hbm_gbs"}
    kernels = {"balance": {"us_per_launch": round(avg["balance"], 2),
                           "launches": "ep_count + ep_plan + ep_reroute, one ep_balance call"},
               "permute": {"us_per_launch": round(avg["permute"], 2),
                           "gbs": roofline["achieved"], "frac": roofline["frac"]}}
    breakdown = {n: {"us_per_launch": round(split[n], 2)} for n in names}
    breakdown["count"].update(gbs=round(gbs(count_bytes, split["count"]), 1),
                              frac=round(gbs(count_bytes, split["count"]) / peak, 4))
    breakdown["reroute"].update(gbs=round(gbs(reroute_bytes, split["reroute"]), 1),
                                frac=round(gbs(reroute_bytes, split["reroute"]) / peak, 4))
    n_iter_mean = float(pipe.n_iter.float().mean().item())
    breakdown["plan"].update(n_iter_mean=n_iter_mean,
                             us_per_move=round(split["plan"] / max(n_iter_mean, 1.0), 3))
    breakdown["note"] = ("one extra step, outside the timed region, with the four calls made "
                         "separately and an event between each")

    # ---- end to end: host (pinned) inputs -> device -> path -> host results
    e2e = None
    if args.e2e_steps > 0:
        ids_h = ids.cpu().pin_memory()
        hid_h = [h.cpu().pin_memory() for h in hiddens]
        ids_d = torch.empty_like(ids)
        hid_d = [torch.empty_like(h) for h in hiddens]
        res_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in pipe.results()]
        dst_h = torch.empty((L, w.N), dtype=torch.int32, pin_memory=True)
        h2d = ids_h.numel() * 4 + sum(h.numel() * 2 for h in hid_h)
        d2h = sum(t.numel() * t.element_size() for t in res_h) + dst_h.numel() * 4
        # every layer's dst_row (the routing result) goes back to pinned host
        # memory on its own stream as soon as the layer is done; the layer two
        # later, which reuses that device buffer, waits for the copy
        d2h_stream = torch.cuda.Stream(device)
        copied = {}

        def before_layer(l):
            if l - 2 in copied:
                stream.wait_event(copied.pop(l - 2))

        def after_layer(l):
            ev_done = torch.cuda.Event()
            ev_done.record(stream)
            d2h_stream.wait_event(ev_done)
            with torch.cuda.stream(d2h_stream):
                dst_h[l].copy_(pipe.outs[l].dst_row[0], non_blocking=True)
            ev_c = torch.cuda.Event()
            ev_c.record(d2h_stream)
            copied[l] = ev_c

        # the inputs are copied in on a second stream, half of the layers' at a
        # time: a step's first-half inputs as soon as the previous step's
        # first half of the layers is done with those device buffers, its
        # second-half inputs once the previous step is done; the layers wait
        # on events.  Every step's inputs are copied inside the timed region.
        copy_stream = torch.cuda.Stream(device)
        half = max(1, L // 2)
        free = {}

        def e2e_step():
            with torch.cuda.stream(copy_stream):
                if "first" in free:
                    copy_stream.wait_event(free["first"])
                else:
                    copy_stream.wait_stream(stream)
                hid_d[0].copy_(hid_h[0], non_blocking=True)
                ids_d[:half].copy_(ids_h[:half], non_blocking=True)
                first = torch.cuda.Event()
                first.record(copy_stream)
                if "second" in free:
                    copy_stream.wait_event(free["second"])
                for d_, h_ in zip(hid_d[1:], hid_h[1:]):
                    d_.copy_(h_, non_blocking=True)
                ids_d[half:].copy_(ids_h[half:], non_blocking=True)
                second = torch.cuda.Event()
                second.record(copy_stream)
            free["first"], free["second"] = torch.cuda.Event(), torch.cuda.Event()
            pipe.step(ids_d, hid_d, stream, ready={0: first, half: second},
                      done={half - 1: free["first"], L - 1: free["second"]},
                      before=before_layer, after=after_layer)
            for h_, d_ in zip(res_h, pipe.results()):
                h_.copy_(d_, non_blocking=True)
            # the step ends when its last rows are on the host
            for ev_c in copied.values():
                stream.wait_event(ev_c)
            copied.clear()

        e2e_step()
        torch.cuda.synchronize(device)
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_stream.wait_event(e0)  # no timed copy starts before the timed region
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(device)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, device)
        # the rows read back match the device path's last step
        if not torch.equal(dst_h[L - 1].to(device), pipe.dst_row[0]):
            raise RuntimeError("rows read back differ from the device's")
        e2e = {"value": round(e2e_ms * 1000.0 / (args.e2e_steps * L * world), 2), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": args.e2e_steps,
               "copies": "in: every layer's ids and the hidden rows (pinned host -> device); "
                         "out: every layer's dst_row and the per-layer plan summary "
                         "(device -> pinned host), all inside the timed region"}

    quality = quality_report(U, w, ids, pipe, microbatch, device) if rank == 0 else None
    if quality is not None and args.extras:
        quality["bruteforce_gap"] = bruteforce_gap(U, device)
    batched = batched_report(U, w, ids, pipe, stream, device, peak) if args.extras else None
    unperm = unpermute_report(U, w, pipe, stream, device, peak) if args.extras else None
    if unperm is not None:
        kernels["unpermute"] = unperm
    if args.extras:
        kernels["combine"] = combine_report(U, w, pipe, stream, device, peak)
        kernels["stage"] = stage_report(U, w, pipe, stream, device, peak)

    # indicative only: a real rank runs 1/R of count, reroute and permute on its own GPU
    per_rank = (split["count"] + split["reroute"] + split["permute"]) / w.R + split["plan"]

    cpu = None
    if rank == 0 and world == 1 and args.cpu_baseline:
        hbits = W.bf16_bits(hiddens[0])
        cpu = cpu_baseline_sample(w, ids[:args.cpu_layers].cpu().numpy(), hbits)
        n_thr = min(os.cpu_count() or 1, 16)
        cpu["nproc"] = os.cpu_count()
        cpu["cpu_model"] = cpu_model()
        cpu["all_cores"] = cpu_baseline_threads(w, ids[:n_thr].cpu().numpy(), hbits, n_thr)

    configs = None
    if args.configs and rank == 0 and world == 1:
        del ids, hiddens, pipe
        torch.cuda.empty_cache()
        configs = configs_report(U, device, peak)

    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "int32", "payload": "bf16", "data": "synthetic",
            "config": {"workload": f"{args.workload}-like: R={w.R} E={w.E} S={w.S} k={w.k} "
                                   f"T={w.T} layers={w.layers} hidden={w.Hd} bf16, "
                                   f"{w.popularity_desc()}",
                       "step": "one microbatch through all layers, per layer "
                               "ep_balance (ep_count -> ep_plan -> ep_reroute chained on the "
                               "device) then ep_permute",
                       "l2": f"inputs larger than L2 ({w.T * w.Hd * 2 / 1e9:.2f} GB hidden per "
                             f"layer, {w.N * w.Hd * 2 / 1e9:.2f} GB permute output per layer)",
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline, "kernels": kernels, "split_breakdown": breakdown,
            "batched": batched, "configs": configs,
            "per_rank_equivalent_us": round(per_rank, 2),
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": 4 * L * args.steps, "clocks": clock_rep, "quality": quality,
            "pages_context": {"critical_path_overhead_us": "< 300 (per rank, hardware not "
                                                           "disclosed)",
                              "planning_us_at_ep64": "< 100",
                              "imbalance": "1.30-4.01 -> 1.01-1.04"}}
    return line


# ------------------------------------------------------------------ the CPU oracle
def cpu_baseline_sample(w, ids_layers, hidden_bits, perm_fraction=8):
    """Time the oracle as it stands (single thread) on a bounded sample: for each
    sampled layer, count + plan + reroute on the whole layer and permute on the
    first 1/perm_fraction of the rows (its time scaled up by perm_fraction)."""
    import oracle
    oracle.lib()
    per_layer = []
    for ids in ids_layers:
        t0 = time.perf_counter()
        c, _, _ = oracle.count(ids, w.R, w.E)
        pl = oracle.plan(c, w.R, w.E, w.S)
        dst, src, off = oracle.reroute(ids, w.R, w.E, w.S, pl)
        t1 = time.perf_counter()
        n = int(off[-1]) // perm_fraction
        oracle.permute(hidden_bits, w.k, src[:n], n)
        t2 = time.perf_counter()
        per_layer.append((t1 - t0) + (t2 - t1) * perm_fraction)
    value = float(np.mean(per_layer)) * 1e6
    return {"value": round(value, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{len(ids_layers)} layer(s) of the same workload: count+plan+reroute on "
                      f"the whole layer, permute on 1/{perm_fraction} of the rows scaled "
                      f"x{perm_fraction}; single-threaded C"}


def run_stress_sweep(args):
    """The stress grid (R in {8,16,32,64}, E = 4R, S in {1,2,4}, k = 8, Zipf
    s in {0.6,1.0,1.6}) at 2048 tokens per rank, 8 layers each: per layer the
    planner alone (separate call), the ep_balance call and ep_permute (hidden
    4096 bf16), with moves per layer and max/mean load before and after."""
    from moe_expert_load_id_b300 import ultraep as U
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)
    grid = W.STRESS_GRID
    rows = []
    for R in grid["R"]:
        for S in grid["S"]:
            for sk in grid["s"]:
                w = dataclasses.replace(W.stress(R, S, 2048, sk), layers=8)
                ids, hiddens = make_inputs(w, 0, device)
                pipe = LayerPipeline(U, w, device)
                L = w.layers
                pipe.step(ids, hiddens, stream)
                ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(L)]
                pipe.step(ids, hiddens, stream, ev)
                sev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(L)]
                pipe.step_split(ids, hiddens, stream, sev)
                torch.cuda.synchronize(device)
                mean = lambda f: float(np.mean([f(l) for l in range(L)]))
                counts = pipe.counts.cpu().numpy().astype(np.int64)
                after = pipe.rank_load.cpu().numpy()
                rows.append({
                    "R": R, "E": w.E, "S": S, "zipf_s": sk, "T": w.T,
                    "plan_us": round(mean(lambda l: sev[l][1].elapsed_time(sev[l][2]) * 1000), 2),
                    "balance_us": round(mean(lambda l: ev[l][0].elapsed_time(ev[l][1]) * 1000), 2),
                    "permute_us": round(mean(lambda l: ev[l][1].elapsed_time(ev[l][2]) * 1000), 2),
                    "moves": round(float(pipe.n_iter.float().mean().item()), 1),
                    "before": round(float(np.median([Q.imbalance(Q.home_load(counts[l], R))
                                                     for l in range(L)])), 4),
                    "after": round(float(np.median([Q.imbalance(after[l]) for l in range(L)])), 4),
                    "status": int(pipe.dev_status.item())})
                del pipe, ids, hiddens
                torch.cuda.empty_cache()
    return {"stress_sweep": rows, "unit": "us per layer (means over 8 layers)",
            "config": "stress grid at 2048 tokens per rank, k=8, hidden 4096 bf16, 8 layers "
                      "per point; plan_us = ep_plan as its own call, balance_us = the ep_balance "
                      "call, permute_us = ep_permute"}


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def cpu_baseline_threads(w, ids_layers, hidden_bits, threads, perm_fraction=32):
    """The same oracle on `threads` host threads at once, one layer each (its C
    calls release the GIL): wall-clock throughput of the whole host.  count +
    plan + reroute run on every sampled layer in parallel, then permute on the
    first 1/perm_fraction of each layer's rows in parallel (its wall time scaled
    up by perm_fraction)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.lib()

    def cpr(ids):
        c, _, _ = oracle.count(ids, w.R, w.E)
        pl = oracle.plan(c, w.R, w.E, w.S)
        return oracle.reroute(ids, w.R, w.E, w.S, pl)

    with ThreadPoolExecutor(threads) as ex:
        t0 = time.perf_counter()
        routes = list(ex.map(cpr, ids_layers))
        t1 = time.perf_counter()
        list(ex.map(lambda r: oracle.permute(hidden_bits, w.k, r[1][:int(r[2][-1]) // perm_fraction],
                                             int(r[2][-1]) // perm_fraction), routes))
        t2 = time.perf_counter()
    n = len(ids_layers)
    value = ((t1 - t0) + (t2 - t1) * perm_fraction) / n * 1e6
    return {"value": round(value, 1), "unit": UNIT, "threads": threads,
            "sample": f"{n} layers at once, one per thread: count+plan+reroute on the whole "
                      f"layer, permute on 1/{perm_fraction} of the rows scaled x{perm_fraction}; "
                      f"wall clock divided by the layers"}


def run_reference(args, rank, world):
    """The oracle as it stands (single-threaded C) on the host cores: each step
    is ONE layer of the workload run whole (count + plan + reroute, and the
    permute of every row), so the timed work is exactly the work done.  The
    metric (microseconds per layer) is the step's time."""
    if rank != 0:
        return None
    import oracle
    oracle.lib()
    w = args.w
    ids = [W.topk_ids(w, l, 3).numpy() for l in range(2)]
    hid = W.bf16_bits(W.hidden(w.T, w.Hd, w.seed(1000, 3)))
    times = []
    t_all0 = time.perf_counter()
    for it in range(args.warmup + args.steps):
        x = ids[it % 2]
        t0 = time.perf_counter()
        c, _, _ = oracle.count(x, w.R, w.E)
        pl = oracle.plan(c, w.R, w.E, w.S)
        dst, src, off = oracle.reroute(x, w.R, w.E, w.S, pl)
        out = oracle.permute(hid, w.k, src, int(off[-1]))
        t1 = time.perf_counter()
        del out
        if it >= args.warmup:
            times.append(t1 - t0)
    wall = time.perf_counter() - t_all0
    value = float(np.mean(times)) * 1e6
    sample = ("each step one whole layer of the workload (two layers' inputs alternating): "
              "count + plan + reroute + the permute of every row, single-threaded C; "
              "no part scaled")
    cpu = {"value": round(value, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": sample}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(value / 1000.0, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32", "payload": "bf16",
            "data": "synthetic",
            "config": {"workload": f"{args.workload}-like: R={w.R} E={w.E} S={w.S} k={w.k} "
                                   f"T={w.T} layers={w.layers} hidden={w.Hd} bf16, "
                                   f"{w.popularity_desc()}",
                       "step": "one layer (a step of all layers would take minutes on the "
                               "host); the metric is per layer either way",
                       "parallelism": "host cores, 1 thread"},
            "cpu_baseline": cpu, "wall_s": round(wall, 1),
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ultraep", "reference"), default="ultraep")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--tokens", type=int, default=0,
                    help="override T (small cases for profiler captures)")
    ap.add_argument("--layers", type=int, default=0, help="override the number of layers")
    ap.add_argument("--hidden", type=int, default=0,
                    help="override the hidden size (small cases for profiler captures)")
    # e2e timed steps: every step's inputs are copied in inside the timed
    # region, and the first step's first half (~1.3 GB on the Qwen3-235B-like
    # workload) cannot overlap anything, so the steps amortise that fill
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-layers", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--stress-sweep", action="store_true",
                    help="instead of the benchmark: planner, ep_balance and ep_permute per layer "
                         "over the stress grid")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="skip the batched count/plan/reroute and unpermute timings")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the other workloads (tiny, DeepSeek-V3-like, GLM-4.5-like, "
                         "stress points)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    w = W.WORKLOADS[args.workload]
    if args.tokens or args.layers or args.hidden:
        w = dataclasses.replace(w, T=args.tokens or w.T, layers=args.layers or w.layers,
                                Hd=args.hidden or w.Hd)
    args.w = w
    rank, world, local = dist_init()
    if args.stress_sweep:
        line = run_stress_sweep(args) if rank == 0 else None
    elif args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ultraep(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
