"""Benchmark of the O = f(A.B).C hot path on GB300.

One step = one pass of every row of the hot path over its full-size
synthetic workload (seeded, inputs resident in HBM for the kernel-only
number), in this order (the rows are independent; those with small inputs go
first so that, end to end, compute starts before all inputs have arrived):
  * causal attention forward 32 x 32768 x 128 (chain_fwd_f16pv: P V as one
    f16 product, V re-encoded by a two-launch pre-pass that is timed with it;
    chain_fwd's compensated form is timed beside the step),
  * GeLU MLP chain 4096x1024 . 1024x4096 . 4096x1024,
  * causal attention backward with recompute 16 x 65536 x 128,
  * the small fp32 attention 1 x 256 x 64,
  * sp_relayout of the Q, K and V sequence shards 4x[32768][32][128] bf16
    to head-major [8][131072][128] (head group 0),
  * causal attention forward on those 8 heads at n = 131072, d = 128
    (chain_fwd_f16pv).
value = algorithmic FLOPs of the chain kernels per step / device time per
step (TFLOP/s).  The relayout contributes bytes, not FLOPs; its GB/s and
every component's share are reported under "components".

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: the
path needs no exchange on one device, so there is no collective.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("f(AB)C TFLOP/s bf16 (attn fwd/bwd, GeLU MLP) and % of tensor peak; "
          "relayout GB/s")
WORKLOAD = ("chain hot path: causal attn fwd 32x32768x128 + GeLU MLP 4096x1024x4096x1024 + "
            "causal attn bwd 16x65536x128 + attn fwd fp32 1x256x64 + 3x sp_relayout "
            "4x[32768][32][128]->[8][131072][128] + causal attn fwd 8x131072x128")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def measured_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.json), or None once the kernel's source file has
    changed since the counters were taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            entry = json.load(f).get(kernel)
        if not entry:
            return None
        with open(os.path.join(ROOT, entry["source"]), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        return entry["dram_bytes_per_launch"] if sha == entry["source_sha256_16"] else None
    except (OSError, ValueError, KeyError):
        return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ FLOPs
def attn_fwd_flops(BH, n, d, causal):
    # 2 products of 2*n*n*d each; causal keeps half (FlashAttention count)
    f = 4.0 * n * n * d * BH
    return f / 2 if causal else f


def attn_bwd_flops(BH, n, d, causal):
    # 5 products of 2*n*n*d each (dV, dP, dS recompute excluded: S counted once)
    f = 10.0 * n * n * d * BH
    return f / 2 if causal else f


def mlp_flops(M, K, N, P):
    return 2.0 * M * K * N + 2.0 * M * N * P


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling during the timed region (reads settings only)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons, pw = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            try:
                pw.append(float(f[3]))
            except ValueError:
                pass
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["no samples"]}
        loaded = [s for s in sm if mx is None or s >= 0.3 * mx] or sm
        # board power beside the clocks: the long attention kernels run at the
        # power cap, which is what sets their clock
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": round(statistics.median(pw), 1) if pw else None,
                "power_w_max": round(max(pw), 1) if pw else None,
                "power_note": "nvidia-smi power.draw, an average over about its last second: "
                              "it lags behind a timed region shorter than that"}


# ------------------------------------------------------------- the step
class HotPath:
    """Buffers and calls of one step; every call goes through the C ABI."""

    def __init__(self, dev, seed_shift=0, only=None):
        import torch
        import chain_gb300 as cg
        import chain_synth as cs
        self.torch, self.cg, self.cs = torch, cg, cs
        self.dev = dev
        self.only = only
        W = cs.WORKLOADS
        g = lambda k: W[k].seed + seed_shift
        want = lambda key: only is None or only in key
        e = torch.empty(0, device=dev)
        u = W["ulysses_128k"].dims
        self.u = u
        Hl, N = u["H"] // u["p"], u["p"] * u["n_loc"]
        if want("sp_relayout") or want("attn_fwd_causal_8x131072x128"):
            self.shards = [cs.shard_inputs(u["p"], u["n_loc"], u["H"], u["d"],
                                           seed=g("ulysses_128k") + t, device=dev) for t in range(3)]
            self.hm = [torch.empty(Hl, N, u["d"], dtype=torch.bfloat16, device=dev) for _ in range(3)]
            for t in range(3):
                cg.sp_relayout(self.shards[t], u["p"], u["g"], self.hm[t])
            self.o4 = torch.empty(Hl, N, u["d"], dtype=torch.bfloat16, device=dev)
            self.l4 = torch.empty(Hl, N, dtype=torch.float32, device=dev)
            self.ws4 = torch.empty(cg.chain_fwd_f16pv_workspace_size(self.hm[0], self.hm[2]),
                                   dtype=torch.uint8, device=dev)
        else:
            self.shards, self.hm, self.o4, self.l4, self.ws4 = [e] * 3, [e] * 3, e, e, e
        c3 = W["causal_attn_32k"].dims
        self.c3 = c3
        if want("attn_fwd_causal_32x32768x128"):
            self.q3, self.k3, self.v3 = cs.attn_inputs(c3["BH"], c3["n"], c3["d"],
                                                       seed=g("causal_attn_32k"), device=dev)
            self.o3 = torch.empty_like(self.q3)
            self.l3 = torch.empty(c3["BH"], c3["n"], dtype=torch.float32, device=dev)
            self.ws3 = torch.empty(cg.chain_fwd_f16pv_workspace_size(self.q3, self.v3),
                                   dtype=torch.uint8, device=dev)
        else:
            self.q3 = self.k3 = self.v3 = self.o3 = self.l3 = self.ws3 = e
        m = W["gelu_mlp"].dims
        self.m = m
        if want("gelu_mlp"):
            self.x, self.w1, self.w2 = cs.mlp_inputs(m["M"], m["K"], m["N"], m["P"],
                                                     seed=g("gelu_mlp"), device=dev)
            self.o2 = torch.empty(m["M"], m["P"], dtype=torch.bfloat16, device=dev)
            self.ws2 = torch.empty(max(cg.chain_fwd_f16h_workspace_size(self.w2), 16),
                                   dtype=torch.uint8, device=dev)
            self.mlp_ok = self._probe_mlp()
        else:
            self.x = self.w1 = self.w2 = self.o2 = self.ws2 = e
            self.mlp_ok = False
        b = W["causal_bwd_64k"].dims
        self.b = b
        if want("attn_bwd"):
            self.q5, self.k5, self.v5, self.do5 = cs.attn_inputs(
                b["BH"], b["n"], b["d"], seed=g("causal_bwd_64k"), device=dev, with_do=True)
            # the forward whose O and LSE the backward consumes (outside the step)
            self.o5, self.l5 = cg.attention_fwd(self.q5, self.k5, self.v5, True)
            self.dq5, self.dk5, self.dv5 = (torch.empty_like(self.q5) for _ in range(3))
            self.ws = torch.empty(cg.chain_bwd_workspace_size(self.q5, self.v5), dtype=torch.uint8,
                                  device=dev)
        else:
            self.q5 = self.k5 = self.v5 = self.do5 = self.o5 = self.l5 = e
            self.dq5 = self.dk5 = self.dv5 = self.ws = e
        t1 = W["tiny_attn_fp32"].dims
        self.t1 = t1
        if want("attn_fwd_fp32"):
            self.q1, self.k1, self.v1 = cs.attn_inputs(t1["BH"], t1["n"], t1["d"],
                                                       seed=g("tiny_attn_fp32"),
                                                       dtype=torch.float32, device=dev)
            self.o1 = torch.empty_like(self.q1)
            self.l1 = torch.empty(t1["BH"], t1["n"], dtype=torch.float32, device=dev)
            self.fp32_ok = self._probe_fp32()
        else:
            self.q1 = self.k1 = self.v1 = self.o1 = self.l1 = e
            self.fp32_ok = False
        self.comp = [c for c in self._components() if only is None or only in c["name"]]

    def _probe_mlp(self):
        try:
            self.cg.chain_fwd_f16h(self.x, self.w1, self.w2, self.cg.F_GELU_TANH, self.o2, self.ws2)
            return True
        except self.cg.ChainError as e:
            if e.status == self.cg.ERR_UNSUPPORTED:
                return False
            raise

    def _probe_fp32(self):
        try:
            self.cg.chain_fwd(self.q1, self.k1, self.v1, self.cg.F_SOFTMAX, 0,
                              self.t1["d"] ** -0.5, self.o1, self.l1)
            return True
        except self.cg.ChainError as e:
            if e.status == self.cg.ERR_UNSUPPORTED:
                return False
            raise

    def _components(self):
        """The step's components, in launch order.  Each lists the device
        tensors it reads from the host ("ins") and the results it returns
        ("outs") for the end-to-end measurement.  The components are
        independent, so those with small inputs go first: end to end, the
        first step starts after 0.8 GB of uploads instead of all 5.4 GB."""
        cg = self.cg
        u, c3, m, b, t1 = self.u, self.c3, self.m, self.b, self.t1
        Hl, N = u["H"] // u["p"], u["p"] * u["n_loc"]
        comps = []
        comps.append(dict(name="attn_fwd_causal_32x32768x128",
                          flops=attn_fwd_flops(c3["BH"], c3["n"], c3["d"], True), bytes=0.0, launches=3,
                          kernels=[("v_absmax_kernel+v_to_f16_kernel", 0.0, 6.0 * c3["BH"] * c3["n"] * c3["d"]),
                                   ("attn_fwd_pv16_kernel",
                                    attn_fwd_flops(c3["BH"], c3["n"], c3["d"], True), 0.0)],
                          ins=[self.q3, self.k3, self.v3], outs=[self.o3, self.l3],
                          fn=lambda: cg.chain_fwd_f16pv(self.q3, self.k3, self.v3, cg.MASK_CAUSAL,
                                                        c3["d"] ** -0.5, self.o3, self.l3,
                                                        self.ws3)))
        if self.mlp_ok:
            # chain_fwd_f16h: the intermediate as one f16 tile; its W2 pre-pass
            # (two HBM-bound launches: 2 + 2 bytes read, 2 written per
            # element) is timed with it, as one span: the main kernel starts
            # while the pre-pass runs
            comps.append(dict(name="gelu_mlp_4096x1024x4096x1024",
                              flops=mlp_flops(m["M"], m["K"], m["N"], m["P"]), bytes=0.0, launches=3,
                              kernels=[("w_absmax_kernel+w_to_f16_kernel+mlp_cluster_kernel",
                                        mlp_flops(m["M"], m["K"], m["N"], m["P"]),
                                        6.0 * m["N"] * m["P"])],
                              ins=[self.x, self.w1, self.w2], outs=[self.o2],
                              fn=lambda: cg.chain_fwd_f16h(self.x, self.w1, self.w2, cg.F_GELU_TANH,
                                                           self.o2, self.ws2)))
        fb = attn_bwd_flops(b["BH"], b["n"], b["d"], True)
        # of the 5 counted products, dK/dV makes S, dP, dV, dK and dQ makes dQ
        # (its recomputed S and dP are not counted)
        comps.append(dict(name="attn_bwd_causal_16x65536x128", flops=fb, bytes=0.0, launches=3,
                          kernels=[("bwd_dkdv_kernel", 0.8 * fb, 0.0), ("bwd_dq_kernel", 0.2 * fb, 0.0)],
                          ins=[self.q5, self.k5, self.v5, self.do5, self.o5, self.l5],
                          outs=[self.dq5, self.dk5, self.dv5],
                          fn=lambda: cg.chain_bwd(self.do5, self.q5, self.k5, self.v5, self.o5, self.l5,
                                                  cg.F_SOFTMAX, cg.MASK_CAUSAL, b["d"] ** -0.5,
                                                  self.dq5, self.dk5, self.dv5, self.ws)))
        if self.fp32_ok:
            comps.append(dict(name="attn_fwd_fp32_1x256x64",
                              flops=attn_fwd_flops(1, t1["n"], t1["d"], False), bytes=0.0, launches=1,
                              kernels=[("attn_fwd_f32_kernel", attn_fwd_flops(1, t1["n"], t1["d"], False),
                                        0.0)],
                              ins=[self.q1, self.k1, self.v1], outs=[self.o1, self.l1],
                              fn=lambda: cg.chain_fwd(self.q1, self.k1, self.v1, cg.F_SOFTMAX,
                                                      cg.MASK_NONE, t1["d"] ** -0.5, self.o1,
                                                      self.l1)))
        for t in range(3):
            comps.append(dict(name=f"sp_relayout[{'QKV'[t]}]", flops=0.0,
                              bytes=2.0 * Hl * N * u["d"] * 2, launches=1,
                              kernels=[("relayout_kernel", 0.0, 2.0 * Hl * N * u["d"] * 2)],
                              ins=[self.shards[t]], outs=[],
                              fn=(lambda t=t: cg.sp_relayout(self.shards[t], u["p"], u["g"], self.hm[t]))))
        # the causal forward on the relayouted heads: chain_fwd_f16pv (P V as
        # one f16 product); its V pre-pass (two HBM-bound launches: 2 + 2
        # bytes read, 2 written per element) is timed with it
        comps.append(dict(name="attn_fwd_causal_8x131072x128", flops=attn_fwd_flops(Hl, N, u["d"], True),
                          bytes=0.0, launches=3,
                          kernels=[("v_absmax_kernel+v_to_f16_kernel", 0.0, 6.0 * Hl * N * u["d"]),
                                   ("attn_fwd_pv16_kernel", attn_fwd_flops(Hl, N, u["d"], True), 0.0)],
                          ins=[], outs=[self.o4, self.l4],
                          fn=lambda: cg.chain_fwd_f16pv(self.hm[0], self.hm[1], self.hm[2],
                                                        cg.MASK_CAUSAL, u["d"] ** -0.5, self.o4,
                                                        self.l4, self.ws4)))
        return comps

    def step(self, events=None):
        """One pass over every component; events[i] (len(kernels) + 1 CUDA
        events) are recorded at the main-kernel boundaries of component i.
        Each component runs inside an NVTX range of its name, so a profiler's
        timeline shows the step's structure."""
        nvtx = self.torch.cuda.nvtx
        for i, c in enumerate(self.comp):
            if events is not None:
                self.cg.set_timing_events(*events[i])
            nvtx.range_push(c["name"])
            c["fn"]()
            nvtx.range_pop()
        if events is not None:
            self.cg.set_timing_events()

    # host <-> device for the end-to-end number
    def host_io(self, make_host=True):
        """Per component: its device input and output tensors and, if
        make_host, pinned host copies of the inputs and pinned host buffers
        for the outputs."""
        torch = self.torch
        res = []
        for c in self.comp:
            ins = [t for t in c["ins"] if t.numel() > 0]
            outs = [t for t in c["outs"] if t.numel() > 0]
            h_in = [t.cpu().pin_memory() for t in ins] if make_host else None
            h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs] if make_host else None
            res.append((ins, h_in, outs, h_out))
        return res

    @property
    def flops(self):
        return sum(c["flops"] for c in self.comp)

    @property
    def launches(self):
        return sum(c["launches"] for c in self.comp)


def dist_setup(gpus):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return rank, world, local, dist
    return 0, 1, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x, dist):
    """Max of a host scalar over all ranks (the timing rule of multi-GPU runs)."""
    if dist is None:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------- CPU baseline
def oracle_sample(scale: int = 3):
    """Time the fp64 oracle on a bounded sample of the same workloads (about
    15 s of host work at scale 1); returns (TFLOP/s, seconds, description,
    threads)."""
    import torch
    import chain_synth as cs
    import oracle
    oracle.build()
    W = cs.WORKLOADS
    flops, secs, parts = 0.0, 0.0, []
    # attention forward rows of the 32k workload (one head), causal
    c3 = W["causal_attn_32k"].dims
    q, k, v = cs.attn_inputs(2, c3["n"], c3["d"], seed=W["causal_attn_32k"].seed)
    nr = 4096 * scale
    rows = [(h, r) for h in range(2) for r in range(c3["n"] - nr // 2, c3["n"])]
    t0 = time.perf_counter()
    oracle.softmax_fwd(q, k, v, c3["d"] ** -0.5, True, rows=rows)
    dt = time.perf_counter() - t0
    f = sum(4.0 * (r + 1) * c3["d"] for _, r in rows)
    flops, secs = flops + f, secs + dt
    parts.append(f"attn fwd {len(rows)} rows (last of 2 heads) of 32x32768x128 ({dt:.1f}s)")
    # backward: last 16 query rows of the 64k workload, one head
    b = W["causal_bwd_64k"].dims
    q, k, v, do = cs.attn_inputs(1, b["n"], b["d"], seed=W["causal_bwd_64k"].seed, with_do=True)
    i0 = b["n"] - 1024 * scale
    t0 = time.perf_counter()
    oracle.softmax_bwd(q, k, v, do, b["d"] ** -0.5, True, row_range=(i0, b["n"]),
                       col_range=(i0, b["n"]))
    dt = time.perf_counter() - t0
    f = sum(8.0 * (r + 1) * b["d"] for r in range(i0, b["n"]))
    flops, secs = flops + f, secs + dt
    parts.append(f"attn bwd {b['n'] - i0} rows of one head of 16x65536x128 ({dt:.1f}s)")
    # MLP rows
    m = W["gelu_mlp"].dims
    x, w1, w2 = cs.mlp_inputs(m["M"], m["K"], m["N"], m["P"], seed=W["gelu_mlp"].seed)
    rows = [r % m["M"] for r in range(0, m["M"] * scale // 2)]
    t0 = time.perf_counter()
    oracle.chain_fwd(x, w1, w2, oracle.F_GELU_TANH, rows=rows)
    dt = time.perf_counter() - t0
    f = len(rows) * (2.0 * m["K"] * m["N"] + 2.0 * m["N"] * m["P"])
    flops, secs = flops + f, secs + dt
    parts.append(f"GeLU MLP {len(rows)} rows of 4096 ({dt:.1f}s)")
    # the fp32 attention of the tiny workload, in full
    c1 = W["tiny_attn_fp32"].dims
    q, k, v = cs.attn_inputs(c1["BH"], c1["n"], c1["d"], seed=W["tiny_attn_fp32"].seed,
                             dtype=torch.float32)
    t0 = time.perf_counter()
    oracle.softmax_fwd(q, k, v, c1["d"] ** -0.5, False)
    dt = time.perf_counter() - t0
    f = 4.0 * c1["BH"] * c1["n"] * c1["n"] * c1["d"]
    flops, secs = flops + f, secs + dt
    parts.append(f"fp32 attention 1x256x64 in full ({dt:.3f}s)")
    return flops / secs / 1e12, secs, "; ".join(parts), oracle.num_threads()


def oracle_relayout_gbps():
    """The oracle's relayout of one full Ulysses tensor (4 x [32768][32][128] bf16 shards to
    the 8 heads of group 0): bytes read plus written per second.  The copy does not depend
    on the values, so the shards are zero-filled rather than drawn."""
    import torch
    import chain_synth as cs
    import oracle
    oracle.build()
    u = cs.WORKLOADS["ulysses_128k"].dims
    shards = torch.zeros((u["p"], u["n_loc"], u["H"], u["d"]), dtype=torch.bfloat16)
    t0 = time.perf_counter()
    out, _ = oracle.relayout(shards, u["p"], u["g"])
    dt = time.perf_counter() - t0
    return 2.0 * out.nbytes / dt / 1e9, dt


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state; warm-up steps are not repeated
    vals, total = [], 0.0
    desc, thr = "", 0
    for _ in range(args.steps):
        v, s, desc, thr = oracle_sample()
        vals.append(v)
        total += s
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * total / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "n/a (host)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def measure_sp_fused(hp, reps=5):
    """The relayout fused into the attention (chain_fwd_sp_f16pv: Q, K read
    from the sequence shards, V's f16 copy written from them by its pre-pass,
    O written back into them) against the unfused sequence sp_relayout x3 +
    chain_fwd_f16pv + sp_relayout_inverse, on the Ulysses workload; and the
    compensated form (chain_fwd_sp).  Measured beside the step, not part of
    its value."""
    torch, cg, u = hp.torch, hp.cg, hp.u
    Hl, N, d = u["H"] // u["p"], u["p"] * u["n_loc"], u["d"]
    o_sh = torch.zeros_like(hp.shards[0])
    l_sh = torch.empty(Hl, N, dtype=torch.float32, device=hp.dev)
    ws = torch.empty(cg.chain_fwd_sp_f16pv_workspace_size(hp.shards[2], u["p"]), dtype=torch.uint8,
                     device=hp.dev)
    scale = d ** -0.5

    def fused():
        cg.chain_fwd_sp_f16pv(hp.shards[0], hp.shards[1], hp.shards[2], u["p"], u["g"],
                              cg.MASK_CAUSAL, scale, o_sh, l_sh, ws)

    def fused_compensated():
        cg.chain_fwd_sp(hp.shards[0], hp.shards[1], hp.shards[2], u["p"], u["g"], cg.MASK_CAUSAL,
                        scale, o_sh, l_sh)

    def unfused():
        for t in range(3):
            cg.sp_relayout(hp.shards[t], u["p"], u["g"], hp.hm[t])
        cg.chain_fwd_f16pv(hp.hm[0], hp.hm[1], hp.hm[2], cg.MASK_CAUSAL, scale, hp.o4, hp.l4, hp.ws4)
        cg.sp_relayout_inverse(hp.o4, u["p"], u["g"], o_sh)

    def timed(fn):
        for _ in range(2):
            fn()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return sorted(ts)[len(ts) // 2]

    ms_f, ms_u, ms_c = timed(fused), timed(unfused), timed(fused_compensated)
    rc, site = cg.chain_check()
    if rc != 0:
        raise RuntimeError(f"device status {rc} site {site:#x} in the fused relayout measurement")
    fl = attn_fwd_flops(Hl, N, d, True)
    del o_sh, l_sh, ws
    return {"attn_fwd_sp_fused_8x131072x128": {
        "ms": round(ms_f, 4), "TFLOPs": round(fl / (ms_f * 1e-3) / 1e12, 1),
        "call": "chain_fwd_sp_f16pv",
        "unfused_ms": round(ms_u, 4),
        "unfused": "sp_relayout x3 + chain_fwd_f16pv + sp_relayout_inverse",
        "compensated_fused_ms": round(ms_c, 4),
        "hbm_bytes_saved": 4 * 2 * Hl * N * d * 2,
        "timing": f"median of {reps} after 2 warm-ups; inputs larger than L2"}}


def measure_relayout_clean(hp, reps=7):
    """sp_relayout of the Q, K and V shards, each launch preceded by a read of
    a 512 MB buffer, so that L2 holds no dirty lines of an earlier kernel when
    it starts.  Inside the step, a relayout that follows a kernel which wrote
    a lot (the previous relayout, the backward) also writes those lines back
    to DRAM during its own launch; this row measures the kernel alone."""
    torch, cg = hp.torch, hp.cg
    u = hp.u
    Hl, N = u["H"] // u["p"], u["p"] * u["n_loc"]
    nbytes = 2.0 * Hl * N * u["d"] * 2
    big = torch.empty(256 * 1024 * 1024, dtype=torch.float16, device=hp.dev)  # 512 MB, > L2
    big.fill_(1.0)
    ts = {t: [] for t in range(3)}
    for _ in range(reps):
        for t in range(3):
            big.sum()
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            cg.set_timing_events(*evs)
            cg.sp_relayout(hp.shards[t], u["p"], u["g"], hp.hm[t])
            cg.set_timing_events()
            torch.cuda.synchronize()
            ts[t].append(evs[0].elapsed_time(evs[1]))
    peaks, _ = load_peaks()
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    out = {}
    for t in range(3):
        ms = statistics.median(ts[t])
        gb = nbytes / (ms * 1e-3) / 1e9
        out["QKV"[t]] = {"ms": round(ms, 4), "GBps": round(gb, 1),
                         "frac_of_measured_hbm": round(gb / hbm, 4), "frac_of_8TBps": round(gb / 8000.0, 4)}
    del big
    return {"sp_relayout_after_clean_l2": dict(out, timing=f"median of {reps}; each launch after a "
                                                             "512 MB read (L2 without dirty lines)")}


def measure_mlp_bwd(hp, reps=10):
    """Backward of the GeLU MLP workload (intermediate recomputed): the
    activation kernel and the batched product kernel, timed at their
    boundaries.  Measured beside the step, not part of its value."""
    torch, cg, m = hp.torch, hp.cg, hp.m
    M, K, N, P = m["M"], m["K"], m["N"], m["P"]
    gen = torch.Generator(device=hp.dev).manual_seed(5)
    do = torch.randn(M, P, device=hp.dev, generator=gen).to(torch.bfloat16)
    dx, dw1, dw2 = torch.empty_like(hp.x), torch.empty_like(hp.w1), torch.empty_like(hp.w2)
    ws = torch.empty(cg.chain_bwd_workspace_size_f(hp.x, hp.w2, cg.F_GELU_TANH), dtype=torch.uint8,
                     device=hp.dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=hp.dev)

    def run(evs=None):
        if evs is not None:
            cg.set_timing_events(*evs)
        cg.chain_bwd(do, hp.x, hp.w1, hp.w2, None, None, cg.F_GELU_TANH, cg.MASK_NONE, 1.0,
                     dx, dw1, dw2, ws)
        if evs is not None:
            cg.set_timing_events()

    for _ in range(3):
        run()
    tot, k1, k2 = [], [], []
    for _ in range(reps):
        flush.zero_()  # L2 flushed between iterations (the inputs fit in L2)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        run(evs)
        torch.cuda.synchronize()
        k1.append(evs[0].elapsed_time(evs[1]))
        k2.append(evs[1].elapsed_time(evs[2]))
        tot.append(evs[0].elapsed_time(evs[2]))
    rc, site = cg.chain_check()
    if rc != 0:
        raise RuntimeError(f"device status {rc} site {site:#x} in the MLP backward measurement")
    med = lambda v: sorted(v)[len(v) // 2]
    fl = 4.0 * M * N * (P + K)  # dH, dW2, dX, dW1; the recomputed X W1 is not counted
    ms = med(tot)
    return {"gelu_mlp_bwd_4096x1024x4096x1024": {
        "ms": round(ms, 4), "TFLOPs": round(fl / (ms * 1e-3) / 1e12, 1),
        "act_kernel_ms": round(med(k1), 4), "gemm_kernel_ms": round(med(k2), 4),
        "flops": fl, "timing": f"median of {reps}, L2 flushed between iterations"}}


def measure_mlp_compensated(hp, reps=10):
    """The GeLU MLP workload through chain_fwd (the intermediate as the bf16
    pair H_hi + H_lo, no workspace), timed beside the step."""
    torch, cg, m = hp.torch, hp.cg, hp.m
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=hp.dev)
    o = torch.empty_like(hp.o2)

    def run():
        cg.chain_fwd(hp.x, hp.w1, hp.w2, cg.F_GELU_TANH, cg.MASK_NONE, 1.0, o, None)

    for _ in range(3):
        run()
    ts = []
    for _ in range(reps):
        flush.zero_()  # L2 flushed between iterations (the inputs fit in L2)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    rc, site = cg.chain_check()
    if rc != 0:
        raise RuntimeError(f"device status {rc} site {site:#x} in the chain_fwd MLP measurement")
    ms = sorted(ts)[len(ts) // 2]
    fl = mlp_flops(m["M"], m["K"], m["N"], m["P"])
    return {"gelu_mlp_compensated_4096x1024x4096x1024": {
        "ms": round(ms, 4), "TFLOPs": round(fl / (ms * 1e-3) / 1e12, 1),
        "kernel": "mlp_cluster_kernel (chain_fwd)",
        "timing": f"median of {reps}, L2 flushed between iterations"}}


def measure_fp8(hp, reps=5):
    """The causal 32 x 32768 x 128 forward on e4m3 Q, K, V (chain_fwd_fp8):
    the V re-encoding kernel and the attention kernel, timed at their
    boundaries.  Measured beside the step, not part of its value."""
    torch, cg, cs = hp.torch, hp.cg, hp.cs
    wl = cs.WORKLOADS["causal_attn_32k_e4m3"]
    dm = wl.dims
    BH, n, d = dm["BH"], dm["n"], dm["d"]
    q, k, v = cs.attn_inputs(BH, n, d, seed=wl.seed, dtype=torch.float8_e4m3fn, device=hp.dev)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=hp.dev)
    lse = torch.empty(BH, n, dtype=torch.float32, device=hp.dev)
    ws = torch.empty(cg.chain_fwd_fp8_workspace_size(v), dtype=torch.uint8, device=hp.dev)

    def run(evs=None):
        if evs is not None:
            cg.set_timing_events(*evs)
        cg.chain_fwd_fp8(q, k, v, cg.MASK_CAUSAL, d ** -0.5, 1.0, o, lse, ws)
        if evs is not None:
            cg.set_timing_events()

    for _ in range(2):
        run()
    tot, conv, attn = [], [], []
    for _ in range(reps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        torch.cuda.synchronize()
        run(evs)
        torch.cuda.synchronize()
        conv.append(evs[0].elapsed_time(evs[1]))
        attn.append(evs[1].elapsed_time(evs[2]))
        tot.append(evs[0].elapsed_time(evs[2]))
    rc, site = cg.chain_check()
    if rc != 0:
        raise RuntimeError(f"device status {rc} site {site:#x} in the e4m3 measurement")
    med = lambda x: sorted(x)[len(x) // 2]
    fl = attn_fwd_flops(BH, n, d, True)
    peaks, src = load_peaks()
    p16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    p16s = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    # half the counted products (Q K^T) run at the 8-bit rate, nominally twice
    # the 16-bit one; the other half (P V) at the 16-bit rate
    peak = 4.0 / 3.0 * p16
    ka = fl / (med(attn) * 1e-3) / 1e12
    vbytes = 3.0 * BH * n * d  # e4m3 read, f16 written
    del q, k, v, o, lse, ws
    return {"attn_fwd_fp8_causal_32x32768x128": {
        "ms": round(med(tot), 4), "TFLOPs": round(fl / (med(tot) * 1e-3) / 1e12, 1),
        "attn_kernel_ms": round(med(attn), 4), "attn_kernel_TFLOPs": round(ka, 1),
        "v_convert_ms": round(med(conv), 4),
        "v_convert_GBps": round(vbytes / (med(conv) * 1e-3) / 1e9, 1),
        "roofline": {"bound": "tensor", "kernel": "attn_fwd_fp8_kernel", "achieved": round(ka, 1),
                     "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(ka / peak, 4),
                     "peak_basis": f"4/3 x {src} burst bf16 (Q K^T at the nominal 2x "
                                   "8-bit rate, P V at the 16-bit rate)",
                     "frac_sustained": round(ka / (4.0 / 3.0 * p16s), 4),
                     "traffic": measured_traffic("attn_fwd_fp8_kernel"),
                     "traffic_unit": "bytes per launch (ncu)"},
        "inputs": "e4m3 Q, K, V (fp32 N(0,1) draws rounded to e4m3), O bf16",
        "timing": f"median of {reps} after 2 warm-ups; inputs larger than L2"}}


def measure_fwd_compensated(hp, reps=5):
    """The causal forwards of the step through chain_fwd (P V as the
    compensated bf16 pair, no workspace), timed beside the step."""
    torch, cg = hp.torch, hp.cg
    out = {}
    cases = []
    if hp.q3.numel():
        cases.append(("attn_fwd_compensated_causal_32x32768x128", hp.q3, hp.k3, hp.v3, hp.o3,
                      hp.l3))
    if hp.hm[0].numel():
        cases.append(("attn_fwd_compensated_causal_8x131072x128", hp.hm[0], hp.hm[1], hp.hm[2],
                      hp.o4, hp.l4))
    for name, q, k, v, o, l in cases:
        d = q.shape[-1]

        def run(evs=None):
            if evs is not None:
                cg.set_timing_events(*evs)
            cg.chain_fwd(q, k, v, cg.F_SOFTMAX, cg.MASK_CAUSAL, d ** -0.5, o, l)
            if evs is not None:
                cg.set_timing_events()

        for _ in range(2):
            run()
        ts = []
        for _ in range(reps):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            torch.cuda.synchronize()
            run(evs)
            torch.cuda.synchronize()
            ts.append(evs[0].elapsed_time(evs[1]))
        rc, site = cg.chain_check()
        if rc != 0:
            raise RuntimeError(f"device status {rc} site {site:#x} in the chain_fwd measurement")
        med = sorted(ts)[len(ts) // 2]
        fl = attn_fwd_flops(q.shape[0], q.shape[1], d, True)
        out[name] = {"ms": round(med, 4), "TFLOPs": round(fl / (med * 1e-3) / 1e12, 1),
                     "kernel": "attn_fwd_kernel (chain_fwd)",
                     "timing": f"median of {reps} after 2 warm-ups"}
    return out


def _median_ms(torch, fn, reps, warm=2):
    """Median device time of fn() over reps calls on the current stream."""
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return sorted(ts)[len(ts) // 2]


def measure_sweep(torch, cg, dev, reps=5):
    """Causal attention forward (chain_fwd_f16pv) and backward (chain_bwd) over
    sequence lengths 2048 ... 131072 at a constant 1,048,576 (head, position)
    pairs, for d = 128 and 64: how the rate holds up as the sequences shorten
    and the heads multiply.  Run on its own (bench.py --sweep), not part of
    the step."""
    import chain_synth as cs
    out = {}
    for d in (128, 64):
        for n in (2048, 8192, 32768, 131072):
            BH = (1 << 20) // n
            q, k, v, do = cs.attn_inputs(BH, n, d, seed=17000 + n + d, device=dev, with_do=True)
            o = torch.empty_like(q)
            lse = torch.empty(BH, n, dtype=torch.float32, device=dev)
            wsf = torch.empty(max(cg.chain_fwd_f16pv_workspace_size(q, v), 16), dtype=torch.uint8,
                              device=dev)
            wsb = torch.empty(cg.chain_bwd_workspace_size(q, v), dtype=torch.uint8, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            scale = d ** -0.5

            def fwd():
                cg.chain_fwd_f16pv(q, k, v, cg.MASK_CAUSAL, scale, o, lse, wsf)

            def bwd():
                cg.chain_bwd(do, q, k, v, o, lse, cg.F_SOFTMAX, cg.MASK_CAUSAL, scale, dq, dk, dv,
                             wsb)

            ms_f = _median_ms(torch, fwd, reps)
            ms_b = _median_ms(torch, bwd, reps)
            rc, site = cg.chain_check()
            if rc != 0:
                raise RuntimeError(f"device status {rc} site {site:#x} in the sweep")
            ff, fb = attn_fwd_flops(BH, n, d, True), attn_bwd_flops(BH, n, d, True)
            out[f"causal_{BH}x{n}x{d}"] = {
                "fwd_ms": round(ms_f, 4), "fwd_TFLOPs": round(ff / (ms_f * 1e-3) / 1e12, 1),
                "bwd_ms": round(ms_b, 4), "bwd_TFLOPs": round(fb / (ms_b * 1e-3) / 1e12, 1)}
            del q, k, v, do, o, lse, wsf, wsb, dq, dk, dv
    return out


def measure_gqa(hp, reps=5):
    """Grouped-query attention, 32 query heads over 8 K/V heads at n = 32768,
    causal: forward (chain_fwd_f16pv) and backward (chain_bwd), each timed
    as one call.  Measured beside the step, not part of its value."""
    torch, cg, cs = hp.torch, hp.cg, hp.cs
    wl = cs.WORKLOADS["gqa_32k"]
    dm = wl.dims
    BH, BHkv, n, d = dm["BH"], dm["BHkv"], dm["n"], dm["d"]
    q, _, _, do = cs.attn_inputs(BH, n, d, seed=wl.seed, device=hp.dev, with_do=True)
    k = cs.normal((BHkv, n, d), wl.seed + cs.OFF_K, device=hp.dev)
    v = cs.normal((BHkv, n, d), wl.seed + cs.OFF_V, device=hp.dev)
    o = torch.empty_like(q)
    lse = torch.empty(BH, n, dtype=torch.float32, device=hp.dev)
    wsf = torch.empty(max(cg.chain_fwd_f16pv_workspace_size(q, v), 16), dtype=torch.uint8,
                      device=hp.dev)
    wsb = torch.empty(cg.chain_bwd_workspace_size(q, v), dtype=torch.uint8, device=hp.dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    scale = d ** -0.5

    def fwd():
        cg.chain_fwd_f16pv(q, k, v, cg.MASK_CAUSAL, scale, o, lse, wsf)

    def bwd():
        cg.chain_bwd(do, q, k, v, o, lse, cg.F_SOFTMAX, cg.MASK_CAUSAL, scale, dq, dk, dv, wsb)

    ms_f = _median_ms(torch, fwd, reps)
    ms_b = _median_ms(torch, bwd, reps)
    rc, site = cg.chain_check()
    if rc != 0:
        raise RuntimeError(f"device status {rc} site {site:#x} in the grouped-query measurement")
    ff, fb = attn_fwd_flops(BH, n, d, True), attn_bwd_flops(BH, n, d, True)
    del q, k, v, do, o, lse, wsf, wsb, dq, dk, dv
    return {"attn_gqa_causal_32q8kv_x32768x128": {
        "fwd_ms": round(ms_f, 4), "fwd_TFLOPs": round(ff / (ms_f * 1e-3) / 1e12, 1),
        "bwd_ms": round(ms_b, 4), "bwd_TFLOPs": round(fb / (ms_b * 1e-3) / 1e12, 1),
        "calls": "chain_fwd_f16pv, chain_bwd",
        "timing": f"median of {reps} after 2 warm-ups; inputs larger than L2"}}


def measure_varlen(hp, reps=5):
    """Sequences of mixed lengths (seeded, 1024..16384) packed end to end into
    131072 positions with 16 heads, causal: forward (chain_fwd_varlen_f16pv;
    the compensated chain_fwd_varlen beside it) and backward
    (chain_bwd_varlen).  FLOPs are counted per sequence.  Measured beside the
    step, not part of its value."""
    torch, cg, cs = hp.torch, hp.cg, hp.cs
    wl = cs.WORKLOADS["varlen_128k"]
    dm = wl.dims
    total, H, d = dm["total"], dm["H"], dm["d"]
    lens = cs.varlen_lengths(total, dm["min_len"], dm["max_len"], wl.seed)
    q = cs.normal((total, H, d), wl.seed + cs.OFF_Q, device=hp.dev)
    k = cs.normal((total, H, d), wl.seed + cs.OFF_K, device=hp.dev)
    v = cs.normal((total, H, d), wl.seed + cs.OFF_V, device=hp.dev)
    do = cs.normal((total, H, d), wl.seed + cs.OFF_DO, device=hp.dev)
    cu_host = [0]
    for L in lens:
        cu_host.append(cu_host[-1] + L)
    cu = torch.tensor(cu_host, dtype=torch.int32, device=hp.dev)
    B, mx = len(lens), max(lens)
    o = torch.empty_like(q)
    lse = torch.empty(H, total, dtype=torch.float32, device=hp.dev)
    ws = torch.empty(cg.chain_bwd_workspace_size(q, q), dtype=torch.uint8, device=hp.dev)
    wsf = torch.empty(cg.chain_fwd_varlen_f16pv_workspace_size(v), dtype=torch.uint8,
                      device=hp.dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    scale = d ** -0.5

    def fwd():
        cg.chain_fwd_varlen_f16pv(q, k, v, cu, B, mx, cg.MASK_CAUSAL, scale, o, lse, wsf)

    def fwd_compensated():
        cg.chain_fwd_varlen(q, k, v, cu, B, mx, cg.MASK_CAUSAL, scale, o, lse)

    def bwd():
        cg.chain_bwd_varlen(do, q, k, v, o, lse, cu, B, mx, cg.MASK_CAUSAL, scale, dq, dk, dv, ws)

    ms_c = _median_ms(torch, fwd_compensated, reps)
    ms_f = _median_ms(torch, fwd, reps)
    ms_b = _median_ms(torch, bwd, reps)
    rc, site = cg.chain_check()
    if rc != 0:
        raise RuntimeError(f"device status {rc} site {site:#x} in the varlen measurement")
    ff = sum(attn_fwd_flops(H, L, d, True) for L in lens)
    fb = sum(attn_bwd_flops(H, L, d, True) for L in lens)
    del q, k, v, do, o, lse, ws, wsf, dq, dk, dv, cu
    return {"attn_varlen_causal_131072x16x128": {
        "fwd_ms": round(ms_f, 4), "fwd_TFLOPs": round(ff / (ms_f * 1e-3) / 1e12, 1),
        "compensated_fwd_ms": round(ms_c, 4),
        "compensated_fwd_TFLOPs": round(ff / (ms_c * 1e-3) / 1e12, 1),
        "bwd_ms": round(ms_b, 4), "bwd_TFLOPs": round(fb / (ms_b * 1e-3) / 1e12, 1),
        "sequences": B, "min_len": min(lens), "max_len": mx,
        "calls": "chain_fwd_varlen_f16pv (compensated: chain_fwd_varlen), chain_bwd_varlen",
        "flops": "per sequence: fwd 2 n^2 d H, bwd 5 n^2 d H (causal)",
        "timing": f"median of {reps} after 2 warm-ups; inputs larger than L2"}}


def host_link_gbps(torch, dev, nbytes=1 << 30, reps=3):
    """Pinned host <-> device copy bandwidth of this machine (one 1 GiB copy
    each way, reps times): the best is the floor under the end-to-end figure,
    the worst shows how much the host side varies between copies."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        times = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            dst.copy_(src, non_blocking=True)
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        out[name] = round(nbytes / (min(times) * 1e-3) / 1e9, 1)
        out[name + "_worst"] = round(nbytes / (max(times) * 1e-3) / 1e9, 1)
    del h, d
    return out


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="chain_gb300")
    ap.add_argument("--only", default=None, help="substring: run only matching components")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="only the sequence-length / head-size sweep of the attention, one JSON line")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        print("bench.py: at least 3 warm-up steps are required", file=sys.stderr)
        args.warmup = 3

    import torch
    import chain_gb300 as cg
    rank, world, local, dist = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cg.lib()
    peaks, peak_src = load_peaks()
    if args.sweep:
        if rank == 0:
            print(json.dumps({"sweep": measure_sweep(torch, cg, dev),
                              "flops": "fwd 2 n^2 d BH, bwd 5 n^2 d BH (causal)",
                              "timing": "median of 5 after 2 warm-ups",
                              "calls": "chain_fwd_f16pv, chain_bwd"}))
        return 0
    hp = HotPath(dev, only=args.only)
    stream = torch.cuda.current_stream()
    if not hp.comp:
        # --only matched no component of the step: the rows measured beside it
        nxt = {}
        if "fp8" in (args.only or ""):
            nxt.update(measure_fp8(hp))
        if "gqa" in (args.only or ""):
            nxt.update(measure_gqa(hp))
        if "varlen" in (args.only or ""):
            nxt.update(measure_varlen(hp))
        if rank == 0:
            print(json.dumps({"only": args.only, "next_rows": nxt or None}))
        if dist is not None:
            dist.destroy_process_group()
        return 0

    ncomp = len(hp.comp)
    for _ in range(args.warmup):
        hp.step()
    torch.cuda.synchronize()
    rc, site = cg.chain_check()
    if rc != 0:
        raise RuntimeError(f"device status {rc} site {site:#x} after warm-up")

    # ---- timed region (kernels only, inputs resident)
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(len(c["kernels"]) + 1)]
             for c in hp.comp] for _ in range(args.steps)]
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    barrier(dist)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        hp.step(evs[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    clocks = clk.stop()
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, dist)
    ms_step = ms_total / args.steps
    rc, site = cg.chain_check()
    if rc != 0:
        raise RuntimeError(f"device status {rc} site {site:#x} in timed region")

    # per component: device time of its main kernels; per kernel function:
    # summed time, algorithmic work and launches over the step
    comp_ms, by_k = [], {}
    for i, c in enumerate(hp.comp):
        tot = 0.0
        for k, (kname, kflops, kbytes) in enumerate(c["kernels"]):
            ms = statistics.mean(evs[s][i][k].elapsed_time(evs[s][i][k + 1])
                                 for s in range(args.steps))
            tot += ms
            e = by_k.setdefault(kname, {"ms": 0.0, "flops": 0.0, "bytes": 0.0, "launches": 0})
            e["ms"] += ms
            e["flops"] += kflops
            e["bytes"] += kbytes
            e["launches"] += 1
        comp_ms.append(tot)
    # Tensor peaks: the burst figure is the headline denominator (the step
    # is tens of milliseconds, not seconds); the sustained one (a seconds-long
    # loop under the power cap) is reported beside it.
    tf_peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    tf_sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    components = {}
    for c, ms in zip(hp.comp, comp_ms):
        e = {"ms": round(ms, 4)}
        if c["flops"]:
            tf = c["flops"] / (ms * 1e-3) / 1e12
            e.update(TFLOPs=round(tf, 1), frac_of_measured_peak=round(tf / tf_peak, 4),
                     frac_of_sustained_peak=round(tf / tf_sus, 4))
        if c["bytes"]:
            gb = c["bytes"] / (ms * 1e-3) / 1e9
            e.update(GBps=round(gb, 1), frac_of_measured_hbm=round(gb / hbm_peak, 4),
                     frac_of_8TBps=round(gb / 8000.0, 4))
        components[c["name"]] = e
    # dominant kernel: the kernel function with the largest share of the
    # step's device time; achieved = its algorithmic work / its time, summed
    # over its launches in the step.
    dom_name = max(by_k, key=lambda k: by_k[k]["ms"])
    dom = by_k[dom_name]
    share = dom["ms"] / sum(v["ms"] for v in by_k.values())
    if dom["flops"]:
        ach = dom["flops"] / (dom["ms"] * 1e-3) / 1e12
        roof = {"kernel": dom_name, "bound": "tensor", "achieved": round(ach, 1),
                "kernel_shares": {k: round(v["ms"] / sum(x["ms"] for x in by_k.values()), 4)
                                  for k, v in by_k.items()},
                "peak": tf_peak, "unit": "TFLOP/s", "frac": round(ach / tf_peak, 4),
                "peak_source": f"{peak_src} bf16_tflops (burst)",
                "peak_sustained": tf_sus, "frac_sustained": round(ach / tf_sus, 4),
                "launches_per_step": dom["launches"], "flops_per_step": dom["flops"],
                "avg_launch_ms": round(dom["ms"] / dom["launches"], 4),
                "share_of_step_device_time": round(share, 4),
                "traffic": measured_traffic(dom_name), "traffic_unit": "bytes per launch (ncu)"}
    else:
        ach = dom["bytes"] / (dom["ms"] * 1e-3) / 1e9
        roof = {"kernel": dom_name, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(ach / hbm_peak, 4), "peak_source": f"{peak_src} hbm_gbs",
                "launches_per_step": dom["launches"], "bytes_per_step": dom["bytes"],
                "avg_launch_ms": round(dom["ms"] / dom["launches"], 4),
                "share_of_step_device_time": round(share, 4),
                "traffic": measured_traffic(dom_name), "traffic_unit": "bytes per launch (ncu)"}
    flops_all = hp.flops * world
    value = flops_all / (ms_step * 1e-3) / 1e12

    # ---- end to end through the C ABI with host buffers.  Every step copies
    # its inputs from pinned host memory and its results back.  NSET sets of
    # device buffers let the uploads of the next steps (own stream) run under
    # step k's kernels, and step k's downloads (own stream) under step k+1's;
    # with three, a step whose uploads run slow (the host side's throughput
    # can swing from step to step) is absorbed by the one before.  Each
    # component waits only for its own inputs, and its results leave as soon
    # as it has finished; events order each copy after the work whose
    # buffers it touches.
    e2e = None
    NSET = 3
    if not args.no_e2e:
        hps = [hp] + [HotPath(dev, only=args.only) for _ in range(NSET - 1)]
        io0 = hp.host_io()
        io = [io0] + [h.host_io(make_host=False) for h in hps[1:]]
        h2d = sum(t.numel() * t.element_size() for _, h_in, _, _ in io0 for t in h_in)
        d2h = sum(t.numel() * t.element_size() for _, _, _, h_out in io0 for t in h_out)
        s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        comp = torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event(enable_timing=False)
        ncomp = len(hp.comp)

        def run(nsteps, t0=None, t1=None, trace=None):
            # trace: if a list, gets per step the host issue time and timing
            # events around each component's upload, compute and download
            done = [ev() for _ in range(NSET)]  # step finished with its buffer set
            down = [ev() for _ in range(NSET)]  # its results are on the host
            tev = lambda: torch.cuda.Event(enable_timing=True)
            if t0 is not None:
                t0.record(s_up)
            for k in range(nsteps):
                h0 = time.perf_counter()
                X = k % NSET
                up_c = [ev() for _ in range(ncomp)]
                done_c = [ev() for _ in range(ncomp)]
                tr = None if trace is None else {n_: [[tev(), tev()] for _ in range(ncomp)]
                                                 for n_ in ("up", "comp", "down")}
                with torch.cuda.stream(s_up):
                    if k >= NSET:
                        s_up.wait_event(done[X])  # step k-NSET no longer reads these inputs
                    for c in range(ncomp):
                        if tr:
                            tr["up"][c][0].record(s_up)
                        for d_, h_ in zip(io[X][c][0], io0[c][1]):
                            d_.copy_(h_, non_blocking=True)
                        up_c[c].record(s_up)
                        if tr:
                            tr["up"][c][1].record(s_up)
                if k >= NSET:
                    comp.wait_event(down[X])  # step k-NSET's results are on the host
                with torch.cuda.stream(comp):
                    for c in range(ncomp):
                        comp.wait_event(up_c[c])
                        if tr:
                            tr["comp"][c][0].record(comp)
                        hps[X].comp[c]["fn"]()
                        done_c[c].record(comp)
                        if tr:
                            tr["comp"][c][1].record(comp)
                    done[X].record(comp)
                with torch.cuda.stream(s_down):
                    for c in range(ncomp):
                        s_down.wait_event(done_c[c])
                        if tr:
                            tr["down"][c][0].record(s_down)
                        for h_, d_ in zip(io0[c][3], io[X][c][2]):
                            h_.copy_(d_, non_blocking=True)
                        if tr:
                            tr["down"][c][1].record(s_down)
                    down[X].record(s_down)
                if tr:
                    tr["host_ms"] = (time.perf_counter() - h0) * 1e3
                    trace.append(tr)
            if t1 is not None:
                s_down.wait_stream(comp)
                t1.record(s_down)

        def timeline(trace):
            # Per step (mean over the traced steps, the first two skipped as
            # pipeline fill): busy time of each stream, the time the compute
            # stream spent waiting between components (for inputs, or for the
            # download that frees its buffer set), and the host's issue time.
            first = 2 if len(trace) > 2 else 1
            steps = range(first, len(trace))
            el = lambda a, b: a.elapsed_time(b)
            out = {}
            for n_ in ("up", "comp", "down"):
                out[f"{n_}_busy_ms"] = round(statistics.mean(
                    sum(el(a, b) for a, b in trace[k][n_]) for k in steps), 3)
            # each traced step's upload time: the host side's throughput can
            # swing within one run, which the mean alone hides
            out["up_busy_ms_per_step"] = [round(sum(el(a, b) for a, b in trace[k]["up"]), 2)
                                          for k in range(len(trace))]

            def wait(k, c):  # gap before component c of step k on the compute stream
                prev_end = trace[k - 1]["comp"][-1][1] if c == 0 else trace[k]["comp"][c - 1][1]
                return max(0.0, el(prev_end, trace[k]["comp"][c][0]))

            out["comp_wait_ms"] = round(statistics.mean(
                sum(wait(k, c) for c in range(ncomp)) for k in steps), 3)
            out["comp_wait_by_component_ms"] = {
                hp.comp[c]["name"]: round(statistics.mean(wait(k, c) for k in steps), 3)
                for c in range(ncomp)}
            out["host_issue_ms"] = round(statistics.mean(trace[k]["host_ms"] for k in steps), 3)
            # one steady-state step in absolute terms: per component, when its
            # upload, compute and download ran (ms from that step's first
            # upload), to show which stream a slow step waited on
            k = len(trace) - 2 if len(trace) >= 3 else len(trace) - 1
            z = trace[k]["up"][0][0]
            out["step_detail_ms"] = {
                hp.comp[c]["name"]: [round(el(z, e), 2) for n_ in ("up", "comp", "down")
                                     for e in trace[k][n_][c]]
                for c in range(ncomp)}
            out["step_detail_fields"] = "up start, up end, compute start, compute end, down start, down end"
            return out

        run(NSET)  # every buffer set used once before timing
        torch.cuda.synchronize()
        link = host_link_gbps(torch, dev)
        barrier(dist)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        run(args.steps, e0, e1)
        torch.cuda.synchronize()
        barrier(dist)
        ms_e2e = max_over_ranks(e0.elapsed_time(e1), dist) / args.steps
        # the same pipeline once more with timing events per component (not
        # part of the figure above)
        trace = []
        run(max(args.steps, 4), trace=trace)
        torch.cuda.synchronize()
        tl = timeline(trace)
        # the link alone again: a change from before the run points at the host
        # side (shared with other work on the machine), not at the pipeline
        link_after = host_link_gbps(torch, dev)
        e2e = {"value": round(flops_all / (ms_e2e * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 3),
               "host_link_GBps": link, "host_link_GBps_after": link_after,
               "upload_floor_ms": round(h2d / (link["h2d"] * 1e9) * 1e3, 3),
               "timeline_per_step": tl,
               "overlap": f"uploads and downloads on their own streams, {NSET} device buffer sets; "
                          "each component waits for its own inputs only and returns its results "
                          "as soon as it has finished"}
        rc, site = cg.chain_check()
        if rc != 0:
            raise RuntimeError(f"device status {rc} site {site:#x} in e2e region")
        del hps

    # ---- NEXT rows, measured beside the step (not part of its value)
    nxt = {}
    if hp.shards[0].numel() and (args.only is None or "sp" in args.only):
        nxt.update(measure_sp_fused(hp))
    if hp.shards[0].numel() and (args.only is None or "relayout" in args.only):
        nxt.update(measure_relayout_clean(hp))
    if hp.mlp_ok:
        nxt.update(measure_mlp_bwd(hp))
        nxt.update(measure_mlp_compensated(hp))
    if args.only is None or "fp8" in args.only:
        nxt.update(measure_fp8(hp))
    if hp.q3.numel() or hp.hm[0].numel():
        nxt.update(measure_fwd_compensated(hp))
    if args.only is None or "gqa" in args.only:
        nxt.update(measure_gqa(hp))
    if args.only is None or "varlen" in args.only:
        nxt.update(measure_varlen(hp))
    nxt = nxt or None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, s, desc, thr = oracle_sample()
        rl_gbps, rl_s = oracle_relayout_gbps()
        cpu = {"value": v, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
               "sample": desc + f"; total {s:.1f}s",
               # the whole step at the sample's rate (its relayouts aside)
               "step_s_extrapolated": round(hp.flops / (v * 1e12), 1),
               "relayout_GBps": round(rl_gbps, 2),
               "relayout_sample": f"one full tensor, 536,870,912 B moved ({rl_s:.2f}s)"}

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic",
                "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}",
                           "l2": "inputs larger than L2 (step working set ~8 GB)",
                           "flops_per_step": hp.flops,
                           "frac_of_measured_peak": round(value / world / tf_peak, 4),
                           "frac_of_sustained_peak": round(value / world / tf_sus, 4)},
                "roofline": roof, "components": components, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": hp.launches * args.steps, "clocks": clocks, "next_rows": nxt}
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
