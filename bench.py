#!/usr/bin/env python
"""MoE decode-layer benchmark: µs per layer-step and achieved HBM GB/s over
the unique weight bytes a step must read, on one GB300 (or N replicas).

Default step (the suite): one decode-layer pass (route -> dispatch -> expert
FFN -> combine, as the library's whole-layer calls run it) of every layer of
the synthetic configurations, each at its batch sizes --
  * vanilla MoE, d=2048, 128 experts, I=768, top-8, bf16: T = 1, 4, 16;
  * DeaMoE ~7B (8 departments of 8, I_sh=1024, I_pr=128, top-8) and its
    budget-matched vanilla twin (64 experts, I=1152): T = 1, 4, 8, 16;
  * DeepSeek-V3-shaped vanilla (256 experts, I=2048, top-8, shared expert
    2048) and DeaMoE (16 departments of 16, I_sh=1792, I_pr=256, same shared
    expert): T = 1, 8, 32, 64;
  * the 7B pair under Zipf(1.1)-skewed routing: T = 1, 2, 4, ..., 128.
Expert weights bf16, router and activations fp32.  Consecutive steps use
different layer replicas (distinct weights and inputs), so the bytes touched
between two uses of a replica exceed the 129 MB L2 many times over: weights
are read cold.

value = unique weight bytes of all timed layer passes / device time (GB/s).
per_batch gives, per layer and batch size, µs per layer, unique MB, GB/s, the
fraction of the measured HBM bandwidth and each stage alone; next_rows the
same for the matrix form P and FP8 weights (not part of the step).
Inputs are synthetic (seeded), see moe_decode_layer_fp32_gb300.synth.

--workload NAME times one layer alone.  --impl reference times the CPU oracle
(the reference arm of this build) on bounded samples of the same workloads.
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

from moe_decode_layer_fp32_gb300 import synth  # noqa: E402

WORKLOADS = {
    "vanilla-128e": synth.VANILLA_128E,
    "deamoe-7b": synth.DEAMOE_7B,
    "vanilla-7b": synth.VANILLA_7B,
    "dsv3-vanilla": synth.DSV3_VANILLA,
    "dsv3-deamoe": synth.DSV3_DEAMOE,
    "zipf-deamoe": synth.ZIPF_DEAMOE,
    "zipf-vanilla": synth.ZIPF_VANILLA,
    "formp-7b": synth.FORMP_7B,
    "formp-dsv3": synth.FORMP_DSV3,
    "dsv3-routed": synth.DSV3_ROUTED,
    "vanilla-128e-fp8": synth.VANILLA_128E_FP8,
    "deamoe-7b-fp8": synth.DEAMOE_7B_FP8,
}
# The default step: every layer of the five configurations that is not a
# correctness case -- the vanilla 128-expert layer, the DeaMoE ~7B layer and its
# budget-matched vanilla twin, the DeepSeek-V3-shaped vanilla and DeaMoE layers,
# and the Zipf-skewed sweep of both 7B layers.
SUITE = ("vanilla-128e", "deamoe-7b", "vanilla-7b", "dsv3-vanilla", "dsv3-deamoe", "zipf-deamoe", "zipf-vanilla")
# Timed after the step, per batch size, outside `value`: the matrix form P at
# its Table 1 shapes next to its baseline, and FP8 weights.
NEXT = ("formp-7b", "formp-dsv3", "dsv3-routed", "vanilla-128e-fp8", "deamoe-7b-fp8")
METRIC = "MoE-layer decode µs and achieved HBM GB/s (unique weight bytes) at batch 1–64"
L2_BYTES = 129 * 2 ** 20


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", choices=["suite"] + sorted(WORKLOADS), default="suite",
                   help="suite (default): one step runs every layer of " + ", ".join(SUITE))
    p.add_argument("--no-next", action="store_true", help="skip the NEXT rows' per-batch timings")
    p.add_argument("--batches", type=str, default="", help="comma list overriding the workload's batches")
    p.add_argument("--replicas", type=int, default=0, help="layer replicas (0 = enough for cold L2)")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU-baseline sample budget")
    p.add_argument("--tc-min-tokens", type=int, default=0,
                   help="tokens per unit from which the tensor-core kernel runs (0 = library default)")
    return p.parse_args(argv)


# --------------------------------------------------------------------------- distributed


def dist_setup(want: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    """Max of a per-rank scalar (the timing rule: slowest rank sets the time)."""
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        self.thread = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.ident = None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.ident:
            cmd += ["-i", self.ident]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm = []
        mx = []
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in self.rows:
            if len(r) < len(self.FIELDS):
                continue
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except ValueError:
                continue
            for name, v in zip(names, r[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- our arm


class Workload:
    """Layer replicas, their inputs, workspaces and outputs on one device."""

    def __init__(self, B, shape: synth.LayerShape, batches, replicas: int, seed: int, device):
        self.B = B
        self.shape = shape
        self.batches = batches
        self.device = device
        s = shape
        self.g = s.g if s.I_sh > 0 else 1
        self.layers = [synth.make_layer(s, seed * 1000 + r, device) for r in range(replicas)]
        self.R = replicas
        self.x, self.ws, self.idx, self.w, self.y = {}, {}, {}, {}, {}
        for r in range(replicas):
            for T in batches:
                key = (r, T)
                self.x[key] = synth.hidden(T, s.d, seed * 1000 + r * 131 + T, device)
                self.ws[key] = (B.new_formp_workspace(T, s.n, s.k, s.g, s.I_sh, device) if s.form_p
                                else B.new_workspace(T, s.n, s.k, self.g, device))
                self.idx[key] = torch.empty((T, s.k), dtype=torch.int32, device=device)
                self.w[key] = torch.empty((T, s.k), dtype=torch.float32, device=device)
                self.y[key] = torch.empty((T, s.d), dtype=torch.float32, device=device)
        # group-limited routing: the departments, or n/8 groups of a vanilla
        # layer; half of them kept per token
        self.rg = s.g if s.I_sh > 0 and s.g > 1 else max(1, s.n // 8)
        self.k_dept = s.k_dept or max(1, (s.n // self.rg) // 2)
        self.gidx = {T: torch.empty((T, s.k), dtype=torch.int32, device=device) for T in batches}
        self.gw = {T: torch.empty((T, s.k), dtype=torch.float32, device=device) for T in batches}
        self.bias_copy = [torch.zeros(s.n, device=device) for _ in range(replicas)]
        self.imbalance = {key: torch.zeros(1, device=device) for key in self.x}
        self.unique = {}
        self.ffn_bytes = {}
        self.counts = {}
        self.choice = {}

    def shared(self, L):
        return None if L["sgate"] is None else (L["sgate"], L["sup"], L["sdown"])

    def scales(self, L):
        """FP8 row scales in the order of the *_fp8 calls (None otherwise)."""
        if self.shape.dtype != "fp8":
            return None
        keys = (("dgate", "dup", "ddown", "pgate", "pup", "pdown") if self.shape.I_sh > 0 else
                ("gate", "up", "down"))
        return [L.get(k_ + "_sc") for k_ in keys + ("sgate", "sup", "sdown")]

    def layer(self, r, T, x=None, y=None):
        s, B, L, key = self.shape, self.B, self.layers[r], (r, T)
        x = self.x[key] if x is None else x
        y = self.y[key] if y is None else y
        if s.form_p:
            B.deamoe_p_layer_forward(x, s.k, 1.0, L["router"], L["bias"], s.g, s.k_dept,
                                     (L["dgate"], L["dup"], L["ddown"]), (L["agate"], L["aup"], L["adown"]),
                                     self.ws[key], self.idx[key], self.w[key], y)
        elif s.I_sh > 0:
            priv = (L["pgate"], L["pup"], L["pdown"]) if s.I_pr > 0 else None
            B.deamoe_layer_forward(x, s.k, 1.0, L["router"], L["bias"], s.g,
                                   (L["dgate"], L["dup"], L["ddown"]), priv, self.shared(L),
                                   self.ws[key], self.idx[key], self.w[key], y, scales=self.scales(L))
        else:
            B.moe_layer_forward(x, s.k, 1.0, L["router"], L["bias"], L["gate"], L["up"], L["down"],
                                self.shared(L), self.ws[key], self.idx[key], self.w[key], y,
                                scales=self.scales(L))

    def route_only(self, r, T):
        s, L, key = self.shape, self.layers[r], (r, T)
        if s.k_dept:
            self.B.moe_route_topk_grouped(self.x[key], L["router"], L["bias"], s.k, s.g, s.k_dept, False, 1.0,
                                          self.idx[key], self.w[key], self.ws[key])
        else:
            self.B.moe_route_topk(self.x[key], L["router"], L["bias"], s.k, 1.0,
                                  self.idx[key], self.w[key], self.ws[key])

    def grouped_only(self, r, T, strict: bool):
        """Group-limited routing of the same inputs (k_dept of the departments,
        or of n/8 expert groups on a vanilla layer) into scratch outputs."""
        L, key = self.layers[r], (r, T)
        self.B.moe_route_topk_grouped(self.x[key], L["router"], L["bias"], self.shape.k, self.rg,
                                      self.k_dept, strict, 1.0, self.gidx[T], self.gw[T], self.ws[key])

    def bias_only(self, r, T):
        """Router-bias update (sign rule) and imbalance ratio from the loads the
        layer pass left in the workspace, on a copy of the bias."""
        key = (r, T)
        counts = self.B.workspace_counts(self.ws[key], T, self.shape.n, self.shape.k, self.g)
        self.B.moe_bias_update(counts, 1e-3, self.B.MOE_BIAS_SIGN, self.bias_copy[r], self.imbalance[key])

    def dispatch_only(self, r, T):
        key = (r, T)
        self.B.moe_dispatch(self.idx[key], self.w[key], self.shape.n, self.g, self.ws[key])

    def ffn_only(self, r, T, out):
        s, B, L, key = self.shape, self.B, self.layers[r], (r, T)
        if s.form_p:
            B.deamoe_p_ffn(self.x[key], s.k, s.g, (L["dgate"], L["dup"], L["ddown"]),
                           (L["agate"], L["aup"], L["adown"]), self.idx[key], self.ws[key], out)
        elif s.I_sh > 0:
            priv = (L["pgate"], L["pup"], L["pdown"]) if s.I_pr > 0 else None
            B.deamoe_ffn(self.x[key], s.k, s.g, (L["dgate"], L["dup"], L["ddown"]), priv,
                         self.shared(L), self.ws[key], B.MOE_OUT_ACCUM, out, scales=self.scales(L))
        else:
            B.moe_ffn_vanilla(self.x[key], s.k, L["gate"], L["up"], L["down"], self.shared(L),
                              self.ws[key], B.MOE_OUT_ACCUM, out, scales=self.scales(L))

    def account(self):
        """Unique weight bytes of every (replica, batch) pass from device counts."""
        s, B = self.shape, self.B
        code = {"bf16": B.MOE_DTYPE_BF16, "f32": B.MOE_DTYPE_F32, "fp8": B.MOE_DTYPE_FP8_E4M3}[s.dtype]
        for key, ws in self.ws.items():
            st, A_e, A_d = B.moe_read_status(ws)
            if st != 0:
                raise RuntimeError(f"device status {st} for {key}")
            if s.form_p:
                U = B.moe_unique_weight_bytes_formp(s.d, s.n, s.I_sh, A_d, A_e)
            elif s.I_sh > 0:
                U = B.moe_unique_weight_bytes_deamoe(s.d, s.n, s.I_sh, s.I_pr, s.I_s, code, A_d, A_e)
            else:
                U = B.moe_unique_weight_bytes_vanilla(s.d, s.n, s.I, s.I_s, code, A_e)
            self.unique[key] = U
            self.ffn_bytes[key] = U - 4 * s.d * s.n
            self.counts[key] = (A_e, A_d)
            lay = B.moe_workspace_layout(key[1], s.n, s.k, self.g)
            self.choice[key] = int(ws[lay["sync"] + 4: lay["sync"] + 8].cpu().view(torch.int32)[0])

    def launches(self, key, thr: int) -> int:
        """Kernels one layer pass launches: form P, the routing kernel and its
        three passes; otherwise the routing kernel and the FFN kernels -- the
        tensor-core kernel alone on its in-CTA routing path (automatic choice,
        rows at most 4096 wide, T <= 32, at most 256 experts), both FFN kernels
        when the tensor-core kernel is launched beside the CUDA-core one, else
        the CUDA-core kernel alone."""
        s, T = self.shape, key[1]
        if s.form_p:
            return 4
        if not self.tc_launched(key, thr):
            return 2
        tc_alone = thr == 0 and s.d <= 4096 and T <= 32 and s.n <= 256 and self.choice[key] == 2
        return 2 if tc_alone else 3

    def tc_launched(self, key, thr: int) -> bool:
        """Whether the layer pass launches the tensor-core FFN kernel: in
        automatic mode exactly when the kernels recorded a choice; with a fixed
        threshold when the weights qualify and T >= thr."""
        s, T = self.shape, key[1]
        if s.form_p:
            return False
        rows = [r for r in (s.I, s.I_sh, s.I_pr, s.I_s) if r > 0]
        ok = s.dtype == "bf16" and s.d % 128 == 0 and all(r % 128 == 0 for r in rows)
        if not ok:
            return False
        if thr > 0:
            return T >= thr
        return self.choice[key] != 0


def capture(fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def time_graphs(graphs, order, world, device):
    """Replay graphs[i] for i in order between two events; max over ranks (s)."""
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for i in order:
        graphs[i].replay()
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(start.elapsed_time(end) / 1e3, world, device)


def replicas_for(shape, R_arg: int) -> int:
    """Layer replicas so that the bytes between two uses of one replica exceed
    4x L2 (from the smallest pass: one token, k experts, one department)."""
    bw = {"bf16": 2, "f32": 4, "fp8": 1}[shape.dtype]
    per_layer_min = (bw * 3 * (shape.d * shape.I_sh + shape.I_sh * shape.I_sh * shape.k) if shape.form_p else
                     bw * 3 * shape.d * (shape.I_pr * shape.k + shape.I_sh + shape.I * shape.k + shape.I_s))
    return R_arg or max(2, min(16, -(-4 * L2_BYTES // max(1, per_layer_min))))


def stage_fns(W, T, scratch):
    """Each stage alone over the replicas: routing with its top-k, dispatch,
    the FFN step, and the NEXT rows on the same inputs (group-limited routing
    soft and strict, router-bias update) for the layers that have them."""
    R = W.R
    fns = [("route_topk", lambda: [W.route_only(r, T) for r in range(R)]),
           ("ffn", lambda: [W.ffn_only(r, T, scratch[r]) for r in range(R)])]
    if not W.shape.form_p:
        fns.insert(1, ("dispatch", lambda: [W.dispatch_only(r, T) for r in range(R)]))
        fns += [("route_topk_grouped", lambda: [W.grouped_only(r, T, False) for r in range(R)]),
                ("route_topk_grouped_strict", lambda: [W.grouped_only(r, T, True) for r in range(R)]),
                ("bias_update", lambda: [W.bias_only(r, T) for r in range(R)])]
    return fns


def measure_batches(W, args, world, device, peak):
    """Per batch size of one workload: µs per layer (graphs of its replicas),
    unique bytes, GB/s, fraction of the HBM peak, and each stage alone."""
    B, shape, R = W.B, W.shape, W.R
    per_batch = {}
    reps = max(3, min(200, args.steps // max(1, R)))
    for T in W.batches:
        gT = capture(lambda T=T: [W.layer(r, T) for r in range(R)])
        time_graphs([gT], [0] * 3, world, device)
        us = time_graphs([gT], [0] * reps, world, device) / (reps * R) * 1e6
        U = sum(W.unique[(r, T)] for r in range(R)) / R
        Uf = sum(W.ffn_bytes[(r, T)] for r in range(R)) / R
        stage_us = {}
        scratch_T = {r: torch.zeros_like(W.y[(r, T)]) for r in range(R)}
        for name, fn in stage_fns(W, T, scratch_T):
            gs = capture(fn)
            time_graphs([gs], [0] * 3, world, device)
            stage_us[name] = round(time_graphs([gs], [0] * reps, world, device) / (reps * R) * 1e6, 2)
        if shape.form_p:
            paths = ["formp passes"]
        else:
            paths = sorted({("tensor-core" if W.choice[(r, T)] == 2 else
                             "cuda-core" if W.choice[(r, T)] == 1 or not W.tc_launched((r, T), args.tc_min_tokens)
                             else "split") for r in range(R)})
        e = {"us_per_layer": round(us, 2), "unique_MB": round(U / 1e6, 2), "GBps": round(U / us / 1e3, 1),
             "frac": round(U / us / 1e3 / peak, 4),
             "ffn_us": stage_us["ffn"], "ffn_frac": round(Uf / stage_us["ffn"] / 1e3 / peak, 4),
             "stage_us": stage_us, "ffn_path": "/".join(paths),
             "active_experts": round(sum(W.counts[(r, T)][0] for r in range(R)) / R, 2)}
        if shape.I_sh > 0:
            e["active_depts"] = round(sum(W.counts[(r, T)][1] for r in range(R)) / R, 2)
        if not shape.form_p:
            e["grouped_routing"] = f"{W.k_dept} of {shape.n // W.rg} groups of {W.rg}"
            e["imbalance"] = round(sum(W.imbalance[(r, T)].item() for r in range(R)) / R, 3)
        per_batch[str(T)] = e
    return per_batch


def run_ours(args, rank, world, local):
    from moe_decode_layer_fp32_gb300 import binding as B
    B.lib()  # fails loudly when the native library is missing
    B.moe_set_tc_min_tokens(args.tc_min_tokens)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    names = SUITE if args.workload == "suite" else (args.workload,)
    override = tuple(int(b) for b in args.batches.split(",")) if args.batches else None
    peaks = load_peaks()
    peak = peaks["hbm_gbs"]

    # one Workload per layer of the step: its replicas, inputs and workspaces
    Ws = []
    for name in names:
        shape = WORKLOADS[name]
        Ws.append(Workload(B, shape, override or shape.batches, replicas_for(shape, args.replicas),
                           args.seed + 17 * rank, device))
        Ws[-1].name = name

    # first pass (eager), then device counts -> unique bytes
    for W in Ws:
        for r in range(W.R):
            for T in W.batches:
                W.layer(r, T)
    torch.cuda.synchronize()
    for W in Ws:
        W.account()

    # a step = one layer pass at every batch size of every workload; step i
    # runs replica i % R of each workload (one graph per workload and replica)
    graphs = [[capture(lambda W=W, r=r: [W.layer(r, T) for T in W.batches]) for r in range(W.R)] for W in Ws]
    flat = [g for gs in graphs for g in gs]
    index = {(w, r): sum(len(gs) for gs in graphs[:w]) + r for w, gs in enumerate(graphs) for r in range(len(gs))}

    def order(steps):
        return [index[(w, i % Ws[w].R)] for i in range(steps) for w in range(len(Ws))]

    time_graphs(flat, order(args.warmup), world, device)
    clocks = ClockSampler(local)
    clocks.start()
    t_step = time_graphs(flat, order(args.steps), world, device)
    clock_info = clocks.stop()
    bytes_rank = sum(W.unique[(i % W.R, T)] for i in range(args.steps) for W in Ws for T in W.batches)
    bytes_all = sum_over_ranks(bytes_rank, world, device)
    value = bytes_all / t_step / 1e9

    per_workload = {W.name: measure_batches(W, args, world, device, peak) for W in Ws}

    # roofline of the dominant kernel (the expert FFN step): FFN launches
    # alone over the same inputs, every workload of the step
    reps_f = max(3, min(50, args.steps // 4))
    t_ffn, ffn_launches, ffn_bytes = 0.0, 0, 0
    for W in Ws:
        scratch = {key: torch.zeros_like(y) for key, y in W.y.items()}
        g_ffn = capture(lambda W=W, scratch=scratch: [W.ffn_only(r, T, scratch[(r, T)])
                                                      for r in range(W.R) for T in W.batches])
        time_graphs([g_ffn], [0] * 3, world, device)
        t_ffn += time_graphs([g_ffn], [0] * reps_f, world, device)
        ffn_launches += reps_f * W.R * len(W.batches)
        ffn_bytes += reps_f * sum(W.ffn_bytes.values())
    achieved = ffn_bytes / t_ffn / 1e9
    kernels = set()
    for W in Ws:
        kernels |= ({"formp_kernel up / private / down passes"} if W.shape.form_p else
                    {"ffn_tc_kernel" if W.choice[key] == 2 else "ffn_stream_kernel" for key in W.ws})
    fracs = [e["frac"] for pb in per_workload.values() for e in pb.values()]
    roofline = {"bound": "hbm", "kernel": "expert FFN step (" + ", ".join(sorted(kernels)) + ")",
                "achieved": round(achieved, 1), "peak": peak, "peak_source": peaks["source"], "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "us_per_launch": round(t_ffn / ffn_launches * 1e6, 2),
                "algorithmic_bytes_per_launch": int(ffn_bytes / ffn_launches),
                "traffic": load_traffic(args.workload) if not args.batches else None,
                "layer_frac_mean": round(sum(fracs) / len(fracs), 4),
                "layer_frac_min": min(fracs),
                "per_workload": {name: {T: {"layer": e["frac"], "ffn": e["ffn_frac"]} for T, e in pb.items()}
                                 for name, pb in per_workload.items()}}

    # end to end through the C ABI with host buffers (copies inside the timed region)
    e2e = None
    if not args.no_e2e:
        hx = [{key: x.cpu().pin_memory() for key, x in W.x.items()} for W in Ws]
        hy = [{key: torch.empty(y.shape, dtype=y.dtype).pin_memory() for key, y in W.y.items()} for W in Ws]
        dx = [{T: torch.empty((T, W.shape.d), device=device) for T in W.batches} for W in Ws]

        def e2e_step(i):
            for w, W in enumerate(Ws):
                r = i % W.R
                for T in W.batches:
                    B.moe_input_from_host(dx[w][T], hx[w][(r, T)])
                    W.layer(r, T, x=dx[w][T])
                    B.moe_output_to_host(hy[w][(r, T)], W.y[(r, T)])

        ke = min(args.steps, 500)
        for i in range(min(args.warmup, 20)):
            e2e_step(i)
        barrier(world)
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record()
        for i in range(ke):
            e2e_step(i)
        s1.record()
        torch.cuda.synchronize()
        barrier(world)
        te = max_over_ranks(s0.elapsed_time(s1) / 1e3, world, device)
        be = sum_over_ranks(sum(W.unique[(i % W.R, T)] for i in range(ke) for W in Ws for T in W.batches),
                            world, device)
        io = sum(T * W.shape.d * 4 for W in Ws for T in W.batches)
        e2e = {"value": round(be / te / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": io,
               "d2h_bytes_per_step": io, "steps": ke, "ms_per_step": round(te / ke * 1e3, 4)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(Ws, args.cpu_seconds)

    # the NEXT rows (matrix form P at its Table 1 shapes beside its baseline,
    # FP8 weights), timed per batch size alone: not part of the step above
    next_rows = None
    if args.workload == "suite" and not args.no_next:
        next_rows = {}
        for name in NEXT:
            shape = WORKLOADS[name]
            W = Workload(B, shape, override or shape.batches, replicas_for(shape, args.replicas),
                         args.seed + 17 * rank, device)
            W.name = name
            for r in range(W.R):
                for T in W.batches:
                    W.layer(r, T)
            torch.cuda.synchronize()
            W.account()
            next_rows[name] = measure_batches(W, args, world, device, peak)
            del W
            torch.cuda.empty_cache()

    launches = sum(W.launches((i % W.R, T), args.tc_min_tokens) for i in range(args.steps) for W in Ws
                   for T in W.batches)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "weights_dtype": "/".join(sorted({W.shape.dtype for W in Ws})), "data": "synthetic",
        "config": {**suite_config(Ws), "tc_min_tokens": args.tc_min_tokens or "default",
                   "l2": "inputs larger than L2: consecutive steps use distinct layer replicas of each "
                         "workload (>=4x L2 between reuses of a replica)",
                   "parallelism": f"replicas x{world}"},
        "per_batch": per_workload,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clock_info,
        "cpu_baseline": cpu,
    }
    if next_rows is not None:
        out["next_rows"] = next_rows
    if rank == 0:
        print(json.dumps(out))


def suite_config(Ws):
    """The `config` of a step over one or more workloads."""
    if len(Ws) == 1:
        W = Ws[0]
        return {**workload_config(W.shape, W.batches), "replicas": W.R}
    return {"workload": "; ".join(f"{W.shape.name} T={'/'.join(map(str, W.batches))}" for W in Ws),
            "layers": {W.name: {**workload_config(W.shape, W.batches), "replicas": W.R} for W in Ws}}


def workload_config(shape, batches):
    """The `config` keys both arms report for a workload."""
    return {"workload": f"{shape.name} T={'/'.join(map(str, batches))}", "d": shape.d,
            "n_experts": shape.n, "top_k": shape.k, "I": shape.I, "I_sh": shape.I_sh,
            "I_pr": shape.I_pr, "experts_per_dept": shape.g, "I_shared": shape.I_s,
            "weights_dtype": shape.dtype, "zipf": shape.zipf, "batches": list(batches),
            "form": "P (eq. 4, r = I_sh)" if shape.form_p else "C" if shape.I_sh > 0 else "vanilla",
            "k_dept": shape.k_dept}


def load_traffic(workload: str):
    """DRAM bytes per FFN launch of this workload from the committed ncu
    summaries (profiles/*.md: `traffic_bytes_per_launch[<workload>]: N`), or
    None when no capture of the current kernels exists for it."""
    import glob
    import re
    pat = re.compile(r"^traffic_bytes_per_launch\[" + re.escape(workload) + r"\]:\s*(\d+)\s*$")
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                m = pat.match(line.strip())
                if m:
                    return int(m.group(1))
    return None


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "source": "fallback"}


# --------------------------------------------------------------------------- oracle arms


class _HostUnits:
    """Host copies of the units of one [units, rows, d] device tensor, made
    on request (outside the oracle's timed sections); FP8 units are decoded
    exactly with their row scales.  Indexing returns the host copy."""

    def __init__(self, O, dev, scales=None):
        self.O, self.dev, self.scales, self.cache = O, dev, scales, {}

    def fetch(self, u):
        if u not in self.cache:
            w = self.dev[u].cpu()
            self.cache[u] = (w if self.scales is None else
                             self.O.dequant_rows_e4m3(w, self.scales[u].cpu()))
        return self.cache[u]

    def __getitem__(self, u):
        return self.cache[u]


class _HostLayer(dict):
    """The oracle's view of one device layer: router, bias and shared expert
    copied whole, every other tensor per unit, only for the units a pass
    touches (a DeepSeek-V3-shaped layer is tens of GB)."""

    UNIT_KEYS = ("gate", "up", "down", "dgate", "dup", "ddown", "pgate", "pup", "pdown", "agate", "aup", "adown")

    def __init__(self, O, shape, L):
        super().__init__()
        self.shape = shape
        self["router"] = L["router"].cpu()
        self["bias"] = None if L["bias"] is None else L["bias"].cpu()
        for key in ("sgate", "sup", "sdown"):
            v = L.get(key)
            if v is not None and shape.dtype == "fp8":
                v = O.dequant_rows_e4m3(v.cpu(), L[key + "_sc"].cpu())
            self[key] = None if v is None else v.cpu() if torch.is_tensor(v) else v
        for key in self.UNIT_KEYS:
            if key in L:
                self[key] = _HostUnits(O, L[key], L.get(key + "_sc"))

    def prefetch(self, idx):
        s = self.shape
        for e in {int(e) for e in idx.ravel()}:
            for key, u in (("gate", e), ("up", e), ("down", e), ("dgate", e // s.g), ("dup", e // s.g),
                           ("ddown", e // s.g), ("pgate", e), ("pup", e), ("pdown", e), ("agate", e),
                           ("aup", e), ("adown", e)):
                if key in self:
                    self[key].fetch(u)


def oracle_route(O, shape, L, x):
    if shape.k_dept:
        return O.route_grouped(x, L["router"], shape.k, shape.g, shape.k_dept, bias=L["bias"])
    return O.route(x, L["router"], shape.k, bias=L["bias"])


def cpu_baseline(Ws, budget_s, max_T=8):
    """The oracle (as it stands) on a bounded sample of the same step: whole
    layer passes of replica 0 of every workload at its batch sizes up to
    max_T, smallest first, repeated until the budget is spent.  Host copies
    of the touched weights are made outside the timed sections."""
    from oracle import moe_oracle as O
    keys = sorted(((T, w) for w, W in enumerate(Ws) for T in W.batches if T <= max_T), key=lambda k: k)
    if not keys:
        keys = [(min(W.batches), w) for w, W in enumerate(Ws)]
    host = {}
    done_bytes = 0
    t_total = 0.0
    passes = 0
    while t_total <= budget_s and passes < 100 * len(keys):
        T, w = keys[passes % len(keys)]
        W = Ws[w]
        if w not in host:
            host[w] = _HostLayer(O, W.shape, W.layers[0])
        L = host[w]
        x = W.x[(0, T)].cpu()
        idx, _, _ = oracle_route(O, W.shape, L, x)      # untimed: which units to copy
        L.prefetch(idx)
        t0 = time.perf_counter()
        idx, p, _ = oracle_route(O, W.shape, L, x)
        oracle_forward(O, W.shape, L, x, idx, p)
        t_total += time.perf_counter() - t0
        done_bytes += W.unique[(0, T)]
        passes += 1
    return {"value": round(done_bytes / t_total / 1e9, 4), "unit": "GB/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{passes} whole layer passes (routing + every selected expert of every token) of "
                      f"replica 0, cycling over {len(keys)} (workload, T <= {max_T}) pairs smallest T first, "
                      f"in {t_total:.1f} s (host copies of the touched weights made outside the timed "
                      "sections)"}


def oracle_forward(O, shape, L, x, idx, p):
    if shape.form_p:
        return O.deamoe_layer_p(x, idx, p, shape.g, L["dgate"], L["dup"], L["ddown"], L["agate"], L["aup"],
                                L["adown"])
    sh = None if L["sgate"] is None else (L["sgate"], L["sup"], L["sdown"])
    if shape.I_sh > 0:
        priv = (L["pgate"], L["pup"], L["pdown"]) if shape.I_pr > 0 else (None, None, None)
        return O.deamoe_layer_c(x, idx, p, shape.g, L["dgate"], L["dup"], L["ddown"], *priv, shared=sh)
    return O.vanilla_layer(x, idx, p, L["gate"], L["up"], L["down"], shared=sh)


class _RefStepper:
    """The reference arm's steps on one workload: step i is selected expert
    i % k of token i // k (its SwiGLU or eq. (4) pass), with the token's
    routing and shared expert on its first step.  Weights of the units the
    steps touch are made on the host before the timed region."""

    def __init__(self, O, s, seed, nsteps):
        self.O, self.s = O, s
        self.router = synth.router(s.d, s.n, seed)
        self.bias = synth.zipf_bias(s.n, s.zipf_g, s.zipf, seed) if s.zipf > 0 else None
        ntok = -(-nsteps // s.k)
        self.xs = synth.hidden(ntok, s.d, seed + 7)
        self.seed = seed
        self.units = {}
        self.row_b = 3 * s.d * {"bf16": 2, "f32": 4, "fp8": 1}[s.dtype] + (12 if s.dtype == "fp8" else 0)
        idx_all, _, _ = self.route(self.xs)      # untimed: the units the steps touch
        self.W = {int(e): self.weights(int(e)) for e in set(idx_all.ravel()[:nsteps].tolist())}
        self.SH = ([self.unit(t, 0, s.I_s) for t in (synth.TID_SGATE, synth.TID_SUP, synth.TID_SDOWN)]
                   if s.I_s else None)
        self.state = {}

    def route(self, x):
        s = self.s
        if s.k_dept:
            return self.O.route_grouped(x, self.router, s.k, s.g, s.k_dept, bias=self.bias)
        return self.O.route(x, self.router, s.k, bias=self.bias)

    def unit(self, tid, u, rows):
        s = self.s
        if (tid, u) not in self.units:
            if s.dtype == "fp8":
                w = synth.normal((rows, s.d), self.seed, tid, synth.WEIGHT_STD, "cpu", salt=u + 1)
                self.units[(tid, u)] = torch.from_numpy(self.O.dequant_rows_e4m3(*synth.quantize_rows_e4m3(w)))
            else:
                self.units[(tid, u)] = synth.normal((rows, s.d), self.seed, tid, synth.WEIGHT_STD, "cpu",
                                                    synth.storage_dtype(s.dtype), salt=u + 1)
        return self.units[(tid, u)]

    def amat(self, tid, e):
        if (tid, e) not in self.units:
            self.units[(tid, e)] = synth.near_identity_unit(e, self.s.I_sh, self.seed, tid, self.s.dtype)
        return self.units[(tid, e)]

    def weights(self, e):
        s = self.s
        if s.form_p:
            j = e // s.g
            return ([self.unit(t, j, s.I_sh) for t in (synth.TID_DGATE, synth.TID_DUP, synth.TID_DDOWN)] +
                    [self.amat(t, e) for t in (synth.TID_AGATE, synth.TID_AUP, synth.TID_ADOWN)])
        if s.I_sh > 0:
            j = e // s.g
            return [torch.cat([self.unit(t1, j, s.I_sh)] + ([self.unit(t2, e, s.I_pr)] if s.I_pr else []))
                    for t1, t2 in ((synth.TID_DGATE, synth.TID_PGATE), (synth.TID_DUP, synth.TID_PUP),
                                   (synth.TID_DDOWN, synth.TID_PDOWN))]
        return [self.unit(t, e, s.I) for t in (synth.TID_GATE, synth.TID_UP, synth.TID_DOWN)]

    def step(self, i):
        O, s, st = self.O, self.s, self.state
        tok, q = divmod(i, s.k)
        nbytes = 0
        if q == 0:
            x = self.xs[tok:tok + 1]
            idx, p, _ = self.route(x)
            st.update(x=x, idx=idx, p=p, depts=set())
            nbytes += 4 * s.d * s.n
            if self.SH is not None:
                O.swiglu_expert(x[0], *self.SH)
                nbytes += self.row_b * s.I_s
        x, idx, p = st["x"], st["idx"], st["p"]
        e = int(idx[0, q])
        if s.form_p:
            p[0, q] * O.deamoe_expert_p(x[0], *self.W[e])
            j = e // s.g
            nbytes += 2 * (3 * s.d * s.I_sh * (j not in st["depts"]) + 3 * s.I_sh * s.I_sh)
            st["depts"].add(j)
        elif s.I_sh > 0:
            p[0, q] * O.swiglu_expert(x[0], *self.W[e])
            j = e // s.g
            nbytes += self.row_b * (s.I_pr + (s.I_sh if j not in st["depts"] else 0))
            st["depts"].add(j)
        else:
            p[0, q] * O.swiglu_expert(x[0], *self.W[e])
            nbytes += self.row_b * s.I
        return nbytes


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle timed on the host cores.  A step is one
    selected expert of one token (its SwiGLU pass, plus the token's routing
    and shared expert on its first step); over the suite, step i runs on
    workload i % (number of workloads)."""
    if rank != 0:
        return
    from oracle import moe_oracle as O
    names = SUITE if args.workload == "suite" else (args.workload,)
    override = tuple(int(b) for b in args.batches.split(",")) if args.batches else None
    total_steps = args.steps + args.warmup
    per = -(-total_steps // len(names))
    steppers = [_RefStepper(O, WORKLOADS[n], args.seed * 1000, per) for n in names]
    counters = [0] * len(names)

    def step(i):
        w = i % len(names)
        j = counters[w]
        counters[w] += 1
        return steppers[w].step(j)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    total = 0
    for i in range(args.steps):
        total += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = total / dt / 1e9

    class _S:     # the configs of the workloads, as our arm reports them
        def __init__(self, name):
            self.name, self.shape = name, WORKLOADS[name]
            self.batches = override or self.shape.batches
            self.R = replicas_for(self.shape, args.replicas)
    config = suite_config([_S(n) for n in names])
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {**config, "sample": "one selected expert of one token per step"
                                          + (", workloads in turn" if len(names) > 1 else "")},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle",
                            "cores": len(os.sched_getaffinity(0)),
                            "sample": "one (token, expert) SwiGLU pass per step; routing and "
                                      "shared expert on each token's first step"},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
