#!/usr/bin/env python
"""MoE decode-layer benchmark: µs per layer-step and achieved HBM GB/s over
the unique weight bytes a step must read, on one GB300 (or N replicas).

Default workload: the vanilla MoE decode layer d=2048, 128 routed experts,
SwiGLU intermediate 768, top-8 softmax-renormalised routing, bf16 expert
weights, fp32 router, no shared expert, at batches T in {1, 4, 16}.  A step is
one decode-layer pass (route -> dispatch -> expert FFN -> combine) at each of
the three batch sizes.  Consecutive steps use different layer replicas
(distinct weights and inputs), so the bytes touched between two uses of the
same replica exceed the 129 MB L2 many times over: weights are read cold.

value = unique weight bytes of all timed layer passes / device time (GB/s).
Inputs are synthetic (seeded), see moe_decode_layer_fp32_gb300.synth.

--impl reference times the CPU oracle (the reference arm of this build) on
bounded samples of the same workload.
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
METRIC = "MoE-layer decode µs and achieved HBM GB/s (unique weight bytes) at batch 1–64"
L2_BYTES = 129 * 2 ** 20


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default="vanilla-128e")
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


def run_ours(args, rank, world, local):
    from moe_decode_layer_fp32_gb300 import binding as B
    B.lib()  # fails loudly when the native library is missing
    B.moe_set_tc_min_tokens(args.tc_min_tokens)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    shape = WORKLOADS[args.workload]
    batches = tuple(int(b) for b in args.batches.split(",")) if args.batches else shape.batches

    # Replicas: enough that the bytes between two uses of a replica exceed 4x L2.
    # (smallest pass: one token, k experts, one department)
    bw = {"bf16": 2, "f32": 4, "fp8": 1}[shape.dtype]
    per_layer_min = (bw * 3 * (shape.d * shape.I_sh + shape.I_sh * shape.I_sh * shape.k) if shape.form_p else
                     bw * 3 * shape.d * (shape.I_pr * shape.k + shape.I_sh + shape.I * shape.k + shape.I_s))
    R = args.replicas or max(2, min(16, -(-4 * L2_BYTES // max(1, per_layer_min))))
    W = Workload(B, shape, batches, R, args.seed + 17 * rank, device)

    # first pass (eager), then device counts -> unique bytes
    for r in range(R):
        for T in batches:
            W.layer(r, T)
    torch.cuda.synchronize()
    W.account()

    # one graph per replica: a step = one layer pass at every batch size
    graphs = [capture(lambda r=r: [W.layer(r, T) for T in batches]) for r in range(R)]
    time_graphs(graphs, [i % R for i in range(args.warmup)], world, device)

    clocks = ClockSampler(local)
    clocks.start()
    t_step = time_graphs(graphs, [i % R for i in range(args.steps)], world, device)
    clock_info = clocks.stop()
    bytes_rank = sum(W.unique[(i % R, T)] for i in range(args.steps) for T in batches)
    bytes_all = sum_over_ranks(bytes_rank, world, device)
    value = bytes_all / t_step / 1e9

    # per-batch µs per layer: graphs of the R replicas at one batch size
    per_batch = {}
    reps = max(3, min(200, args.steps // max(1, R)))
    for T in batches:
        gT = capture(lambda T=T: [W.layer(r, T) for r in range(R)])
        time_graphs([gT], [0] * 3, world, device)
        t = time_graphs([gT], [0] * reps, world, device)
        us = t / (reps * R) * 1e6
        U = sum(W.unique[(r, T)] for r in range(R)) / R
        # each stage alone (route+top-k, dispatch, expert FFN), as graphs over the replicas
        stage_us = {}
        scratch_T = {r: torch.zeros_like(W.y[(r, T)]) for r in range(R)}
        for name, fn in (("route_topk", lambda T=T: [W.route_only(r, T) for r in range(R)]),
                         ("dispatch", lambda T=T: [W.dispatch_only(r, T) for r in range(R)]),
                         ("ffn", lambda T=T: [W.ffn_only(r, T, scratch_T[r]) for r in range(R)]),
                         ("route_topk_grouped", lambda T=T: [W.grouped_only(r, T, False) for r in range(R)]),
                         ("route_topk_grouped_strict", lambda T=T: [W.grouped_only(r, T, True) for r in range(R)]),
                         ("bias_update", lambda T=T: [W.bias_only(r, T) for r in range(R)])):
            gs = capture(fn)
            time_graphs([gs], [0] * 3, world, device)
            stage_us[name] = round(time_graphs([gs], [0] * reps, world, device) / (reps * R) * 1e6, 2)
        paths = sorted({("tensor-core" if W.choice[(r, T)] == 2 else
                         "cuda-core" if W.choice[(r, T)] == 1 or not W.tc_launched((r, T), args.tc_min_tokens)
                         else "split") for r in range(R)})
        per_batch[str(T)] = {"us_per_layer": round(us, 2), "unique_MB": round(U / 1e6, 2),
                             "GBps": round(U / us / 1e3, 1), "stage_us": stage_us,
                             "grouped_routing": f"{W.k_dept} of {shape.n // W.rg} groups of {W.rg}",
                             "imbalance": round(sum(W.imbalance[(r, T)].item() for r in range(R)) / R, 3),
                             "ffn_path": "/".join(paths),
                             "active_experts": round(sum(W.counts[(r, T)][0] for r in range(R)) / R, 2)}
        if shape.I_sh > 0:
            per_batch[str(T)]["active_depts"] = round(sum(W.counts[(r, T)][1] for r in range(R)) / R, 2)

    # roofline of the dominant kernel (the expert FFN): FFN launches alone, same inputs
    scratch = {key: torch.zeros_like(y) for key, y in W.y.items()}
    g_ffn = capture(lambda: [W.ffn_only(r, T, scratch[(r, T)]) for r in range(R) for T in batches])
    time_graphs([g_ffn], [0] * 3, world, device)
    reps_f = max(3, min(100, args.steps // max(1, R)))
    t_ffn = time_graphs([g_ffn], [0] * reps_f, world, device)
    ffn_launches = reps_f * R * len(batches)
    ffn_bytes = reps_f * sum(W.ffn_bytes.values())
    peaks = load_peaks()
    achieved = ffn_bytes / t_ffn / 1e9
    ffn_kernels = (["formp_kernel up / private / down passes"] if shape.form_p else
                   sorted({"ffn_tc_kernel" if W.choice[key] == 2 else "ffn_stream_kernel" for key in W.ws}))
    roofline = {"bound": "hbm", "kernel": "expert FFN step (" + ", ".join(ffn_kernels) + ")",
                "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "peak_source": peaks["source"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4),
                "us_per_launch": round(t_ffn / ffn_launches * 1e6, 2),
                "algorithmic_bytes_per_launch": int(sum(W.ffn_bytes.values()) / (R * len(batches))),
                "traffic": load_traffic(args.workload) if not args.batches else None}

    # end to end through the C ABI with host buffers (copies inside the timed region)
    e2e = None
    if not args.no_e2e:
        hx = {key: x.cpu().pin_memory() for key, x in W.x.items()}
        hy = {key: torch.empty(y.shape, dtype=y.dtype).pin_memory() for key, y in W.y.items()}
        dx = {T: torch.empty((T, shape.d), device=device) for T in batches}
        ke = min(args.steps, 500)
        for i in range(min(args.warmup, 20)):
            for T in batches:
                B.moe_input_from_host(dx[T], hx[(i % R, T)])
                W.layer(i % R, T, x=dx[T])
                B.moe_output_to_host(hy[(i % R, T)], W.y[(i % R, T)])
        barrier(world)
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record()
        for i in range(ke):
            r = i % R
            for T in batches:
                B.moe_input_from_host(dx[T], hx[(r, T)])
                W.layer(r, T, x=dx[T])
                B.moe_output_to_host(hy[(r, T)], W.y[(r, T)])
        s1.record()
        torch.cuda.synchronize()
        barrier(world)
        te = max_over_ranks(s0.elapsed_time(s1) / 1e3, world, device)
        be = sum_over_ranks(sum(W.unique[(i % R, T)] for i in range(ke) for T in batches), world, device)
        io = sum(T * shape.d * 4 for T in batches)
        e2e = {"value": round(be / te / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": io,
               "d2h_bytes_per_step": io, "steps": ke, "ms_per_step": round(te / ke * 1e3, 4)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(W, shape, batches, args.cpu_seconds)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "weights_dtype": shape.dtype, "data": "synthetic",
        "config": {**workload_config(shape, batches), "replicas": R,
                   "tc_min_tokens": args.tc_min_tokens or "default",
                   "l2": "inputs larger than L2: consecutive steps use distinct layer replicas "
                         f"({R} replicas, >=4x L2 between reuses)",
                   "parallelism": f"replicas x{world}"},
        "per_batch": per_batch,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": sum(W.launches((i % R, T), args.tc_min_tokens) for i in range(args.steps) for T in batches),
        "clocks": clock_info,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(out))


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


def cpu_baseline(W, shape, batches, budget_s):
    """The oracle (as it stands) on a bounded sample of the same workload:
    whole layer passes of replicas 0-1 at every batch size, repeated until the
    budget is spent."""
    from oracle import moe_oracle as O
    import numpy as np  # noqa: F401
    done_bytes = 0
    t_total = 0.0
    passes = 0
    keys = [(r, T) for r in range(min(2, W.R)) for T in sorted(batches)]   # host copies of <= 2 layers
    host = {}
    while t_total <= budget_s and passes < 100 * len(keys):
        r, T = keys[passes % len(keys)]
        if shape.form_p:
            # form P: host copies of the units this pass touches only (a
            # whole layer can be tens of GB)
            L = W.layers[r]
            Wl = host.setdefault(r, {"router": L["router"].cpu(), "bias": None if L["bias"] is None else L["bias"].cpu()})
            sel, _, _ = O.route_grouped(W.x[(r, T)].cpu(), Wl["router"], shape.k, shape.g, shape.k_dept or
                                        shape.n // shape.g, bias=Wl["bias"])          # untimed: units to copy
            for e in set(sel.ravel().tolist()):
                for key_, src, u in (("dgate", "dgate", e // shape.g), ("dup", "dup", e // shape.g),
                                     ("ddown", "ddown", e // shape.g), ("agate", "agate", e),
                                     ("aup", "aup", e), ("adown", "adown", e)):
                    Wl.setdefault(key_, {})
                    if u not in Wl[key_]:
                        Wl[key_][u] = L[src][u].cpu()
        else:
            if r not in host:
                L = W.layers[r]
                host[r] = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in L.items()}
                if shape.dtype == "fp8":
                    # the oracle decodes each unit it reads (codes and row scales)
                    for k_ in [k_ for k_ in host[r] if k_ + "_sc" in host[r]]:
                        host[r][k_] = _Fp8Units(O, host[r][k_], host[r][k_ + "_sc"])
        L = host[r]
        x = W.x[(r, T)].cpu()
        t0 = time.perf_counter()
        if shape.k_dept:
            idx, p, _ = O.route_grouped(x, L["router"], shape.k, shape.g, shape.k_dept, bias=L["bias"])
        else:
            idx, p, _ = O.route(x, L["router"], shape.k, bias=L["bias"])
        oracle_forward(O, shape, L, x, idx, p)
        t_total += time.perf_counter() - t0
        done_bytes += W.unique[(r, T)]
        passes += 1
    return {"value": round(done_bytes / t_total / 1e9, 4), "unit": "GB/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{passes} full layer passes cycling over (replica, T) for T in "
                      f"{sorted(batches)}, {min(passes, len(keys))} distinct, in {t_total:.1f} s "
                      "(host copies of the weights made outside the timed sections)"}


class _Fp8Units:
    """FP8 unit tensor for the oracle: indexing a unit decodes it exactly."""

    def __init__(self, O, codes, scales):
        self.O, self.codes, self.scales = O, codes, scales

    def __getitem__(self, u):
        return self.O.dequant_rows_e4m3(self.codes[u], self.scales[u])


def oracle_forward(O, shape, L, x, idx, p):
    if shape.form_p:
        return O.deamoe_layer_p(x, idx, p, shape.g, L["dgate"], L["dup"], L["ddown"], L["agate"], L["aup"],
                                L["adown"])
    sh = None if L["sgate"] is None else (L["sgate"], L["sup"], L["sdown"])
    if shape.I_sh > 0:
        priv = (L["pgate"], L["pup"], L["pdown"]) if shape.I_pr > 0 else (None, None, None)
        return O.deamoe_layer_c(x, idx, p, shape.g, L["dgate"], L["dup"], L["ddown"], *priv, shared=sh)
    return O.vanilla_layer(x, idx, p, L["gate"], L["up"], L["down"], shared=sh)


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle timed on the host cores.  A step is one
    selected expert of one token (its SwiGLU pass, plus the token's routing
    and shared expert on its first step).  The weights of every unit the
    steps touch are generated on the host before the timed region."""
    if rank != 0:
        return
    from oracle import moe_oracle as O
    s = WORKLOADS[args.workload]
    batches = tuple(int(b) for b in args.batches.split(",")) if args.batches else s.batches
    bw = {"bf16": 2, "f32": 4, "fp8": 1}[s.dtype]
    row_b = 3 * s.d * bw + (12 if s.dtype == "fp8" else 0)    # one intermediate row: weights (+ FP8 scales)
    seed = args.seed * 1000
    router = synth.router(s.d, s.n, seed)
    bias = synth.zipf_bias(s.n, s.zipf_g, s.zipf, seed) if s.zipf > 0 else None
    ntok = -(-(args.steps + args.warmup) // s.k)
    xs = synth.hidden(ntok, s.d, seed + 7)

    def route(x):
        if s.k_dept:
            return O.route_grouped(x, router, s.k, s.g, s.k_dept, bias=bias)
        return O.route(x, router, s.k, bias=bias)

    idx_all, _, _ = route(xs)       # untimed: which units to make
    units = {}

    def unit(tid, u, rows):
        if (tid, u) not in units:
            if s.dtype == "fp8":
                w = synth.normal((rows, s.d), seed, tid, synth.WEIGHT_STD, "cpu", salt=u + 1)
                units[(tid, u)] = torch.from_numpy(O.dequant_rows_e4m3(*synth.quantize_rows_e4m3(w)))
            else:
                units[(tid, u)] = synth.normal((rows, s.d), seed, tid, synth.WEIGHT_STD, "cpu",
                                               synth.storage_dtype(s.dtype), salt=u + 1)
        return units[(tid, u)]

    def amat(tid, e):
        if (tid, e) not in units:
            units[(tid, e)] = synth.near_identity_unit(e, s.I_sh, seed, tid, s.dtype)
        return units[(tid, e)]

    def weights(e):
        if s.form_p:
            j = e // s.g
            return ([unit(t, j, s.I_sh) for t in (synth.TID_DGATE, synth.TID_DUP, synth.TID_DDOWN)] +
                    [amat(t, e) for t in (synth.TID_AGATE, synth.TID_AUP, synth.TID_ADOWN)])
        if s.I_sh > 0:
            j = e // s.g
            return [torch.cat([unit(t1, j, s.I_sh)] + ([unit(t2, e, s.I_pr)] if s.I_pr else []))
                    for t1, t2 in ((synth.TID_DGATE, synth.TID_PGATE), (synth.TID_DUP, synth.TID_PUP),
                                   (synth.TID_DDOWN, synth.TID_PDOWN))]
        return [unit(t, e, s.I) for t in (synth.TID_GATE, synth.TID_UP, synth.TID_DOWN)]

    W = {int(e): weights(int(e)) for e in set(idx_all.ravel().tolist())}
    SH = ([unit(t, 0, s.I_s) for t in (synth.TID_SGATE, synth.TID_SUP, synth.TID_SDOWN)]
          if s.I_s else None)
    state = {}

    def step(i):
        tok, q = divmod(i, s.k)
        nbytes = 0
        if q == 0:
            x = xs[tok:tok + 1]
            idx, p, _ = route(x)
            state.update(x=x, idx=idx, p=p, depts=set())
            nbytes += 4 * s.d * s.n
            if SH is not None:
                O.swiglu_expert(x[0], *SH)
                nbytes += row_b * s.I_s
        x, idx, p = state["x"], state["idx"], state["p"]
        e = int(idx[0, q])
        if s.form_p:
            p[0, q] * O.deamoe_expert_p(x[0], *W[e])
            j = e // s.g
            nbytes += 2 * (3 * s.d * s.I_sh * (j not in state["depts"]) + 3 * s.I_sh * s.I_sh)
            state["depts"].add(j)
        elif s.I_sh > 0:
            p[0, q] * O.swiglu_expert(x[0], *W[e])
            j = e // s.g
            nbytes += row_b * (s.I_pr + (s.I_sh if j not in state["depts"] else 0))
            state["depts"].add(j)
        else:
            p[0, q] * O.swiglu_expert(x[0], *W[e])
            nbytes += row_b * s.I
        return nbytes

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    total = 0
    for i in range(args.steps):
        total += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = total / dt / 1e9
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {**workload_config(s, batches),
                      "sample": "one selected expert of one token per step"},
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
