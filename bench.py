"""Benchmark of the routed-MoE NVFP4 (W4A16) prefill path on GB300 through the C ABI.

One step = one ``moe_prefill_forward`` over one prefill chunk (routing, expert sort, grouped
gate/up GEMM with the fused SwiGLU, grouped down GEMM, combine), inputs already resident in
HBM.  The headline workload is the largest single-GPU configuration: Zipf(1.2)-skewed routing
at GLM shapes (hidden 5120, moe_intermediate 1536, 160 experts, top-8), one 8192-row chunk.
L2 is flushed between timed steps by writing a 256 MiB buffer outside the timed events.

The same JSON line also carries, as extra keys, the other workloads of the path:
* ``workloads.c1`` / ``workloads.c2``: the full routed-MoE block on a 256-row chunk (hidden
  2048, 64 experts, router GEMM) and the balanced 2048-row GLM chunk, each with its own
  roofline, CPU-oracle baseline and end-to-end number;
* ``c0``: the single grouped GEMM (64 tokens, 16 experts, N 256, K 512), whose time is launch
  latency, reported as such;
* ``c4_sweep``: the row-count sweep at GLM shapes (8 ... 16384 rows) with tokens/s, TFLOP/s,
  the binding roofline fraction of each grouped GEMM, and the weight bytes read per launch
  against the once-per-expert minimum.

Prints ONE JSON line.  ``--impl reference`` times the CPU oracle instead, on a bounded sample
of the same workload.  One GPU only: the grouped GEMM's activation loads multicast within a
thread-block cluster of this GPU's memory, so ``--gpus`` > 1 is refused.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

WORKLOAD_DESC = {
    "c1": "routed-MoE block, one 256-row prefill chunk: hidden 2048, moe_intermediate 768, 64 experts, top-8, "
          "BF16 router GEMM, NVFP4 gate/up [1536,2048] and down [2048,768] per expert",
    "c2": "GLM-scale routed MoE, 2048-row prefill chunk: hidden 5120, moe_intermediate 1536, 160 experts, top-8, "
          "synthetic logits N(0,1)+bias N(0,0.1)",
    "c3": "Zipf(1.2) skewed routing at GLM shapes (hidden 5120, moe_intermediate 1536, 160 experts, top-8), "
          "8192-row prefill chunk, 16 experts never chosen",
    "c1s": "the 256-row chunk of c1 plus the shared expert (dense BF16 SwiGLU MLP, intermediate 768) on a second "
           "stream, joined in the combine",
}
C0_DESC = "single grouped W4A16 GEMM: 64 tokens x top-8 of 16 experts (512 sorted rows), N 256, K 512, gathered rows"
C4_DESC = "row-count sweep at GLM shapes (hidden 5120, moe_intermediate 1536, 160 experts, top-8), balanced routing"
HEADLINE = "c3"
METRIC = "routed-MoE prefill tokens/s/layer"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------ arithmetic


def weight_bytes_min(E_touched: int, N: int, K: int) -> int:
    """Each touched expert's packed weights, E4M3 scales and FP32 scale2, read once."""
    return E_touched * (N * K // 2 + N * K // 16 + 4)


def gemm_bytes(case, off: np.ndarray, proj: str) -> int:
    """Algorithmic bytes of one grouped GEMM launch: every touched expert's packed weights and
    scales once (+ its scale2), the unique A rows, and the output written once (the gate/up
    launch writes the SwiGLU activation [R, I] from its epilogue, not G [R, 2I])."""
    E = case.E
    touched = int((np.diff(off[:E + 1]) > 0).sum())
    R = int(off[E])
    if proj == "gate_up":
        N, K, a_bytes, c_bytes = 2 * case.I, case.H, case.T * case.H * 2, R * case.I * 2
    else:
        N, K, a_bytes, c_bytes = case.H, case.I, R * case.I * 2, R * case.H * 2
    return weight_bytes_min(touched, N, K) + a_bytes + c_bytes


def gemm_flops(case, proj: str) -> int:
    R = case.T * case.k
    return 2 * R * 2 * case.I * case.H if proj == "gate_up" else 2 * R * case.H * case.I


def roofline_entry(name: str, nbytes: int, flops: int, dur_s: float, peaks: dict, src: str, traffic) -> dict:
    """Binding roofline of one launch: HBM when bytes/peak_HBM >= flops/peak_TC, else tensor."""
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        ach = nbytes / dur_s / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": traffic, "algorithmic_bytes": int(nbytes),
                "algorithmic_flops": int(flops), "us": round(dur_s * 1e6, 2), "peak_source": src}
    ach = flops / dur_s / 1e12
    return {"kernel": name, "bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4), "traffic": traffic,
            "algorithmic_bytes": int(nbytes), "algorithmic_flops": int(flops), "us": round(dur_s * 1e6, 2),
            "peak_source": src}


def max_over_ranks(x: float, device) -> float:
    """The slowest rank's time: every replica's timed region ends when the slowest one does."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(n_ranks: int, rows_per_step: int, steps: int, max_ms: float) -> float:
    """Whole-job tokens/s of N independent replicas (weak scaling): every rank processes its own
    chunk of `rows_per_step` rows per step; the job takes the slowest rank's time."""
    return n_ranks * rows_per_step * steps / (max_ms / 1e3)


GEMM_SOURCES = ("grouped_gemm.cu", "pair_gemm.cu", "common.cuh", "internal.h")


def gemm_sources_digest() -> str:
    """SHA-256 of the grouped GEMM's sources (concatenated in GEMM_SOURCES order) with C/C++
    comments removed and whitespace runs collapsed: an edit of a comment keeps the counters valid,
    any change of code does not."""
    import hashlib
    import re

    csrc = os.path.join(ROOT, "moe_prefill_nvfp4_gb300", "csrc")
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        # string literals of these files hold inline PTX, whose "//" never starts a comment there;
        # keep literals, drop comments
        tok = re.compile(r'"(?:\\.|[^"\\])*"|//[^\n]*|/\*.*?\*/', re.S)
        text = tok.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def measured_traffic(workload: str, launch: str, kind: str = "total"):
    """DRAM bytes per launch from the committed ncu summary (read + write for ``total``, read
    only for ``read``), or None when the kernel's sources changed since those counters were
    taken or the workload was not captured."""
    digest = gemm_sources_digest()
    path = os.path.join(ROOT, "profiles", "grouped_gemm_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            p = line.split()
            if len(p) == 5 and not line.startswith("#") and p[0] == workload and p[1] == launch and p[2] == digest:
                return int(p[3]) + (int(p[4]) if kind == "total" else 0)
    return None


# ---------------------------------------------------------------------------------------------- GPU


class GpuBench:
    """Device state shared by the workloads of one run: the flush buffer, peaks, the stream."""

    def __init__(self, args, dev):
        import torch

        self.torch = torch
        self.args = args
        self.dev = dev
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        self.peaks, self.peak_src = _peaks()

    def timed(self, run, n):
        """n runs, each bracketed by CUDA events on the launching stream, L2 flushed before each
        (outside the events)."""
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            self.flush.fill_(1)
            evs[i][0].record(self.stream)
            run()
            evs[i][1].record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def capture(self, fn):
        torch = self.torch
        cap = torch.cuda.Stream(self.dev)
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(self.stream)
        with torch.cuda.graph(g, stream=cap):
            fn(cap)
        torch.cuda.synchronize()
        return g

    # -------------------------------------------------------------------------- a routed block

    def block(self, name: str, case, steps: int, warmup: int, e2e: bool = True, clocks=None, tag=None) -> dict:
        """Time one routed-MoE block workload: graph replays of the forward (value), the stage
        graph (per-stage times and the GEMM rooflines), the end-to-end graph on pinned host
        buffers, and eager launches."""
        import moe_prefill_nvfp4_gb300 as moe
        from moe_prefill_nvfp4_gb300.weights import upload_projection

        torch = self.torch
        dev = self.dev
        T, H, I, E, k = case.T, case.H, case.I, case.E, case.k
        x = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).to(dev)
        wr = (torch.from_numpy(case.router_w.view(np.int16)).view(torch.bfloat16).to(dev)
              if case.router_w is not None else None)
        logits = torch.from_numpy(case.logits).to(dev) if case.logits is not None else None
        gu = getattr(case, "_dev_gu", None) or upload_projection(case.gate_up.packed, case.gate_up.scales,
                                                                 case.gate_up.scale2, 2 * I, H, device=str(dev))
        dn = getattr(case, "_dev_dn", None) or upload_projection(case.down.packed, case.down.scales, case.down.scale2,
                                                                 H, I, device=str(dev))
        cfg = moe.MoePrefillConfig(hidden=H, moe_intermediate=I, num_experts=E, top_k=k, swiglu_limit=7.0,
                                   renormalize=1, routed_scale=1.0)
        lay = moe.moe_workspace_layout(cfg, T)
        ws = torch.empty(lay.total, dtype=torch.uint8, device=dev)
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        NEV = moe.MOE_FWD_NUM_EVENTS
        sh = None
        if case.shared is not None:  # shared expert on a second stream, joined before the combine
            bits = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
            sh = dict(gate=bits(case.shared.gate), up=bits(case.shared.up), down=bits(case.shared.down),
                      out=torch.empty(T, H, dtype=torch.bfloat16, device=dev),
                      ws=torch.empty(moe.moe_shared_expert_workspace_bytes(T, H, case.shared.I), dtype=torch.uint8,
                                     device=dev),
                      side=torch.cuda.Stream(dev), fork=torch.cuda.Event(), ready=torch.cuda.Event())

        def step(events=None, st=None, dst=None, src=None, lg=None):
            st = st if st is not None else self.stream
            dst = dst if dst is not None else out
            src = src if src is not None else x
            lg = lg if lg is not None else logits
            ready = None
            if sh is not None:
                sh["fork"].record(st)
                sh["side"].wait_event(sh["fork"])
                moe.moe_shared_expert_forward(x, sh["gate"], sh["up"], sh["down"], 7.0, ws=sh["ws"], out=sh["out"],
                                              stream=sh["side"])
                sh["ready"].record(sh["side"])
                ready = sh["ready"]
            moe.moe_prefill_forward(cfg, src, gu.table, dn.table, ws, w_router=wr, logits=lg, out=dst,
                                    stage_events=events, stream=st, shared_out=sh["out"] if sh else None,
                                    shared_ready=ready)
            if sh is not None:
                st.wait_stream(sh["side"])

        for _ in range(warmup):
            self.flush.fill_(1)
            step()
        torch.cuda.synchronize()
        if moe.moe_get_device_error() != 0:
            raise RuntimeError(f"{name}: device error during warm-up")

        # The forward makes no host round trip, so one chunk's whole forward is captured once into
        # a CUDA graph and replayed per step (the launch-bound host work is paid once, as a serving
        # loop with fixed chunk shapes does).  A second graph carries the per-stage events.
        stage_ev = [torch.cuda.Event(enable_timing=True) for _ in range(NEV)]
        for e in stage_ev:  # torch creates the CUDA event on first record; the library records it afterwards
            e.record(self.stream)
        torch.cuda.synchronize()
        g_step = self.capture(lambda st: step(None, st))
        g_stage = self.capture(lambda st: step(stage_ev, st))
        graphs = [g_step, g_stage]
        if e2e:
            x_host = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).pin_memory()
            lg_host = torch.from_numpy(case.logits).pin_memory() if case.logits is not None else None
            out_host = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()

            def e2e_body(st):
                # The step's inputs and result live in pinned host memory, which the device reaches
                # over the coherent CPU-GPU link: the forward stages x into its workspace as the router
                # reads it (without a router, with one copy), the top-k reads host logits in place and
                # the combine stores out into the host buffer.  With a shared expert (which reads x
                # from device memory) x is copied to the device first.
                if sh is not None:
                    x.copy_(x_host, non_blocking=True)
                    step(None, st, dst=out_host, lg=lg_host)
                else:
                    step(None, st, dst=out_host, src=x_host, lg=lg_host)

            g_e2e = self.capture(e2e_body)
            graphs.append(g_e2e)
        for g in graphs:
            for _ in range(3):
                self.flush.fill_(1)
                g.replay()
        torch.cuda.synchronize()

        if clocks is not None:
            clocks.start()
            time.sleep(0.3)
        t_wall0 = time.perf_counter()
        step_ms = self.timed(g_step.replay, steps)
        t_wall = time.perf_counter() - t_wall0
        # per-stage times: the same graph with the stage events, one step at a time
        stage_rows = []
        for _ in range(steps):
            self.flush.fill_(1)
            g_stage.replay()
            torch.cuda.synchronize()
            stage_rows.append([stage_ev[j].elapsed_time(stage_ev[j + 1]) for j in range(NEV - 1)])
        stage_ms = np.array(stage_rows)
        e2e_list = self.timed(g_e2e.replay, steps) if e2e else None
        eager_list = self.timed(step, steps)
        clk = clocks.stop() if clocks is not None else None
        if moe.moe_get_device_error() != 0:
            raise RuntimeError(f"{name}: device error during timed steps")
        total_ms = max_over_ranks(float(sum(step_ms)), dev)
        eager_ms = max_over_ranks(float(sum(eager_list)), dev)

        off = ws[lay.expert_offsets:lay.expert_offsets + 4 * (E + 1)].view(torch.int32).cpu().numpy()
        # stage intervals between the forward's 8 events; with a router (E <= 64) the router GEMM and
        # the top-k are one launch ("route_topk" is then an empty interval), and with the fused SwiGLU
        # the "swiglu" interval is empty (each interval carries the event node's own ~2 us)
        names = ["router_logits", "route_topk", "sort", "grouped_gemm_gate_up", "swiglu", "grouped_gemm_down",
                 "combine"]
        mean_stage = stage_ms.mean(axis=0)
        gemms = {}
        for proj, idx in (("gate_up", 3), ("down", 5)):
            gemms[proj] = roofline_entry(f"grouped_gemm_{proj}", gemm_bytes(case, off, proj), gemm_flops(case, proj),
                                         mean_stage[idx] / 1e3, self.peaks, self.peak_src,
                                         measured_traffic(tag or name, proj))
        dom = "gate_up" if mean_stage[3] >= mean_stage[5] else "down"
        R = T * k
        launches = (((2 if E > 64 else 1) if wr is not None else 1) + (1 if R <= 2048 else 2) + 3
                    + (3 if sh is not None else 0))
        res = {
            "workload": WORKLOAD_DESC.get(name, name), "rows": T, "hidden": H, "moe_intermediate": I, "experts": E,
            "top_k": k, "experts_touched": int((np.diff(off[:E + 1]) > 0).sum()),
            "max_rows_per_expert": int(np.diff(off[:E + 1]).max()),
            "value": round(replica_throughput(1, T, steps, total_ms), 1), "unit": "tokens/s",
            "ms_per_step": round(total_ms / steps, 5),
            "routed_tflops": round((gemm_flops(case, "gate_up") + gemm_flops(case, "down")) / (total_ms / steps / 1e3)
                                   / 1e12, 1),
            "eager": {"value": round(replica_throughput(1, T, steps, eager_ms), 1), "unit": "tokens/s",
                      "ms_per_step": round(eager_ms / steps, 5),
                      "how": "moe_prefill_forward launched from the host every step (no graph)"},
            "roofline": gemms[dom],
            "gemm_roofline": gemms,
            "stage_ms": {n: round(float(v), 5) for n, v in zip(names, mean_stage)},
            # routing (router GEMM + top-k as one launch for E <= 64, else two; top-k alone on given
            # logits), sort (one launch up to 2048 slots, else two), gate/up GEMM with the fused
            # SwiGLU (the CTA-pair kernel also stores its token rows in expert order), down GEMM,
            # combine (+ the shared expert's gate/up GEMM, SwiGLU and down GEMM)
            "gpu_launches_per_step": launches,
            "wall_s_timed": round(t_wall, 4),
        }
        if e2e:
            e2e_ms = max_over_ranks(float(sum(e2e_list)), dev)
            res["e2e"] = {"value": round(replica_throughput(1, T, steps, e2e_ms), 1), "unit": "tokens/s",
                          "h2d_bytes_per_step": x_host.numel() * 2 + (lg_host.numel() * 4 if lg_host is not None else 0),
                          "d2h_bytes_per_step": out_host.numel() * 2,
                          "how": "CUDA graph of moe_prefill_forward on pinned host x/logits/out (x staged to the "
                                 "device by the router kernel or one copy, logits read in place, out stored by the "
                                 "combine), replayed per step"}
        if clk is not None:
            res["clocks"] = clk
        del ws, out
        if getattr(case, "_dev_gu", None) is None:
            gu.close()
            dn.close()
        return res

    # --------------------------------------------------------------------- the single GEMM (c0)

    def single_gemm(self, steps: int) -> dict:
        """c0: one grouped W4A16 GEMM launch over 512 gathered rows.  Its algorithmic time is far
        below a launch (0.15 us of HBM at the measured peak), so the number is launch latency:
        a graph of one launch replayed per step (L2 flushed), and a graph of 20 back-to-back
        launches (L2 warm after the first) for the per-launch cost in a stream."""
        import moe_prefill_nvfp4_gb300 as moe
        from moe_prefill_nvfp4_gb300.weights import upload_projection
        from synth import inputs as S

        torch = self.torch
        c = S.workload("c0")
        dev = self.dev
        A = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).to(dev)
        ids = torch.from_numpy(c.ids).to(dev)
        w = upload_projection(c.w.packed, c.w.scales, c.w.scale2, c.N, c.K, device=str(dev))
        srt = moe.moe_sort_by_expert(ids, c.E)
        R = c.T * c.k
        C = torch.empty(R, c.N, dtype=torch.bfloat16, device=dev)

        def one(st):
            moe.moe_w4a16_grouped_gemm(A, w.table, srt["expert_offsets"], R, gather_ids=srt["sorted_token_ids"],
                                       out=C, stream=st)

        for _ in range(5):
            one(self.stream)
        torch.cuda.synchronize()
        g1 = self.capture(one)
        nb = 20
        g20 = self.capture(lambda st: [one(st) for _ in range(nb)])
        for g in (g1, g20):
            g.replay()
        torch.cuda.synchronize()
        cold = self.timed(g1.replay, steps)
        burst = self.timed(g20.replay, max(3, steps // 4))
        if moe.moe_get_device_error() != 0:
            raise RuntimeError("c0: device error")
        off = srt["expert_offsets"].cpu().numpy()
        touched = int((np.diff(off) > 0).sum())
        nbytes = weight_bytes_min(touched, c.N, c.K) + c.T * c.K * 2 + R * c.N * 2
        flops = 2 * R * c.N * c.K
        us_cold = float(np.mean(cold)) * 1e3
        us_burst = float(np.mean(burst)) * 1e3 / nb
        w.close()
        return {"workload": C0_DESC, "rows": c.T, "sorted_rows": R, "experts": c.E, "top_k": c.k, "N": c.N, "K": c.K,
                "bound": "latency", "us_per_launch_cold": round(us_cold, 2),
                "us_per_launch_back_to_back": round(us_burst, 2),
                "tflops_back_to_back": round(flops / (us_burst * 1e-6) / 1e12, 3),
                "gbs_back_to_back": round(nbytes / (us_burst * 1e-6) / 1e9, 1),
                "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                "roofline_us": round(max(nbytes / (self.peaks["hbm_gbs"] * 1e9),
                                         flops / (self.peaks["bf16_tflops"] * 1e12)) * 1e6, 3),
                "note": "the roofline time is far below one launch: the launch latency binds, 70% of roofline "
                        "is unreachable at this size",
                "how": "CUDA events around a graph of one launch (L2 flushed before each) and around a graph of "
                       f"{nb} back-to-back launches"}

    # --------------------------------------------------------------------------- the sweep (c4)

    def sweep(self, rows, steps: int, warmup: int) -> list:
        """c4: the forward at each row count, one set of GLM-shape expert weights (seed of the
        sweep) on the device for every point."""
        from moe_prefill_nvfp4_gb300.weights import upload_projection
        from synth import inputs as S

        base = S.workload("c4", T=8)
        H, I = base.H, base.I
        gu = upload_projection(base.gate_up.packed, base.gate_up.scales, base.gate_up.scale2, 2 * I, H,
                               device=str(self.dev))
        dn = upload_projection(base.down.packed, base.down.scales, base.down.scale2, H, I, device=str(self.dev))
        out = []
        for T in rows:
            c = S.make_block_case(T=T, H=H, I=I, E=base.E, k=base.k, routing="biased", seed=S.WORKLOADS["c4"]["seed"],
                                  with_weights=False)
            c.gate_up, c.down = base.gate_up, base.down
            c._dev_gu, c._dev_dn = gu, dn
            r = self.block(f"c4 T={T}", c, steps, warmup, e2e=False, tag=f"c4_{T}")
            entry = {"rows": T, "value": r["value"], "unit": "tokens/s", "ms_per_step": r["ms_per_step"],
                     "routed_tflops": r["routed_tflops"], "experts_touched": r["experts_touched"],
                     "stage_ms": {k2: r["stage_ms"][k2] for k2 in ("grouped_gemm_gate_up", "grouped_gemm_down")}}
            for proj in ("gate_up", "down"):
                g = r["gemm_roofline"][proj]
                N, K = (2 * I, H) if proj == "gate_up" else (H, I)
                bmin = weight_bytes_min(r["experts_touched"], N, K)
                read = measured_traffic(f"c4_{T}", proj, kind="read")
                entry[proj] = {"bound": g["bound"], "frac": g["frac"], "achieved": g["achieved"], "unit": g["unit"],
                               "us": g["us"], "weight_bytes_min": bmin,
                               "weight_bytes_read": read if read is not None else bmin,
                               "weight_bytes_read_source": ("ncu dram__bytes_read.sum (all bytes of the launch)"
                                                            if read is not None else
                                                            "algorithmic: each touched expert once (no capture of "
                                                            "the current kernel at this row count)")}
            out.append(entry)
        gu.close()
        dn.close()
        return out


def run_gemm_only(args):
    """Profiling driver: the two grouped GEMMs alone (gate/up with the fused SwiGLU, then down),
    `args.gemm_only` times, on a small Zipf case at GLM widths (40 experts, 4096 rows, top-8:
    every expert takes the wide 384-token tiles; 0.5 GB of weights), sized for an ncu capture.  The token
    rows are put into expert order with torch indexing (in the forward the CTA-pair gate/up launch
    stores them itself)."""
    import torch

    import moe_prefill_nvfp4_gb300 as moe
    from moe_prefill_nvfp4_gb300.weights import upload_projection
    from synth import inputs as S

    torch.cuda.set_device(0)
    case = S.make_block_case(T=4096, H=5120, I=1536, E=40, k=8, routing="zipf", seed=1003)
    T, H, I, E, k = case.T, case.H, case.I, case.E, case.k
    x = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).cuda()
    ids, _ = moe.moe_route_topk(torch.from_numpy(case.logits).cuda(), k)
    srt = moe.moe_sort_by_expert(ids, E)
    gu = upload_projection(case.gate_up.packed, case.gate_up.scales, case.gate_up.scale2, 2 * I, H, device="cuda")
    dn = upload_projection(case.down.packed, case.down.scales, case.down.scale2, H, I, device="cuda")
    R = T * k
    xs = x[srt["sorted_token_ids"].long()].contiguous()
    act = torch.empty(R, I, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(R, H, dtype=torch.bfloat16, device="cuda")
    for _ in range(args.gemm_only):
        moe.moe_w4a16_grouped_gemm_swiglu(xs, gu.table, srt["expert_offsets"], R, limit=7.0, out=act)
        moe.moe_w4a16_grouped_gemm(act, dn.table, srt["expert_offsets"], R, out=Y)
    torch.cuda.synchronize()
    err = moe.moe_get_device_error()
    counts = np.diff(srt["expert_offsets"].cpu().numpy())
    print(json.dumps({"gemm_only": args.gemm_only, "rows_per_expert_max": int(counts.max()),
                      "rows_per_expert_mean": R / E, "device_error": err}), flush=True)
    gu.close()
    dn.close()
    if err:
        sys.exit(1)


def run_gpu(args):
    import torch

    import moe_prefill_nvfp4_gb300 as moe  # noqa: F401  (loads the library)
    from synth import inputs as S

    ws_n, rank, local = _dist()
    if ws_n > 1 or args.gpus > 1:
        print("bench.py runs on one GPU: the grouped GEMM multicasts activation rows within a thread-block "
              "cluster, which stays in single-GPU runs", file=sys.stderr)
        sys.exit(2)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gb = GpuBench(args, dev)
    if args.sweep_only:  # profiling driver: the c4 forward at the given row counts, nothing else
        rows = S.SWEEP_ROWS if args.sweep_rows is None else tuple(int(v) for v in args.sweep_rows.split(","))
        print(json.dumps({"c4_sweep": {"workload": C4_DESC, "points": gb.sweep(rows, args.steps, args.warmup)}}),
              flush=True)
        return
    clocks = ClockSampler(local)
    head = gb.block(args.workload, S.workload(args.workload), args.steps, args.warmup, clocks=clocks)
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(S.workload(args.workload), args.cpu_budget_s)
    reports = [r for r in args.reports.split(",") if r and r != "none"]
    extra = {}
    c0 = None
    sweep = None
    for r in reports:
        if r in ("c1", "c2", "c1s"):
            case = S.workload(r)
            extra[r] = gb.block(r, case, args.steps, args.warmup)
            if not args.no_cpu_baseline:
                extra[r]["cpu_baseline"] = cpu_baseline(case, args.cpu_budget_s)
        elif r == "c0":
            c0 = gb.single_gemm(args.steps)
        elif r == "c4":
            rows = S.SWEEP_ROWS if args.sweep_rows is None else tuple(int(v) for v in args.sweep_rows.split(","))
            sweep = gb.sweep(rows, max(3, args.steps // 2), 3)
    res = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (NVFP4 weights dequantised to BF16, FP32 accumulate)",
        "data": "synthetic (seeded; random NVFP4 weights, no trained checkpoint)",
        "config": {"workload": head["workload"], "rows": head["rows"], "hidden": head["hidden"],
                   "moe_intermediate": head["moe_intermediate"], "experts": head["experts"], "top_k": head["top_k"],
                   "l2": "flushed between timed steps (256 MiB write outside the step events)"},
        "e2e": head["e2e"],
        "eager": head["eager"],
        "timing": "CUDA events around each graph replay of the forward; stage_ms from a second graph with "
                  "stage events, replayed one step at a time",
        "roofline": head["roofline"],
        "gemm_roofline": head["gemm_roofline"],
        "stage_ms": head["stage_ms"],
        "routed_tflops": head["routed_tflops"],
        "experts_touched": head["experts_touched"],
        "max_rows_per_expert": head["max_rows_per_expert"],
        "gpu_launches": head["gpu_launches_per_step"] * args.steps,
        "clocks": head.get("clocks"),
        "wall_s_timed": head["wall_s_timed"],
    }
    if cpu is not None:
        res["cpu_baseline"] = cpu
    if extra:
        res["workloads"] = extra
    if c0 is not None:
        res["c0"] = c0
    if sweep is not None:
        res["c4_sweep"] = {"workload": C4_DESC, "points": sweep}
    print(json.dumps(res), flush=True)


# ---------------------------------------------------------------------------------------------- CPU


def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample_rows(case) -> int:
    """Rows of one bounded oracle sample: the whole chunk for the 256-row block, one row at GLM
    shapes (where the oracle's per-expert dequantisation of the 8 touched experts alone takes
    seconds)."""
    return case.T if case.H * case.I <= 2048 * 768 else 1


def _head_rows(case, n: int):
    """The first n rows of a block workload (same weights)."""
    import copy

    c = copy.copy(case)
    c.T = n
    c.x = case.x[:n]
    if case.logits is not None:
        c.logits = case.logits[:n]
    return c


def cpu_baseline(case, budget_s: float = 20.0) -> dict:
    """The oracle (BF16 variant) as it stands, on the host cores: samples of the workload's first
    rows while the budget lasts (at least one).  Returns tokens/s of the oracle."""
    from oracle import moe_oracle as O

    n_rows = oracle_sample_rows(case)
    sub = _head_rows(case, n_rows)
    t0 = time.perf_counter()
    n = 0
    while True:
        O.prefill_forward(sub, "bf16")
        n += 1
        if time.perf_counter() - t0 > budget_s / 2 or n >= 3:
            break
    dt = time.perf_counter() - t0
    what = f"{n} full {case.T}-row chunk(s)" if n_rows == case.T else \
        f"{n} sample(s) of the chunk's first {n_rows} row(s) (each its own oracle call, dequantising its experts)"
    return {"value": round(n * n_rows / dt, 3), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{what} of the same workload through the fp64 numpy oracle (BF16 variant), {dt:.1f} s; "
                      f"numpy elementwise single-threaded, BLAS matmuls on the cores listed"}


def run_reference(args):
    ws_n, rank, _ = _dist()
    if rank != 0:
        return
    from synth import inputs as S

    case = S.workload(args.workload)
    from oracle import moe_oracle as O

    n_rows = oracle_sample_rows(case)
    sub = _head_rows(case, n_rows)
    # The oracle holds no warm state: one untimed sample warms imports and page faults; the
    # remaining warm-up steps would only repeat it.
    if args.warmup > 0:
        O.prefill_forward(sub, "bf16")
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.prefill_forward(sub, "bf16")
    dt = time.perf_counter() - t0
    value = n_rows * args.steps / dt
    what = f"{args.steps} full {case.T}-row chunk(s), one per step" if n_rows == case.T else \
        f"{args.steps} samples of the chunk's first {n_rows} row(s), one per step"
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": ws_n,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded)",
           "config": {"workload": WORKLOAD_DESC[args.workload], "rows": case.T, "hidden": case.H,
                      "moe_intermediate": case.I, "experts": case.E, "top_k": case.k},
           "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
                            "sample": what},
           "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOAD_DESC))
    ap.add_argument("--reports", default="c1,c2,c1s,c0,c4",
                    help="extra workloads in the same line: any of c0,c1,c2,c1s,c4 (comma-separated) or none")
    ap.add_argument("--sweep-rows", default=None, help="row counts of the c4 sweep (default: all eleven)")
    ap.add_argument("--sweep-only", action="store_true",
                    help="profiling driver: run only the c4 sweep (at --sweep-rows) and print its points")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gemm-only", type=int, default=0,
                    help="profiling driver: run the two grouped GEMMs this many times on a small Zipf case and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gemm_only:
        run_gemm_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
