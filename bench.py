"""Benchmark of the routed-MoE NVFP4 (W4A16) prefill path on GB300 through the C ABI.

One step = one ``moe_prefill_forward`` over one prefill chunk (router GEMM, top-k, expert
sort, grouped gate/up GEMM, SwiGLU, grouped down GEMM, combine), inputs already resident in
HBM.  Default workload: the full routed-MoE block on one 256-row chunk (hidden 2048,
moe_intermediate 768, 64 experts, top-8, BF16 router [64, 2048]).  L2 is flushed between
timed steps by writing a 256 MiB buffer outside the timed events.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead, on a
bounded sample of the same workload.  Multi-GPU (torchrun): independent replicas, one chunk
per rank per step ("replicas only": the path has no exchange step on one node of this design).
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
    "c3": "Zipf(1.2) skewed routing at GLM shapes, 8192 rows, 16 experts never chosen",
    "c1s": "the 256-row chunk of c1 plus the shared expert (dense BF16 SwiGLU MLP, intermediate 768, cuBLAS "
           "GEMMs) on a second stream, joined in the combine",
}
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


# ---------------------------------------------------------------------------------------------- GPU


def build_case(name: str):
    from synth import inputs as S

    return S.workload(name)


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
    w = touched * (N * K // 2 + N * K // 16 + 4)
    return w + a_bytes + c_bytes


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


GEMM_SOURCES = ("grouped_gemm.cu", "common.cuh", "internal.h")


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


def measured_traffic(workload: str, launch: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary, or None when the
    kernel's sources changed since those counters were taken (or the workload was not captured)."""
    digest = gemm_sources_digest()
    path = os.path.join(ROOT, "profiles", "grouped_gemm_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            p = line.split()
            if len(p) == 5 and not line.startswith("#") and p[0] == workload and p[1] == launch and p[2] == digest:
                return int(p[3]) + int(p[4])
    return None


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import moe_prefill_nvfp4_gb300 as moe
    from moe_prefill_nvfp4_gb300.weights import upload_projection

    ws_n, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws_n > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    case = build_case(args.workload)
    T, H, I, E, k = case.T, case.H, case.I, case.E, case.k
    x = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).to(dev)
    wr = torch.from_numpy(case.router_w.view(np.int16)).view(torch.bfloat16).to(dev) if case.router_w is not None else None
    logits = torch.from_numpy(case.logits).to(dev) if case.logits is not None else None
    gu = upload_projection(case.gate_up.packed, case.gate_up.scales, case.gate_up.scale2, 2 * I, H, device=str(dev))
    dn = upload_projection(case.down.packed, case.down.scales, case.down.scale2, H, I, device=str(dev))
    cfg = moe.MoePrefillConfig(hidden=H, moe_intermediate=I, num_experts=E, top_k=k, swiglu_limit=7.0,
                               renormalize=1, routed_scale=1.0)
    lay = moe.moe_workspace_layout(cfg, T)
    ws = torch.empty(lay.total, dtype=torch.uint8, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
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
        st = st if st is not None else stream
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

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if moe.moe_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    # The forward makes no host round trip, so one chunk's whole forward is captured once into a
    # CUDA graph and replayed per step (the launch-bound host work is paid once, as a serving
    # loop with fixed chunk shapes does).  A second graph carries the per-stage events.
    x_host = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    lg_host = torch.from_numpy(case.logits).pin_memory() if case.logits is not None else None
    out_host = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    stage_ev = [torch.cuda.Event(enable_timing=True) for _ in range(NEV)]
    for e in stage_ev:  # torch creates the CUDA event on first record; the library records it afterwards
        e.record(stream)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            fn(cap)
        torch.cuda.synchronize()
        return g

    def e2e_body(st):
        # The step's inputs and result live in pinned host memory, which the device reaches over
        # the coherent CPU-GPU link: the forward stages x into its workspace as the router reads
        # it (without a router, with one copy), the top-k reads host logits in place and the
        # combine stores out into the host buffer.  With a shared expert (which reads x from
        # device memory) x is copied to the device first.
        if sh is not None:
            x.copy_(x_host, non_blocking=True)
            step(None, st, dst=out_host, lg=lg_host)
        else:
            step(None, st, dst=out_host, src=x_host, lg=lg_host)

    g_step = capture(lambda st: step(None, st))
    g_stage = capture(lambda st: step(stage_ev, st))
    g_e2e = capture(e2e_body)
    for g in (g_step, g_stage, g_e2e):
        for _ in range(3):
            flush.fill_(1)
            g.replay()
    torch.cuda.synchronize()

    def timed(run, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            flush.fill_(1)  # L2 flush, outside the step's events
            evs[i][0].record(stream)
            run()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    clocks = ClockSampler(local)
    if ws_n > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_wall0 = time.perf_counter()
    step_ms = timed(g_step.replay, args.steps)
    t_wall = time.perf_counter() - t_wall0
    # per-stage times: the same graph with the stage events, one step at a time
    stage_rows = []
    for _ in range(args.steps):
        flush.fill_(1)
        g_stage.replay()
        torch.cuda.synchronize()
        stage_rows.append([stage_ev[j].elapsed_time(stage_ev[j + 1]) for j in range(NEV - 1)])
    stage_ms = np.array(stage_rows)
    # end to end: pinned host x (and logits) -> device, forward, out -> pinned host, every step
    e2e_list = timed(g_e2e.replay, args.steps)
    # the same forward launched eagerly from the host every step (no graph)
    eager_list = timed(step, args.steps)
    clk = clocks.stop()
    if moe.moe_get_device_error() != 0:
        raise RuntimeError("device error during timed steps")
    total_ms = max_over_ranks(float(sum(step_ms)), dev)
    value = replica_throughput(ws_n, T, args.steps, total_ms)
    e2e_ms = max_over_ranks(float(sum(e2e_list)), dev)
    eager_ms = max_over_ranks(float(sum(eager_list)), dev)
    h2d = x_host.numel() * 2 + (lg_host.numel() * 4 if lg_host is not None else 0)
    d2h = out_host.numel() * 2

    # ---- roofline of the dominant kernel (largest mean stage time)
    off = ws[lay.expert_offsets:lay.expert_offsets + 4 * (E + 1)].view(torch.int32).cpu().numpy()
    # stage intervals between the forward's 8 events; with a router (E <= 64) the router GEMM and the top-k
    # are one launch ("route_topk" is then an empty interval), and with the fused SwiGLU the
    # "swiglu" interval is empty (each interval carries the event node's own ~2 us)
    names = ["router_logits", "route_topk", "sort", "grouped_gemm_gate_up", "swiglu", "grouped_gemm_down", "combine"]
    mean_stage = stage_ms.mean(axis=0)
    dom = int(np.argmax(mean_stage))
    peaks, src = _peaks()
    R = T * k
    flops = {"grouped_gemm_gate_up": 2 * R * 2 * I * H, "grouped_gemm_down": 2 * R * H * I}
    bytes_ = {"grouped_gemm_gate_up": gemm_bytes(case, off, "gate_up"), "grouped_gemm_down": gemm_bytes(case, off, "down")}
    dname = names[dom]
    dur_s = mean_stage[dom] / 1e3
    roof = None
    traffic = measured_traffic(args.workload, dname.replace("grouped_gemm_", "")) if dname in bytes_ else None
    if dname in bytes_:
        t_hbm = bytes_[dname] / (peaks["hbm_gbs"] * 1e9)
        t_tc = flops[dname] / (peaks["bf16_tflops"] * 1e12)
        if t_hbm >= t_tc:
            ach = bytes_[dname] / dur_s / 1e9
            roof = {"kernel": dname, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": traffic,
                    "algorithmic_bytes": bytes_[dname], "peak_source": src}
        else:
            ach = flops[dname] / dur_s / 1e12
            roof = {"kernel": dname, "bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4), "traffic": traffic,
                    "algorithmic_flops": flops[dname], "peak_source": src}
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (NVFP4 weights dequantised to BF16, FP32 accumulate)",
        "data": "synthetic (seeded; random NVFP4 weights, no trained checkpoint)",
        "config": {"workload": WORKLOAD_DESC[args.workload], "rows": T, "hidden": H, "moe_intermediate": I,
                   "experts": E, "top_k": k, "parallelism": f"replicas x{ws_n}",
                   "l2": "flushed between timed steps (256 MiB write outside the step events)"},
        "e2e": {"value": round(replica_throughput(ws_n, T, args.steps, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "CUDA graph of moe_prefill_forward on pinned host x/logits/out (x staged to the device "
                       "by the router kernel or one copy, logits read in place, out stored by the combine), "
                       "replayed per step"},
        "eager": {"value": round(replica_throughput(ws_n, T, args.steps, eager_ms), 1), "unit": "tokens/s",
                  "ms_per_step": round(eager_ms / args.steps, 5),
                  "how": "moe_prefill_forward launched from the host every step (no graph)"},
        "timing": "CUDA events around each graph replay of the forward; stage_ms from a second graph with "
                  "stage events, replayed one step at a time",
        "roofline": roof,
        "stage_ms": {n: round(float(v), 5) for n, v in zip(names, mean_stage)},
        # routing (router GEMM + top-k as one launch for E <= 64, else two; top-k alone on given
        # logits), sort (one launch up to 2048 slots, else two), gate/up GEMM with the fused
        # SwiGLU, down GEMM, combine (+ the shared expert's SwiGLU; its GEMMs are cuBLAS kernels)
        "gpu_launches": (((2 if E > 64 else 1) if wr is not None else 1) + (1 if T * k <= 2048 else 2) + 3
                         + (1 if sh is not None else 0)) * args.steps,
        "clocks": clk,
        "wall_s_timed": round(t_wall, 4),
    }
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(case, args.cpu_budget_s)
    gu.close()
    dn.close()
    if ws_n > 1:
        dist.destroy_process_group()
    if rank == 0:
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


def cpu_baseline(case, budget_s: float = 20.0) -> dict:
    """The oracle (BF16 variant) as it stands, on the host cores: whole chunks while the budget
    lasts (at least one).  Returns tokens/s of the oracle."""
    from oracle import moe_oracle as O

    t0 = time.perf_counter()
    n = 0
    while True:
        O.prefill_forward(case, "bf16")
        n += 1
        if time.perf_counter() - t0 > budget_s / 2 or n >= 3:
            break
    dt = time.perf_counter() - t0
    return {"value": round(n * case.T / dt, 2), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{n} full {case.T}-row chunk(s) of the same workload through the fp64 numpy oracle "
                      f"(BF16 variant), {dt:.1f} s; numpy elementwise single-threaded, BLAS matmuls on the cores listed"}


def run_reference(args):
    ws_n, rank, _ = _dist()
    if rank != 0:
        return
    case = build_case(args.workload)
    from oracle import moe_oracle as O

    # The oracle holds no warm state: one untimed chunk warms imports and page faults; the
    # remaining warm-up steps would only repeat it.
    if args.warmup > 0:
        O.prefill_forward(case, "bf16")
    t0 = time.perf_counter()

    for _ in range(args.steps):
        O.prefill_forward(case, "bf16")
    dt = time.perf_counter() - t0
    value = case.T * args.steps / dt
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws_n,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded)",
           "config": {"workload": WORKLOAD_DESC[args.workload], "rows": case.T, "hidden": case.H,
                      "moe_intermediate": case.I, "experts": case.E, "top_k": case.k},
           "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
                            "sample": f"{args.steps} full {case.T}-row chunk(s), one per step"},
           "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c1", choices=sorted(WORKLOAD_DESC))
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
