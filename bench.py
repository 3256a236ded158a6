"""Throughput of the GB300 routed int4-g128 MoE layer (one JSON line on stdout).

Default workload: the decode MoE layer — hidden 4096, expert inter 1536, 288 routed experts
top-8 + 1 shared expert, int4 g128 experts quantized on the device, bf16 activations, Zipf(1.1)
router bias — at a batch of 16 tokens (the largest batch of its sweep; the other batches are
reported under "sweep"). A step is one strata_moe_forward: router + softmax + top-k, grouping,
gate/up grouped GEMM with SiLU, down grouped GEMM, weighted combine.

Cold L2: every step uses another of 8 copies of the layer's quantized experts (identical
values, distinct addresses: 8 x 2.8 GB, far above the 129 MB L2) and another of 8 token
batches, so no step finds its weights in L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl strata|reference] [--batch T]

The default single-GPU run also reports, each under its own key with its own roofline:
"padded_graph" (one CUDA graph captured at 16 tokens replayed with 1/5/16 live tokens),
"prefill_c5" (on-device quantization GB/s and the 4096-token tensor-core layer's TFLOP/s against
the burst bf16 peak), "prefill_c3" (the 512-token layer against its HBM roof) and "stack_c4" (the
8-layer decode stack at 1..32 tokens). Their experts are drawn N(0, 0.02) on the device (the same
distribution as the host generator) and quantized there; --no-extras skips them.

Under torchrun (N > 1) each rank runs its own replica of the layer on its own GPU (the layer is
data-parallel over tokens: no exchange step); the time is the max over ranks and the value the
tokens all ranks processed per second.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import CONFIGS, gen  # noqa: E402

WORKLOAD = "c2"
METRIC = "MoE-layer tokens/s (decode)"
N_LAYER_COPIES = 8
N_TOKEN_BATCHES = 8


# ----------------------------------------------------------------------------- distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value: float) -> float:
    """Max of a per-rank float over all ranks (the value itself on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(tokens_per_rank: int, elapsed_s: float, world: int) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world / max_over_ranks(elapsed_s)


# ----------------------------------------------------------------------------- clocks

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.proc = None
        self.path = os.path.join("/tmp", f"strata_clocks_{os.getpid()}.csv")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            p = [c.strip() for c in line.split(",")]
            if len(p) >= 9:
                rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": float(np.nanmedian(sm)), "sm_max_mhz": num(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": float(np.nanmax([num(r[3]) for r in rows]))}


# ----------------------------------------------------------------------------- workload

def build_layer(wl, threads=0, group=128, bits=4):
    """One device layer quantized from the seeded fp16 experts (strata_quantize_groups_bits).
    Its calls skip the per-call clearing of the workspace header (STRATA_WS_REUSE): every
    workspace here is zero-filled once and then reused by completed calls only."""
    import torch
    import int4_grouped_expert_gb300 as st
    from int4_grouped_expert_gb300 import MoELayer
    L = MoELayer(wl.H, wl.I, wl.E, wl.k, wl.shared, group=group, bits=bits,
                 flags=st.STRATA_WS_REUSE)
    L.set_router(gen.router_weight(wl), gen.router_bias(wl))
    n = wl.E + wl.shared
    for s in range(0, n, 16):
        es = list(range(s, min(n, s + 16)))
        for e, m in zip(es, gen.expert_weights_many(wl, es, 0, threads)):
            L.load_expert_fp16(e, *m)
    torch.cuda.synchronize()
    L.check_status()
    return L


def layer_copies(L0, n):
    """n layers sharing L0's router and values but with their own expert storage."""
    from int4_grouped_expert_gb300 import MoELayer
    out = [L0]
    for _ in range(n - 1):
        L = MoELayer(L0.H, L0.I, L0.E, L0.k, L0.shared, group=L0.group, bits=L0.bits)
        L.w_router = L0.w_router.clone()
        L.flags = L0.flags
        L.bias = L0.bias
        L.copy_expert_from(L0)
        out.append(L)
    return out


def token_batches(wl, T, n):
    import torch
    xs = [gen.activations(T, wl.H, wl.seed, name=f"bench/{T}/{i}") for i in range(n)]
    return xs, [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for x in xs]


def routed_experts(L, x_dev, T):
    """Distinct experts (incl. shared) the batch activates, read back from the GPU routing."""
    import torch
    import int4_grouped_expert_gb300 as st
    ws = torch.zeros(L.workspace_size(T), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(x_dev)
    counts = torch.zeros(L.E, dtype=torch.int32, device="cuda")
    st.check(st.strata_moe_forward_ex(L.struct(), x_dev, T, out, counts=counts, workspace=ws,
                                      ws_bytes=ws.numel()), "forward_ex")
    c = counts.cpu().numpy()
    return int((c > 0).sum()) + L.shared


# ----------------------------------------------------------------------------- strata arm

def time_steps(layers, xs_dev, T, steps, warmup, stream, ws, ws_bytes, out, profiled=False):
    import torch
    import int4_grouped_expert_gb300 as st
    structs = [L.struct() for L in layers]
    nL, nX = len(structs), len(xs_dev)

    def one(i, evs=None):
        s = structs[i % nL]
        x = xs_dev[i % nX]
        if evs is None:
            rc = st.strata_moe_forward(s, x, T, out, ws, ws_bytes, stream)
        else:
            rc = st.strata_moe_forward_profiled(s, x, T, out, ws, ws_bytes, evs, stream)
        if rc:
            st.check(rc, "strata_moe_forward")

    with torch.cuda.stream(stream):
        for i in range(warmup):
            one(i)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        stage_ev = None
        if profiled:
            stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
            for evs in stage_ev:          # torch creates the CUDA event on its first record
                for ev in evs:
                    ev.record(stream)
            torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(steps):
            one(warmup + i, stage_ev[i] if profiled else None)
        stop.record(stream)
        torch.cuda.synchronize()
        barrier()
    elapsed_ms = start.elapsed_time(stop)
    stages = None
    if profiled:
        names = ["router", "grouping", "gate_up_gemm", "down_gemm", "combine"]
        acc = np.zeros(5)
        for ev in stage_ev:
            acc += [ev[j].elapsed_time(ev[j + 1]) for j in range(5)]
        stages = {n: float(a / steps) for n, a in zip(names, acc)}
    return elapsed_ms, stages


def step_percentiles(layers, xs_dev, T, steps, stream, ws, ws_bytes, out):
    """p10 / p50 / p90 of single-step device times (an event pair around every step)."""
    import torch
    import int4_grouped_expert_gb300 as st
    structs = [L.struct() for L in layers]
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i, (a, b) in enumerate(evs):
            a.record(stream)
            st.check(st.strata_moe_forward(structs[i % len(structs)], xs_dev[i % len(xs_dev)], T,
                                           out, ws, ws_bytes, stream), "forward")
            b.record(stream)
        torch.cuda.synchronize()
    us = np.array([a.elapsed_time(b) * 1e3 for a, b in evs])
    return {"p10": float(np.percentile(us, 10)), "p50": float(np.percentile(us, 50)),
            "p90": float(np.percentile(us, 90)), "steps": steps}


def time_e2e(L, xs_host, T, steps, warmup, stream):
    """Through the C ABI with host buffers: H2D of x and D2H of out inside every call."""
    import torch
    import int4_grouped_expert_gb300 as st
    s = L.struct()
    need = st.strata_moe_workspace_size(s, T) + st.strata_moe_host_staging_size(s, T)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    xh = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs_host]
    oh = torch.empty_like(xh[0]).pin_memory()
    for i in range(warmup):
        st.check(st.strata_moe_forward_host(s, xh[i % len(xh)], T, oh, ws, need, stream), "host")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        st.check(st.strata_moe_forward_host(s, xh[i % len(xh)], T, oh, ws, need, stream), "host")
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    nbytes = xh[0].numel() * 2
    return dt, nbytes


def oracle_one_thread(T):
    """The same oracle sample in a child process with every BLAS pool limited to one thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", str(T)],
                           env=env, capture_output=True, text=True, timeout=300)
        return float(r.stdout.strip().splitlines()[-1])
    except Exception:  # noqa: BLE001 - reported as missing, not fatal
        return None


def cpu_baseline(wl, xs_host, T, budget_s=20.0, one_thread=True):
    """The fp64 oracle on the host cores, on a bounded sample of the batch's tokens."""
    import oracle
    from workloads.gen import router_bias, router_weight
    wr, b = router_weight(wl), router_bias(wl)
    x = xs_host[0]
    cache = {}

    def experts(e):
        if e not in cache:
            cache[e] = tuple(oracle.quantize_groups(m) for m in gen.expert_weights(wl, e))
        return cache[e]
    r = oracle.route_topk(x, wr, b, wl.k)
    # quantization is part of loading, as on the GPU: pre-quantize the sampled tokens' experts
    n_tok = 1
    for e in sorted(set(r["ids"][:n_tok].reshape(-1).tolist()) | ({wl.E} if wl.shared else set())):
        experts(e)
    tokens = 0
    t0 = time.perf_counter()
    while True:
        oracle.moe_forward(x, wr, b, wl.k, experts, wl.E, wl.shared, tokens=np.arange(n_tok))
        tokens += n_tok
        if time.perf_counter() - t0 > budget_s / 4 or tokens >= 4:
            break
    dt = time.perf_counter() - t0
    threads = os.environ.get("OMP_NUM_THREADS") or os.environ.get("OPENBLAS_NUM_THREADS")
    rec = {"value": tokens / dt, "unit": "tokens/s", "cores": int(threads) if threads else
           (os.cpu_count() or 1), "kind": "oracle",
            "sample": f"{n_tok} token of the T={T} batch per pass ({tokens} tokens, {dt:.1f} s): "
                      f"fp64 routing over all {wl.E} experts, dequant + FFN of its "
                      f"{wl.k} routed experts and the shared one; experts pre-quantized"}
    if one_thread:
        rec["one_thread_value"] = oracle_one_thread(T)
    return rec


def kernels_per_forward(T):
    """Kernels one strata_moe_forward launches (the workspace-header memset not counted): up to
    64 tokens the one-launch router (logits, softmax, top-k, grouping) + gate/up + down + combine;
    above, router logits + top-k + grouping + row gather + gate/up + down + combine."""
    return 4 if T <= 64 else 7


def measured_traffic(key):
    """DRAM bytes per launch of a kernel from a committed ncu capture (profiles/dram_traffic.json),
    or None when the kernel's source has changed since the capture."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))[key]
        src = open(os.path.join(ROOT, rec["source"]), "rb").read()
        if hashlib.sha256(src).hexdigest() != rec["source_sha256"]:
            return None
        return float(rec["bytes_per_launch"])
    except Exception:
        return None


def stale_traffic_note(key):
    """When measured_traffic(key) is None because the source changed: the last capture's figure and
    profile, for context (it no longer describes the current kernel)."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))[key]
    except Exception:
        return None
    if measured_traffic(key) is not None:
        return None
    return (f"no capture of the current {rec['source']}; the last one measured "
            f"{rec['bytes_per_launch'] / 1e6:.1f} MB per launch ({rec['profile']})")


def peak_numbers():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def run_strata(args):
    import torch
    ws_n, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    import int4_grouped_expert_gb300 as st
    st.lib()
    wl = CONFIGS[WORKLOAD]
    T = args.batch
    L0 = build_layer(wl, group=args.group, bits=args.bits)
    if args.router_fp16:
        L0.set_router(gen.router_weight(wl), gen.router_bias(wl), fp16=True)
    layers = layer_copies(L0, max(1, args.copies))
    stream = torch.cuda.Stream()
    xs_host, xs_dev = token_batches(wl, T, N_TOKEN_BATCHES)
    ws_bytes = L0.workspace_size(T)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(T, wl.H, dtype=torch.bfloat16, device="cuda")

    # distinct activated experts per step (all batches): bytes the layer must stream
    experts = [routed_experts(L0, x, T) for x in xs_dev]
    n_exp = float(np.mean(experts))
    eb = L0.expert_bytes()
    gu_bytes = n_exp * (2 * wl.H * wl.I) * (args.bits / 8 + 2 / args.group)

    clocks = ClockSampler(local)
    time.sleep(0.3)
    torch.cuda.nvtx.range_push("timed")
    elapsed_ms, _ = time_steps(layers, xs_dev, T, args.steps, args.warmup, stream, ws, ws_bytes, out)
    torch.cuda.nvtx.range_pop()
    clk = clocks.stop()
    # per-stage times from a second, profiled pass (events between the kernels)
    _, stages = time_steps(layers, xs_dev, T, min(args.steps, 2000), args.warmup, stream, ws,
                           ws_bytes, out, profiled=True)
    step_pct = step_percentiles(layers, xs_dev, T, min(args.steps, 1000), stream, ws, ws_bytes, out)
    elapsed_s = elapsed_ms / 1e3
    value = aggregate_throughput(T * args.steps, elapsed_s, ws_n)
    ms_step = max_over_ranks(elapsed_ms) / args.steps

    sweep = {}
    for Tb in (() if args.quick else (1, 4, 8, 16)):
        if Tb == T:
            continue
        xh_b, xd_b = token_batches(wl, Tb, N_TOKEN_BATCHES)
        wsb = torch.zeros(L0.workspace_size(Tb), dtype=torch.uint8, device="cuda")
        ob = torch.empty(Tb, wl.H, dtype=torch.bfloat16, device="cuda")
        eb_n = float(np.mean([routed_experts(L0, x, Tb) for x in xd_b]))
        ms, _ = time_steps(layers, xd_b, Tb, min(args.steps, 2000), args.warmup, stream, wsb,
                           wsb.numel(), ob)
        per = ms / min(args.steps, 2000)
        sweep[str(Tb)] = {"tokens_per_s": Tb / (per / 1e3), "us_per_layer": per * 1e3,
                          "experts": eb_n, "layer_hbm_gbs": eb_n * eb / (per / 1e3) / 1e9}
    per = ms_step
    sweep[str(T)] = {"tokens_per_s": T / (per / 1e3), "us_per_layer": per * 1e3, "experts": n_exp,
                     "layer_hbm_gbs": n_exp * eb / (per / 1e3) / 1e9}

    e2e = None
    if not args.quick:
        e2e_steps = max(10, min(args.steps, 500))
        e2e_dt, xbytes = time_e2e(L0, xs_host, T, e2e_steps, args.warmup, stream)
        e2e = {"value": aggregate_throughput(T * e2e_steps, e2e_dt, ws_n), "unit": "tokens/s",
               "h2d_bytes_per_step": xbytes, "d2h_bytes_per_step": xbytes}

    peak, peak_kind = peak_numbers()
    gu_ms = stages["gate_up_gemm"]
    achieved = gu_bytes / (gu_ms / 1e3) / 1e9
    layer_gbs = n_exp * eb / (ms_step / 1e3) / 1e9
    rec = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "tokens_per_step": T, "H": wl.H, "I": wl.I, "E": wl.E,
                   "k": wl.k, "shared": wl.shared, "router": "zipf(s=1.1), top-20% take 80%",
                   "weights": f"int{args.bits} g{args.group} codes + fp16 scales, quantized on device",
                   "router_weights": "fp16" if args.router_fp16 else "fp32",
                   "l2": f"inputs larger than L2: {N_LAYER_COPIES} expert-storage copies x "
                         f"{N_TOKEN_BATCHES} token batches rotated per step",
                   "workspace": "zero-filled once, reused by every step (STRATA_WS_REUSE)",
                   "parallelism": f"replicas x{ws_n}"},
        "roofline": {"kernel": ("gate_up_gemm (grouped W4A16 GEMM + SiLU)" if args.bits == 4 else
                                "gate_up_gemm (tcgen05 grouped W8A16 GEMM + SiLU)"),
                     "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": gu_bytes,
                     "traffic": (measured_traffic("decode_gate_up")
                                 if args.bits == 4 and args.group == 128 else None),
                     "traffic_note": (stale_traffic_note("decode_gate_up")
                                      if args.bits == 4 and args.group == 128 else None)},
        "layer_hbm": {"achieved_gbs": layer_gbs, "frac": layer_gbs / peak,
                      "bytes_per_step": n_exp * eb, "experts_per_step": n_exp},
        "stages_us": {k: v * 1e3 for k, v in stages.items()},
        "step_us_percentiles": step_pct,
        "sweep": sweep,
        "e2e": e2e,
        "gpu_launches": kernels_per_forward(T) * args.steps,
        "clocks": clk,
    }
    if ws_n == 1 and not args.quick and not args.no_extras:
        # the rest of the metric on the same GPU, each under its own key with its own roofline:
        # the padded fixed-max-batch graph (this layer), the prefill layers and the decode stack
        t0 = time.perf_counter()
        rec["padded_graph"] = guarded(padded_graph_measure, layers, wl, 16, (1, 5, 16), 200,
                                      args.warmup)
        rec["prefill_c5"] = guarded(prefill_measure, "c5", 10, 3, local=local)
        rec["prefill_c3"] = guarded(prefill_measure, "c3", 50, 5, local=local)
        rec["stack_c4"] = guarded(stack_measure, 200, 5, CONFIGS["c4"].batches, local=local)
        rec["extras_wall_s"] = time.perf_counter() - t0
    if rank == 0:
        if ws_n == 1 and not args.quick:
            rec["cpu_baseline"] = cpu_baseline(wl, xs_host, T)
        print(json.dumps(rec), flush=True)


def guarded(fn, *a, **kw):
    """fn's record, or the error it raised (an extra measurement never hides the headline)."""
    try:
        return fn(*a, **kw)
    except Exception as exc:  # noqa: BLE001 - reported in the JSON line
        import traceback
        traceback.print_exc(file=sys.stderr)
        return {"error": f"{type(exc).__name__}: {exc}"}


def device_random_experts(L, seed, chunk=16):
    """Fill every expert slot of L with codes quantized on the device (strata_quantize_groups_bits)
    from fp16 weights drawn N(0, 0.02) on the device by torch's seeded CUDA generator: the
    workloads' distribution, drawn where it is used (tens of GB of fp16 would take minutes in the
    host generator). The timings depend on the shapes and on the routing, not on these values."""
    import torch
    import int4_grouped_expert_gb300 as st
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    n = L.E + L.shared
    for codes, scales, rows, cols in ((L.gate_codes, L.gate_scales, L.I, L.H),
                                      (L.up_codes, L.up_scales, L.I, L.H),
                                      (L.down_codes, L.down_scales, L.H, L.I)):
        for e0 in range(0, n, chunk):
            e1 = min(n, e0 + chunk)
            w = (torch.randn((e1 - e0) * rows, cols, generator=g, device="cuda") * 0.02).half()
            st.check(st.strata_quantize_groups_bits(w, (e1 - e0) * rows, cols, codes[e0:e1],
                                                    scales[e0:e1], L._status, group_size=L.group,
                                                    bits=L.bits), "strata_quantize_groups_bits")
            del w
    torch.cuda.synchronize()
    L.check_status()


def tensor_peak(timed_s):
    """Dense bf16 tensor peak (TFLOP/s) for a kernel timed over timed_s seconds: the burst figure
    below a second, the sustained one (power cap) above. f16 operands run at the bf16 rate."""
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        if timed_s < 1.0:
            return float(d["bf16_tflops"]), "measured burst"
        return float(d["bf16_tflops_sustained"]), "measured sustained"
    except Exception:
        return (1900.0, "fallback burst") if timed_s < 1.0 else (1700.0, "fallback sustained")


def prefill_measure(key, steps, warmup, experts=0, tokens=0, router=None, host_weights=False,
                    local=0):
    """A prefill layer (c3: 512 tokens over 64 experts; c5: 4096 tokens over 256 + shared, with its
    experts quantized on the device from resident fp16 stacks, timed) on the tensor-core path:
    tokens/s, gate/up and down TFLOP/s, the gate/up roofline and, for c5, quantize GB/s."""
    import torch
    import int4_grouped_expert_gb300 as st
    from int4_grouped_expert_gb300 import MoELayer
    wl = CONFIGS[key]
    if experts:  # a smaller layer of the same shapes (e.g. for profiler captures)
        import dataclasses
        wl = dataclasses.replace(wl, E=experts)
    T = tokens or wl.batches[0]
    L = MoELayer(wl.H, wl.I, wl.E, wl.k, wl.shared, flags=st.STRATA_WS_REUSE)
    L.set_router(gen.router_weight(wl), gen.router_bias(wl, 0, router) if not experts else None)
    n = wl.E + wl.shared
    quant = None
    hbm_peak, hbm_kind = peak_numbers()
    if key == "c5" and not experts:
        # fp16 experts resident on the device, then one quantize launch per projection stack
        g = torch.Generator(device="cuda")
        g.manual_seed(wl.seed)
        w16 = {}
        for name, rows, cols in (("gate", wl.I, wl.H), ("up", wl.I, wl.H), ("down", wl.H, wl.I)):
            t = torch.empty(n, rows, cols, dtype=torch.float16, device="cuda")
            for e0 in range(0, n, 16):
                e1 = min(n, e0 + 16)
                t[e0:e1].copy_(torch.randn(e1 - e0, rows, cols, generator=g, device="cuda") * 0.02)
            w16[name] = t
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        jobs = [(w16["gate"], L.gate_codes, L.gate_scales, wl.I * n, wl.H),
                (w16["up"], L.up_codes, L.up_scales, wl.I * n, wl.H),
                (w16["down"], L.down_codes, L.down_scales, wl.H * n, wl.I)]

        def quantize_all():
            for w, c, sc, rows, cols in jobs:
                st.check(st.strata_quantize_groups(w, rows, cols, c, sc, status), "quantize")
        for _ in range(2):
            quantize_all()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 3
        e0.record()
        for _ in range(reps):
            quantize_all()
        e1.record()
        torch.cuda.synchronize()
        qs = e0.elapsed_time(e1) / reps / 1e3
        nw = 3 * n * wl.H * wl.I
        qbytes = nw * 2 + nw // 2 + 2 * (nw // 128)  # fp16 in, int4 codes + fp16 scales out
        gbs = qbytes / qs / 1e9
        quant = {"seconds_per_layer": qs, "weights": nw, "launches_per_layer": 3,
                 "roofline": {"kernel": "quantize_groups_kernel", "bound": "hbm", "achieved": gbs,
                              "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                              "peak_kind": hbm_kind,
                              "algorithmic_bytes_per_launch": qbytes / 3,
                              "traffic": measured_traffic("quantize_c5")}}
        rc, v = st.strata_read_status(status)
        assert rc == 0, hex(v)
        del w16, jobs
        torch.cuda.empty_cache()
    elif host_weights:
        for s0 in range(0, n, 16):
            es = list(range(s0, min(n, s0 + 16)))
            for e, m in zip(es, gen.expert_weights_many(wl, es)):
                L.load_expert_fp16(e, *m)
        torch.cuda.synchronize()
        L.check_status()
    else:
        device_random_experts(L, wl.seed)
    xs_host, xs_dev = token_batches(wl, T, 2)
    ws_bytes = L.workspace_size(T)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(T, wl.H, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    clocks = ClockSampler(local)
    elapsed_ms, _ = time_steps([L], xs_dev, T, steps, warmup, stream, ws, ws_bytes, out)
    clk = clocks.stop()
    _, stages = time_steps([L], xs_dev, T, steps, warmup, stream, ws, ws_bytes, out, profiled=True)
    rows = T * wl.k + wl.shared * T
    gu_flops = 2 * 2 * wl.H * wl.I * rows
    dn_flops = 2 * wl.H * wl.I * rows
    ms = elapsed_ms / steps
    peak_tf, tf_kind = tensor_peak(elapsed_ms / 1e3)
    gu_tf = gu_flops / (stages["gate_up_gemm"] / 1e3) / 1e12
    dn_tf = dn_flops / (stages["down_gemm"] / 1e3) / 1e12
    layer_tf = (gu_flops + dn_flops) / (ms / 1e3) / 1e12
    # binding roof of the gate/up GEMM: its flops per algorithmic byte (the activated experts'
    # gate + up codes and scales) against the ridge of the measured peaks
    n_exp = float(np.mean([routed_experts(L, x, T) for x in xs_dev]))
    gu_bytes = n_exp * 2 * wl.H * wl.I * (0.5 + 2 / 128)
    hbm_bound = gu_flops / gu_bytes < peak_tf * 1e12 / (hbm_peak * 1e9)
    traffic_key = {"c5": "prefill_gate_up_c5", "c3": "prefill_gate_up_c3"}.get(key)
    traffic = measured_traffic(traffic_key) if traffic_key and not experts and not tokens else None
    kname = "gate_up_gemm (tcgen05 grouped W4A16 GEMM + SiLU, f16 operands)"
    if hbm_bound:
        gu_gbs = gu_bytes / (stages["gate_up_gemm"] / 1e3) / 1e9
        roof = {"kernel": kname, "bound": "hbm", "achieved": gu_gbs, "peak": hbm_peak,
                "unit": "GB/s", "frac": gu_gbs / hbm_peak, "peak_kind": hbm_kind,
                "algorithmic_bytes_per_launch": gu_bytes, "traffic": traffic, "tflops": gu_tf,
                "tensor_frac": gu_tf / peak_tf}
    else:
        roof = {"kernel": kname, "bound": "tensor", "achieved": gu_tf, "peak": peak_tf,
                "unit": "TFLOP/s", "frac": gu_tf / peak_tf, "peak_kind": tf_kind,
                "algorithmic_flops_per_launch": gu_flops, "traffic": traffic}
    rec = {"workload": wl.name, "tokens_per_step": T, "router": router or wl.router,
           "tokens_per_s": T / (ms / 1e3), "ms_per_step": ms, "steps": steps, "warmup": warmup,
           "roofline": roof, "experts_per_step": n_exp,
           "layer_tflops": layer_tf, "layer_frac": layer_tf / peak_tf,
           "down_tflops": dn_tf, "down_frac": dn_tf / peak_tf, "tensor_peak": peak_tf,
           "tensor_peak_kind": tf_kind,
           "stages_us": {k: v * 1e3 for k, v in stages.items()}, "quantize": quant,
           "weights": ("host-generated (workloads.gen)" if host_weights else
                       "N(0,0.02) fp16 drawn on the device, quantized on the device"),
           "gpu_launches": kernels_per_forward(T) * steps, "clocks": clk}
    del L, ws
    torch.cuda.empty_cache()
    return rec


def run_prefill(args):
    """Prefill workloads alone (c3 / c5), one JSON line."""
    import torch
    import int4_grouped_expert_gb300 as st
    ws_n, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    st.lib()
    r = prefill_measure(args.workload, args.steps, args.warmup, experts=args.experts,
                        tokens=args.tokens, router=args.router, host_weights=args.host_weights,
                        local=local)
    rec = {"metric": f"MoE-layer tokens/s (prefill, {args.workload})", "value": r["tokens_per_s"],
           "unit": "tokens/s", "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": r["workload"], "tokens_per_step": r["tokens_per_step"],
                      "router": r["router"], "weights": r["weights"]},
           "roofline": r["roofline"], "gpu_launches": r["gpu_launches"], "clocks": r["clocks"],
           "prefill": r}
    if rank == 0:
        print(json.dumps(rec), flush=True)


def stack_graph_us(structs, xs_dev, T, out, ws, need, steps, warmup):
    """The same stack call captured once in a CUDA graph and replayed (no per-launch host work):
    mean microseconds per replay, or None if capture is not possible here."""
    import torch
    import int4_grouped_expert_gb300 as st
    try:
        xg = xs_dev[0].clone()
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):  # first call outside the capture (one-time host set-up)
            st.check(st.strata_moe_stack_forward(structs, xg, T, out, ws, need, side), "stack")
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            s = torch.cuda.current_stream()
            st.check(st.strata_moe_stack_forward(structs, xg, T, out, ws, need, s), "stack")
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps * 1e3
    except Exception as exc:  # noqa: BLE001 - reported, not fatal
        print(f"stack graph capture unavailable: {exc}", file=sys.stderr)
        return None


def stack_measure(steps, warmup, batches, host_weights=False, local=0):
    """The 8-layer decode stack (hidden 4096, expert inter 2048, 128 experts top-4 + shared, a
    Zipf router per layer, residual add between layers) through strata_moe_stack_forward, for each
    batch: stack and per-layer tokens/s, HBM GB/s of the activated experts, graph replay."""
    import torch
    import int4_grouped_expert_gb300 as st
    from int4_grouped_expert_gb300 import MoELayer
    wl = CONFIGS["c4"]
    # layer 0's experts are quantized on the device; every other layer gets its own copy of those
    # values at its own addresses (the same bytes stream from HBM) and its own router
    if host_weights:
        L0 = build_layer(wl)
    else:
        L0 = MoELayer(wl.H, wl.I, wl.E, wl.k, wl.shared, flags=st.STRATA_WS_REUSE)
        L0.set_router(gen.router_weight(wl), gen.router_bias(wl))
        device_random_experts(L0, wl.seed)
    layers = [L0]
    for l in range(1, wl.layers):
        L = MoELayer(wl.H, wl.I, wl.E, wl.k, wl.shared,
                     flags=st.STRATA_ADD_RESIDUAL | st.STRATA_WS_REUSE)
        L.set_router(gen.router_weight(wl, l), gen.router_bias(wl, l))
        L.copy_expert_from(L0)
        layers.append(L)
    L0.flags |= st.STRATA_ADD_RESIDUAL
    structs = [L.struct() for L in layers]
    stream = torch.cuda.Stream()
    eb = wl.expert_bytes()
    peak, peak_kind = peak_numbers()
    sweep = {}
    clocks = ClockSampler(local)
    for T in batches:
        xs_host, xs_dev = token_batches(wl, T, N_TOKEN_BATCHES)
        need = st.strata_moe_stack_workspace_size(structs, T)
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        out = torch.empty(T, wl.H, dtype=torch.bfloat16, device="cuda")
        # distinct experts each layer streams: route the layer-by-layer activations
        n_exp = []
        cur = xs_dev[0]
        for L in layers:
            nxt = torch.empty_like(cur)
            counts = torch.zeros(wl.E, dtype=torch.int32, device="cuda")
            wsl = torch.zeros(L.workspace_size(T), dtype=torch.uint8, device="cuda")
            st.check(st.strata_moe_forward_ex(L.struct(), cur, T, nxt, counts=counts,
                                              workspace=wsl, ws_bytes=wsl.numel()), "forward_ex")
            n_exp.append(int((counts.cpu().numpy() > 0).sum()) + wl.shared)
            cur = nxt
        with torch.cuda.stream(stream):
            for i in range(warmup):
                st.check(st.strata_moe_stack_forward(structs, xs_dev[i % N_TOKEN_BATCHES], T, out,
                                                     ws, need, stream), "stack")
            torch.cuda.synchronize()
            barrier()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(steps):
                rc = st.strata_moe_stack_forward(structs, xs_dev[i % N_TOKEN_BATCHES], T, out, ws,
                                                 need, stream)
                if rc:
                    st.check(rc, "stack")
            e1.record(stream)
            torch.cuda.synchronize()
            barrier()
        ms = max_over_ranks(e0.elapsed_time(e1)) / steps
        graph_us = stack_graph_us(structs, xs_dev, T, out, ws, need, steps, warmup)
        # per-stage times of single layers (events between the kernels), same inputs and layers
        wsl = torch.zeros(max(L.workspace_size(T) for L in layers), dtype=torch.uint8, device="cuda")
        _, stages = time_steps(layers, xs_dev, T, min(steps, 400), warmup, stream, wsl,
                               wsl.numel(), out, profiled=True)
        st_bytes = float(sum(n_exp)) * eb
        gbs = st_bytes / (ms / 1e3) / 1e9
        sweep[str(T)] = {"stack_tokens_per_s": T / (ms / 1e3),
                         "layer_tokens_per_s": T / (ms / wl.layers / 1e3),
                         "us_per_stack": ms * 1e3, "us_per_layer": ms * 1e3 / wl.layers,
                         "experts_per_layer": float(np.mean(n_exp)),
                         "hbm_gbs": gbs, "hbm_frac": gbs / peak, "steps": steps,
                         "us_per_stack_graph": graph_us,
                         "stages_us": {k: v * 1e3 for k, v in stages.items()}}
        del ws, wsl
    clk = clocks.stop()
    head = str(max(batches))
    h = sweep[head]
    rec = {"workload": wl.name, "layers": wl.layers, "tokens_per_step": int(head),
           "roofline": {"kernel": "whole stack (all kernels)", "bound": "hbm",
                        "achieved": h["hbm_gbs"], "peak": peak, "unit": "GB/s",
                        "frac": h["hbm_gbs"] / peak, "peak_kind": peak_kind,
                        "algorithmic_bytes_per_step": h["experts_per_layer"] * wl.layers * eb,
                        "traffic": None},
           "sweep": sweep,
           "weights": ("layer 0's int4 g128 experts ("
                       + ("host-generated" if host_weights else "N(0,0.02) drawn on the device")
                       + ", quantized on the device) copied into each layer's own storage; "
                         "per-layer Zipf routers"),
           "l2": f"each step streams {wl.layers} layers' activated experts (GBs) > L2",
           "gpu_launches": kernels_per_forward(int(head)) * wl.layers * h["steps"], "clocks": clk}
    del layers, L0
    torch.cuda.empty_cache()
    return rec


def run_stack(args):
    """The 8-layer decode stack alone, one JSON line."""
    import torch
    import int4_grouped_expert_gb300 as st
    ws_n, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    st.lib()
    wl = CONFIGS["c4"]
    batches = (args.tokens,) if args.tokens else wl.batches
    r = stack_measure(args.steps, args.warmup, batches, host_weights=args.host_weights, local=local)
    h = r["sweep"][str(r["tokens_per_step"])]
    rec = {"metric": "MoE stack tokens/s (decode, 8 layers)",
           "value": aggregate_throughput(r["tokens_per_step"] * h["steps"],
                                         h["us_per_stack"] * h["steps"] / 1e6, ws_n),
           "unit": "tokens/s", "n_gpus": ws_n, "steps": h["steps"], "warmup": args.warmup,
           "ms_per_step": h["us_per_stack"] / 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": r["workload"], "tokens_per_step": r["tokens_per_step"],
                      "layers": r["layers"], "weights": r["weights"], "l2": r["l2"]},
           "roofline": r["roofline"], "sweep": r["sweep"], "gpu_launches": r["gpu_launches"],
           "clocks": r["clocks"]}
    if rank == 0:
        print(json.dumps(rec), flush=True)


def padded_graph_measure(layers, wl, T_max, batches, steps, warmup):
    """One CUDA graph holding a strata_moe_forward_padded call per layer copy (each copy's own
    expert storage, so every layer streams its weights from HBM), captured once at T_max and
    replayed with each batch's live count written to the device: microseconds per layer."""
    import torch
    import int4_grouped_expert_gb300 as st
    n_tok = torch.full((1,), T_max, dtype=torch.int32, device="cuda")
    xs_host, _ = token_batches(wl, T_max, 1)
    x_static = torch.from_numpy(xs_host[0].view(np.int16)).view(torch.bfloat16).cuda()
    out = torch.empty_like(x_static)
    ws = torch.zeros(max(L.workspace_size(T_max) for L in layers), dtype=torch.uint8, device="cuda")
    structs = [L.struct() for L in layers]
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):  # first calls outside the capture (one-time host set-up)
        for s in structs:
            st.check(st.strata_moe_forward_padded(s, x_static, n_tok, T_max, out, ws, ws.numel(),
                                                  side), "padded")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for s in structs:
            st.check(st.strata_moe_forward_padded(s, x_static, n_tok, T_max, out, ws, ws.numel(),
                                                  cs), "capture")
    res = {}
    for T in batches:
        n_tok.fill_(T)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / steps / len(structs) * 1e3
        res[str(T)] = {"us_per_layer": us, "tokens_per_s": T / (us / 1e6)}
    rc, v = st.strata_workspace_status(ws)
    assert rc == 0, hex(v)
    return {"T_max": T_max, "layers_per_replay": len(structs), "replays": steps, "batches": res}


def run_reference(args):
    """The oracle on the host cores, same metric and workload, each step a bounded sample."""
    ws_n, rank = init_dist("gloo")
    if rank != 0:
        return
    import oracle
    wl = CONFIGS[WORKLOAD]
    T = args.batch
    x = gen.activations(T, wl.H, wl.seed, name=f"bench/{T}/0")
    wr, b = gen.router_weight(wl), gen.router_bias(wl)
    cache = {}

    def experts(e):
        if e not in cache:
            cache[e] = tuple(oracle.quantize_groups(m) for m in gen.expert_weights(wl, e))
        return cache[e]
    r = oracle.route_topk(x, wr, b, wl.k)
    sample = max(1, min(T, int(args.ref_tokens)))
    order = [t % T for t in range(args.warmup + args.steps)]
    need = set()
    for t in order:
        need |= set(r["ids"][t].tolist())
    for e in sorted(need | ({wl.E} if wl.shared else set())):
        experts(e)
    for i in range(args.warmup):
        oracle.moe_forward(x, wr, b, wl.k, experts, wl.E, wl.shared, tokens=[order[i]])
    t0 = time.perf_counter()
    done = 0
    for i in range(args.steps):
        t = order[args.warmup + i]
        oracle.moe_forward(x, wr, b, wl.k, experts, wl.E, wl.shared,
                           tokens=[(t + j) % T for j in range(sample)])
        done += 1
        if time.perf_counter() - t0 > args.ref_budget_s:
            break                                   # a bounded run: steps_timed says how many
    dt = time.perf_counter() - t0
    val = sample * done / dt
    cores = os.cpu_count() or 1
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": ws_n,
        "steps": args.steps, "steps_timed": done, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / done,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": wl.name, "tokens_per_step": sample, "H": wl.H, "I": wl.I,
                   "E": wl.E, "k": wl.k, "shared": wl.shared},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample} token(s) of the T={T} batch per step: fp64 routing, "
                                   "dequant + FFN of its experts; experts pre-quantized"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps (default 5000; 10 for --impl reference)")
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--copies", type=int, default=N_LAYER_COPIES,
                   help="expert-storage copies rotated per step (cold L2)")
    p.add_argument("--quick", action="store_true",
                   help="headline only: no batch sweep, no host-buffer run, no CPU baseline")
    p.add_argument("--batch", type=int, default=16)
    p.add_argument("--impl", choices=["strata", "reference"], default="strata")
    p.add_argument("--ref-tokens", type=int, default=1)
    p.add_argument("--ref-budget-s", type=float, default=240.0)
    p.add_argument("--workload", choices=["c2", "c3", "c4", "c5"], default="c2",
                   help="c2: the decode layer (default, the headline); c3 / c5: prefill layers; "
                        "c4: the 8-layer decode stack")
    p.add_argument("--router", choices=["uniform", "zipf"], default=None)
    p.add_argument("--group", type=int, choices=[64, 128, 256], default=128,
                   help="decode: scale group size of the experts")
    p.add_argument("--bits", type=int, choices=[4, 8], default=4,
                   help="decode: code width of the experts (8: the tensor-core W8A16 path)")
    p.add_argument("--router-fp16", action="store_true",
                   help="decode: store the router weights as fp16 (STRATA_ROUTER_FP16)")
    p.add_argument("--experts", type=int, default=0, help="prefill: override the routed expert count")
    p.add_argument("--tokens", type=int, default=0,
                   help="prefill: override the batch; c4: run this batch only")
    p.add_argument("--no-extras", action="store_true",
                   help="c2: skip the padded-graph, prefill and stack measurements of the default run")
    p.add_argument("--host-weights", action="store_true",
                   help="c3/c4/c5: draw the experts with the host generator (workloads.gen) instead "
                        "of on the device")
    p.add_argument("--oracle-sample", type=int, default=0, help=argparse.SUPPRESS)
    args = p.parse_args(argv)
    if args.oracle_sample:  # child of cpu_baseline: the oracle sample alone, tokens/s on stdout
        wl = CONFIGS[WORKLOAD]
        xs = [gen.activations(args.oracle_sample, wl.H, wl.seed, name=f"bench/{args.oracle_sample}/0")]
        print(cpu_baseline(wl, xs, args.oracle_sample, one_thread=False)["value"])
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.steps is None:
        args.steps = 10 if args.impl == "reference" else 5000
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "c4":
        if args.steps == 5000:
            args.steps = 500
        run_stack(args)
    elif args.workload != "c2":
        if args.steps == 5000:
            args.steps = 50
        run_prefill(args)
    else:
        run_strata(args)


if __name__ == "__main__":
    main()
