"""Benchmark of the MoE expert FFN forward on one GB300 (or N replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one pass of the whole path (rms_norm, router softmax/top-k,
permute, FC1 + silu_and_mul, FC2 + routing weight, combine) over one batch of
the workload.  Prints ONE JSON line (rank 0).

Timed regions (CUDA events on the launching stream, after W warm-up steps):
  value     K calls of moe_ffn_forward with device-resident inputs.
  roofline  K steps through the step entry points (the same kernels), with
            events around each stage; achieved = algorithmic bytes (decode)
            or flops (prefill) of the dominant kernel / its mean duration.
  e2e       K calls of moe_ffn_forward whose inputs come from pinned host
            memory and whose output goes back to pinned host memory, copies
            inside the timed region.
The expert weights of every workload but the tiny one are larger than L2, so
each step reads them from HBM; for the tiny workload L2 is flushed (a 512 MB
write) between timed steps.

--impl reference times the CPU oracle (fp64 numpy, one thread) on a bounded
token sample of the same workload and prints the same line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MoE FFN fwd: HBM TB/s vs peak & tokens/s (T≤64); TFLOP/s vs peak (T=4096)"
DEFAULT_WORKLOAD = "c2_decode_balanced"
NOMINAL_HBM_GBS = 8000.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# --------------------------------------------------------------- algorithm --

def algorithmic_work(inp, offsets_np):
    """Expert-weight bytes each GEMM reads (experts with >= 1 row) and the
    GEMM flops over unpadded rows."""
    E, H, I = inp["E"], inp["H"], inp["I"]
    counts = np.diff(offsets_np)
    active = int((counts > 0).sum())
    if inp.get("nvfp4"):
        # E2M1 codes (1/2 B), one E4M3 block scale per 16 (1/16 B), an fp32 matrix scale
        fc1_bytes = active * (2 * I * H // 2 + 2 * I * H // 16 + 4)
        fc2_bytes = active * (H * I // 2 + H * I // 16 + 4)
    elif inp["fp8"] == "block":
        # E4M3 codes (1 B) and one fp32 scale per 128 x 128 tile
        fc1_bytes = active * (2 * I * H + (2 * I // 128) * (H // 128) * 4)
        fc2_bytes = active * (H * I + (H // 128) * (I // 128) * 4)
    else:
        elem = 1 if inp["fp8"] else 2
        fc1_bytes = active * 2 * I * H * elem + (active * 2 * I * 4 if inp["fp8"] else 0)
        fc2_bytes = active * H * I * elem + (active * H * 4 if inp["fp8"] else 0)
    rows = int(counts.sum())
    fc1_flops = 2.0 * rows * H * 2 * I
    fc2_flops = 2.0 * rows * I * H
    return dict(active_experts=active, rows=rows, fc1_bytes=fc1_bytes, fc2_bytes=fc2_bytes,
                fc1_flops=fc1_flops, fc2_flops=fc2_flops)


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                     power=float(parts[3]) if parts[3] not in ("[N/A]", "") else 0.0,
                                     hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        load = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(load)}


# -------------------------------------------------------------- CPU oracle --

def _save_sample(inp, toks, path):
    """Writes the inputs the oracle needs for the sampled tokens."""
    import torch
    k = inp["k"]
    d = dict(x=inp["x"][toks].float().cpu().numpy(), norm_w=inp["norm_w"].float().cpu().numpy(),
             eps=np.array(inp["eps"]), k=np.array(k), fp8=np.array(str(inp["fp8"])),
             nvfp4=np.array(bool(inp.get("nvfp4"))))
    if inp["router_logits"] is not None:
        d["logits"] = inp["router_logits"][toks].cpu().numpy()
        l = inp["router_logits"][toks].cpu().numpy()
        experts = sorted(set(np.argsort(-l, axis=1, kind="stable")[:, :k].reshape(-1).tolist()))
    else:
        d["router_w"] = inp["router_w"].cpu().numpy()
        if inp["router_bias"] is not None:
            d["router_bias"] = inp["router_bias"].cpu().numpy()
        experts = list(range(inp["E"]))
        # only experts some sampled token can select are needed: the oracle's
        # own routing decides; keep all when E is small, else the candidates
        # with the largest logits (fp32 estimate) plus a margin of 4 per token.
        if inp["E"] > 16:
            x = inp["x"][toks].float()
            xh = x * torch.rsqrt(x.pow(2).mean(-1, keepdim=True) + inp["eps"]) * inp["norm_w"].float()
            l = (xh @ inp["router_w"])
            if inp["router_bias"] is not None:
                l = l + inp["router_bias"]
            cand = torch.topk(l, min(inp["E"], k + 4), dim=1).indices.cpu().numpy()
            experts = sorted(set(cand.reshape(-1).tolist()))
    d["experts"] = np.array(experts, dtype=np.int64)
    d["E"] = np.array(inp["E"])
    for e in experts:
        d[f"w13_{e}"] = inp["w13"][e].view(torch.int16).cpu().numpy()
        d[f"w2_{e}"] = inp["w2"][e].view(torch.int16).cpu().numpy()
    np.savez(path, **d)


ORACLE_CHILD = r"""
import sys, time, json, os
import numpy as np
sys.path.insert(0, sys.argv[2])
import oracle as O
d = np.load(sys.argv[1])
def bf(a):
    return (a.astype(np.int32).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
W13 = {int(e): bf(d[f"w13_{e}"]) for e in d["experts"]}
W2 = {int(e): bf(d[f"w2_{e}"]) for e in d["experts"]}
kw = {}
if "logits" in d: kw["logits"] = d["logits"].astype(np.float64)
else:
    kw["router_w"] = d["router_w"].astype(np.float64)
    if "router_bias" in d: kw["router_bias"] = d["router_bias"].astype(np.float64)
if "nvfp4" in d and bool(d["nvfp4"]):
    # NVFP4 weights: quantised once, like the GPU path's offline quantisation
    W13 = {e: O.dequantize_nvfp4(*O.quantize_nvfp4(w)) for e, w in W13.items()}
    W2 = {e: O.dequantize_nvfp4(*O.quantize_nvfp4(w)) for e, w in W2.items()}
fp8 = str(d["fp8"])
fp8 = "block" if fp8 == "block" else fp8 == "True"
reps = int(sys.argv[3])
min_seconds = float(sys.argv[4])
t0 = time.perf_counter()
done = 0
while done < reps or time.perf_counter() - t0 < min_seconds:
    res = O.moe_ffn_forward(d["x"].astype(np.float64), d["norm_w"].astype(np.float64),
                            float(d["eps"]), int(d["k"]), lambda e: W13[e], lambda e: W2[e],
                            fp8=fp8, **kw)
    assert set(res["ids"].reshape(-1).tolist()) <= set(W13), "sample needs more experts"
    done += 1
dt = time.perf_counter() - t0
print(json.dumps({"seconds": dt, "tokens": int(d["x"].shape[0]) * done, "passes": done}))
"""


def run_oracle_sample(inp, n_tokens, reps=1, seed=0, min_seconds=10.0):
    """Times the CPU oracle (one thread) on n_tokens sampled tokens, repeated
    for at least `reps` passes and `min_seconds`; returns (tokens/s, seconds,
    description)."""
    T = inp["T"]
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(T, size=min(n_tokens, T), replace=False))
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "sample.npz")
        _save_sample(inp, toks, path)
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
                   CUDA_VISIBLE_DEVICES="")
        p = subprocess.run([sys.executable, "-c", ORACLE_CHILD, path, ROOT, str(reps),
                            str(min_seconds)],
                           capture_output=True, text=True, env=env, timeout=1800)
        if p.returncode != 0:
            raise RuntimeError("oracle baseline failed:\n" + p.stderr[-2000:])
        r = json.loads(p.stdout.strip().splitlines()[-1])
    desc = (f"{len(toks)} of {T} tokens (seeded sample) x {r['passes']} passes: oracle "
            f"moe_ffn_forward on the sample (weights of the experts it needs preloaded as "
            f"fp64), 1 thread")
    return r["tokens"] / r["seconds"], r["seconds"], desc


# -------------------------------------------------------------------- main --

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=0, help="oracle sample size (0 = auto)")
    ap.add_argument("--shape", default=None,
                    help="T,H,E,k,I: the workload's recipe at another shape (smaller cases for "
                         "profiling); the JSON line names it in config")
    ap.add_argument("--no-more", action="store_true",
                    help="measure only --workload (no prefill entries under \"more\")")
    return ap.parse_args()


def dist_setup(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def max_over_ranks(value: float, world: int) -> float:
    """Max of a float over ranks (timing only; no data-path collective)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def auto_cpu_tokens(workload):
    return {"c1_tiny": 4, "c2_decode_balanced": 2, "c3_decode_skewed": 1,
            "c4_decode_fp8": 2, "c5_prefill": 2, "c6_decode_nvfp4": 2,
            "c7_decode_fp8_block": 2, "c8_prefill_fp8": 2, "c9_prefill_fp8_block": 2}.get(workload, 1)


def main_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    import workloads
    inp = workloads.make_inputs(args.workload, "cpu" if not torch.cuda.is_available() else "cuda")
    n = args.cpu_tokens or auto_cpu_tokens(args.workload)
    # warm-up steps are untimed oracle runs on the same sample
    for _ in range(min(args.warmup, 1)):
        run_oracle_sample(inp, n, 1, min_seconds=0.0)
    tps, secs, desc = run_oracle_sample(inp, n, max(1, args.steps), min_seconds=0.0)
    ms = secs / max(1, args.steps) * 1e3
    cfg = inp
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "T": cfg["T"], "H": cfg["H"], "E": cfg["E"],
                   "top_k": cfg["k"], "I": cfg["I"], "fp8": cfg["fp8"]},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": 1,
                         "host_cores": os.cpu_count(), "kind": "oracle",
                         "sample": desc + f"; each step = one pass over the sample"},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_workload(args, workload, dev, rank, world, local, steps, warmup, cpu_ok):
    """Measures one workload (regions A, B and e2e); returns rank 0's JSON
    record (None on other ranks)."""
    import torch
    import moe_expert_ffn_rms_gb300 as M
    import workloads

    shape_over = None
    if args.shape and workload == args.workload:
        T_, H_, E_, k_, I_ = (int(v) for v in args.shape.split(","))
        shape_over = workloads.Shape(T=T_, H=H_, E=E_, k=k_, I=I_)
    inp = workloads.make_inputs(workload, dev, shape=shape_over)
    # committed DRAM traffic records are per full-size workload
    traffic_key = workload if shape_over is None else None
    T, H, E, k, I, fp8 = inp["T"], inp["H"], inp["E"], inp["k"], inp["I"], inp["fp8"]
    nvfp4 = bool(inp.get("nvfp4"))
    fb = fp8 == "block"
    R = T * k
    shape = M.make_shape(T, H, E, I, k, inp["eps"], fp8=fp8, nvfp4=nvfp4)
    ws = M.alloc_workspace(M.moe_ffn_workspace_size(shape), dev)
    w13, w2, s13, s2 = inp["w13"], inp["w2"], None, None
    if fb:
        # E4M3 codes with one fp32 scale per 128 x 128 tile
        w13 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=dev)
        s13 = torch.empty((E, 2 * I // 128, H // 128), dtype=torch.float32, device=dev)
        w2 = torch.empty((E, H, I), dtype=torch.uint8, device=dev)
        s2 = torch.empty((E, H // 128, I // 128), dtype=torch.float32, device=dev)
        M.moe_quantize_fp8_blocks(inp["w13"], w13, s13, 128)
        M.moe_quantize_fp8_blocks(inp["w2"], w2, s2, 128)
    elif fp8:
        w13 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=dev)
        s13 = torch.empty((E, 2 * I), dtype=torch.float32, device=dev)
        w2 = torch.empty((E, H, I), dtype=torch.uint8, device=dev)
        s2 = torch.empty((E, H), dtype=torch.float32, device=dev)
        M.moe_quantize_fp8_rows(inp["w13"], w13, s13)
        M.moe_quantize_fp8_rows(inp["w2"], w2, s2)
    nv = None
    if nvfp4:
        # NVFP4 codes [E, N, K/2], E4M3 block scales [E, N, K/16], fp32 matrix scales [E]
        nv = []
        for w in (inp["w13"], inp["w2"]):
            n_, k_ = w.shape[1], w.shape[2]
            q = torch.empty((E, n_, k_ // 2), dtype=torch.uint8, device=dev)
            sbq = torch.empty((E, n_, k_ // 16), dtype=torch.uint8, device=dev)
            sgq = torch.empty((E,), dtype=torch.float32, device=dev)
            M.moe_quantize_nvfp4(w, q, sbq, sgq)
            nv.append((q, sbq, sgq))
        torch.cuda.synchronize()
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    tw = torch.empty((T, k), dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream()
    wbytes = 3 * H * I * E * (0.5625 if nvfp4 else (1 if fp8 else 2))  # fp8: True or "block"
    small = wbytes < 256 * 2 ** 20
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev) if small else None

    def fwd(x=None, out_=None, logits=None):
        xi = inp["x"] if x is None else x
        lg = inp["router_logits"] if logits is None else logits
        o = out if out_ is None else out_
        if nvfp4:
            (q13, sb13, sg13), (q2, sb2, sg2) = nv
            M.moe_ffn_forward_nvfp4(shape, xi, inp["norm_w"], q13, sb13, sg13, q2, sb2, sg2, o, ws,
                                    router_w=inp["router_w"], router_logits=lg,
                                    router_bias=inp["router_bias"], topk_ids_out=ids,
                                    topk_w_out=tw)
        else:
            M.moe_ffn_forward(shape, xi, inp["norm_w"], w13, w2, o, ws, router_w=inp["router_w"],
                              router_logits=lg, router_bias=inp["router_bias"],
                              w13_scale=s13, w2_scale=s2, topk_ids_out=ids, topk_w_out=tw)

    # ---- region A: the product call, device-resident inputs
    for _ in range(warmup):
        fwd()
    torch.cuda.synchronize()
    offsets_np = None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    lc0 = M.lib.moe_launch_count()  # the library's own host-side launch counter
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(st)
        fwd()
        ev[i][1].record(st)
    torch.cuda.synchronize()
    launches_timed = M.lib.moe_launch_count() - lc0
    wall_a = time.perf_counter() - t_wall
    step_ms = [a.elapsed_time(b) for a, b in ev]
    # keep the same load for a moment so the clock sampler sees it
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < max(0.0, 1.5 - wall_a):
        fwd()
        torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    mean_ms = sum(step_ms) / len(step_ms)
    mean_ms = max_over_ranks(mean_ms, world)
    value = world * T / (mean_ms * 1e-3)

    # ---- region B: the same kernels through the step entry points, with
    # events around each stage (per-kernel durations for the roofline)
    xhat = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    xq = torch.empty((T, H), dtype=torch.uint8, device=dev) if fp8 else None
    hs = H // 128 if fb else 1  # activation scales per row
    xs = torch.empty((T, hs), dtype=torch.float32, device=dev).squeeze(1) if fp8 else None
    rws = M.alloc_workspace(max(256, M.moe_route_workspace_size(T, H, E)), dev)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=dev)
    row_src = torch.empty((R,), dtype=torch.int32, device=dev)
    rop = torch.empty((R,), dtype=torch.int32, device=dev)
    xp = torch.empty((R, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    xps = torch.empty((R, hs), dtype=torch.float32, device=dev).squeeze(1) if fp8 else None
    act = torch.empty((R, I), dtype=torch.bfloat16, device=dev)
    actq = torch.empty((R, I), dtype=torch.uint8, device=dev) if fp8 else None
    if fb:
        # the scale rows are gathered like the code rows (a second permute
        # call moves them as rows of H/128 fp32 values)
        assert (hs * 4) % 16 == 0, "block-wise FP8 stage path needs H % 512 == 0"
        pxs = torch.empty((R,), dtype=torch.int32, device=dev)
    acts = torch.empty((R,), dtype=torch.float32, device=dev) if fp8 else None
    y = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    pws = M.alloc_workspace(max(256, M.moe_permute_workspace_size(T, E, k)), dev)
    out_b = torch.empty_like(out)
    # The decode engine with bf16 weights runs FC1 and FC2 in one fused launch:
    # time that launch (moe_grouped_ffn) as one stage; otherwise FC1 and FC2.
    fused = nvfp4 or fb or ((T * k / E <= 96.0) and os.environ.get("MOE_FUSE", "1") != "0")
    xp16 = torch.empty((R, H), dtype=torch.float16, device=dev) if nvfp4 else None
    act16 = torch.empty((R, I), dtype=torch.float16, device=dev) if nvfp4 else None
    fws = M.alloc_workspace(max(256, M.moe_grouped_ffn_workspace_size(shape)), dev)
    stages = (["rmsnorm", "route", "permute", "ffn", "combine"] if fused else
              ["rmsnorm", "route", "permute", "fc1", "quant", "fc2", "combine"] if fp8 else
              ["rmsnorm", "route", "permute", "fc1", "fc2", "combine"])

    def step_b(evs=None):
        def mark(i):
            if evs is not None:
                evs[i].record(st)
        mark(0)
        if fb:
            M.moe_rmsnorm(inp["x"], inp["norm_w"], inp["eps"], xhat)
            M.moe_quantize_fp8_blocks(xhat, xq, xs, 1)
        else:
            M.moe_rmsnorm(inp["x"], inp["norm_w"], inp["eps"], xhat, xq, xs)
        mark(1)
        M.moe_route_topk(T, H, E, k, ids, tw, xhat=xhat, router_w=inp["router_w"],
                         router_bias=inp["router_bias"], logits_in=inp["router_logits"],
                         workspace=rws)
        mark(2)
        if fb:
            M.moe_permute(ids, T, E, k, offsets, row_src, rop, xhat=xq, xp=xp, row_bytes=H,
                          workspace=pws)
            M.moe_permute(ids, T, E, k, offsets, row_src, pxs, xhat=xs, xp=xps,
                          row_bytes=hs * 4, workspace=pws)
        else:
            M.moe_permute(ids, T, E, k, offsets, row_src, rop, xhat=xq if fp8 else xhat, xp=xp,
                          row_bytes=H * (1 if fp8 else 2), xscale=xs, xp_scale=xps, workspace=pws)
        if nvfp4:
            xp16.copy_(xp)   # fp16 rows for the NVFP4 FFN step (counted in the permute stage)
        mark(3)
        if nvfp4:
            (q13, sb13, sg13), (q2, sb2, sg2) = nv
            M.moe_grouped_ffn_nvfp4(shape, xp16, q13, sb13, sg13, q2, sb2, sg2, offsets, row_src,
                                    tw, act16, y, fws)
        elif fused:
            M.moe_grouped_ffn(shape, xp, w13, w2, offsets, row_src, tw, actq if fb else act, y, fws,
                              xp_scale=xps, w13_scale=s13, w2_scale=s2)
        else:
            M.moe_grouped_gemm(shape, M.GEMM_FC1_SILU, xp, w13, offsets, act, a_scale=xps,
                               w_scale=s13)
            mark(4)
            if fp8:
                M.lib.moe_quantize_fp8_rows(act.data_ptr(), R, I, actq.data_ptr(),
                                            acts.data_ptr(), st.cuda_stream)
                mark(5)
            M.moe_grouped_gemm(shape, M.GEMM_FC2_BF16, actq if fp8 else act, w2, offsets, y,
                               a_scale=acts, w_scale=s2, row_src=row_src, topk_w=tw)
        mark(len(stages) - 1)
        M.moe_combine(y, rop, T, k, out_b, pair_order=True)
        mark(len(stages))

    for _ in range(warmup):
        step_b()
    torch.cuda.synchronize()
    fwd()
    torch.cuda.synchronize()
    same = bool(torch.equal(out, out_b)) if warmup > 0 else None
    evs_all = []
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
        step_b(evs)
        evs_all.append(evs)
    torch.cuda.synchronize()
    stage_ms = {s: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs_all)
                for i, s in enumerate(stages)}
    offsets_np = offsets.cpu().numpy()
    work = algorithmic_work(dict(inp, fp8=fp8, nvfp4=nvfp4), offsets_np)
    peaks = load_peaks()
    # a contraction takes the peak of its own dtype: E4M3 = measured bf16 x the
    # nominal fp8 / bf16 dense ratio (4.5 / 2.25 = 2)
    tmul = 2.0 if fp8 else 1.0
    tpeak, tpeak_sus = peaks["bf16_tflops"] * tmul, peaks["bf16_tflops_sustained"] * tmul
    tsrc = peaks["source"] + (" bf16 x nominal fp8/bf16 ratio 2" if fp8 else "")
    decode = T <= 64
    if decode and fused:
        ffn_bytes = work["fc1_bytes"] + work["fc2_bytes"]
        achieved = ffn_bytes / (stage_ms["ffn"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": read_traffic("ffn", traffic_key),
                "kernel": "fused decode FFN (FC1 + silu_and_mul + FC2 + routing weight, one launch)",
                "peak_source": peaks["source"],
                "frac_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS,
                "algorithmic_bytes_per_launch": ffn_bytes}
    elif decode:
        achieved = work["fc1_bytes"] / (stage_ms["fc1"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": read_traffic("fc1", traffic_key),
                "kernel": "grouped GEMM FC1 + silu_and_mul",
                "peak_source": peaks["source"],
                "frac_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS,
                "fc2_GBs": work["fc2_bytes"] / (stage_ms["fc2"] * 1e-3) / 1e9,
                "ffn_GBs": (work["fc1_bytes"] + work["fc2_bytes"]) /
                           ((stage_ms["fc1"] + stage_ms["fc2"]) * 1e-3) / 1e9,
                "algorithmic_bytes_per_launch": work["fc1_bytes"]}
    elif fused:
        # block-wise FP8 at prefill sizes: one moe_grouped_ffn call, three
        # launches (FC1 tiles, the intermediate's group quantiser, FC2 tiles)
        flops = work["fc1_flops"] + work["fc2_flops"]
        achieved = flops / (stage_ms["ffn"] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                "frac": achieved / tpeak, "traffic": read_traffic("ffn", traffic_key),
                "kernel": "block-wise FP8 FFN: FC1 tiles + silu_and_mul, 1x128 group quantiser, "
                          "FC2 tiles + routing weight (three launches timed together)",
                "peak_source": tsrc, "frac_of_sustained": achieved / tpeak_sus,
                "algorithmic_flops_per_launch": flops,
                "weight_GBs": (work["fc1_bytes"] + work["fc2_bytes"]) / (stage_ms["ffn"] * 1e-3) / 1e9}
    else:
        dom = "fc1"
        achieved = work["fc1_flops"] / (stage_ms["fc1"] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tpeak,
                "unit": "TFLOP/s", "frac": achieved / tpeak,
                "traffic": read_traffic("fc1", traffic_key),
                "kernel": "grouped GEMM FC1 + silu_and_mul", "peak_source": tsrc,
                "frac_of_sustained": achieved / tpeak_sus,
                "fc2_TFLOPs": work["fc2_flops"] / (stage_ms["fc2"] * 1e-3) / 1e12,
                "ffn_TFLOPs": (work["fc1_flops"] + work["fc2_flops"]) /
                              ((stage_ms["fc1"] + stage_ms["fc2"]) * 1e-3) / 1e12,
                "algorithmic_flops_per_launch": work["fc1_flops"]}
        roof["fc2_frac"] = roof["fc2_TFLOPs"] / tpeak
        roof["ffn_frac"] = roof["ffn_TFLOPs"] / tpeak

    # ---- e2e: host buffers in, host buffer out, copies inside the timed region.
    # Every step uploads its inputs from pinned host memory, runs the forward
    # and downloads its output to pinned host memory.  Uploads and downloads
    # run on their own streams with two device buffers each way, ordered by
    # events, so step i+1's upload and step i-1's download overlap step i's
    # forward (as a serving loop would run them).  For forwards under 0.1 ms
    # (the tiny workload) the cross-stream hand-offs cost more than they hide,
    # and the steps run on the compute stream alone.
    x_h = inp["x"].cpu().pin_memory()
    lg_h = inp["router_logits"].cpu().pin_memory() if inp["router_logits"] is not None else None
    out_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(inp["x"]) for _ in range(2)]
    lg_d = [torch.empty_like(inp["router_logits"]) if lg_h is not None else None for _ in range(2)]
    out_d = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_fwd = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]

    overlap = mean_ms >= 0.1

    def e2e_step(i):
        b = i & 1
        if not overlap:
            x_d[b].copy_(x_h, non_blocking=True)
            if lg_h is not None:
                lg_d[b].copy_(lg_h, non_blocking=True)
            fwd(x=x_d[b], out_=out_d[b], logits=lg_d[b])
            out_h[b].copy_(out_d[b], non_blocking=True)
            ev_down[b].record(st)
            return
        if i >= 2:
            up.wait_event(ev_fwd[b])      # forward i-2 has read x_d[b]
        with torch.cuda.stream(up):
            x_d[b].copy_(x_h, non_blocking=True)
            if lg_h is not None:
                lg_d[b].copy_(lg_h, non_blocking=True)
            ev_up[b].record(up)
        st.wait_event(ev_up[b])
        if i >= 2:
            st.wait_event(ev_down[b])     # download i-2 has read out_d[b]
        fwd(x=x_d[b], out_=out_d[b], logits=lg_d[b])
        ev_fwd[b].record(st)
        down.wait_event(ev_fwd[b])
        with torch.cuda.stream(down):
            out_h[b].copy_(out_d[b], non_blocking=True)
            ev_down[b].record(down)

    for i in range(warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    up.wait_event(e0)
    for i in range(steps):
        e2e_step(i)
    st.wait_event(ev_down[(steps - 1) & 1])
    e1.record(st)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    e2e_same = bool(torch.equal(out_h[(steps - 1) & 1], out.cpu()))
    h2d = x_h.numel() * 2 + (lg_h.numel() * 4 if lg_h is not None else 0)
    d2h = out_h[0].numel() * 2

    cpu = None
    if rank == 0 and world == 1 and cpu_ok and not args.no_cpu_baseline:
        n = args.cpu_tokens or auto_cpu_tokens(workload)
        # FP8 workloads: the oracle gets the bf16 originals and quantises them itself
        tps, secs, desc = run_oracle_sample(inp, n)
        cpu = {"value": tps, "unit": "tokens/s", "cores": 1, "host_cores": os.cpu_count(),
               "kind": "oracle", "sample": desc, "seconds": secs}
    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": steps, "warmup": warmup, "ms_per_step": mean_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("fp16 x fp16 -> f32 (NVFP4 weights dequantised exactly, bf16 activations)"
                      if nvfp4 else
                      "fp8-e4m3 x fp8-e4m3 -> f32 per 128-wide K group, scaled and summed in f32"
                      if fb else "fp8-e4m3 x fp8-e4m3 -> f32" if fp8 else "bf16 x bf16 -> f32"),
            "data": "synthetic (seeded torch generator; random-init weights)",
            "config": {"workload": workload + ("" if shape_over is None else " (reduced shape)"),
                       "T": T, "H": H, "E": E, "top_k": k, "I": I,
                       "fp8": fp8,
                       "weights": ("nvfp4" if nvfp4 else "e4m3, 128x128 tile scales" if fb else
                                   ("e4m3" if fp8 else "bf16")),
                       "routing": inp["routing"],
                       "active_experts": work["active_experts"],
                       "l2": ("flushed between steps (512 MB write)" if flush is not None else
                              f"inputs larger than L2: expert weights "
                              f"{wbytes / 1e9:.2f} GB"),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof,
            "stages_ms": stage_ms,
            "stage_path_equals_forward": same,
            "e2e": {"value": world * T / (e2e_ms * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "copies": ("upload and download streams, two device buffers each way"
                               if overlap else "on the compute stream (forward under 0.1 ms)"),
                    "output_equals_forward": e2e_same},
            "gpu_launches": launches_timed,
            "launches_per_step": launches_timed / steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "wall_s_region_a": wall_a,
        }
    del inp, ws
    torch.cuda.empty_cache()
    return line


# Workloads measured after the headline one in a default single-GPU run: the
# prefill (T = 4096) half of the metric, bf16 and FP8 W8A8.
MORE_WORKLOADS = ("c5_prefill", "c8_prefill_fp8")
MORE_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "dtype", "config", "roofline",
             "stages_ms", "e2e", "clocks", "launches_per_step", "stage_path_equals_forward")


def main_native(args):
    import torch
    rank, world, local = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import moe_expert_ffn_rms_gb300 as M
    M.check_device()
    line = run_workload(args, args.workload, dev, rank, world, local, args.steps, args.warmup,
                        cpu_ok=True)
    if rank == 0 and line is not None and line["roofline"]["bound"] == "hbm":
        # The measured HBM peak is a copy (read + write bytes counted); a
        # decode FFN only reads, and a read stream can run a little faster
        # than a copy, so the fraction can read slightly above 1.  The
        # fraction of the nominal 8 TB/s sits beside it.
        line["roofline"]["peak_kind"] = "copy bandwidth (read + write bytes), measured"
    more = [w for w in MORE_WORKLOADS if w != args.workload] if (
        world == 1 and args.workload == DEFAULT_WORKLOAD and not args.no_more and
        not args.shape) else []
    if more and rank == 0:
        line["more"] = {}
        for w in more:
            sub = run_workload(args, w, dev, rank, world, local, min(args.steps, 100),
                               max(3, min(args.warmup, 10)), cpu_ok=False)
            line["more"][w] = {k: sub[k] for k in MORE_KEYS if k in sub}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def kernel_source_sha(workload):
    """sha256 (12 hex digits) of the source that defines the workload's GEMM
    kernel: its .cu file and the device headers it includes."""
    import hashlib
    import workloads
    cfg = workloads.CONFIGS[workload]
    src = os.path.join(ROOT, "moe_expert_ffn_rms_gb300", "csrc")
    main = ("gemm_nvfp4.cu" if cfg.nvfp4 else "gemm_fp8b.cu" if cfg.fp8 == "block" else
            "gemm_tc.cu")
    h = hashlib.sha256()
    for fn in [main] + sorted(f for f in os.listdir(src) if f.endswith(".cuh")):
        h.update(open(os.path.join(src, fn), "rb").read())
    return h.hexdigest()[:12]


def read_traffic(kernel, workload):
    """DRAM traffic per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    import workloads
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p) or workload is None or workload not in workloads.CONFIGS:
        return None
    sha = kernel_source_sha(workload)
    with open(p) as f:
        for ln in f:
            parts = ln.split()
            if len(parts) >= 4 and not ln.startswith("#") and parts[0] == kernel and \
                    parts[1] == workload and parts[2] == sha:
                return float(parts[3])
    return None


if __name__ == "__main__":
    if len(sys.argv) == 3 and sys.argv[1] == "--kernel-sha":
        print(kernel_source_sha(sys.argv[2]))
        sys.exit(0)
    a = parse()
    if a.impl == "reference":
        main_reference(a)
    else:
        main_native(a)
