#!/usr/bin/env python3
"""Throughput of the single-GPU MoE layer (tokens/s, TFLOP/s, % of peak).

One step = one forward pass of the whole layer over one batch of synthetic
tokens: route -> plan -> dispatch -> grouped up/gate + SwiGLU -> grouped
down -> combine (the shared expert's tiles run inside the two grouped
launches), every kernel launched through the C ABI
of libmok.so on the current stream (the same kernels, in the same order, as
one mok_moe_fwd call).  The default workload is the DSV3-shaped BF16
forward (T 7168, D 7168, I 2048, 256 experts top-8 + one shared expert,
I 2048).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config NAME]

N > 1 runs under torch.distributed (one process per GPU, NCCL barrier and a
MAX reduction of the timed region): independent replicas, each on its own
tokens, no collective on the data path ("scaling": "weak").

--impl reference times the CPU oracle (oracle/, numpy) on the host cores on
a bounded sample of the same workload and prints the same JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
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
import torch  # noqa: E402

from routing_grouped_expert_device_gb300 import workloads as W  # noqa: E402

METRIC = "MoE layer fwd/bwd tokens/s and TFLOP/s (% dense tensor peak), 1×GB300"
KERNEL_SOURCES = ["common.cuh", "gemm_core.cuh", "pair.cuh", "gemm_pair.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "upgate_gemm_dsv3_bf16_fwd_traffic.txt")
NOMINAL_BF16_TFLOPS = 2250.0  # GB300 dense bf16 datasheet figure (no 2:4 sparsity)


# ---------------------------------------------------------------------------
def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=30)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="dsv3_bf16_fwd")
    p.add_argument("--cpu-slice-experts", type=int, default=0,
                   help="experts in the cpu_baseline slice (0 = a per-workload default)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--chunk-rows", type=int, default=0,
                   help="BF16 forward: gather through a ring of chunks of this many routed rows "
                        "(512..32768; -1 = whole-batch dispatch; 0 = as mok_moe_fwd chooses: the ring "
                        "with 2048-row chunks for layers of 512 or more routed rows per expert, else "
                        "the whole-batch dispatch)")
    p.add_argument("--producer-sms", type=int, default=0,
                   help="SMs left to route, plan and the dispatch while the shared expert's up/gate "
                        "runs on the others (mok_shape.producer_sms; 0 = the shared expert takes every SM)")
    p.add_argument("--bwd-shared-sms", type=int, default=0,
                   help="fwd+bwd: SMs the shared expert's backward takes on a side stream while the routed "
                        "dgrad and dX run on the others (mok_shape.bwd_shared_sms; 0 = no side stream, which "
                        "measured fastest)")
    p.add_argument("--mx-pair-scales", action="store_true",
                   help="MXFP8: give the paired W_up / W_gate scale blocks, so that the up/gate takes the "
                        "routed rows as N (measured slower than the row-major up/gate on GB300)")
    p.add_argument("--act-rows", type=int, default=-1,
                   help="fwd+bwd: rows of the forward's kept h, u store (-1 = every routed row, and the "
                        "shared expert's h, u kept too; "
                        "0 = none: the backward replays every expert)")
    p.add_argument("--protocol-warmup", type=int, default=500,
                   help="the pages' protocol: warm-up calls of the public entry point")
    p.add_argument("--protocol-runs", type=int, default=100,
                   help="the pages' protocol: timed calls (median reported)")
    return p.parse_args()


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device: str = "cuda") -> float:
    """The slowest rank's time: the job ends when its last replica does."""
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank_step: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput of N replicas: every rank's tokens over the
    slowest rank's time (weak scaling: per-rank work is fixed)."""
    return world * tokens_per_rank_step * steps / (max_ms / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sustained=d.get("bf16_tflops_sustained"),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.3)

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
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------------------
def source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "routing_grouped_expert_device_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(cfg_name: str):
    """DRAM bytes per launch of the up/gate kernel from the committed ncu
    summary, if it was taken on the current kernel source and workload."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    kv = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("source_sha256") != source_hash() or kv.get("workload") != cfg_name:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


# ---------------------------------------------------------------------------
class OracleSlice:
    """The CPU oracle on a batched slice of the workload (host cores).

    A slice is every routed row of a few experts of the full workload, plus
    the shared expert on the same fraction of the tokens: per expert the
    oracle's own per-expert steps as the layer functions run them (the
    bf16 -> fp32 weight conversion inside, MXFP8 quantisation of the weights
    and rows for MXFP8 experts, the SwiGLU FFN; for fwd+bwd also the
    backward of those rows and the expert's weight gradients).  Routing is
    computed once beforehand.  Its work is scaled to layer tokens by FLOPs:
    tokens = T * slice FLOPs / layer FLOPs."""

    def __init__(self, cfg, d):
        import oracle as O
        self.O, self.cfg = O, cfg
        self.mx = cfg.dtype == "mxfp8"
        s_host = d["s"].cpu().numpy()
        self.idx, self.g, _ = O.route(s_host, cfg.K)
        self.counts = np.bincount(self.idx.reshape(-1), minlength=cfg.E)
        self.nonempty = [int(e) for e in np.flatnonzero(self.counts)]
        self.x = W.bf16_bits(d["x"])
        self.dy = W.bf16_bits(d["dy"]) if cfg.backward else None
        self.d = d
        self.shared = None
        if cfg.I_shared:
            self.shared = (W.bf16_bits(d["ws_gate"]), W.bf16_bits(d["ws_up"]), W.bf16_bits(d["ws_down"]))
        self.layer_flops = cfg.fwd_flops() + (cfg.bwd_flops() if cfg.backward else 0.0)

    def weights(self, e):
        d = self.d
        return W.bf16_bits(d["w_gate"][e]), W.bf16_bits(d["w_up"][e]), W.bf16_bits(d["w_down"][e])

    def _expert(self, rows, g_rows, wts, shared=False):
        O, cfg = self.O, self.cfg
        mx = self.mx and not shared
        if mx:
            O.expert_ffn_rows_mxfp8(self.x[rows], *wts)
        else:
            O.expert_ffn_rows(self.x[rows], *wts)
        if cfg.backward:
            fn = O.route_backward_rows_mxfp8 if mx else O.route_backward_rows
            b = fn(self.x[rows], self.dy[rows], g_rows, *wts)
            X = O.bf16_to_f32(self.x[rows])
            dY = O.bf16_to_f32(self.dy[rows])
            O.round_bf16(dY.T @ b["a_g"])
            O.round_bf16(b["dh"].T @ X)
            O.round_bf16(b["du"].T @ X)

    def run(self, experts):
        """Time the slice of the given experts: (layer tokens, seconds)."""
        cfg = self.cfg
        jobs = []
        for e in experts:
            hit = self.idx == e
            rows = np.flatnonzero(hit.any(1))
            jobs.append((rows, self.g[hit], self.weights(e)))  # host copies before the clock starts
        routed = sum(len(r) for r, _, _ in jobs)
        n_sh = 0
        if self.shared is not None:
            n_sh = max(1, round(cfg.T * len(experts) / max(1, len(self.nonempty))))
        t0 = time.perf_counter()
        for rows, g_rows, wts in jobs:
            self._expert(rows, g_rows, wts)
        if n_sh:
            self._expert(np.arange(n_sh), np.ones(n_sh, np.float32), self.shared, shared=True)
        dt = time.perf_counter() - t0
        per = 3.0 if cfg.backward else 1.0  # backward = twice the forward
        flops = per * (6.0 * routed * cfg.D * cfg.I + 6.0 * n_sh * cfg.D * cfg.I_shared)
        return cfg.T * flops / self.layer_flops, dt

    def describe(self, experts, dt):
        cfg = self.cfg
        what = ("MXFP8 " if self.mx else "") + ("forward+backward incl. weight gradients" if cfg.backward
                                                else "forward")
        sh = " + the shared expert on the same fraction of tokens" if self.shared is not None else ""
        return (f"all routed rows of {len(experts)} of {len(self.nonempty)} non-empty experts of {cfg.name}{sh}, "
                f"oracle {what}, {dt:.1f} s; scaled to layer tokens by FLOPs")


def slice_experts(sl, n, seed=0):
    rng = np.random.default_rng(seed)
    return [int(e) for e in rng.choice(sl.nonempty, min(n, len(sl.nonempty)), replace=False)]


# experts per cpu_baseline slice (about 10-30 s on 16 host cores; all of
# them for the BF16 forwards, which is then the whole layer)
CPU_SLICE_EXPERTS = {("bf16", False): 256, ("bf16", True): 64, ("mxfp8", False): 16, ("mxfp8", True): 6}


def roofline_of(cfg, nonempty: int, part_ms: float, peaks: dict, capped: bool, chunk_rows: int = 0,
                traffic=None):
    """The roofline object of the bench line for the timed kernel (the routed
    up/gate launch of a forward, the whole mok_moe_bwd call of fwd+bwd):
    algorithmic bytes and FLOPs per launch, its bound (arithmetic intensity
    against the ridge point of the measured peaks), achieved / peak / frac
    against that bound, and the other figure beside it.  Returns
    (roofline, tensor_peak, burst_peak, bf16_peak) in TFLOP/s."""
    mx = cfg.dtype == "mxfp8"
    ring = chunk_rows > 0
    T, D, I, Is, R = cfg.T, cfg.D, cfg.I, cfg.I_shared, cfg.R
    bf16_peak = peaks["bf16_sustained"] if (capped and peaks.get("bf16_sustained")) else peaks["bf16"]
    # fp8 dense rate is twice bf16 on this part (nominal 4.5 vs 2.25 PFLOP/s)
    tensor_peak = bf16_peak * (2.0 if mx else 1.0)
    burst_peak = peaks["bf16"] * (2.0 if mx else 1.0)
    wbytes = 1 if mx else 2  # bytes per weight / activation element on the routed path
    if cfg.backward:
        # the whole backward call: ideal bytes = every weight read once (the
        # routed ones as fp8 codes + scales for MXFP8) + every weight
        # gradient written once (bf16) + x, dY, dX
        wread = nonempty * 3 * I * D * (wbytes + (1 / 32 if mx else 0.0)) + 3 * Is * D * 2
        alg_bytes = int(wread + (nonempty * 3 * I * D + 3 * Is * D) * 2 + 3 * T * D * 2)
        kernel = "backward (mok_moe_bwd: gathers, dgrad+replay, dx, combine, wgrad, router grad)"
        part_flops = cfg.bwd_flops()
    else:
        # grouped up/gate + SwiGLU: each expert's W_gate/W_up tile is read once
        # per 128..256 routed rows
        scale_b = (1 / 32) if mx else 0.0
        # (with the ring: x read once instead of xg; the ring itself stays on chip)
        alg_bytes = int(nonempty * 2 * I * D * wbytes * (1 + scale_b) + (T if ring else R) * D * wbytes * (1 + scale_b)
                        + R * I * wbytes * (1 + scale_b))
        part_flops = 4.0 * R * D * I
        kernel = (f"grouped up/gate + SwiGLU GEMM (tcgen05 cta_group::2"
                  f"{', MXFP8 block-scaled' if mx else ''}, routed experts"
                  f"{f', ring dispatch in the same launch, chunk {chunk_rows} rows' if ring else ''})")
    part_tflops = part_flops / (part_ms / 1e3) / 1e12
    achieved = alg_bytes / (part_ms / 1e3) / 1e9
    if ring:
        traffic = None
    intensity = part_flops / alg_bytes
    ridge = tensor_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if intensity > ridge:
        roofline = {"kernel": kernel, "bound": "tensor", "achieved": round(part_tflops, 1), "peak": tensor_peak,
                    "unit": "TFLOP/s", "frac": round(part_tflops / tensor_peak, 4), "traffic": traffic,
                    "gbs": round(achieved, 1), "hbm_frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        roofline = {"kernel": kernel, "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                    "tflops": round(part_tflops, 1), "tensor_frac": round(part_tflops / tensor_peak, 4)}
    roofline.update({"algorithmic_bytes": alg_bytes, "algorithmic_flops": part_flops,
                     "intensity_flop_per_byte": round(intensity, 1), "ridge_flop_per_byte": round(ridge, 1),
                     "avg_launch_ms": round(part_ms, 4), "peak_source": peaks["source"]})
    return roofline, tensor_peak, burst_peak, bf16_peak


# ---------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    from routing_grouped_expert_device_gb300 import mok as M
    M._lib_handle()
    cfg = W.CONFIGS[args.config]
    mx = cfg.dtype == "mxfp8"
    dev = torch.device("cuda", torch.cuda.current_device())
    d = W.make_inputs(cfg, dev, seed=rank)
    T, D, I, E, K, Is, R = cfg.T, cfg.D, cfg.I, cfg.E, cfg.K, cfg.I_shared, cfg.R
    # the gather of mok_moe_fwd's automatic choice (chunk_rows 0): the ring
    # of 2048-row chunks where the GEMMs run row-major tiles (512 or more
    # routed rows per expert), else the whole-batch dispatch
    ring = not mx and not cfg.backward and (args.chunk_rows > 0 or (args.chunk_rows == 0 and R >= 512 * E))
    chunk = args.chunk_rows if args.chunk_rows > 0 else 2048
    shape = M.shape_of(cfg, chunk_rows=chunk if ring else (args.chunk_rows if cfg.backward else -1),
                       producer_sms=args.producer_sms,
                       bwd_shared_sms=args.bwd_shared_sms)
    i32, f32, bf, u8 = torch.int32, torch.float32, torch.bfloat16, torch.uint8
    if mx:
        # weights are model parameters: quantised once, outside the timed region
        for name, key in (("gate", "w_gate"), ("up", "w_up"), ("down", "w_down")):
            wt = d[key].reshape(-1, d[key].shape[-1])
            q = torch.empty(wt.shape, dtype=u8, device=dev)
            sc = torch.empty(M.mx_scale_words(*wt.shape), dtype=i32, device=dev)
            M.quantize_mxfp8(wt, q, sc)
            d["q_" + name], d["sc_" + name] = q, sc
        if args.mx_pair_scales:
            # the paired W_up / W_gate scale blocks: the up/gate with the routed rows as N
            d["sc_gu_pair"] = torch.empty(M.mx_scale_words(2 * E * I, D), dtype=i32, device=dev)
            M.mxfp8_pair_scales(shape, M.make_weights(d), d["sc_gu_pair"])
        if cfg.backward:
            # the backward's copies: W_down^T along D, [W_gate^T | W_up^T] along 2I
            d["qt_down"] = torch.empty(E * I, D, dtype=u8, device=dev)
            d["sct_down"] = torch.empty(M.mx_scale_words(E * I, D), dtype=i32, device=dev)
            d["qt_gu"] = torch.empty(E * D, 2 * I, dtype=u8, device=dev)
            d["sct_gu"] = torch.empty(M.mx_scale_words(E * D, 2 * I), dtype=i32, device=dev)
            M.quantize_mxfp8_bwd_weights(shape, M.make_weights(d), d["qt_down"], d["sct_down"], d["qt_gu"],
                                         d["sct_gu"])
        torch.cuda.synchronize()
    w = M.make_weights(d)
    topk = torch.empty(T, K, dtype=i32, device=dev)
    g = torch.empty(T, K, dtype=f32, device=dev)
    counts = torch.empty(E, dtype=i32, device=dev)
    offsets = torch.empty(E + 1, dtype=i32, device=dev)
    table = torch.empty(R, 3, dtype=i32, device=dev)
    route_dst = torch.empty(R, dtype=i32, device=dev)
    pws = torch.empty(M.workspace_bytes(shape, M.OP_PLAN), dtype=u8, device=dev)
    xg = None if ring else torch.empty(R, D, dtype=u8 if mx else bf, device=dev)
    rws = torch.empty(M.workspace_bytes(shape, M.OP_RING), dtype=u8, device=dev) if ring else None
    xs = torch.empty(M.mx_scale_words(R, D, E), dtype=i32, device=dev) if mx else None
    a = torch.empty(R, I, dtype=u8 if mx else bf, device=dev)
    asc = torch.empty(M.mx_scale_words(R, I, E), dtype=i32, device=dev) if mx else None
    yg = torch.empty(R, D, dtype=bf, device=dev)
    ys = torch.empty(T, D, dtype=bf, device=dev) if Is else None
    a_s = torch.empty(T, Is, dtype=bf, device=dev) if Is else None
    out = torch.empty(T, D, dtype=bf, device=dev)
    stream = torch.cuda.current_stream()
    # route, plan (3), dispatch, up/gate, down, combine; the shared expert's
    # up/gate (BF16) or whole FFN (MXFP8) on the side stream
    launches_per_step = 1 + 3 + (0 if ring else 1) + 1 + 1 + 1 + ((2 if mx else 1) if Is else 0)
    side = torch.cuda.Stream() if Is else None
    sws = torch.empty(M.workspace_bytes(shape, M.OP_SHARED_FFN), dtype=u8, device=dev) if (Is and mx) else None

    if cfg.backward:
        bws = torch.empty(max(M.workspace_bytes(shape, M.OP_FWD), M.workspace_bytes(shape, M.OP_BWD)),
                          dtype=u8, device=dev)
        saved = dict(topk_idx=topk, g=g, counts=counts, offsets=offsets, table=table, route_dst=route_dst)
        act_rows = R if args.act_rows < 0 else min(args.act_rows, R)
        if act_rows > 0:
            # the forward keeps h, u (fp32) of the experts that fit, and the
            # shared expert's; the backward replays only the others
            saved["act"] = torch.empty(act_rows, 2 * I, dtype=f32, device=dev)
            if Is:
                saved["act_shared"] = torch.empty(T, 2 * Is, dtype=f32, device=dev)
        pb = M.make_plan_buf(saved)
        gr = dict(dx=torch.empty(T, D, dtype=bf, device=dev), dw_gate=torch.empty(E, I, D, dtype=bf, device=dev),
                  dw_up=torch.empty(E, I, D, dtype=bf, device=dev), dw_down=torch.empty(E, D, I, dtype=bf, device=dev),
                  dws_gate=torch.empty(Is, D, dtype=bf, device=dev) if Is else None,
                  dws_up=torch.empty(Is, D, dtype=bf, device=dev) if Is else None,
                  dws_down=torch.empty(D, Is, dtype=bf, device=dev) if Is else None,
                  ds=torch.empty(T, E, dtype=f32, device=dev), dg=torch.empty(T, K, dtype=f32, device=dev))
        # forward: route, plan (3), dispatch, up/gate, down, combine, the
        # shared expert's up/gate (BF16) or FFN (MXFP8); backward: gathers
        # (2), dgrad of the kept experts and / or dgrad with replay, dx
        # (BF16), or the quantising dispatch of dY (and of x with a replay),
        # the replay, t, activation gradient, dX (MXFP8); reverse combine,
        # 3 wgrad, router grad, and the shared expert's dgrad, dx and 3 wgrad
        all_kept = act_rows >= R
        some_kept = act_rows > 0
        bwd_routed = (4 if all_kept else 6) if mx else ((1 if all_kept else 2 if some_kept else 1) + 1)
        launches_per_step = ((1 + 3 + 1 + 2 + 1 + ((2 if mx else 1) if Is else 0))
                             + (2 + bwd_routed + 1 + 3 + 1 + (5 if Is else 0)))

    def step(ev0=None, ev1=None):
        if cfg.backward:
            M.moe_fwd(shape, w, d["x"], d["s"], out, bws, pb)
            if ev0 is not None:
                ev0.record(stream)
            M.moe_bwd(shape, w, d["x"], d["s"], pb, d["dy"], gr["dx"], gr["dw_gate"], gr["dw_up"],
                      gr["dw_down"], gr["dws_gate"], gr["dws_up"], gr["dws_down"], gr["ds"], gr["dg"], bws)
            if ev1 is not None:
                ev1.record(stream)
            return
        # the same schedule as mok_moe_fwd: the shared expert depends on x
        # alone and runs on a side stream next to route, plan and dispatch
        # (and, for MXFP8, the routed up/gate)
        if Is:
            side.wait_stream(stream)
            if mx:
                M.shared_ffn(shape, w, d["x"], ys, sws, stream=side)
            else:
                M.expert_upgate(shape, w, None, None, None, x_shared=d["x"], a_shared=a_s, stream=side)
        M.route(d["s"], K, topk, g)
        M.plan(topk, E, counts, offsets, table, route_dst, pws)
        if not ring:
            M.dispatch(shape, d["x"], table, route_dst, xg, xs, offsets=offsets)
        if Is and not mx and not ring:
            # as mok_moe_fwd: the BF16 routed up/gate waits for the shared up/gate
            stream.wait_stream(side)
        if ev0 is not None:
            ev0.record(stream)
        if ring:  # the dispatch runs inside the up/gate launch (producer warps, ring of chunks)
            M.expert_upgate_ring(shape, w, d["x"], table, offsets, a, rws)
        else:
            M.expert_upgate(shape, w, xg, offsets, a, xg_scale=xs, a_scale=asc)
        if ev1 is not None:
            ev1.record(stream)
        if Is:
            stream.wait_stream(side)
        # BF16: the shared expert's down tiles run inside the routed down launch
        M.expert_down(shape, w, a, offsets, yg, a_scale=asc, a_shared=None if mx else a_s,
                      ys=None if mx else ys)
        M.combine(shape, yg, ys, g, route_dst, out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    M.check_device_status()
    nonempty = int((counts > 0).sum().item())

    K_steps = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_steps)]
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t_start.record(stream)
    for i in range(K_steps):
        step(*evs[i])
    t_stop.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    M.check_device_status()
    total_ms = max_over_ranks(t_start.elapsed_time(t_stop), world)
    part_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    # schedule construction (route + plan) timed on its own: inside the step
    # it queues behind the shared expert's up/gate, whose launch holds every SM
    sched_ms = None
    if not cfg.backward:
        sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
        for e0, e1 in sev:
            e0.record(stream)
            M.route(d["s"], K, topk, g)
            M.plan(topk, E, counts, offsets, table, route_dst, pws)
            e1.record(stream)
        torch.cuda.synchronize()
        sched_ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in sev[5:])
    ms_step = total_ms / K_steps
    value = job_tokens_per_s(world, T, K_steps, total_ms)
    flops = cfg.fwd_flops() + (cfg.bwd_flops() if cfg.backward else 0.0)
    tflops = flops / (ms_step / 1e3) / 1e12
    peaks = measured_peaks()
    # A long timed region runs under the 1.4 kW power cap, so its peak is the
    # sustained cuBLAS figure (measured the same way); a short one that kept
    # the SM clock near its maximum is compared with the burst figure.
    ck = clk or {}
    capped = bool(ck.get("sm_mhz") and ck.get("sm_max_mhz") and ck["sm_mhz"] < 0.95 * ck["sm_max_mhz"])
    roofline, tensor_peak, burst_peak, bf16_peak = roofline_of(
        cfg, nonempty, part_ms, peaks, capped, chunk if ring else 0, recorded_traffic(cfg.name))

    # end to end through the public entry points with pinned host buffers:
    # every step copies its inputs in and reads its result back.  The copies
    # run on their own streams into two device slots, so step i+1's inputs
    # arrive and step i-1's result leaves while step i computes (the way a
    # serving loop drives the layer).
    ws = bws if cfg.backward else torch.empty(M.workspace_bytes(shape, M.OP_FWD), dtype=u8, device=dev)
    names_in = ["x", "s"] + (["dy"] if cfg.backward else [])
    host_in = {n: d[n].cpu().pin_memory() for n in names_in}
    host_out = {n: torch.empty(T, D, dtype=bf, pin_memory=True) for n in (["out", "dx"] if cfg.backward else ["out"])}
    slots = [{n: torch.empty_like(d[n]) for n in names_in} for _ in range(2)]
    for sl in slots:
        sl["out"] = torch.empty(T, D, dtype=bf, device=dev)
        if cfg.backward:
            sl["dx"] = torch.empty(T, D, dtype=bf, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(3, min(K_steps, 100))

    def e2e_step(i):
        j = i % 2
        sl = slots[j]
        if i >= 2:
            h2d_s.wait_event(free[j])  # step i-2 has read slot j and its result is out
        with torch.cuda.stream(h2d_s):
            for n in names_in:
                sl[n].copy_(host_in[n], non_blocking=True)
            in_ready[j].record(h2d_s)
        stream.wait_event(in_ready[j])
        if cfg.backward:
            M.moe_fwd(shape, w, sl["x"], sl["s"], sl["out"], ws, pb)
            M.moe_bwd(shape, w, sl["x"], sl["s"], pb, sl["dy"], sl["dx"], gr["dw_gate"], gr["dw_up"],
                      gr["dw_down"], gr["dws_gate"], gr["dws_up"], gr["dws_down"], gr["ds"], gr["dg"], ws)
        else:
            M.moe_fwd(shape, w, sl["x"], sl["s"], sl["out"], ws)
        done[j].record(stream)
        d2h_s.wait_event(done[j])
        with torch.cuda.stream(d2h_s):
            for n, h in host_out.items():
                h.copy_(sl[n], non_blocking=True)
            free[j].record(d2h_s)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_s.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(d2h_s)  # the last result is on the host
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
    M.check_device_status()
    e2e = {"value": round(world * T / (e2e_ms / 1e3), 1), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
           "copies": "H2D of step i+1 and D2H of step i-1 overlap step i (two device slots, copy streams)"}

    # the pages' protocol (paper note, "Results": median of 100 runs after
    # 500 warm-ups, schedule construction included): each call of the public
    # entry point (mok_moe_fwd, or mok_moe_fwd + mok_moe_bwd) on
    # device-resident inputs, timed alone with CUDA events
    def call():
        if cfg.backward:
            M.moe_fwd(shape, w, d["x"], d["s"], out, ws, pb)
            M.moe_bwd(shape, w, d["x"], d["s"], pb, d["dy"], gr["dx"], gr["dw_gate"], gr["dw_up"],
                      gr["dw_down"], gr["dws_gate"], gr["dws_up"], gr["dws_down"], gr["ds"], gr["dg"], ws)
        else:
            M.moe_fwd(shape, w, d["x"], d["s"], out, ws)

    for _ in range(args.protocol_warmup):
        call()
    pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.protocol_runs)]
    for e0, e1 in pev:
        e0.record(stream)
        call()
        e1.record(stream)
    torch.cuda.synchronize()
    M.check_device_status()
    per_call = sorted(e0.elapsed_time(e1) for e0, e1 in pev)
    med = max_over_ranks(per_call[len(per_call) // 2], world) if per_call else None
    protocol = None if med is None else {
        "warmup": args.protocol_warmup, "runs": args.protocol_runs, "median_ms": round(med, 4),
        "tokens_per_s": round(world * T / (med / 1e3), 1),
        "entry": "mok_moe_fwd + mok_moe_bwd" if cfg.backward else "mok_moe_fwd"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sl = OracleSlice(cfg, d)
        ex = slice_experts(sl, args.cpu_slice_experts or CPU_SLICE_EXPERTS[(cfg.dtype, cfg.backward)])
        toks, dt = sl.run(ex)
        cpu = {"value": round(toks / dt, 4), "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
               "sample": sl.describe(ex, dt)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": K_steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3+e8m0 (routed), bf16 (shared)" if mx else "bf16",
            "data": "synthetic (seeded; x~N(0,1), W~N(0,1/fan_in), logits~N(0,1) softmax; bf16)",
            "config": {"workload": cfg.name, "T": T, "D": D, "I": I, "E": E, "K": K, "I_shared": Is,
                       "global_batch": world * T, "parallelism": f"replicas x{world}",
                       "chunk_rows": chunk if ring else 0, "producer_sms": args.producer_sms,
                       "kept_act_rows": (act_rows if cfg.backward else None),
                       "bwd_shared_sms": (M.bwd_shared_sms(shape) if cfg.backward else None),
                       "l2": "inputs larger than L2: every step streams all expert weights "
                             f"({(nonempty * 3 * I * D + 3 * Is * D) * 2 / 1e9:.1f} GB)"},
            "tflops": round(tflops, 1), "tensor_frac": round(tflops / tensor_peak, 4),
            "tensor_peak": tensor_peak,
            "tensor_peak_source": peaks["source"] + (" sustained" if bf16_peak != peaks["bf16"] else " burst")
                                  + (" bf16 x 2 (fp8)" if mx else " bf16")
                                  + (" (SM clock below 95 % of max under load: power cap)" if capped else ""),
            "tensor_frac_burst": round(tflops / burst_peak, 4),
            # against the datasheet's dense peak (2.25 PFLOP/s bf16, 4.5 fp8)
            "tensor_frac_nominal": round(tflops / (NOMINAL_BF16_TFLOPS * (2.0 if mx else 1.0)), 4),
            "pass": "fwd+bwd" if cfg.backward else "fwd",
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "pages_protocol": protocol,
            "schedule_share": None if sched_ms is None else {
                "route_plan_ms": round(sched_ms, 4), "share": round(sched_ms / ms_step, 4),
                "pages": "under 3 % (blog), 2.1-7.7 % (note) of MoE runtime"},
            "gpu_launches": launches_per_step * K_steps, "clocks": clk,
        }
        print(json.dumps(line), flush=True)


def run_reference(args, world, rank, local):
    """The CPU oracle as the reference arm, on the host cores.  Each step is
    the oracle on every routed row of one expert of the workload (plus the
    shared expert on the same fraction of tokens), as OracleSlice runs it,
    cycling over the non-empty experts; its work counts as the layer tokens
    of the same FLOPs.  Only rank 0 works; other ranks exit."""
    if rank != 0:
        return
    cfg = W.CONFIGS[args.config]
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    d = W.make_inputs(cfg, dev, seed=0)
    sl = OracleSlice(cfg, d)
    order = slice_experts(sl, len(sl.nonempty), seed=1)
    for i in range(args.warmup):
        sl.run([order[i % len(order)]])
    toks = total = 0.0
    for i in range(args.steps):
        t, dt = sl.run([order[(args.warmup + i) % len(order)]])
        toks += t
        total += dt
    value = toks / total
    line = {
        "metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (oracle" + (", MXFP8 operands)" if cfg.dtype == "mxfp8" else ")"),
        "data": "synthetic (seeded)", "config": {"workload": cfg.name, "T": cfg.T, "D": cfg.D, "I": cfg.I,
                                                 "E": cfg.E, "K": cfg.K, "I_shared": cfg.I_shared},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": "per step: " + sl.describe([0], total / max(1, args.steps))},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        # the oracle runs on the host cores: rank 0 alone, no process group
        env = lambda k: int(os.environ.get(k, "0"))
        run_reference(args, max(1, env("WORLD_SIZE")), env("RANK"), env("LOCAL_RANK"))
        return
    world, rank, local = dist_setup(args.gpus)
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
