"""Benchmark of the sparse self-speculative decoding attention hot path on GB300.

One step = one speculative round of every layer of a synthetic multi-layer cache in the
Qwen3-8B attention shape (32 requests, lengths U[2048, 8192], 32/8 heads, d = 128, bf16, pages of
16 tokens, k = 4, top-K = 5%): for each layer verify (+ fused criticality) and Top-K select, then the
k drafts of every layer (draft j of all layers, then draft j+1).  The step is captured once in a
CUDA graph and replayed; each layer's KV (671 MB) is larger than L2 and the layers are cycled, so
no timed kernel finds its inputs in L2 from a previous use.

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU oracle instead, on a
bounded sample of the same workload.  Multi-GPU (torchrun): every rank runs its own independent
batch (weak scaling, no collective on the data path); timings are the max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import glob
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

import torch  # noqa: E402

from sparse_self_speculative_verify_gb300 import metrics as M  # noqa: E402
from sparse_self_speculative_verify_gb300 import workloads as W  # noqa: E402

METRIC = "spec-decode attention HBM GB/s (% of ~8 TB/s peak); verify+draft rounds/s"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "verify_qwen3_8b_traffic.json")


# --------------------------------------------------------------------------------------------
# Distributed helpers (host side; tested with gloo on CPU).
# --------------------------------------------------------------------------------------------


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws an independent batch of the same shape."""
    return base + 7919 * rank


def max_over_ranks(value: float, device=None) -> float:
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, device=None) -> float:
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------------------------------------
# Clock sampling during the timed region.
# --------------------------------------------------------------------------------------------

CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
                "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
                "clocks_event_reasons.sw_power_cap"]
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.gpu_id = gpu_id
        self.period_ms = period_ms
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--id={self.gpu_id}", "--query-gpu=" + ",".join(CLOCK_FIELDS),
               "--format=csv,noheader,nounits", "-lms", str(self.period_ms)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(CLOCK_FIELDS):
                self.rows.append((time.time(), parts))

    def stop(self, t_begin: float = 0.0, t_end: float = float("inf")) -> dict:
        """Stops sampling; summarises the samples taken between t_begin and t_end (host time)."""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        sm = []
        smax = None
        reasons = set()
        for ts, r in self.rows:
            if ts < t_begin or ts > t_end:
                continue
            try:
                sm.append(float(r[0]))
                smax = float(r[1])
            except ValueError:
                continue
            for name, v in zip(REASON_NAMES, r[3:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(device) -> str:
    try:
        u = torch.cuda.get_device_properties(device).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return str(torch.cuda.current_device())


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# Sources of the dominant calls (ssd_verify_select: tensor-core verify kernel + criticality/Top-K
# pass; ssd_verify_attn: verify kernel + finalize); a change to any of them makes the committed
# DRAM-traffic capture stale.
VERIFY_SOURCES = ("ssd_common.cuh", "ssd_finalize.cuh", "ssd_host.h", "ssd_sm100.cuh", "ssd_topk.cuh",
                  "ssd_verify.cu", "ssd_verify_tc.cu", "ssd_verify_tile.cuh")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for p in sorted(os.path.join(ROOT, "sparse_self_speculative_verify_gb300", "csrc", n) for n in VERIFY_SOURCES):
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(launch_units: int, call: str = "ssd_verify_select"):
    """DRAM bytes of one `call` (the sum over its kernels in the committed ncu summary), scaled from
    the capture's units to this launch's; None when the kernels changed since the capture or the
    capture lacks one of the call's kernels."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        d = json.load(f)
    if d.get("kernel_src_sha") != kernel_source_sha():
        return None
    kernels = d.get("calls", {}).get(call)
    if not kernels or any(k not in d.get("kernel_dram_bytes", {}) for k in kernels):
        return None
    return sum(d["kernel_dram_bytes"][k] for k in kernels) / d["units"] * launch_units


# --------------------------------------------------------------------------------------------
# Workload.
# --------------------------------------------------------------------------------------------


def make_layers(spec, n_layers: int, seed: int, device):
    """n_layers independent caches of the same requests (shared lengths, own pages and values)."""
    first = W.make_workload(spec, seed=seed, device=device)
    lens = first.seq_lens.cpu().tolist()
    layers = [first]
    for l in range(1, n_layers):
        layers.append(W.make_workload(spec, seed=seed + 101 * l, device=device, lengths=lens))
    return layers


# --------------------------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm).
# --------------------------------------------------------------------------------------------


def oracle_round_time(layer, reqs, threads: int):
    """Time one round (verify + select + k drafts) of requests ``reqs`` of one layer with the
    float64 oracle.  Returns (seconds, KV bytes of the round)."""
    import numpy as np

    import oracle
    spec = layer.spec
    ps = spec.page_size
    lens = layer.seq_lens.cpu()[reqs]
    pt = layer.page_table.cpu()[reqs]
    npg = [(int(L) + ps - 1) // ps for L in lens.tolist()]
    pages = torch.cat([pt[i, :n] for i, n in enumerate(npg)]).to(torch.int64)
    pool = layer.pool[pages.to(layer.pool.device)].cpu()
    new_pt = torch.full((len(reqs), max(npg)), -1, dtype=torch.int32)
    off = 0
    for i, n in enumerate(npg):
        new_pt[i, :n] = torch.arange(off, off + n, dtype=torch.int32)
        off += n
    kv = oracle.PagedKV(pool, new_pt, lens)
    qv = layer.q_verify.cpu()[reqs]
    qd = layer.q_draft.cpu()[:, reqs]
    kpr = layer.k_per_req.cpu()[reqs].numpy()
    k_max = int(kpr.max())
    scale = 1.0 / math.sqrt(spec.d)
    t0 = time.perf_counter()
    ref = oracle.verify(kv, qv, scale, threads=threads)
    S = ref["crit"].astype(np.float32)
    idx, cnt = oracle.topk(S.reshape(-1, S.shape[-1]), lens.numpy(), kpr, k_max, rows_per_group=spec.h_kv)
    idx = idx.reshape(len(reqs), spec.h_kv, k_max)
    cnt = cnt.reshape(len(reqs), spec.h_kv)
    for j in range(spec.k):
        oracle.draft(kv, qd[j], idx, cnt, scale, threads=threads)
    dt = time.perf_counter() - t0
    nbytes = M.round_kv_bytes(lens.tolist(), kpr.tolist(), spec.h_kv, spec.d, spec.elem_bytes, spec.k)
    return dt, nbytes


def cpu_baseline(layers, budget_s: float = 12.0) -> dict:
    import oracle
    threads = oracle.default_threads()
    B = layers[0].spec.batch
    total_t, total_b, done = 0.0, 0, []
    for li, layer in enumerate(layers):
        for b in range(B):
            dt, nb = oracle_round_time(layer, [b], threads)
            total_t += dt
            total_b += nb
            done.append((li, b))
            if total_t >= budget_s:
                break
        if total_t >= budget_s:
            break
    return {"value": total_b / total_t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(done)} (layer, request) rounds of verify + select + {layers[0].spec.k} drafts, "
                      f"{total_t:.1f} s of float64 oracle time on {threads} threads"}


# --------------------------------------------------------------------------------------------
# Arms.
# --------------------------------------------------------------------------------------------


def run_reference(args, spec, rank, world):
    """The reference arm: the float64 CPU oracle as it stands, each step one bounded sample."""
    import oracle
    if rank != 0:
        return None
    layers = make_layers(spec, 1, W.spec_seed(spec.name), "cpu")
    layer = layers[0]
    threads = oracle.default_threads()
    reqs = list(range(min(args.ref_requests, spec.batch)))
    for _ in range(args.warmup):
        oracle_round_time(layer, reqs[:1], threads)
    tt, tb = 0.0, 0
    for _ in range(args.steps):
        dt, nb = oracle_round_time(layer, reqs, threads)
        tt += dt
        tb += nb
    value = tb / tt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{spec.name}: {spec.batch} requests, L~U[{spec.len_lo},{spec.len_hi}], "
                                   f"{spec.h_q}/{spec.h_kv} heads, d={spec.d}, bf16 paged (16), k={spec.k}, top-K 5%",
                       "sample_per_step": f"requests 0..{len(reqs) - 1} of layer 0, one round"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{len(reqs)} requests x 1 round per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


def run_ours(args, spec, rank, world, local):
    from sparse_self_speculative_verify_gb300 import KVCache, SpecRound, ssd_status
    from sparse_self_speculative_verify_gb300 import build as libbuild
    from sparse_self_speculative_verify_gb300 import binding

    libbuild.build()
    binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    seed = rank_seed(W.spec_seed(spec.name), rank)
    layers = make_layers(spec, args.layers, seed, dev)
    scale = 1.0 / math.sqrt(spec.d)
    k_max = max(int(l.k_per_req.max()) for l in layers)
    rounds = [SpecRound(KVCache.from_workload(l), spec.h_q, spec.n_cand, k_max, scale, pack_rows=not args.no_pack)
              for l in layers]
    outs = [torch.empty((spec.k, spec.batch, spec.h_q, spec.d), dtype=torch.float32, device=dev) for _ in layers]
    # The step's inputs (the queries of every layer) and outputs (the verify and draft outputs of every
    # layer) each live in one buffer, so that a step's host copies are one per direction.
    q_arena = torch.empty(sum(l.q_verify.numel() + l.q_draft.numel() for l in layers), dtype=layers[0].q_verify.dtype,
                          device=dev)
    off = 0
    for l in layers:
        for name in ("q_verify", "q_draft"):
            t = getattr(l, name)
            v = q_arena[off:off + t.numel()].view(t.shape)
            v.copy_(t)
            setattr(l, name, v)
            off += t.numel()
    o_arena = torch.empty(sum(r.out_v.numel() + o.numel() for r, o in zip(rounds, outs)), dtype=torch.float32,
                          device=dev)
    off, arena_outs = 0, []
    for r, o in zip(rounds, outs):
        r.out_v = o_arena[off:off + r.out_v.numel()].view(r.out_v.shape)
        off += r.out_v.numel()
        arena_outs.append(o_arena[off:off + o.numel()].view(o.shape))
        off += o.numel()
    outs = arena_outs
    stream = torch.cuda.Stream(device=dev)

    def step():
        for r, l in zip(rounds, layers):
            if args.separate_select:
                r.verify(l.q_verify)
                r.select(l.k_per_req)
            else:
                r.verify_select(l.q_verify, l.k_per_req)
        for j in range(spec.k):
            for r, l, o in zip(rounds, layers, outs):
                r.draft(l.q_draft[j], out=o[j], last=j == spec.k - 1)

    launches_per_step = args.layers * ((3 if args.separate_select else 2) + spec.k)
    with torch.cuda.stream(stream):
        step()  # eager warm-up (also sets kernel attributes outside capture)
    stream.synchronize()
    assert ssd_status() == 0, "device status fault in warm-up"
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step()
    stream.synchronize()

    # Work per step (this rank).
    lens = layers[0].seq_lens.cpu().tolist()
    kv_step = sum(M.round_kv_bytes(lens, l.k_per_req.cpu().tolist(), spec.h_kv, spec.d, spec.elem_bytes, spec.k)
                  for l in layers)

    wv0, wv1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        wv0.record(stream)
        for _ in range(args.warmup):
            graph.replay()
        wv1.record(stream)
    stream.synchronize()
    ms_warm = wv0.elapsed_time(wv1) / max(args.warmup, 1)
    barrier()
    clocks = ClockSampler(gpu_id_for(dev))
    clocks.start()
    time.sleep(0.3)
    # Clock window: the same replays for about a second right before the timed region (untimed),
    # so that the 50 ms clock samples see the load the timed steps run under even when the timed
    # region itself is shorter than a sampling period; samples from the window's start to the end
    # of the timed region are summarised.
    n_pre = int(args.clock_window / max(ms_warm * 1e-3, 1e-4))
    torch.cuda.synchronize(dev)
    t_window = time.time()
    with torch.cuda.stream(stream):
        for _ in range(n_pre):
            graph.replay()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    ms_total = ev0.elapsed_time(ev1)
    clk = clocks.stop(t_window, t_end)
    clk["window"] = (f"{n_pre} untimed replays of the step directly before the {args.steps} timed ones, "
                     f"sampled every {clocks.period_ms} ms with them")
    barrier()
    ms_total = max_over_ranks(ms_total, dev)
    bytes_all = sum_over_ranks(float(kv_step * args.steps), dev)
    value = bytes_all / (ms_total * 1e-3) / 1e9
    ms_step = ms_total / args.steps
    rounds_per_s = world * args.layers / (ms_step * 1e-3)
    assert ssd_status() == 0, "device status fault in the timed region"

    # Dominant call: the round's verify call, layers cycled (cold L2): the mean time per call of a
    # CUDA graph of consecutive calls, timed with events on its stream.  The step runs
    # ssd_verify_select (verify kernel + criticality and Top-K pass); ssd_verify_attn (verify
    # kernel + finalize, no selection) is timed beside it.
    reps = max(2, min(args.steps, 10))
    va_ms = graph_mean_ms([(lambda r=r, l=l: r.verify(l.q_verify, stream=stream)) for r, l in zip(rounds, layers)],
                          reps, stream)
    vs_ms = graph_mean_ms([(lambda r=r, l=l: r.verify_select(l.q_verify, l.k_per_req, stream=stream))
                           for r, l in zip(rounds, layers)], reps, stream)
    peaks = measured_peaks()
    va_bytes = M.verify_call_bytes(lens, spec.batch, spec.h_q, spec.h_kv, spec.d, spec.elem_bytes, spec.n_cand)
    vs_bytes = va_bytes + spec.batch * spec.h_kv * (k_max + 1) * 4  # + the selected indices and counts
    if args.separate_select:
        v_ms, v_bytes, v_kernel = va_ms, va_bytes, "ssd_verify_attn (verify_tc_kernel + finalize_kernel)"
    else:
        v_ms, v_bytes, v_kernel = vs_ms, vs_bytes, "ssd_verify_select (verify_tc_kernel + crit_select_kernel)"
    achieved = v_bytes / (v_ms * 1e-3) / 1e9
    units = sum(lens) * spec.h_kv
    roofline = {"bound": "hbm", "kernel": v_kernel,
                "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"],
                "traffic": profiled_traffic(units, "ssd_verify_attn" if args.separate_select else "ssd_verify_select"),
                "verify_attn_ms": va_ms, "verify_attn_frac": va_bytes / (va_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "peak_source": peaks["source"], "launch_ms": v_ms, "algorithmic_bytes": v_bytes,
                "timing": f"mean per call over a CUDA graph of {reps} x {args.layers} consecutive calls, layers cycled",
                "verify_tflops": M.verify_flops(lens, spec.h_q, spec.d, spec.n_cand) / (v_ms * 1e-3) / 1e12}

    # Draft calls of the round, layers cycled (the other layers' drafts evict a layer's selected rows
    # from L2 in between), as the mean time per call of a CUDA graph of consecutive calls: the later
    # drafts of a round read the row pack the first one stored; the first gathers through the index
    # list and stores the pack.
    d_bytes = M.draft_kv_bytes(layers[0].k_per_req.cpu().tolist(), lens, spec.h_kv, spec.d, spec.elem_bytes)
    d_call_bytes = d_bytes + spec.batch * spec.h_q * (spec.d * spec.elem_bytes + (spec.d + 1) * 4)

    from sparse_self_speculative_verify_gb300 import binding as Bd

    def draft_call(r, l, o, mode):
        idx = r.idx.view(spec.batch, spec.h_kv, r.k_max)
        cnt = r.cnt.view(spec.batch, spec.h_kv)
        return lambda: Bd.ssd_draft_attn_packed(r.kv, l.q_draft[1], idx, cnt, r.scale, r.pack, mode, out=o[1],
                                                lse=r.lse_d, workspace=r.ws, stream=stream)

    def plain_call(r, l, o):
        idx = r.idx.view(spec.batch, spec.h_kv, r.k_max)
        cnt = r.cnt.view(spec.batch, spec.h_kv)
        return lambda: Bd.ssd_draft_attn(r.kv, l.q_draft[1], idx, cnt, r.scale, out=o[1], lse=r.lse_d,
                                         workspace=r.ws, stream=stream)

    if args.no_pack:
        dw_ms = dr_ms = None
    else:
        dw_ms = graph_mean_ms([draft_call(r, l, o, Bd.PACK_WRITE) for r, l, o in zip(rounds, layers, outs)], reps,
                              stream)
        dr_ms = graph_mean_ms([draft_call(r, l, o, Bd.PACK_READ) for r, l, o in zip(rounds, layers, outs)], reps,
                              stream)
    dp_ms = graph_mean_ms([plain_call(r, l, o) for r, l, o in zip(rounds, layers, outs)], reps, stream)
    assert ssd_status() == 0, "device status fault in the draft timing"
    def draft_rec(ms, kernel):
        return {"kernel": kernel, "launch_ms": ms, "achieved": d_call_bytes / (ms * 1e-3) / 1e9,
                "frac": d_call_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}

    plain_kernel = "ssd_draft_attn (rows gathered through the index list, draft_kernel)"
    main_ms = dp_ms if args.no_pack else dr_ms
    roofline_draft = {"bound": "hbm",
                      "kernel": plain_kernel if args.no_pack else "ssd_draft_attn_packed, row pack read (draft_pack_kernel)",
                      "timing": f"mean per call over a CUDA graph of {reps} x {args.layers} consecutive calls, "
                                f"layers cycled",
                      "achieved": d_call_bytes / (main_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": d_call_bytes / (main_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], "traffic": None,
                      "peak_source": peaks["source"], "launch_ms": main_ms, "algorithmic_bytes": d_call_bytes,
                      "plain": draft_rec(dp_ms, plain_kernel)}
    if not args.no_pack:
        roofline_draft["first_draft"] = draft_rec(dw_ms, "ssd_draft_attn_packed, row pack written (draft_kernel)")

    # End to end through the API with host buffers: per step, the queries of every layer (and the
    # lengths / page table) go host -> device from pinned memory, the attention outputs device ->
    # host.  As a serving loop would run it, the copies are pipelined on a second stream: step s+1's
    # inputs are uploaded and step s-1's outputs read back while step s computes, through two sets of
    # device staging buffers (device-to-device copies into and out of the step's own buffers, captured
    # with the step in one graph per staging set).
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)  # noqa: E731
    h_in = pin(q_arena)
    h_meta = (pin(layers[0].seq_lens), pin(layers[0].page_table))
    h_out = torch.empty(o_arena.shape, dtype=o_arena.dtype, pin_memory=True)
    h2d = h_in.numel() * h_in.element_size() + sum(t.numel() * t.element_size() for t in h_meta)
    d2h = h_out.numel() * h_out.element_size()
    st_in = [torch.empty_like(q_arena) for _ in range(2)]
    st_meta = [(torch.empty_like(layers[0].seq_lens), torch.empty_like(layers[0].page_table)) for _ in range(2)]
    st_out = [torch.empty_like(o_arena) for _ in range(2)]
    # One graph per staging set: the staged inputs copied into the step's buffers, the step, and the
    # step's outputs copied out to the staging set, all captured together (no host launch between the
    # copies and the step).
    g_io = []
    for b in range(2):
        g_b = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g_b, stream=stream):
                q_arena.copy_(st_in[b], non_blocking=True)
                layers[0].seq_lens.copy_(st_meta[b][0], non_blocking=True)
                layers[0].page_table.copy_(st_meta[b][1], non_blocking=True)
                step()
                st_out[b].copy_(o_arena, non_blocking=True)
        g_io.append(g_b)
    stream.synchronize()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    cstream = torch.cuda.Stream(dev)
    e2e_steps = max(1, min(args.steps, 20))

    def upload(s):
        b = s % 2
        if s >= 2:
            cstream.wait_event(in_free[b])
        st_in[b].copy_(h_in, non_blocking=True)
        st_meta[b][0].copy_(h_meta[0], non_blocking=True)
        st_meta[b][1].copy_(h_meta[1], non_blocking=True)
        in_ready[b].record(cstream)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream.wait_stream(torch.cuda.current_stream(dev))
    cstream.wait_stream(stream)
    with torch.cuda.stream(cstream):
        e0.record(cstream)
        upload(0)
    for s in range(e2e_steps):
        b = s % 2
        with torch.cuda.stream(stream):
            stream.wait_event(in_ready[b])
            if s >= 2:
                stream.wait_event(out_free[b])
            g_io[b].replay()
            in_free[b].record(stream)
            out_ready[b].record(stream)
        with torch.cuda.stream(cstream):
            if s + 1 < e2e_steps:
                upload(s + 1)
            cstream.wait_event(out_ready[b])
            h_out.copy_(st_out[b], non_blocking=True)
            out_free[b].record(cstream)
    with torch.cuda.stream(cstream):
        e1.record(cstream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    e2e_value = sum_over_ranks(float(kv_step * e2e_steps), dev) / (e2e_ms * 1e-3) / 1e9

    cfg_records = None
    if rank == 0 and not args.no_configs:
        cfg_records = config_records(peaks["hbm_gbs"], dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(layers, args.cpu_budget)
    if rank != 0:
        return None
    return {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "rounds_per_s": rounds_per_s,
            "hbm_frac": value / peaks["hbm_gbs"],
            "config": {"workload": f"{spec.name}: {spec.batch} requests, L~U[{spec.len_lo},{spec.len_hi}], "
                                   f"{spec.h_q}/{spec.h_kv} heads, d={spec.d}, bf16 paged KV (page {spec.page_size}, "
                                   f"shuffled), k={spec.k}, top-K ceil(5% L)",
                       "layers": args.layers, "kv_bytes_per_step_per_gpu": kv_step,
                       "step": ("per layer: verify + criticality, then select" if args.separate_select else
                                "per layer: verify + criticality + select (ssd_verify_select)") +
                               "; then k drafts of every layer",
                       "l2": f"inputs larger than L2: {args.layers} layers x "
                             f"{M.verify_kv_bytes(lens, spec.h_kv, spec.d, spec.elem_bytes) / 1e6:.0f} MB KV, cycled",
                       "timing": "CUDA graph of one step, replayed; CUDA events on the replay stream"},
            "roofline": roofline, "roofline_draft": roofline_draft, "configs": cfg_records, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps,
                    "copies": "pinned host buffers; step s+1 uploaded and step s-1 read back on a second "
                              "stream while step s runs (one copy per direction: every layer's queries in one "
                              "buffer, every output in another); the device staging copies into and out of the "
                              "step's buffers captured with the step (one graph per staging set)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk}


def graph_mean_ms(calls, reps: int, stream) -> float:
    """Mean device time per call of ``reps`` passes over ``calls`` (cycled in order), captured as
    one CUDA graph after a warm-up pass and timed with CUDA events on ``stream`` around two
    replays of it (the graph is replayed once before, untimed)."""
    with torch.cuda.stream(stream):
        for c in calls:
            c()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                for c in calls:
                    c()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        g.replay()
        g.replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / (2 * reps * len(calls))


def _time_calls(fn, reps: int = 20, warm: int = 3) -> float:
    """Mean device time of fn() in ms with a cold L2: [L2 flush, fn] and [L2 flush] are each captured
    once as a CUDA graph (after warm-up calls) and replayed `reps` times between CUDA events on their
    stream; the call's time is the difference, so neither host overhead nor the flush is counted."""
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    flush = W.flush_buffer(torch.device("cuda", torch.cuda.current_device()))
    with torch.cuda.stream(st):
        for _ in range(warm):
            fn()
    st.synchronize()
    graphs = []
    for with_fn in (True, False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            with torch.cuda.graph(g, stream=st):
                flush.fill_(1.0)
                if with_fn:
                    fn()
        graphs.append(g)
    st.synchronize()
    ms = []
    for g in graphs:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            g.replay()
            e0.record(st)
            for _ in range(reps):
                g.replay()
            e1.record(st)
        st.synchronize()
        ms.append(e0.elapsed_time(e1) / reps)
    return ms[0] - ms[1]


def config_records(peak_gbs: float, dev) -> dict:
    """One record per other workload of the hot path, each on one GPU: ms per round (per call for
    the unified batch), algorithmic KV bytes per round, KV GB/s and the fraction of the measured HBM
    peak.  Each round is captured as a CUDA graph and timed after an L2 flush (``_time_calls``).
    A workload that fails records its error instead of stopping the benchmark."""
    from sparse_self_speculative_verify_gb300 import binding as Bd
    from sparse_self_speculative_verify_gb300 import KVCache, SpecRound

    def rec(ms, nbytes, **extra):
        gbs = nbytes / (ms * 1e-3) / 1e9
        d = {"ms_per_round": ms, "kv_bytes_per_round": nbytes, "kv_GB_s": gbs, "frac_of_measured_hbm": gbs / peak_gbs,
             "rounds_per_s": 1e3 / ms}
        d.update(extra)
        return d

    def spec_round(name):
        spec = W.SPECS[name]
        w = W.make_workload(spec, seed=W.spec_seed(name), device=dev)
        kv = KVCache.from_workload(w)
        k_max = int(w.k_per_req.max())
        rnd = SpecRound(kv, spec.h_q, spec.n_cand, k_max, 1.0 / math.sqrt(spec.d))
        outs = torch.empty((spec.k, spec.batch, spec.h_q, spec.d), dtype=torch.float32, device=dev)
        ms = _time_calls(lambda: rnd.run(w.q_verify, w.q_draft, w.k_per_req, draft_outs=outs, fused_select=True),
                         reps=10)
        lens, kpr = w.seq_lens.cpu().tolist(), w.k_per_req.cpu().tolist()
        nbytes = M.round_kv_bytes(lens, kpr, spec.h_kv, spec.d, spec.elem_bytes, spec.k)
        return spec, ms, nbytes

    out = {}
    for name in ("tiny", "b128_l8k", "qwen3_14b_unified", "block_131k"):
        try:
            if name in ("tiny", "b128_l8k"):
                spec, ms, nbytes = spec_round(name)
                extra = {"round": f"verify + select + {spec.k} drafts (row pack)"}
                if name == "b128_l8k":
                    extra["ideal_rounds_per_s_at_8TBs"] = 8e12 / nbytes
                    extra["ideal_rounds_per_s_at_measured_peak"] = peak_gbs * 1e9 / nbytes
                out[name] = rec(ms, nbytes, **extra)
            elif name == "qwen3_14b_unified":
                spec = W.SPECS[name]
                w = W.make_workload(spec, seed=W.spec_seed(name), device=dev)
                kv = Bd.KVCache.from_workload(w)
                scale = 1.0 / math.sqrt(spec.d)
                k_max = int(w.k_per_req.max())
                uidx, ucnt = W.random_index_sets(w.seq_lens, spec.h_kv, w.k_per_req, k_max, seed=w.seed)
                uidx, ucnt = uidx.to(dev), ucnt.to(dev)
                phase = w.phase.cpu().numpy()
                lens = w.seq_lens.cpu().tolist()
                vreq = [b for b in range(spec.batch) if phase[b] == 1]
                dreq = [b for b in range(spec.batch) if phase[b] == 0]
                scores = torch.zeros((spec.batch, spec.h_kv, kv.max_seq_len), device=dev)
                nbytes = (M.verify_kv_bytes([lens[b] for b in vreq], spec.h_kv, spec.d, spec.elem_bytes) +
                          int(ucnt[dreq].sum().item()) * M.kv_bytes_per_token_head(spec.d, spec.elem_bytes))
                wsu = Bd.Workspace()
                ms = _time_calls(lambda: Bd.ssd_unified_attn(kv, w.phase, w.q_verify, w.q_draft[0], spec.n_cand,
                                                             uidx, ucnt, scale, scores=scores, workspace=wsu), reps=10)
                vi, di = torch.tensor(vreq, device=dev), torch.tensor(dreq, device=dev)
                kv_v = Bd.KVCache(kv.pool, kv.page_table[vi].contiguous(), kv.seq_lens[vi].contiguous(),
                                  kv.max_seq_len)
                kv_d = Bd.KVCache(kv.pool, kv.page_table[di].contiguous(), kv.seq_lens[di].contiguous(),
                                  kv.max_seq_len)
                qv, qd = w.q_verify[vi].contiguous(), w.q_draft[0][di].contiguous()
                di_idx, di_cnt = uidx[di].contiguous(), ucnt[di].contiguous()

                def separate():
                    Bd.ssd_verify_attn(kv_v, qv, spec.n_cand, scale, workspace=wsu)
                    Bd.ssd_draft_attn(kv_d, qd, di_idx, di_cnt, scale, workspace=wsu)
                ms_sep = _time_calls(separate, reps=10)
                out[name] = rec(ms, nbytes, round="one ssd_unified_attn call (verify-phase requests: verify + "
                                                  "criticality; draft-phase requests: sparse draft)",
                                verify_requests=len(vreq), draft_requests=len(dreq), separate_calls_ms=ms_sep,
                                unified_over_separate=ms / ms_sep)
            else:
                spec = W.SPECS[name]
                w = W.make_workload(spec, seed=W.spec_seed(name), device=dev)
                kv = Bd.KVCache.from_workload(w)
                scale = 1.0 / math.sqrt(spec.d)
                nb = (kv.max_seq_len + 63) // 64
                bs = torch.zeros((spec.batch, spec.h_kv, spec.n_cand, nb), device=dev)
                wsb = Bd.Workspace()
                kb = spec.top_blocks
                ks = torch.full((spec.batch,), kb, dtype=torch.int32, device=dev)
                umax = spec.n_cand * kb
                bi = torch.empty((spec.batch * spec.h_kv * spec.n_cand, kb), dtype=torch.int32, device=dev)
                bc = torch.empty((spec.batch * spec.h_kv * spec.n_cand,), dtype=torch.int32, device=dev)
                un_i = torch.empty((spec.batch * spec.h_kv, umax), dtype=torch.int32, device=dev)
                un_m = torch.empty((spec.batch * spec.h_kv, umax), dtype=torch.int32, device=dev)
                un_c = torch.empty((spec.batch * spec.h_kv,), dtype=torch.int32, device=dev)
                out_b = torch.empty((spec.batch, spec.n_cand, spec.h_q, spec.d), dtype=torch.float32, device=dev)

                def block_round():
                    Bd.ssd_verify_attn(kv, w.q_verify, spec.n_cand, scale, bscores=bs, want_scores=False,
                                       workspace=wsb)
                    Bd.ssd_select_topk(bs, kv.seq_lens, ks, kb, spec.h_kv * spec.n_cand, len_div=64, max_len=nb,
                                       idx=bi, cnt=bc)
                    Bd.ssd_block_union(bi.view(-1, spec.n_cand, kb), bc.view(-1, spec.n_cand), nb, umax,
                                       uidx=un_i, umask=un_m, ucnt=un_c)
                    Bd.ssd_block_sparse_attn(kv, w.q_verify, spec.n_cand, un_i, un_m, un_c, scale, out=out_b,
                                             workspace=wsb)
                ms = _time_calls(block_round, reps=5)
                lens = w.seq_lens.cpu().tolist()
                ublocks = int(un_c.sum().item())
                nbytes = (M.verify_kv_bytes(lens, spec.h_kv, spec.d, spec.elem_bytes) +
                          ublocks * 64 * M.kv_bytes_per_token_head(spec.d, spec.elem_bytes))
                out[name] = rec(ms, nbytes, round="verify with per-candidate block scores + block Top-16 + union "
                                                  "+ block-sparse attention", union_blocks=ublocks)
            assert Bd.ssd_status() == 0, "device status fault"
        except Exception as e:  # a failing workload is reported, the benchmark goes on
            out[name] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    return out


def run_rows(args) -> list:
    """One line per hot-path call on its own workload (the verify, select and draft of the Qwen3-8B
    round, the unified launch on the Qwen3-14B mixed batch against separate verify and draft calls on
    the same requests, and the block path on 8 x 131072): device time per call, L2 flushed before
    each call, and algorithmic bytes."""
    from sparse_self_speculative_verify_gb300 import binding as Bd
    from sparse_self_speculative_verify_gb300 import build as libbuild
    libbuild.build()
    Bd.load()
    dev = torch.device("cuda", 0)
    peak = measured_peaks()["hbm_gbs"]
    out = []

    def line(row, workload, ms, nbytes, **extra):
        gbs = nbytes / (ms * 1e-3) / 1e9
        d = {"row": row, "workload": workload, "us_per_call": ms * 1e3, "algorithmic_bytes": nbytes,
             "GB_s": gbs, "frac_of_measured_hbm": gbs / peak}
        d.update(extra)
        out.append(d)

    # Qwen3-8B round: verify, select, draft.
    spec = W.SPECS["qwen3_8b"]
    w = W.make_workload(spec, seed=1002, device=dev)
    kv = Bd.KVCache.from_workload(w)
    scale = 1.0 / math.sqrt(spec.d)
    lens = w.seq_lens.cpu().tolist()
    kpr = w.k_per_req.cpu().tolist()
    k_max = max(kpr)
    ws = Bd.Workspace()
    r = {}

    def verify():
        r.update(Bd.ssd_verify_attn(kv, w.q_verify, spec.n_cand, scale, workspace=ws))
    ms = _time_calls(verify)
    line("a1-a3 verify + criticality + combine", spec.name, ms,
         M.verify_call_bytes(lens, spec.batch, spec.h_q, spec.h_kv, spec.d, spec.elem_bytes, spec.n_cand))
    sel = {}

    def select():
        sel["idx"], sel["cnt"] = Bd.ssd_select_topk(r["scores"], kv.seq_lens, w.k_per_req, k_max, spec.h_kv,
                                                    max_len=kv.max_seq_len)
    ms = _time_calls(select)
    line("a4 top-K select", spec.name, ms, sum(lens) * spec.h_kv * 4)
    idx = sel["idx"].view(spec.batch, spec.h_kv, k_max)
    cnt = sel["cnt"].view(spec.batch, spec.h_kv)
    ms = _time_calls(lambda: Bd.ssd_draft_attn(kv, w.q_draft[0], idx, cnt, scale, workspace=ws))
    dbytes = M.draft_kv_bytes(kpr, lens, spec.h_kv, spec.d, spec.elem_bytes)
    line("a5 sparse draft", spec.name, ms, dbytes)
    # The same draft through the row pack: the round's first draft (gathers and stores the rows) and
    # each later one (reads them back).
    npk = Bd.ssd_draft_pack_bytes(kv, k_max)
    pk = torch.empty(npk + 256, dtype=torch.uint8, device=dev)
    pk = pk[(-pk.data_ptr()) % 256:][:npk]
    ms = _time_calls(lambda: Bd.ssd_draft_attn_packed(kv, w.q_draft[0], idx, cnt, scale, pk, Bd.PACK_WRITE,
                                                      workspace=ws))
    line("a5 sparse draft, first of a round (row pack written)", spec.name, ms, dbytes)
    ms = _time_calls(lambda: Bd.ssd_draft_attn_packed(kv, w.q_draft[1], None, cnt, scale, pk, Bd.PACK_READ,
                                                      k_max=k_max, workspace=ws))
    line("a5 sparse draft, later in a round (row pack read)", spec.name, ms, dbytes)
    del w, kv, r, sel, idx, cnt, pk
    torch.cuda.empty_cache()

    # Qwen3-14B mixed batch: one unified launch against a verify call and a draft call on the two
    # request subsets.
    spec = W.SPECS["qwen3_14b_unified"]
    w = W.make_workload(spec, seed=1004, device=dev)
    kv = Bd.KVCache.from_workload(w)
    scale = 1.0 / math.sqrt(spec.d)
    k_max = int(w.k_per_req.max())
    uidx, ucnt = W.random_index_sets(w.seq_lens, spec.h_kv, w.k_per_req, k_max, seed=w.seed)
    uidx, ucnt = uidx.to(dev), ucnt.to(dev)
    phase = w.phase.cpu().numpy()
    lens = w.seq_lens.cpu().tolist()
    vreq = [b for b in range(spec.batch) if phase[b] == 1]
    dreq = [b for b in range(spec.batch) if phase[b] == 0]
    nbytes = (M.verify_kv_bytes([lens[b] for b in vreq], spec.h_kv, spec.d, spec.elem_bytes) +
              int(ucnt[dreq].sum().item()) * M.kv_bytes_per_token_head(spec.d, spec.elem_bytes))
    wsu = Bd.Workspace()
    ms = _time_calls(lambda: Bd.ssd_unified_attn(kv, w.phase, w.q_verify, w.q_draft[0], spec.n_cand, uidx, ucnt,
                                                 scale, workspace=wsu))
    vi = torch.tensor(vreq, device=dev)
    di = torch.tensor(dreq, device=dev)
    kv_v = Bd.KVCache(kv.pool, kv.page_table[vi].contiguous(), kv.seq_lens[vi].contiguous(), kv.max_seq_len)
    kv_d = Bd.KVCache(kv.pool, kv.page_table[di].contiguous(), kv.seq_lens[di].contiguous(), kv.max_seq_len)
    qv = w.q_verify[vi].contiguous()
    qd = w.q_draft[0][di].contiguous()
    di_idx, di_cnt = uidx[di].contiguous(), ucnt[di].contiguous()

    def separate():
        Bd.ssd_verify_attn(kv_v, qv, spec.n_cand, scale, workspace=wsu)
        Bd.ssd_draft_attn(kv_d, qd, di_idx, di_cnt, scale, workspace=wsu)
    ms_sep = _time_calls(separate)
    line("a6 unified launch", spec.name, ms, nbytes, verify_requests=len(vreq), draft_requests=len(dreq),
         separate_calls_us=ms_sep * 1e3, speedup_over_separate=ms_sep / ms)
    del w, kv, kv_v, kv_d, uidx, ucnt
    torch.cuda.empty_cache()

    # Block path on 8 x 131072: per-candidate block scores, block Top-16, union, block-sparse attention.
    spec = W.SPECS["block_131k"]
    w = W.make_workload(spec, seed=1005, device=dev)
    kv = Bd.KVCache.from_workload(w)
    scale = 1.0 / math.sqrt(spec.d)
    nb = (kv.max_seq_len + 63) // 64
    bs = torch.zeros((spec.batch, spec.h_kv, spec.n_cand, nb), device=dev)
    wsb = Bd.Workspace()
    lens = w.seq_lens.cpu().tolist()
    ms_v = _time_calls(lambda: Bd.ssd_verify_attn(kv, w.q_verify, spec.n_cand, scale, bscores=bs, want_scores=False,
                                                  workspace=wsb), reps=5)
    kb = spec.top_blocks
    ks = torch.full((spec.batch,), kb, dtype=torch.int32, device=dev)
    bi, bc = Bd.ssd_select_topk(bs, kv.seq_lens, ks, kb, spec.h_kv * spec.n_cand, len_div=64, max_len=nb)
    blocks = bi.view(spec.batch * spec.h_kv, spec.n_cand, kb)
    bcnt = bc.view(spec.batch * spec.h_kv, spec.n_cand)
    un = {}

    def union():
        un["i"], un["m"], un["c"] = Bd.ssd_block_union(blocks, bcnt, nb)
    ms_u = _time_calls(union)
    ms_b = _time_calls(lambda: Bd.ssd_block_sparse_attn(kv, w.q_verify, spec.n_cand, un["i"], un["m"], un["c"], scale,
                                                        workspace=wsb))
    ublocks = int(un["c"].sum().item())
    line("a7 block-sparse attention over the union", spec.name, ms_b,
         ublocks * 64 * M.kv_bytes_per_token_head(spec.d, spec.elem_bytes), union_blocks=ublocks,
         union_us=ms_u * 1e3, block_scores_verify_us=ms_v * 1e3,
         block_scores_verify_frac=M.verify_kv_bytes(lens, spec.h_kv, spec.d, spec.elem_bytes) / (ms_v * 1e-3) / 1e9
         / peak)
    assert Bd.ssd_status() == 0, "device status fault"
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="qwen3_8b", choices=sorted(W.SPECS))
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload records of the other configs")
    ap.add_argument("--clock-window", type=float, default=1.0,
                    help="seconds of untimed replays sampled for clocks before the timed steps (0: none)")
    ap.add_argument("--separate-select", action="store_true",
                    help="run each layer's verify and select as two calls instead of ssd_verify_select")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-requests", type=int, default=2)
    ap.add_argument("--rows", action="store_true", help="time each hot-path call on its own workload (1 GPU)")
    ap.add_argument("--no-pack", action="store_true",
                    help="every draft of the round gathers its rows (no row pack written by the first draft)")
    args = ap.parse_args(argv)
    if args.rows:
        for d in run_rows(args):
            print(json.dumps(d), flush=True)
        return
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    spec = W.SPECS[args.config]
    if args.impl == "reference":
        line = run_reference(args, spec, rank, world)
    else:
        line = run_ours(args, spec, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
