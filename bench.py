"""Benchmark: injected KV tokens/s of retrieve + Chunked RoPE + paged scatter.

One step = one is_retrieve_and_inject call over one batch of the workload
(cosine similarity, top-k, segment plan, gather + rotate + scatter for every
layer and KV head).  Default workload: the Llama-3.1-8B KV shape (32 layers, 8
KV heads, head_dim 128, bf16), 2000 stored facts of U[10, 40] tokens, one query,
k = 50, block size 16; synthetic, seeded.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica on its own store (weak scaling, no collective on the data path); the
timing is the max over ranks after a barrier.  ``--impl reference`` times the
fp64 CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "injected KV tokens/s (retrieve+RoPE+paged scatter) at k=50; % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "inject_traffic.json")
INJECT_SRC = os.path.join(ROOT, "kv_cache_injection_gb300", "csrc", "inject.cu")


# ----------------------------------------------------------------------------- helpers

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank's replica draws its own store (weak scaling)."""
    return base_seed + 1000 * rank


def reduce_max(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


def inject_source_hash() -> str:
    with open(INJECT_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def library_source_hash() -> str:
    """Hash of every source file the library is built from, and of this file."""
    h = hashlib.sha256()
    csrc = os.path.dirname(INJECT_SRC)
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc)) + [
        os.path.join(ROOT, "include", "injectscale.h"), os.path.abspath(__file__)]
    for path in files:
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def ncu_traffic_per_token_layer(key: str):
    """DRAM bytes per injected token and layer from the committed ncu summary
    for this workload, budget k, cache type and placement (key
    "workload/k<k>/cache dtype/placement"), if it was taken on the current
    inject kernel source; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    if d.get("inject_cu_sha256_16") != inject_source_hash():
        return None
    c = d.get("captures", {}).get(key)
    return float(c["dram_bytes_per_token_layer"]) if c else None


class L2Flush:
    """Evicts L2 between steps: writes a buffer larger than L2, then reads
    another one, so that the lines the write left dirty are written back
    during the flush and the next step starts from a clean, cold L2."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not self.out:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- our arm

def measure_h2d_gbs(dev, nbytes: int = 1 << 30, reps: int = 5) -> float:
    """Best of ``reps`` pinned host-to-device copies of ``nbytes``, in GB/s."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = float("inf")
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        d.copy_(h, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b))
    del h, d
    return nbytes / (best * 1e-3) / 1e9


def workload_description(s) -> str:
    Q, k = s.n_queries, s.k
    return (f"{s.name}: {s.num_layers} layers x {s.num_kv_heads} KV heads x head_dim {s.head_dim} "
            f"{s.kv_dtype}; {s.n_facts} facts {s.length_dist}; {Q} quer{'y' if Q == 1 else 'ies'}, "
            f"k={k}, block {s.block_size}")


def prepare(args, rank, local_rank, extra_facts=0, extra_tokens=0):
    """Builds the library, the workload's store (with room for extra_facts
    facts of extra_tokens tokens more) and its device inputs."""
    import torch

    from kv_cache_injection_gb300 import _lib, api
    from kv_cache_injection_gb300 import build as kbuild
    from synth import staging, workloads

    kbuild.build()
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    spec = workloads.SPECS[args.workload]
    overrides = {"seed": rank_seed(spec.seed, rank)}
    if args.facts:
        overrides["facts_per_user"] = args.facts
    if args.layers:
        overrides["num_layers"] = args.layers
    if args.k:
        overrides["k"] = args.k
        overrides["tokens_cap"] = args.k * int(spec.length_dist[2] if spec.length_dist[0] == "uniform"
                                                else spec.tokens_cap // spec.k)
    wl = workloads.get(args.workload, **overrides)
    store = staging.load_store(wl, api, device=local_rank, kv_placement=args.kv_placement,
                               max_facts=wl.spec.n_facts + extra_facts,
                               max_facts_per_user=wl.spec.facts_per_user + extra_facts,
                               max_tokens=wl.total_tokens + extra_tokens)
    api.is_set_retrieval_mode(store, {"auto": _lib.IS_RETRIEVAL_AUTO, "per_query": _lib.IS_RETRIEVAL_PER_QUERY,
                                      "batched": _lib.IS_RETRIEVAL_BATCHED}[args.retrieval])
    inp = staging.device_inputs(wl, local_rank)
    return api, staging, wl, store, inp, dev


def run_ours(args, rank, world, local_rank):
    import torch

    api, staging, wl, store, inp, dev = prepare(args, rank, local_rank)
    s = wl.spec
    cache = staging.canary_cache(wl, local_rank, cache_dtype=args.cache_dtype)
    Q, k = s.n_queries, s.k
    ids = torch.empty((Q, k), dtype=torch.int64, device=dev)
    scores = torch.empty((Q, k), dtype=torch.float32, device=dev)
    seg_len = torch.empty(Q, dtype=torch.int32, device=dev)
    rope = staging.rope_params(wl, api)
    cache_dtype = args.cache_dtype or s.kv_dtype
    cdesc = api.make_cache_desc(s.block_size, wl.num_blocks, cache_dtype)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def step():
        api.is_retrieve_and_inject(store, inp["users"], inp["q_emb"], k, inp["seg_start"], rope,
                                   inp["block_table"], cdesc, cache, ids, scores, seg_len, None,
                                   stream=stream)

    # The clock sampler runs from the warm-up through the end of the timed region.
    clocks = ClockSampler(local_rank).__enter__()
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    bits = api.is_get_status(store)
    if bits:
        raise RuntimeError(f"device status bits 0x{bits:x} during warm-up")
    tokens_per_step = int(seg_len.sum().item())

    # Timed region: per-step CUDA events around the call, L2 flushed between
    # steps (outside the events).  Kernels inside a step overlap their launches
    # (programmatic dependent launch), so no event sits between them here.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms_local = sum(step_ms)
    bits = api.is_get_status(store)
    if bits:
        raise RuntimeError(f"device status bits 0x{bits:x} in the timed region")

    # Stage pass: the same steps with CUDA events around every kernel launch
    # (on the launching stream), for the per-kernel durations of the roofline.
    stage_steps = min(args.steps, 500)
    api.is_reset_timing(store)
    api.is_set_timing(store, True)
    for i in range(stage_steps):
        flush()
        step()
    torch.cuda.synchronize()
    clocks.__exit__(None, None, None)
    api.is_set_timing(store, False)
    stage_ms, stage_n = {}, {}
    for name, st in (("similarity", 0), ("topk", 1), ("plan", 2), ("inject", 3)):
        stage_ms[name], stage_n[name] = api.is_get_timing(store, st)
    launches_per_step = sum(stage_n.values()) / stage_steps
    gpu_launches = int(round(launches_per_step * args.steps))

    total_ms = reduce_max(total_ms_local, dev)
    total_tokens = reduce_sum(float(tokens_per_step * args.steps), dev)

    # End to end through the public API with host buffers: the C-ABI call
    # that takes the step's inputs (users, queries, starts, block table) in
    # host memory, copies them into the library's page-locked buffer, runs the
    # path and returns the ids, scores and segment lengths in host memory
    # (synchronous).  Up to 16 KiB of inputs the kernels read them, and write
    # the outputs, over the host link; larger inputs go in one host-to-device
    # copy and the outputs return in one device-to-host copy.
    edt = np.float16 if s.emb_dtype == "f16" else np.float32
    h_users = np.ascontiguousarray(wl.users, dtype=np.int32)
    h_q = np.ascontiguousarray(wl.queries, dtype=edt)
    h_start = np.ascontiguousarray(wl.seg_start, dtype=np.int32)
    h_bt = np.ascontiguousarray(wl.block_table, dtype=np.int32)
    h_ids = np.empty((Q, k), dtype=np.int64)
    h_scores = np.empty((Q, k), dtype=np.float32)
    h_len = np.empty(Q, dtype=np.int32)
    h2d = h_users.nbytes + h_q.nbytes + h_start.nbytes + h_bt.nbytes
    d2h = h_ids.nbytes + h_scores.nbytes + h_len.nbytes
    call = api.prepare_retrieve_and_inject_host(store, h_users, h_q, k, h_start, rope, h_bt, cdesc, cache,
                                                h_ids, h_scores, h_len, stream=stream)
    e2e_steps = max(3, args.steps)
    e2e_s = 0.0
    for i in range(args.warmup + e2e_steps):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        call()
        if i >= args.warmup:
            e2e_s += time.perf_counter() - t0
    assert np.array_equal(h_ids, ids.cpu().numpy()), "end-to-end ids differ from the timed run"
    e2e_s = reduce_max(e2e_s, dev)
    e2e_tokens = reduce_sum(float(int(h_len.sum()) * e2e_steps), dev)

    result = None
    if rank == 0:
        peaks = measured_peaks()
        per_tok = 2 * s.token_elems * s.elt_bytes            # K + V read per token
        per_tok_w = 2 * s.token_elems * (1 if cache_dtype == "e4m3" else s.elt_bytes)   # written
        inject_bytes = (per_tok + per_tok_w) * tokens_per_step  # read + write per launch
        inject_ms = stage_ms["inject"] / max(1, stage_n["inject"])
        achieved = inject_bytes / (inject_ms * 1e-3) / 1e9
        traffic_tl = ncu_traffic_per_token_layer(f"{s.name}/k{s.k}/{cache_dtype}/{args.kv_placement}")
        emb_bytes = 0
        for u in np.unique(wl.users):
            emb_bytes += int((wl.fact_user == u).sum()) * s.emb_dim * (2 if s.emb_dtype == "f16" else 4)
        path_bytes = inject_bytes + emb_bytes
        step_avg_ms = total_ms_local / args.steps
        if args.kv_placement == "host":
            # Only the reads cross the CPU-GPU link; the writes land in HBM.
            link_gbs = measure_h2d_gbs(dev)
            link_achieved = per_tok * tokens_per_step / (inject_ms * 1e-3) / 1e9
            roofline = {
                "bound": "link",
                "kernel": "inject from host memory (gather over the CPU-GPU link + Chunked RoPE + "
                          "paged scatter)",
                "achieved": link_achieved,
                "peak": link_gbs,
                "peak_source": "pinned host-to-device cudaMemcpyAsync of 1 GiB, measured in this run",
                "unit": "GB/s",
                "frac": link_achieved / link_gbs,
                "traffic": None,
                "algorithmic_bytes": per_tok * tokens_per_step,
                "avg_launch_ms": inject_ms,
            }
        else:
            roofline = {
                "bound": "hbm",
                "kernel": "inject (gather + Chunked RoPE + paged scatter)",
                "achieved": achieved,
                "peak": peaks["hbm_gbs"],
                "peak_source": peaks["source"],
                "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"],
                "frac_of_nominal_8tbs": achieved / 8000.0,
                "traffic": (traffic_tl * tokens_per_step * s.num_layers) if traffic_tl else None,
                "algorithmic_bytes": inject_bytes,
                "avg_launch_ms": inject_ms,
            }
            if roofline["traffic"]:
                # What DRAM saw during the launch: writes still in L2 when the
                # launch ends are written back later (during the flush), so
                # this is below the algorithmic rate whenever the cache tail
                # fits in L2.
                dram = roofline["traffic"] / (inject_ms * 1e-3) / 1e9
                roofline["dram_achieved"] = dram
                roofline["dram_frac"] = dram / peaks["hbm_gbs"]
        roofline["timing"] = (f"CUDA events around each inject launch over {stage_steps} steps of the "
                              "same workload right after the timed region (events between kernels "
                              "disable launch overlap, so this duration includes the launch gap)")
        result = {
            "metric": METRIC,
            "value": total_tokens / (total_ms * 1e-3),
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps,
            "step_ms_distribution": {"median": statistics.median(step_ms),
                                     "p10": float(np.percentile(step_ms, 10)),
                                     "p90": float(np.percentile(step_ms, 90))},
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": s.kv_dtype,
            "data": "synthetic (seeded; LoCoMo and model weights not available)",
            "config": {
                "workload": workload_description(s),
                "tokens_per_step": tokens_per_step,
                "bytes_per_step": path_bytes,
                "l2": (f"flushed between steps, outside the events: {L2_FLUSH_BYTES >> 20} MiB write "
                       f"then {L2_FLUSH_BYTES >> 20} MiB read (clean, cold L2 at each step)"),
                "parallelism": f"replicas x{world} (one store per GPU, no collective)",
                "kv_placement": args.kv_placement,
                "cache_dtype": cache_dtype,
                "retrieval": args.retrieval,
            },
            "roofline": roofline,
            "path_roofline": {
                "bytes": path_bytes,
                "achieved": path_bytes / (step_avg_ms * 1e-3) / 1e9,
                "frac": path_bytes / (step_avg_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "unit": "GB/s",
            },
            "stage_ms": {n: stage_ms[n] / max(1, stage_n[n]) for n in stage_ms},
            "e2e": {"value": e2e_tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": gpu_launches,
            "clocks": clocks.summary(),
            "source_sha16": library_source_hash(),
        }
        if args.cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_budget,
                                                  tokens_per_step=tokens_per_step)
    store.destroy()
    return result


# ----------------------------------------------------------------------------- other entry points

def _per_launch(events):
    return [a.elapsed_time(b) for a, b in events]


def run_layerwise(args, rank, world, local_rank):
    """Layer-wise injection as a layer-by-layer KV connector calls it: the ids
    of one retrieval, then one is_inject_layer call per layer into that layer's
    own cache tensor (the first call plans the segments, the others reuse the
    plan).  CUDA events around every call, L2 flushed between steps."""
    import torch

    api, staging, wl, store, inp, dev = prepare(args, rank, local_rank)
    s = wl.spec
    Q, k, L = s.n_queries, s.k, s.num_layers
    cache_dtype = args.cache_dtype or s.kv_dtype
    ids = torch.empty((Q, k), dtype=torch.int64, device=dev)
    scores = torch.empty((Q, k), dtype=torch.float32, device=dev)
    api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, scores)
    n_ids = (ids >= 0).sum(dim=1).to(torch.int32)
    shape = (2, wl.num_blocks, s.block_size, s.num_kv_heads, s.head_dim)
    caches = [torch.empty(shape, dtype=staging.torch_dtype(cache_dtype), device=dev) for _ in range(L)]
    for c in caches:
        staging.refill_canary(c, cache_dtype)
    seg_len = torch.empty(Q, dtype=torch.int32, device=dev)
    rope = staging.rope_params(wl, api)
    cdesc = api.make_cache_desc(s.block_size, wl.num_blocks, cache_dtype)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    G = max(1, args.layer_group)
    groups = [(l0, min(L, l0 + G)) for l0 in range(0, L, G)]

    def step(events=None):
        for gi, (l0, l1) in enumerate(groups):
            if events is not None:
                events[gi][0].record(stream)
            first = gi == 0
            if G == 1:
                api.is_inject_layer(store, l0, Q, inp["seg_start"], rope, inp["block_table"], cdesc, caches[l0],
                                    fact_ids=ids if first else None, n_ids=n_ids if first else None,
                                    users=inp["users"] if first else None,
                                    seg_len_out=seg_len if first else None, stream=stream)
            else:
                api.is_inject_layers(store, l0, Q, inp["seg_start"], rope, inp["block_table"], cdesc,
                                     caches[l0:l1], fact_ids=ids if first else None,
                                     n_ids=n_ids if first else None, users=inp["users"] if first else None,
                                     seg_len_out=seg_len if first else None, stream=stream)
            if events is not None:
                events[gi][1].record(stream)

    clocks = ClockSampler(local_rank).__enter__()
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if api.is_get_status(store):
        raise RuntimeError("device status bits set during warm-up")
    tokens = int(seg_len.sum().item())
    # Two passes: "host-paced", the calls submitted as the GPU runs them (each
    # call's host cost shows); "queued", the stream held by a short GPU delay
    # while the host submits all L calls, so the events time the GPU side.
    res = {}
    for mode in ("host_paced", "queued"):
        first, later, total = [], [], []
        for _ in range(args.steps):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(len(groups))]
            flush()
            if mode == "queued":
                torch.cuda._sleep(int(len(groups) * 40e-6 * 2.0e9))   # ~40 us of GPU time per call
            step(ev)
            torch.cuda.synchronize()
            d = _per_launch(ev)
            first.append(d[0])
            later.extend(d[1:])
            total.append(ev[0][0].elapsed_time(ev[-1][1]))
        res[mode] = (first, later, total)
    clocks.__exit__(None, None, None)
    first, later, total = res["queued"]
    if api.is_get_status(store):
        raise RuntimeError("device status bits set in the timed region")
    store.destroy()
    elt = 1 if cache_dtype == "e4m3" else s.elt_bytes
    layer_bytes = tokens * 2 * s.num_kv_heads * s.head_dim * (s.elt_bytes + elt) * G   # K+V read and written
    later_ms = statistics.mean(later) if later else statistics.mean(first)
    peaks = measured_peaks()
    achieved = layer_bytes / (later_ms * 1e-3) / 1e9
    step_ms = statistics.mean(total)
    return {"metric": ("layer-wise injected KV tokens/s (one is_inject_layer call per layer, plan from the first)"
                       if G == 1 else f"layer-wise injected KV tokens/s (one is_inject_layers call per {G} layers, "
                       "plan from the first)"),
            "value": tokens / (step_ms * 1e-3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "dtype": s.kv_dtype,
            "data": "synthetic (seeded)",
            "config": {"workload": workload_description(s), "tokens_per_step": tokens, "layers": L,
                       "layers_per_call": G,
                       "cache_dtype": cache_dtype,
                       "l2": "flushed between steps, outside the events; events around every layer call",
                       "timing": "queued: a GPU delay holds the stream while the host submits the L calls"},
            "per_call_us": {"first_with_plan": statistics.mean(first) * 1e3, "later": later_ms * 1e3},
            "host_paced": {"ms_per_step": statistics.mean(res["host_paced"][2]),
                           "per_call_us": statistics.mean(res["host_paced"][1] or res["host_paced"][0]) * 1e3,
                           "value": tokens / (statistics.mean(res["host_paced"][2]) * 1e-3)},
            "roofline": {"bound": "hbm", "kernel": f"inject, {G} layer(s) per launch", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "algorithmic_bytes": layer_bytes, "traffic": None},
            "clocks": clocks.summary(),
            "source_sha16": library_source_hash(),
            "cpu_baseline": (cpu_baseline(wl, budget_s=args.cpu_budget, tokens_per_step=tokens)
                             if args.cpu_baseline and rank == 0 else None)}


def run_capture(args, rank, world, local_rank):
    """Context-Window Encoding capture: per step, is_store_capture_begin for
    --capture-facts facts (fact lengths from the workload, windows of
    --window tokens before each), one is_store_capture_layer call per layer
    from synthetic engine layer buffers, and is_store_capture_abort (so the
    store does not grow).  CUDA events around every layer call."""
    import numpy as np
    import torch

    from synth import workloads
    n = args.capture_facts
    lengths = np.resize(workloads.get(args.workload).lengths, n).astype(np.int32)
    api, staging, wl, store, inp, dev = prepare(args, rank, local_rank, extra_facts=n,
                                                extra_tokens=int(lengths.sum()))
    s = wl.spec
    L = s.num_layers
    rng = np.random.default_rng(5)
    window = np.full(n, args.window, dtype=np.int32)
    src_tokens = int((lengths + window).sum())
    fact_tokens = int(lengths.sum())
    row = s.num_kv_heads * s.head_dim
    tdt = staging.torch_dtype(s.kv_dtype)
    k_buf = torch.empty(src_tokens * row, dtype=tdt, device=dev)
    v_buf = torch.empty_like(k_buf)
    from synth import kvgen
    staging.fill_kv(k_buf, s.kv_dtype, 99, kvgen.STREAM_K, 0)
    staging.fill_kv(v_buf, s.kv_dtype, 99, kvgen.STREAM_V, 0)
    edt = torch.float16 if s.emb_dtype == "f16" else torch.float32
    emb = torch.from_numpy(rng.standard_normal((n, s.emb_dim))).to(edt).to(dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local_rank).__enter__()

    def step(events=None):
        api.is_store_capture_begin(store, 0, window, lengths, emb, stream=stream)
        if events is not None:
            # hold the stream while the host submits the L calls, so the
            # events time the GPU side
            torch.cuda._sleep(int(L * 40e-6 * 2.0e9))
        for l in range(L):
            if events is not None:
                events[l][0].record(stream)
            api.is_store_capture_layer(store, l, k_buf, v_buf, stream=stream)
            if events is not None:
                events[l][1].record(stream)
        torch.cuda.synchronize()
        api.is_store_capture_abort(store)

    for _ in range(args.warmup):
        flush()
        step()
    per_layer, layers_ms, wall = [], [], []
    for _ in range(args.steps):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step(ev)
        wall.append(time.perf_counter() - t0)
        d = _per_launch(ev)
        per_layer.extend(d)
        layers_ms.append(ev[0][0].elapsed_time(ev[-1][1]))
    clocks.__exit__(None, None, None)
    if api.is_get_status(store):
        raise RuntimeError("device status bits set during the capture")
    store.destroy()
    layer_bytes = fact_tokens * 2 * row * s.elt_bytes * 2     # the facts' K+V rows read and written
    mean_layer = statistics.mean(per_layer)
    peaks = measured_peaks()
    achieved = layer_bytes / (mean_layer * 1e-3) / 1e9
    return {"metric": "captured KV tokens/s (Context-Window Encoding: fact rows of every layer into the store)",
            "value": fact_tokens / (statistics.mean(layers_ms) * 1e-3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(layers_ms),
            "higher_is_better": True, "dtype": s.kv_dtype, "data": "synthetic (seeded)",
            "config": {"workload": workload_description(s), "facts": n, "window_tokens": args.window,
                       "fact_tokens": fact_tokens, "source_tokens": src_tokens, "layers": L,
                       "l2": "flushed between steps, outside the events; events around every layer call",
                       "timing": "a GPU delay holds the stream while the host submits the L calls"},
            "per_layer_us": mean_layer * 1e3,
            "host_wall_ms_per_capture": statistics.mean(wall) * 1e3,
            "roofline": {"bound": "hbm", "kernel": "capture_layer (one layer per launch)", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "algorithmic_bytes": layer_bytes, "traffic": None},
            "clocks": clocks.summary(),
            "source_sha16": library_source_hash(),
            "cpu_baseline": (cpu_baseline_capture(s, lengths, args.window, fact_tokens, budget_s=args.cpu_budget)
                             if args.cpu_baseline and rank == 0 else None)}


# ----------------------------------------------------------------------------- oracle arm

def oracle_step(wl, q: int, max_facts: int | None, kv_cache_fn):
    """One query through the fp64 oracle: cosine top-k, then rotation and
    scatter of (at most max_facts of) the retrieved facts into a host cache."""
    from oracle import inject as oinject
    from oracle import retrieval, rope
    s = wl.spec
    facts = wl.user_facts(int(wl.users[q]))
    ids, _ = retrieval.retrieve(wl.queries[q].astype(np.float64), wl.emb[facts].astype(np.float64),
                                facts, s.k)
    use = ids if max_facts is None else ids[:max_facts]
    r = s.rope
    freqs = rope.inv_freq(s.head_dim, r.theta, r.scaling, r.factor, r.low_freq_factor,
                          r.high_freq_factor, r.original_max_pos)
    cache = kv_cache_fn()
    _, T, _ = oinject.inject(cache, s.kv_dtype, wl_fact_kv(wl), use, wl.lengths,
                             int(wl.seg_start[q]), wl.block_table[q], s.block_size, freqs, r.style)
    return T


_FACT_MEMO = {}


def wl_fact_kv(wl):
    from synth import kvgen

    def get(f):
        key = (wl.spec.name, wl.spec.seed, int(f))
        if key not in _FACT_MEMO:
            _FACT_MEMO[key] = (wl.fact_kv(int(f), kvgen.STREAM_K), wl.fact_kv(int(f), kvgen.STREAM_V))
        return _FACT_MEMO[key]
    return get


def _prefetch_facts(wl, q, max_facts):
    from oracle import retrieval
    facts = wl.user_facts(int(wl.users[q]))
    ids, _ = retrieval.retrieve(wl.queries[q].astype(np.float64), wl.emb[facts].astype(np.float64),
                                facts, wl.spec.k)
    get = wl_fact_kv(wl)
    for f in ids[:max_facts]:
        get(f)


def _host_cache(wl):
    from synth.workloads import cache_shape
    s = wl.spec
    shape = cache_shape(s, wl.num_blocks)
    dt = np.float32 if s.kv_dtype == "f32" else np.uint16
    return lambda: np.zeros(shape, dtype=dt)


_ONE_THREAD = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _oracle_worker(spec, max_facts, warmup, steps, budget_s, barrier, out_q, queries=(0,)):
    """One oracle process: build the workload from its spec, warm up, wait for
    the others, then run ``steps`` oracle steps (or until ``budget_s``), step i
    on query queries[i % len(queries)]."""
    from synth import workloads
    wl = workloads.generate(spec)
    for q in queries:
        _prefetch_facts(wl, q, max_facts)
    cache = _host_cache(wl)()
    for i in range(warmup):
        oracle_step(wl, queries[i % len(queries)], max_facts, lambda: cache)
    barrier.wait()
    t0 = time.monotonic()
    tokens = reps = 0
    while reps < steps and (budget_s is None or time.monotonic() - t0 < budget_s):
        tokens += oracle_step(wl, queries[reps % len(queries)], max_facts, lambda: cache)
        reps += 1
    out_q.put((tokens, reps, t0, time.monotonic()))


def oracle_pool(spec, max_facts: int, workers: int, steps: list[int], warmup: int = 1,
                budget_s: float | None = None, queries=(0,)) -> dict:
    """Run the oracle in ``workers`` spawned processes at once (each with its
    BLAS held to one thread, so ``workers`` is the number of threads used).
    Worker i runs ``steps[i]`` steps; the rate is all tokens over the span from
    the first start to the last end (system-wide monotonic clock)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    barrier, out_q = ctx.Barrier(workers), ctx.Queue()
    saved = {v: os.environ.get(v) for v in _ONE_THREAD}
    os.environ.update({v: "1" for v in _ONE_THREAD})
    try:
        procs = [ctx.Process(target=_oracle_worker,
                             args=(spec, max_facts, warmup, steps[i], budget_s, barrier, out_q,
                                   tuple(queries)))
                 for i in range(workers)]
        for p in procs:
            p.start()
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    res = [out_q.get(timeout=600) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        if p.exitcode != 0:
            raise RuntimeError(f"oracle worker exited with {p.exitcode}")
    wall = max(r[3] for r in res) - min(r[2] for r in res)
    tokens = sum(r[0] for r in res)
    return {"tokens": tokens, "reps": sum(r[1] for r in res), "wall_s": wall,
            "value": tokens / wall}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl, budget_s: float = 20.0, max_facts: int = 10, tokens_per_step: int | None = None,
                 n_sample_queries: int = 4) -> dict:
    """Time the oracle, as it stands, on a bounded sample of the workload: per
    sampled query, the retrieval over its user's store plus rotation and
    scatter of its first ``max_facts`` retrieved facts, repeated (at most 50
    times or about ``budget_s``) in one process with one thread, then in one
    process per host core at once.  A workload of one query samples that
    query; with more, a seeded random subset of ``n_sample_queries`` of them,
    taken in turn.  The rate is per injected token, so the time the oracle
    would take for the whole step is an extrapolation, labelled as such."""
    Q = int(wl.spec.n_queries)
    if Q == 1:
        queries = [0]
    else:
        queries = sorted(np.random.default_rng(12345).choice(Q, size=min(n_sample_queries, Q),
                                                             replace=False).tolist())
    n_user = [int((wl.fact_user == wl.users[q]).sum()) for q in queries]
    what = (f"cosine top-{wl.spec.k} over the user's {n_user[0] if len(set(n_user)) == 1 else n_user} "
            f"facts + fp64 RoPE/scatter of the first {max_facts} retrieved facts")
    if Q > 1:
        what = f"queries {queries} of {Q} (seeded random subset) in turn, each: " + what
    one = oracle_pool(wl.spec, max_facts, 1, [50], budget_s=budget_s, queries=queries)
    cores = host_cores()
    many = oracle_pool(wl.spec, max_facts, cores, [50] * cores, budget_s=budget_s, queries=queries)
    out = {"value": one["value"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": (f"{one['reps']} x ({what}); {one['tokens']} tokens in {one['wall_s']:.1f} s, "
                      f"numpy fp64, 1 process, BLAS on 1 thread"),
           "all_cores": {"value": many["value"], "unit": "tokens/s", "cores": cores,
                         "sample": (f"{cores} processes at once, each {many['reps'] // cores} x the "
                                    f"same sample; {many['tokens']} tokens in {many['wall_s']:.1f} s")}}
    if tokens_per_step:
        out["extrapolated_s_per_step"] = {
            "cores_1": tokens_per_step / one["value"], "all_cores": tokens_per_step / many["value"],
            "note": (f"the step's {tokens_per_step} injected tokens at the sampled per-token rate: "
                     "an extrapolation, not a measurement of the whole step")}
    return out


def cpu_baseline_capture(spec, lengths, window: int, fact_tokens: int, budget_s: float = 20.0,
                         sample_facts: int = 64) -> dict:
    """Time the oracle's capture step, as it stands, on a bounded sample: for
    each of the first ``sample_facts`` facts, an engine layer output of its
    [window || fact] sequence (seeded values) for every layer, from which
    oracle.cwe.capture keeps the fact's rows; one process, one thread.  The
    rate is per captured fact token over all layers, and the time for the
    whole capture is an extrapolation, labelled as such."""
    from oracle import cwe
    rng = np.random.default_rng(7)
    L, H, D = spec.num_layers, spec.num_kv_heads, spec.head_dim
    seqs = []
    for n in lengths[:sample_facts]:
        T = int(n) + int(window)
        kv = [(rng.standard_normal((T, H, D)), rng.standard_normal((T, H, D))) for _ in range(L)]
        seqs.append((kv, int(window)))
    toks = reps = 0
    t0 = time.monotonic()
    while reps < 50 and time.monotonic() - t0 < budget_s:
        for kv, wl_ in seqs:
            K, V = cwe.capture(kv, wl_)
            toks += K.shape[0]
        reps += 1
    wall = time.monotonic() - t0
    value = toks / wall
    return {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": (f"{reps} x oracle.cwe.capture over {len(seqs)} facts' [window ({window} tokens) || fact] "
                       f"layer outputs, {L} layers x {H} x {D} fp64; {toks} fact tokens in {wall:.1f} s, "
                       "1 process"),
            "extrapolated_s_per_step": {"cores_1": fact_tokens / value,
                                        "note": "the capture's fact tokens at the sampled rate: an extrapolation"}}


def run_reference(args, rank, world):
    from synth import workloads
    if rank != 0:
        return None
    spec = workloads.SPECS[args.workload]
    overrides = {"k": args.k} if args.k else {}
    wl = workloads.get(args.workload, **overrides)
    max_facts = 4
    cores = host_cores()
    steps = [args.steps // cores + (i < args.steps % cores) for i in range(cores)]
    run = oracle_pool(wl.spec, max_facts, cores, steps, warmup=args.warmup)
    value = run["value"]
    sample = (f"per step: cosine top-{wl.spec.k} over {spec.facts_per_user} facts + fp64 RoPE/scatter "
              f"of the first {max_facts} retrieved facts ({run['tokens'] // max(1, args.steps)} tokens); "
              f"the {args.steps} steps spread over {cores} processes (one per host core, BLAS on 1 "
              f"thread each), each after {args.warmup} untimed steps")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": run["wall_s"] * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": workload_description(wl.spec),
                       "parallelism": f"oracle on {cores} host cores (rank 0), bounded sample",
                       "kv_placement": args.kv_placement, "cache_dtype": args.cache_dtype or wl.spec.kv_dtype,
                       "retrieval": args.retrieval},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama31_8b")
    ap.add_argument("--k", type=int, default=0)
    ap.add_argument("--facts", type=int, default=0,
                    help="facts per user (smaller store for profiling captures)")
    ap.add_argument("--layers", type=int, default=0,
                    help="model layers (smaller K/V for profiling the retrieval kernels)")
    ap.add_argument("--kv-placement", choices=["device", "host"], default="device",
                    help="where the store's K/V arena lives (host: page-locked host DRAM)")
    ap.add_argument("--cache-dtype", choices=["e4m3"], default=None,
                    help="paged-cache type when it differs from the store's (e4m3: FP8, scales 1.0)")
    ap.add_argument("--retrieval", choices=["auto", "per_query", "batched"], default="auto",
                    help="similarity path: per-query kernel, tcgen05 batched contraction, or automatic")
    ap.add_argument("--mode", choices=["step", "layerwise", "capture"], default="step",
                    help="step: the fused retrieve+inject step (the headline); layerwise: one "
                         "is_inject_layer call per layer; capture: Context-Window Encoding capture")
    ap.add_argument("--capture-facts", type=int, default=256, help="facts per capture (--mode capture)")
    ap.add_argument("--layer-group", type=int, default=1,
                    help="layers per call in --mode layerwise (1: is_inject_layer; more: is_inject_layers)")
    ap.add_argument("--window", type=int, default=64, help="window tokens before each fact (--mode capture)")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return 0
        else:
            import torch
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    elif args.mode == "layerwise":
        out = run_layerwise(args, rank, world, local_rank)
    elif args.mode == "capture":
        out = run_capture(args, rank, world, local_rank)
    else:
        out = run_ours(args, rank, world, local_rank)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
