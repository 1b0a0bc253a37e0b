"""Benchmark of the verify step on one B300 per process.

Workload (the headline one): single-request verify of an 8B-class bf16
decoder — 36 layers, d_model 4096, 32 q / 8 kv heads x 128, SwiGLU ffn 12288,
vocab 151936 — with a 4096-position KV context of random bf16 N(0,1) values,
batch 1, gamma = 16 drafts (M = 17 rows), temperature 0. Drafts follow a
greedy-decoding run of the same model on the GPU: draft i (0-based) is the
greedy token with probability 0.9^(i+1), else a uniform token. Weights are
random N(0, 0.02) (no checkpoint), so the data is synthetic.

One step = one sv_verify of that block (embedding, 36 layers, LM head,
acceptance, KV commit) with its inputs resident in HBM. The decode plan
(anchor and drafts of every step) is computed before the timed region from
the greedy run, so the timed loop issues verifies back to back; after it the
accepted lengths are checked against the plan (near-tie flips are counted).

Prints one JSON line (rank 0). Under torchrun (N > 1) each rank runs an
independent replica of the workload (the verify step has no cross-request
exchange), and value is the sum over ranks divided by the slowest rank's time.

--impl reference times the CPU oracle (float64 numpy) on a bounded sample of
the same workload: one decoder layer of the step's block per step, scaled to
the 36 layers plus the LM head.
--sweep gemm times the skinny GEMM alone on the workload's projection shapes.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "accepted tokens/s (verify-step us and weight+KV HBM fraction alongside)"
CONTEXT = 4096
GAMMA = 16
PAGE = 16
P_KEEP = 0.9


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", choices=["none", "gemm", "step", "schedule"], default="none",
                    help="gemm: the skinny GEMM alone per projection shape; step: the whole verify step of the "
                         "8B-class model per block size M (the step-cost table a prefix scheduler takes)")
    ap.add_argument("--sweep-m", default="17", help="comma-separated block sizes M for --sweep gemm")
    ap.add_argument("--sweep-dtype", choices=["bf16", "w12"], default="bf16")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cuda-core-gemm", action="store_true",
                    help="with --sweep step: run the projections on the CUDA-core (FMA) kernel instead of tcgen05")
    ap.add_argument("--no-graph", action="store_true",
                    help="time only direct launches (default: the headline steps are replayed from a CUDA graph "
                         "captured once, with the direct launches timed and reported beside them)")
    ap.add_argument("--trace", action="store_true",
                    help="after the timed steps, run two traced steps and add a per-kernel timeline summary "
                         "(device %globaltimer per CTA) to the JSON line")
    ap.add_argument("--trace-out", default=None, help="with --trace: also save the raw per-CTA records (.npz)")
    ap.add_argument("--workload", choices=["8b", "tiny", "27b", "w12", "w12g", "sampled", "tree"], default="8b",
                    help="8b: the headline line (default); the others time the other verify configurations "
                         "(tiny greedy, 27B-class ragged batch 32, W12 weights at the 8B-class shapes, sampled "
                         "batch 64) and print their own line")
    ap.add_argument("--layers", type=int, default=None,
                    help="decoder layers (default: the workload's own, 36 for the 8B-class model; fewer only "
                         "for small profiling runs, which the JSON line's config then names)")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce(x, world, op):
    """One float reduced over the ranks (NCCL on the GPU, or gloo on the CPU)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def all_max(x, world):
    import torch.distributed as dist
    return _reduce(x, world, dist.ReduceOp.MAX if world > 1 else None)


def all_sum(x, world):
    import torch.distributed as dist
    return _reduce(x, world, dist.ReduceOp.SUM if world > 1 else None)


def aggregate(tokens, t_ms, world):
    """Whole-job throughput of independent replicas: all ranks' tokens over the slowest rank's time."""
    t_max = all_max(t_ms, world)
    return all_sum(tokens, world) / (t_max * 1e-3), t_max


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        smax = float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s, pw in zip(sm, power) if pw > 0.35 * max(power)] if power else sm
        return {"sm_mhz": statistics.median(loaded or sm), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "verify_step_02_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# the projection kernel's sources: a recorded DRAM traffic holds only while they are unchanged
GEMM_SOURCES = ["gemm_tc.cu", "gemm_tc.cuh", "gemm_tc_plan.h", "epilogue.cuh", "tc_ptx.cuh", "internal.h"]


def traffic_record(kernel, workload, files):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's sources are unchanged since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(f"{kernel}@{workload}")
    if not rec or rec.get("source_hash") != kernel_source_hash(files):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ device timeline
LAYER_KERNELS = ("qkv", "attention", "o", "gate_up", "down")


# trace words past the common ones (1 start, 2 wait, 3 first operands, 4 last MMA, 6 exit)
GEMM_MARKS = (("t_acc", 7), ("t_x", 12), ("t_stored", 8), ("t_counted", 9), ("t_summed", 13), ("t_reduced", 10),
              ("t_epilogue", 11))
ATTN_MARKS = (("s0_ready", 12), ("p0_ready", 13), ("kv_last", 10), ("p_last", 11), ("pv_done", 14),
              ("sets_merged", 15), ("partial", 7), ("cluster_synced", 8), ("merge_weights", 9))


def trace_summary(records, launches, n_layers):
    """Per-kernel critical-path timeline of traced verify steps (microseconds).

    records: uint64 [n, 8] per-CTA records; launches: [(first, ctas, kind)] in
    launch order (the layer kernels of each step, then the LM head). For each
    kernel, times are measured from the moment the previous kernel's last CTA
    exited: its first CTA start, its median dependency-wait return, its median
    first operands, its median and last MMA issue, the latest CTA at each step
    of the last tile's hand-off (projections), and its last CTA exit (= the
    time it adds to the step). Layer 0 is skipped (its predecessor is not
    traced).
    """
    nk = len(LAYER_KERNELS)
    per_step = nk * n_layers + 1
    names = []
    for i in range(len(launches)):
        j = i % per_step
        names.append("lm_head" if j == per_step - 1 else LAYER_KERNELS[j % nk])
    acc = {}
    prev_exit = None
    for i, (first, ctas, kind) in enumerate(launches):
        r = records[first:first + ctas].astype(np.float64)
        w = lambda k: r[:, k][r[:, k] > 0]
        starts, waits, mma0, mma1, exits = w(1), w(2), w(3), w(4), w(6)
        marks = ATTN_MARKS if names[i] == "attention" else GEMM_MARKS
        tail = {n: w(k) for n, k in marks}
        if len(exits) == 0:
            prev_exit = None
            continue
        ex = exits.max()
        j = i % per_step
        if prev_exit is not None and j >= nk:
            d = acc.setdefault(names[i], {k: [] for k in ("ctas", "start", "wait", "first_mma", "last_mma_median",
                                                           "last_mma", *(n for n, _ in marks), "exit")})
            d["ctas"].append(ctas)
            d["start"].append(starts.min() - prev_exit)
            if len(mma1):
                d["last_mma_median"].append(np.median(mma1) - prev_exit)
            for n, v in tail.items():
                if len(v):
                    d[n].append(v.max() - prev_exit)
            if len(waits):
                d["wait"].append(np.median(waits) - prev_exit)
            if len(mma0):
                d["first_mma"].append(np.median(mma0) - prev_exit)
            if len(mma1):
                d["last_mma"].append(mma1.max() - prev_exit)
            d["exit"].append(ex - prev_exit)
        prev_exit = ex
    out = {}
    for name, d in acc.items():
        out[name] = {k: (int(np.mean(v)) if k == "ctas" else round(float(np.mean(v)) / 1e3, 2))
                     for k, v in d.items() if v}
    layer_us = sum(out[n]["exit"] for n in LAYER_KERNELS if n in out)
    return {"per_kernel_us_after_previous_exit": out, "layer_us": round(layer_us, 2),
            "note": "device %globaltimer per CTA, means over layers 1.. of two traced steps"}


# ------------------------------------------------------------------ workload
def build_workload(steps_total, layers=36, flags=0):
    import torch

    import synth
    import synth.device as sd
    import verify_step_02_b300 as vs

    shape = dict(synth.SHAPES["8b"], n_layers=layers)
    max_seq = CONTEXT + (steps_total + 2) * (GAMMA + 1) + 64
    max_seq = (max_seq + PAGE - 1) // PAGE * PAGE
    wdev = sd.random_bf16_model(shape)
    table, n_pages = synth.contiguous_page_table([max_seq], PAGE, max_seq // PAGE + 1)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="normal")
    seq = torch.tensor([CONTEXT], dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    cfg = vs.make_config(shape, vs.SV_BF16, 1, GAMMA, max_seq, PAGE, flags=flags)
    model = vs.Model(cfg, wdev)
    return shape, wdev, kv, model, table, cfg


def greedy_reference(model, kv, anchor, n_tokens, width=GAMMA + 1):
    """Greedy decoding with the same engine (one row per step, no drafts)."""
    import torch
    tok = torch.zeros((1, width), dtype=torch.int32, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(n_tokens, dtype=torch.int32, device="cuda")
    tok[0, 0] = anchor
    for i in range(n_tokens):
        model.verify(tok, [0], kv, acc, nxt[i:i + 1])
        tok[0, 0:1].copy_(nxt[i:i + 1])
    return [anchor] + [int(x) for x in nxt.cpu().numpy()]


def make_plan(g, steps, vocab, gamma=GAMMA, p_keep=P_KEEP):
    """Blocks [anchor, d_1..d_gamma] of each step, assuming the engine accepts exactly as greedy decoding."""
    import synth
    blocks, expect = [], []
    off = 0  # index in g of the current anchor
    for s in range(steps):
        want = g[off + 1: off + 1 + gamma]
        if len(want) < gamma:
            want = list(want) + [0] * (gamma - len(want))
        drafts = synth.greedy_mix_drafts(want, gamma, p_keep, vocab, 40, s)
        k = 0
        while k < gamma and off + 1 + k < len(g) and drafts[k] == g[off + 1 + k]:
            k += 1
        blocks.append([g[off]] + [int(x) for x in drafts])
        expect.append(k)
        off = min(off + k + 1, len(g) - 1)
    return np.array(blocks, np.int32), np.array(expect, np.int32)


TREE_NODES = 32


def make_tree_plan(g, steps, vocab):
    """Token trees of each step and their parents; the anchor advances as greedy tree acceptance
    would (the deepest node whose path spells the greedy continuation)."""
    import synth
    blocks, parents = [], []
    off = 0  # index in g of the current anchor
    for s in range(steps):
        par = synth.random_tree(TREE_NODES, 3, 60, s)
        want = [int(x) for x in g[off + 1: off + 1 + TREE_NODES]]
        tok = synth.tree_drafts(par, g[off], want, 0.9, vocab, 61, s)
        depth, ok, k = [0] * TREE_NODES, [True] + [False] * (TREE_NODES - 1), 0
        for i in range(1, TREE_NODES):
            depth[i] = depth[par[i]] + 1
            ok[i] = ok[par[i]] and depth[i] <= len(want) and int(tok[i]) == want[depth[i] - 1]
            if ok[i]:
                k = max(k, depth[i])
        blocks.append([int(t) for t in tok])
        parents.append([int(p) for p in par])
        off = min(off + k + 1, len(g) - 1)
    return np.array(blocks, np.int32), np.array(parents, np.int32)


def graph_replay(model, kv, blocks_d, args, stream, world, gamma=GAMMA, context=CONTEXT):
    """The same steps replayed from one CUDA graph of a verify (captured after a warm-up call with
    the same shape); each step copies its block into the graph's input buffer first. Returns timing
    and whether the replays accepted exactly as the direct launches did (one request of `gamma`
    drafts whose KV context starts at `context` tokens)."""
    import torch
    tok = torch.zeros((1, gamma + 1), dtype=torch.int32, device="cuda")
    acc1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = args.warmup + args.steps
    accs = torch.zeros(n, dtype=torch.int32, device="cuda")
    kv.seq_len.fill_(context)
    tok.copy_(blocks_d[0:1])
    model.verify(tok, [gamma], kv, acc1, nxt1)   # warm-up: first-call setup outside the capture
    torch.cuda.synchronize()
    kv.seq_len.fill_(context)
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g):
            model.verify(tok, [gamma], kv, acc1, nxt1)
    except Exception as e:  # noqa: BLE001 - reported, not fatal
        return {"unavailable": f"capture failed: {e}"}
    kv.seq_len.fill_(context)   # the capture ran nothing; start from the same context
    for i in range(args.warmup):
        tok.copy_(blocks_d[i:i + 1])
        g.replay()
        accs[i:i + 1].copy_(acc1)
    barrier(world)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for j in range(args.steps):
        i = args.warmup + j
        tok.copy_(blocks_d[i:i + 1])
        g.replay()
        accs[i:i + 1].copy_(acc1)
        ev[j + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = ev[0].elapsed_time(ev[-1]) / args.steps
    return {"ms_per_step": round(ms, 4), "accepted": accs.cpu().numpy().tolist(),
            "per_step": [ev[j].elapsed_time(ev[j + 1]) for j in range(args.steps)],
            "note": "one CUDA graph of the verify launches (programmatic dependencies kept), replayed per step "
                    "after a device copy of the step's block into its input buffer"}


def step_bytes(shape):
    """Algorithmic HBM bytes of one verify step: every weight once + the KV rows read and written."""
    s = shape
    d, f, v = s["d_model"], s["ffn"], s["vocab"]
    nq, nkv = s["n_heads"] * s["head_dim"], s["n_kv_heads"] * s["head_dim"]
    per_layer = ((nq + 2 * nkv) * d + d * nq + 2 * f * d + d * f) * 2
    weights = s["n_layers"] * per_layer + v * d * 2
    kv_row = s["n_layers"] * 2 * nkv * 2
    return per_layer, weights, kv_row


def run_ours(args, world, rank, local):
    import torch

    import verify_step_02_b300 as vs

    torch.cuda.set_device(local)
    steps_total = args.warmup + args.steps
    shape, wdev, kv, model, table, cfg = build_workload(3 * steps_total, args.layers or 36)
    vocab = shape["vocab"]
    anchor = int(np.random.default_rng(20261202).integers(0, vocab))
    n_ref = int(steps_total * (1 + sum(P_KEEP ** (i + 1) for i in range(GAMMA))) * 1.5) + GAMMA + 8
    g = greedy_reference(model, kv, anchor, n_ref)
    blocks, expect = make_plan(g, steps_total, vocab)
    blocks_d = torch.from_numpy(blocks).cuda()
    acc = torch.zeros(steps_total, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(steps_total, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def run(i):
        model.verify(blocks_d[i:i + 1], [GAMMA], kv, acc[i:i + 1], nxt[i:i + 1])

    # ---- device-timed region: inputs resident in HBM
    clocks = ClockSampler(local)
    kv.seq_len.fill_(CONTEXT)
    for i in range(args.warmup):
        run(i)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")  # lets a profiler select the timed launches
    ev[0].record(stream)
    for j in range(args.steps):
        run(args.warmup + j)
        ev[j + 1].record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier(world)
    per_step = [ev[j].elapsed_time(ev[j + 1]) for j in range(args.steps)]
    t_ms = ev[0].elapsed_time(ev[-1])
    graph = None
    if not args.no_graph:
        graph = graph_replay(model, kv, blocks_d, args, stream, world)
    acc_np = acc.cpu().numpy()[args.warmup:]
    direct_ms = t_ms / args.steps
    if graph is not None and "accepted" in graph:
        graph["same_decisions_as_direct"] = graph.pop("accepted")[args.warmup:] == acc_np.tolist()
        g_steps = graph.pop("per_step")
        if graph["same_decisions_as_direct"]:   # the headline steps are the graph replays
            t_ms = graph["ms_per_step"] * args.steps
            per_step = g_steps
    tokens = float((acc_np + 1).sum())
    flips = int((acc.cpu().numpy() != expect).sum())

    # ---- end to end through the host-buffer entry point
    kv.seq_len.fill_(CONTEXT)
    host_blocks = torch.from_numpy(blocks).pin_memory()
    out_acc = torch.zeros(1, dtype=torch.int32).pin_memory()
    out_nxt = torch.zeros(1, dtype=torch.int32).pin_memory()
    for i in range(args.warmup):
        model.verify_host(host_blocks[i:i + 1], [GAMMA], kv, out=(out_acc, out_nxt))
    barrier(world)
    torch.cuda.synchronize()
    e2e_tokens = 0
    t0 = time.perf_counter()
    for j in range(args.steps):
        i = args.warmup + j
        model.verify_host(host_blocks[i:i + 1], [GAMMA], kv, out=(out_acc, out_nxt))
        e2e_tokens += int(out_acc[0]) + 1
    t_e2e = time.perf_counter() - t0
    barrier(world)

    # ---- instrumented pass: per-kernel-class device time from CUDA events around
    # every launch, on a second engine over the same weights whose kernels run
    # one after another (no programmatic dependent launch), so the classes add
    # up to that pass's step time
    import ctypes
    cfg_np = vs.Config.from_buffer_copy(cfg)
    cfg_np.flags |= vs.SV_FLAG_NO_PDL
    model_np = vs.Model(cfg_np, wdev)
    kv.seq_len.fill_(CONTEXT)

    def run_np(i):
        model_np.verify(blocks_d[i:i + 1], [GAMMA], kv, acc[i:i + 1], nxt[i:i + 1])
    for i in range(args.warmup):
        run_np(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for j in range(args.steps):
        run_np(args.warmup + j)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_np = e0.elapsed_time(e1) / args.steps
    kv.seq_len.fill_(CONTEXT)
    for i in range(args.warmup):
        run_np(i)
    torch.cuda.synchronize()
    model_np.set_timing(True)
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for j in range(args.steps):
        run_np(args.warmup + j)
    e3.record(stream)
    torch.cuda.synchronize()
    ms_instr = e2.elapsed_time(e3) / args.steps
    tim = model_np.timing()
    model_np.set_timing(False)
    model_np.close()
    clk = clocks.stop()

    # ---- optional device timeline of two steps (the default engine)
    trace = None
    if args.trace:
        n_layers = args.layers or 36
        cap = 2 * (n_layers * (4 * 148 + 8 * 16 * 2) + 148 + 64)
        recs = torch.zeros((cap, 16), dtype=torch.int64, device="cuda")
        kv.seq_len.fill_(CONTEXT)
        for i in range(args.warmup):
            run(i)
        torch.cuda.synchronize()
        model.set_trace(recs)
        for j in range(2):
            run(args.warmup + j)
        torch.cuda.synchronize()
        launches = model.trace_launches()
        model.set_trace(None)
        raw = recs.cpu().numpy().view(np.uint64)
        trace = trace_summary(raw, launches, n_layers)
        if args.trace_out:
            np.savez_compressed(args.trace_out, records=raw, launches=np.array([l[:2] for l in launches]),
                                kinds=np.array([l[2] for l in launches]))

    value, t_max = aggregate(tokens, t_ms, world)
    e2e_all, _ = aggregate(e2e_tokens, t_e2e * 1e3, world)
    result = None
    if rank == 0:
        peak, peak_kind = measured_peaks()
        per_layer, wbytes, kv_row = step_bytes(shape)
        ctx_mean = CONTEXT + float(np.mean(np.cumsum(np.r_[0, (acc.cpu().numpy() + 1)[:-1]])[args.warmup:]))
        kv_read = kv_row * (ctx_mean + GAMMA + 1)
        step_alg = wbytes + kv_read + kv_row * (GAMMA + 1)
        gemm_ms, gemm_n = tim["gemm"]
        gemm_bytes_launch = per_layer / 4.0                     # 4 projections per layer
        achieved = gemm_bytes_launch / (gemm_ms / gemm_n * 1e-3) / 1e9 if gemm_n else None
        traffic = traffic_record("gemm", "8b_m17", GEMM_SOURCES)
        launches = sum(n for _, n in tim.values()) / args.steps
        ms_step = t_max / args.steps
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (random N(0,0.02) weights, random N(0,1) KV context, greedy-mix drafts)",
            "config": {"workload": "8B-class bf16 single-request verify, gamma 16 (M=17), context 4096, T=0",
                       "batch": 1, "gamma": GAMMA, "context": CONTEXT, "layers": args.layers or 36, "d_model": 4096,
                       "vocab": 151936, "l2": "inputs larger than L2 (15.1 GB of weights per step)",
                       "parallelism": f"replicas x{world}"},
            "verify_us": {"median": round(1e3 * statistics.median(per_step), 1),
                          "p90": round(1e3 * float(np.percentile(per_step, 90)), 1)},
            "tokens_per_step": round(tokens / args.steps, 3),
            "hbm": {"bytes_per_step": step_alg, "gbs": round(step_alg / (ms_step * 1e-3) / 1e9, 1),
                    "frac_of_peak": round(step_alg / (ms_step * 1e-3) / 1e9 / peak, 4), "peak_gbs": peak,
                    "peak_kind": peak_kind, "bound_ms": round(step_alg / (peak * 1e9) * 1e3, 4)},
            "roofline": {"kernel": "skinny GEMM (q|k|v, o, gate|up, down projections)", "bound": "hbm",
                         "achieved": round(achieved, 1) if achieved else None, "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4) if achieved else None, "traffic": traffic,
                         "peak_kind": peak_kind, "launches": gemm_n,
                         "bytes_per_launch": gemm_bytes_launch,
                         "avg_launch_us": round(gemm_ms / gemm_n * 1e3, 2) if gemm_n else None,
                         "timing": "CUDA events around each launch in a pass without programmatic dependent "
                                   "launch (each kernel alone, start to finish)"},
            "kernel_ms_per_step": {k: round(v[0] / args.steps, 4) for k, v in tim.items()},
            "kernel_ms_timing": {"pass": "no programmatic dependent launch; events around every launch",
                                 "ms_per_step_of_that_pass": round(ms_np, 4),
                                 "ms_per_step_with_the_events": round(ms_instr, 4),
                                 "sum_of_classes": round(sum(v[0] for v in tim.values()) / args.steps, 4),
                                 "note": "the classes add up to the instrumented pass (<= its time with the events); "
                                         "the default step is shorter because neighbouring kernels overlap"},
            "e2e": {"value": round(e2e_all, 2), "unit": "tokens/s", "h2d_bytes_per_step": 4 * (GAMMA + 1),
                    "d2h_bytes_per_step": 8},
            "gpu_launches": int(round(launches * args.steps)),
            "launches_per_step": launches,
            "near_tie_flips_vs_plan": flips,
            "clocks": clk,
        }
        if trace is not None:
            result["trace"] = trace
        result["launch"] = {"headline": "cuda_graph" if graph and graph.get("same_decisions_as_direct") else "direct",
                            "direct_ms_per_step": round(direct_ms, 4), **({"graph": graph} if graph else {})}
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(wdev, kv, table, blocks[args.warmup], tokens / args.steps)
    return result


# ------------------------------------------------------------------ oracle timing
def oracle_sample(wdev, kv, table, block, layers):
    """Host copies of the sampled layers' weights and KV context, as the oracle takes them."""
    import synth
    import synth.device as sd
    from oracle.decoder import Config, DenseWeights
    shape = synth.SHAPES["8b"]
    host_layers = [{k: sd.bf16_to_bits(v) for k, v in wdev["layers"][l].items()} for l in layers]
    cfg = Config(**dict(shape, n_layers=len(layers)), kv_dtype="bf16")
    embed = sd.bf16_to_bits(wdev["embed"])
    lm = sd.bf16_to_bits(wdev["lm_head"])
    W = DenseWeights(cfg, host_layers, embed, sd.bf16_to_bits(wdev["final_norm"]), lm, bf16=True)
    pos = np.arange(CONTEXT)
    ck = [sd.read_positions(kv.k_pools[l], table[0], pos, PAGE).float().cpu().numpy().astype(np.float64)
          for l in layers]
    cv = [sd.read_positions(kv.v_pools[l], table[0], pos, PAGE).float().cpu().numpy().astype(np.float64)
          for l in layers]
    return cfg, W, ck, cv


def time_oracle_layers(cfg, W, ck, cv, block):
    """Seconds for the oracle's decoder layers of one block (the LM head excluded)."""
    from oracle import decoder

    class NoHead:
        def __init__(self, w):
            self.w = w
            self.cfg = w.cfg

        def embed(self, t):
            return self.w.embed(t)

        def layer(self, l):
            return self.w.layer(l)

        def final_norm(self):
            return self.w.final_norm()

        def logits(self, x, rowwise):
            return np.zeros((x.shape[0], 1))

    t0 = time.perf_counter()
    decoder.forward_block(cfg, NoHead(W), ck, cv, block, CONTEXT, rowwise=False)
    return time.perf_counter() - t0


def time_oracle_head(W, block_rows):
    x = np.random.default_rng(0).standard_normal((block_rows, W.cfg.d_model))
    t0 = time.perf_counter()
    W.logits(x, False)
    return time.perf_counter() - t0


def cpu_baseline(wdev, kv, table, block, tokens_per_step):
    cores = len(os.sched_getaffinity(0))
    cfg, W, ck, cv = oracle_sample(wdev, kv, table, block, [0, 1])
    t_layers = time_oracle_layers(cfg, W, ck, cv, block)
    t_head = time_oracle_head(W, len(block))
    t_step = t_layers / 2 * 36 + t_head
    return {"value": round(tokens_per_step / t_step, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "seconds_per_step": round(t_step, 3),
            "sample": "float64 numpy oracle forward of decoder layers 0-1 for one 17-row block at context 4096, "
                      "plus the full LM head; step time = 18 x (two-layer time) + LM-head time; tokens/step "
                      "from the GPU run (the same decode plan)"}


def expected_tokens_per_step(p_keep=P_KEEP, gamma=GAMMA):
    """Tokens per verify of the prefix rule when draft i (1-based) matches w.p. p^i, independently.

    accepted >= i needs drafts 1..i all to match: P = prod_{j<=i} p^j = p^(i(i+1)/2); one more
    token (correction or bonus) is always emitted.
    """
    return 1.0 + sum(p_keep ** (i * (i + 1) // 2) for i in range(1, gamma + 1))


def reference_inputs(layers):
    """Host inputs of the oracle sample, drawn like the GPU workload's, without the CUDA library.

    The sampled layers' weights, the embedding and the LM head come from the same per-tensor
    streams as synth.device.random_bf16_model (drawn on the device by torch, then copied to the
    host); the context keys/values are N(0,1) rounded to bf16.
    """
    import torch

    import synth
    from oracle.decoder import Config, DenseWeights
    shape = synth.SHAPES["8b"]
    ms = synth.matrix_shapes(shape)
    d = shape["d_model"]
    bits = lambda t: t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    one = np.full(d, 0x3F80, np.uint16)  # bf16 1.0
    host_layers = []
    for l in layers:
        host_layers.append({
            "attn_norm": one, "mlp_norm": one,
            "wqkv": bits(synth.device_bf16_normal(ms["wqkv"], 0.02, (l, synth.T_WQKV), "cuda")),
            "wo": bits(synth.device_bf16_normal(ms["wo"], 0.02, (l, synth.T_WO), "cuda")),
            "wgu": bits(synth.device_bf16_normal(ms["wgu"], 0.02, (l, synth.T_WGU), "cuda")),
            "wd": bits(synth.device_bf16_normal(ms["wd"], 0.02, (l, synth.T_WD), "cuda")),
        })
    embed = bits(synth.device_bf16_normal((shape["vocab"], d), 0.02, (0, synth.T_EMBED), "cuda"))
    lm = bits(synth.device_bf16_normal((shape["vocab"], d), 0.02, (0, synth.T_LM_HEAD), "cuda"))
    torch.cuda.empty_cache()
    cfg = Config(**dict(shape, n_layers=len(layers)), kv_dtype="bf16")
    W = DenseWeights(cfg, host_layers, embed, one, lm, bf16=True)
    rng = synth.rng(7, 0)
    kvshape = (CONTEXT, shape["n_kv_heads"], shape["head_dim"])
    to_bf16 = lambda a: torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    ck = [to_bf16(rng.standard_normal(kvshape)) for _ in layers]
    cv = [to_bf16(rng.standard_normal(kvshape)) for _ in layers]
    return cfg, W, ck, cv


def run_reference(args, world, rank, local):
    """The CPU oracle on the same workload; each timed step runs one decoder layer of a verify block.

    The oracle is the reference arm (the pages publish no code). A whole oracle step (36 layers and
    the LM head of a 17-row block) takes minutes, so every step times one layer (layers 0 and 1
    alternating) and the reported step time is extrapolated: 36 x that layer's time + the LM head's
    time (measured once). The CUDA library is not loaded by this arm.
    """
    if rank != 0:
        return None
    import torch
    torch.cuda.set_device(local)
    cfg, W, ck, cv = reference_inputs([0, 1])
    rng = np.random.default_rng(20261202)
    block = [int(rng.integers(0, cfg.vocab))] + [int(x) for x in rng.integers(0, cfg.vocab, size=GAMMA)]
    t_head = time_oracle_head(W, len(block))
    tokens_per_step = expected_tokens_per_step()
    one = cfg.__class__(**dict(cfg.__dict__, n_layers=1))

    class OneLayer:
        def __init__(self, w, l):
            self.w, self.l, self.cfg = w, l, one

        def embed(self, t):
            return self.w.embed(t)

        def layer(self, _):
            return self.w.layer(self.l)

        def final_norm(self):
            return self.w.final_norm()

        def logits(self, x, rowwise):
            return np.zeros((x.shape[0], 1))

    from oracle import decoder
    layer_s = []
    t_run0 = time.perf_counter()
    for s in range(args.warmup + args.steps):
        l = s % 2
        t0 = time.perf_counter()
        decoder.forward_block(one, OneLayer(W, l), [ck[l]], [cv[l]], block, CONTEXT, rowwise=False)
        if s >= args.warmup:
            layer_s.append(time.perf_counter() - t0)
    run_s = time.perf_counter() - t_run0
    t_layer = statistics.mean(layer_s)
    t_step = t_layer * 36 + t_head
    value = tokens_per_step / t_step
    cores = len(os.sched_getaffinity(0))
    sample = ("per timed step: the float64 numpy oracle forward of one decoder layer (layers 0 and 1 "
              "alternating) of one 17-row block at context 4096; the step time is extrapolated as 36 x the "
              "mean layer time + the LM head's time (measured once); tokens/step = 1 + the expected accepted "
              f"drafts of the workload's draft rule ({tokens_per_step:.3f})")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 1),
        "extrapolated_from": {"sample": "one decoder layer per timed step",
                              "sample_ms_per_step": round(t_layer * 1e3, 1),
                              "lm_head_ms": round(t_head * 1e3, 1), "scale": "36 layers + LM head",
                              "timed_loop_s": round(run_s, 2)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (random N(0,0.02) weights, random N(0,1) KV context, random drafts)",
        "config": {"workload": "8B-class bf16 single-request verify, gamma 16 (M=17), context 4096, T=0",
                   "batch": 1, "gamma": GAMMA, "context": CONTEXT, "layers": 36, "d_model": 4096,
                   "vocab": 151936, "parallelism": "rank 0 only"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ GEMM sweep
def run_sweep(args, local):
    """The skinny GEMM alone (sv_linear) on the 8B-class projection and LM-head shapes.

    Activations are a hi/lo bf16 pair, as the verify step passes them. Each shape
    rotates enough weight copies to exceed L2, and the timed launches replay from
    a CUDA graph, so the time is the kernels' alone (no host work between them).
    """
    import ctypes

    import torch

    import synth
    import verify_step_02_b300 as vs
    torch.cuda.set_device(local)
    s = synth.SHAPES["8b"]
    shapes = {"qkv": ((s["n_heads"] + 2 * s["n_kv_heads"]) * s["head_dim"], s["d_model"]),
              "o": (s["d_model"], s["n_heads"] * s["head_dim"]), "gate_up": (2 * s["ffn"], s["d_model"]),
              "down": (s["d_model"], s["ffn"]), "lm_head": (s["vocab"], s["d_model"])}
    peak, peak_kind = measured_peaks()
    ms = [int(v) for v in str(args.sweep_m).split(",")]
    out = {}
    stream = torch.cuda.Stream()
    for name, (n, k) in shapes.items():
        copies = max(1, int(np.ceil(512e6 / (n * k * 2))))
        ws = [synth.device_bf16_normal((n, k), 0.02, (900 + i, 0), "cuda") for i in range(copies)]
        wdtype, bases, bpe = vs.SV_BF16, [0] * copies, 2.0
        if args.sweep_dtype == "w12":
            wdtype, bpe = vs.SV_W12, 1.5
            packed, bases = [], []
            for w in ws:
                bits = torch.randint(0, 2, w.shape, device="cuda", dtype=torch.int32) << 15 | \
                    torch.randint(111, 127, w.shape, device="cuda", dtype=torch.int32) << 7 | \
                    torch.randint(0, 128, w.shape, device="cuda", dtype=torch.int32)
                planes, base = vs.pack_w12(bits.to(torch.int16).view(torch.bfloat16))
                packed.append(planes)
                bases.append(base)
            ws = packed
        for m in ms:
            xf = torch.randn((m, k), device="cuda")
            hi = xf.to(torch.bfloat16)
            x = torch.stack([hi, (xf - hi.float()).to(torch.bfloat16)]).contiguous()
            y = torch.empty((m, n), dtype=torch.float32, device="cuda")
            need = int(vs.lib.sv_linear_workspace_bytes(wdtype, m, n, k))
            wsp = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
            mats = [vs.Matrix(w.data_ptr(), int(b)) for w, b in zip(ws, bases)]
            reps = max(4, min(40, int(4e9 / (n * k * bpe))))

            def launch(i):
                st = vs.lib.sv_linear(wdtype, ctypes.byref(mats[i % copies]), n, k, ctypes.c_void_p(x.data_ptr()),
                                      2, m, ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(wsp.data_ptr()),
                                      wsp.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
                assert st == vs.SV_OK, vs.lib.sv_last_error()

            with torch.cuda.stream(stream):
                for i in range(3):
                    launch(i)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(reps):
                    launch(i)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record()
                g.replay()
                e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) / reps * 1e3
            gbs = n * k * bpe / (us * 1e-6) / 1e9
            out[f"{name}@M{m}"] = {"n": n, "k": k, "m": m, "us": round(us, 2), "gbs": round(gbs, 1),
                                   "frac": round(gbs / peak, 4)}
            del g
        del ws
        torch.cuda.empty_cache()
    return {"sweep": "gemm", "dtype": args.sweep_dtype, "x": "hi/lo bf16 pair", "peak_gbs": peak,
            "peak_kind": peak_kind, "timing": "CUDA-graph replay of back-to-back launches", "shapes": out}


# ------------------------------------------------------------------ step-cost table
STEP_SWEEP_M = (1, 2, 4, 8, 16, 17, 24, 32, 48, 64, 96, 128, 192, 256)
STEP_SWEEP_M_FMA = (1, 2, 4, 8, 16, 17)


def run_sweep_step(args, local):
    """Verify-step time of the 8B-class model per block size M (requests of up to 64 rows).

    M = 1 is one step of plain autoregressive greedy decoding; the table (step
    time and steps per second per M) is what the prefix scheduler
    (sv_schedule_prefix) maximizes tau / T(M) over. Context 4096 per request,
    drafts random (the step's work does not depend on acceptance).
    """
    import torch

    import synth
    import synth.device as sd
    import verify_step_02_b300 as vs
    torch.cuda.set_device(local)
    shape = dict(synth.SHAPES["8b"], n_layers=args.layers or 36)
    max_b, max_g = 4, 63
    steps = args.steps
    reps = len(STEP_SWEEP_M) * (steps + args.warmup)
    max_seq = CONTEXT + reps + 128
    max_seq = (max_seq + PAGE - 1) // PAGE * PAGE
    wdev = sd.random_bf16_model(shape)
    table, n_pages = synth.contiguous_page_table([max_seq] * max_b, PAGE, max_seq // PAGE + 1)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="normal")
    seq = torch.full((max_b,), CONTEXT, dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    flags = vs.SV_FLAG_CUDA_CORE_GEMM if args.cuda_core_gemm else 0
    model = vs.Model(vs.make_config(shape, vs.SV_BF16, max_b, max_g, max_seq, PAGE, flags=flags), wdev)
    rng = np.random.default_rng(5)
    tok = torch.from_numpy(rng.integers(0, shape["vocab"], size=(max_b, max_g + 1)).astype(np.int32)).cuda()
    acc = torch.zeros(max_b, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(max_b, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peaks()
    per_layer, wbytes, kv_row = step_bytes(shape)
    rows = {}
    for M in (STEP_SWEEP_M_FMA if args.cuda_core_gemm else STEP_SWEEP_M):
        b = (M + max_g) // (max_g + 1)
        lens = [M // b - 1 + (1 if r < M % b else 0) for r in range(b)]
        for _ in range(args.warmup):
            model.verify(tok[:b], lens, kv, acc[:b], nxt[:b])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            model.verify(tok[:b], lens, kv, acc[:b], nxt[:b])
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / steps * 1e3
        ctx = float(seq[:b].float().mean().item())
        alg = wbytes + kv_row * b * (ctx + M / b) + kv_row * M
        rows[str(M)] = {"batch": b, "us": round(us, 1), "steps_per_s": round(1e6 / us, 1),
                        "hbm_frac": round(alg / (us * 1e-6) / 1e9 / peak, 4)}
    model.close()
    return {"sweep": "step", "model": "8B-class bf16, 36 layers", "context": CONTEXT, "layers": shape["n_layers"],
            "gemm": "CUDA-core FMA" if args.cuda_core_gemm else "tcgen05 tensor cores",
            "table": rows, "ar_greedy_tokens_per_s": rows["1"]["steps_per_s"], "peak_gbs": peak,
            "peak_kind": peak_kind,
            "note": "M rows per step (requests of up to 64 rows); M = 1 is autoregressive greedy decoding"}


SCHED_B, SCHED_G = 8, 16
SCHED_M = (8, 16, 24, 32, 40, 48, 64, 80, 96, 112, 136)


def run_sweep_schedule(args, local):
    """The prefix scheduler on the device's own step costs (8B-class model, 8 requests at context 4096).

    Measures T(M) for M = 8 .. 136 rows (the requests' lengths as even as possible), takes for every
    M the cost of the next measured point at or above it, draws per-draft confidences c ~ Beta(8, 2) (the 27B workload's draft model),
    chooses the verify lengths with sv_schedule_prefix (with and without early stop), times the
    chosen lengths on the device and compares the expected throughput tau / T with two fixed
    rules: all 16 drafts, and drafts kept while the survival probability stays >= 0.3.
    """
    import torch

    import synth
    import synth.device as sd
    import verify_step_02_b300 as vs
    torch.cuda.set_device(local)
    shape = dict(synth.SHAPES["8b"], n_layers=args.layers or 36)
    B, G = SCHED_B, SCHED_G
    reps = (len(SCHED_M) + 4) * (args.steps + args.warmup)
    max_seq = (CONTEXT + reps + 128 + PAGE - 1) // PAGE * PAGE
    wdev = sd.random_bf16_model(shape)
    table, n_pages = synth.contiguous_page_table([max_seq] * B, PAGE, max_seq // PAGE + 1)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="normal")
    seq = torch.full((B,), CONTEXT, dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    model = vs.Model(vs.make_config(shape, vs.SV_BF16, B, G, max_seq, PAGE), wdev)
    rng = np.random.default_rng(8)
    tok = torch.from_numpy(rng.integers(0, shape["vocab"], size=(B, G + 1)).astype(np.int32)).cuda()
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step_us(lens):
        for _ in range(args.warmup):
            model.verify(tok, lens, kv, acc, nxt)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            model.verify(tok, lens, kv, acc, nxt)
        e1.record(stream)
        torch.cuda.synchronize()
        seq.fill_(CONTEXT)
        return e0.elapsed_time(e1) / args.steps * 1e3

    measured = {}
    for M in SCHED_M:
        lens = [M // B - 1 + (1 if r < M % B else 0) for r in range(B)]
        measured[M] = step_us(lens)
    # T(M) between measured points: the cost of the next measured M at or above it (the step cost
    # rises in steps at token-tile boundaries, so a straight line between points would understate it)
    table_us = np.array([measured[min(m for m in SCHED_M if m >= M)] for M in range(1, SCHED_M[-1] + 1)])
    conf = synth.rng(31, 1).beta(8.0, 2.0, size=(B, G)).astype(np.float32)
    surv = np.cumprod(conf.astype(np.float64), axis=1)

    def tau(lens):
        return float(sum(1.0 + surv[r, :lens[r]].sum() for r in range(B)))

    rules = {}
    for name, lens in (("fixed gamma 16", [G] * B),
                       ("survival >= 0.3", [max(1, int((surv[r] >= 0.3).sum())) for r in range(B)])):
        rules[name] = [int(x) for x in lens]
    for early in (False, True):
        lens, _, _ = vs.schedule_prefix(conf, table_us.astype(np.float32), early_stop=early)
        rules["scheduler" + (" (early stop)" if early else "")] = [int(x) for x in lens]
    out = {}
    for name, lens in rules.items():
        M = int(sum(l + 1 for l in lens))
        t_tab = float(table_us[M - 1])
        t_dev = step_us(lens)
        out[name] = {"verify_lens": lens, "M": M, "expected_tokens": round(tau(lens), 3),
                     "table_us": round(t_tab, 1), "device_us": round(t_dev, 1),
                     "expected_tokens_per_s": round(tau(lens) / (t_dev * 1e-6), 1)}
    model.close()
    return {"sweep": "schedule", "model": "8B-class bf16", "layers": shape["n_layers"], "batch": B, "gamma": G,
            "context": CONTEXT, "step_us_measured": {str(m): round(v, 1) for m, v in measured.items()},
            "rules": out,
            "note": "expected tokens = sum_r (1 + sum_{j <= L_r} prod_{i <= j} c_{r,i}), c ~ Beta(8, 2); "
                    "device_us times the chosen lengths on this GPU"}


# ------------------------------------------------------------------ the other configurations
WORKLOADS = {
    "tiny": "tiny fp32 greedy verify: 2 layers, d 256, 4 x 64 heads, vocab 1024; batch 1, gamma 4, context 64",
    "27b": "27B-class bf16 ragged verify: 64 layers, d 5120, 40 q / 8 kv heads; batch 32, contexts uniform "
           "512-8192 on shuffled 16-token pages, verify lengths 1-16 by confidence truncation; greedy",
    "w12": "8B-class verify with W12 weights (16-binade window): batch 1, gamma 16, context 4096; greedy",
    "tree": "8B-class bf16 token-tree verify: batch 1, random 32-node trees (at most 3 children per node) whose "
            "drafts follow the engine's greedy continuation w.p. 0.9 per node, context 4096; greedy",
    "w12g": "8B-class verify with grouped W12 weights (N(0, 0.02) bf16 weights, per-64-row bases and escapes): "
            "batch 1, gamma 16, context 4096; greedy",
    "sampled": "tiny fp32 sampled verify: batch 64, context 2048, gamma 8, T = 1, rejection sampling",
}


def run_workload(args, world, rank, local):
    """Time one of the other verify configurations (timing only; parity is in the tests)."""
    import torch

    import synth
    import synth.device as sd
    import verify_step_02_b300 as vs

    torch.cuda.set_device(local)
    wl = args.workload
    rng = np.random.default_rng(20261202)
    steps_total = args.warmup + args.steps
    temperature, probs = 0.0, None

    def shape_of(name):
        sh = synth.SHAPES[name]
        return dict(sh, n_layers=args.layers) if args.layers else sh
    if wl in ("tiny", "sampled"):
        shape = shape_of("tiny")
        kind, wdtype, kvdt = "f32", vs.SV_F32, torch.float32
        B, gamma = (1, 4) if wl == "tiny" else (64, 8)
        ctx = np.full(B, 64 if wl == "tiny" else 2048)
        lens = np.full(B, gamma)
        wdev = sd.host_to_device_weights(synth.host_weights(shape, "f32"), "f32")
    elif wl == "27b":
        shape = shape_of("27b")
        kind, wdtype, kvdt = "bf16", vs.SV_BF16, torch.bfloat16
        B, gamma = 32, 16
        ctx = rng.integers(512, 8193, size=B)
        lens = synth.truncated_verify_lens(B, gamma, 0.3, 31, 0)
        wdev = sd.random_bf16_model(shape)
    elif wl == "tree":
        shape = shape_of("8b")
        kind, wdtype, kvdt = "bf16", vs.SV_BF16, torch.bfloat16
        B, gamma = 1, TREE_NODES - 1
        ctx = np.full(B, CONTEXT)
        lens = np.full(B, gamma)
        wdev = sd.random_bf16_model(shape)
    elif wl == "w12g":  # the random N(0, 0.02) bf16 model itself, packed losslessly
        shape = shape_of("8b")
        kind, wdtype, kvdt = "w12", vs.SV_W12, torch.bfloat16
        B, gamma = 1, 16
        ctx = np.full(B, CONTEXT)
        lens = np.full(B, gamma)
        wdev = sd.random_bf16_model(shape)
        for lay in wdev["layers"]:
            for name in ("wqkv", "wo", "wgu", "wd"):
                lay[name] = vs.pack_w12_grouped(lay[name])
        wdev["lm_head"] = vs.pack_w12_grouped(wdev["lm_head"])
    else:  # w12
        shape = shape_of("8b")
        kind, wdtype, kvdt = "w12", vs.SV_W12, torch.bfloat16
        B, gamma = 1, 16
        ctx = np.full(B, CONTEXT)
        lens = np.full(B, gamma)
        wdev = sd.random_bf16_model(shape)

        def w12(t, seed):
            g = torch.Generator(device="cuda")
            g.manual_seed(seed)
            bits = (torch.randint(0, 2, t.shape, device="cuda", generator=g, dtype=torch.int32) << 15) | \
                (torch.randint(111, 127, t.shape, device="cuda", generator=g, dtype=torch.int32) << 7) | \
                torch.randint(0, 128, t.shape, device="cuda", generator=g, dtype=torch.int32)
            return vs.pack_w12(bits.to(torch.int16).view(torch.bfloat16))
        for l, lay in enumerate(wdev["layers"]):
            for i, name in enumerate(("wqkv", "wo", "wgu", "wd")):
                lay[name] = w12(lay[name], 1000 * l + i)
        wdev["lm_head"] = w12(wdev["lm_head"], 99999)
    V = shape["vocab"]
    lengths = [int(c) + steps_total * (gamma + 1) + 16 for c in ctx]
    max_pages = max((n + PAGE - 1) // PAGE for n in lengths) + 1
    table, n_pages = synth.shuffled_page_table(lengths, PAGE, max_pages, 77, 0)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, kvdt, fill="normal")
    seq = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    max_seq = max(lengths) + 16
    model = vs.Model(vs.make_config(shape, wdtype, B, gamma, max_seq, PAGE), wdev)
    tok = torch.from_numpy(rng.integers(0, V, size=(B, gamma + 1)).astype(np.int32)).cuda()
    if wl == "sampled":
        temperature = 1.0
        z = torch.randn((B, gamma, V), device="cuda") * 3.0
        probs = torch.softmax(z, dim=-1).contiguous()
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    rid = torch.arange(B, dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream()

    blocks_d = None
    if wl == "tree":
        g = greedy_reference(model, kv, int(tok[0, 0].item()), steps_total * 12 + 24, gamma + 1)
        tblocks, tparents = make_tree_plan(g, steps_total, V)
        blocks_d = torch.from_numpy(tblocks).cuda()
        parents_d = torch.from_numpy(tparents).cuda()
        nodes = torch.zeros((1, gamma + 1), dtype=torch.int32, device="cuda")
        seq.copy_(torch.from_numpy(ctx.astype(np.int32)))
    elif wl == "tiny":
        # the configuration's draft rule: draft i is the target's greedy token with probability
        # 0.8^(i+1), from the same engine's greedy run (then the KV context is reset)
        g = greedy_reference(model, kv, int(tok[0, 0].item()), steps_total * (gamma + 1) + gamma + 8, gamma + 1)
        blocks, _ = make_plan(g, steps_total, V, gamma, 0.8)
        blocks_d = torch.from_numpy(blocks).cuda()
        seq.copy_(torch.from_numpy(ctx.astype(np.int32)))

    # one request: every step's accepted count kept apart (compared with the graph replays)
    acc_steps = torch.zeros(steps_total, dtype=torch.int32, device="cuda")

    def run(i):
        if wl == "tree":
            model.verify_tree(blocks_d[i:i + 1], parents_d[i:i + 1], lens, kv, acc, nxt, nodes)
            return
        a_out = acc_steps[i:i + 1] if wl == "tiny" else acc
        model.verify(tok if blocks_d is None else blocks_d[i:i + 1], lens, kv, a_out, nxt, draft_probs=probs,
                     temperature=temperature, seed=1234 + i, request_ids=rid)

    clocks = ClockSampler(local)
    for i in range(args.warmup):
        run(i)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    acc_sum = torch.zeros(B, dtype=torch.int64, device="cuda")
    barrier(world)
    torch.cuda.synchronize()
    seq_start = seq.cpu().numpy().astype(np.int64)
    ev[0].record(stream)
    for j in range(args.steps):
        run(args.warmup + j)
        ev[j + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    seq_end = seq.cpu().numpy().astype(np.int64)
    graph = None
    if wl == "tiny" and not args.no_graph:
        # the same steps replayed from one CUDA graph of the verify; the headline when the
        # replays accept exactly as the direct launches did
        direct = acc_steps.cpu().numpy()[args.warmup:].tolist()
        graph = graph_replay(model, kv, blocks_d, args, stream, world, gamma=gamma, context=int(ctx[0]))
        if "accepted" in graph:
            graph["same_decisions_as_direct"] = graph.pop("accepted")[args.warmup:] == direct
            g_steps = graph.pop("per_step")
            graph["direct_ms_per_step"] = round(ev[0].elapsed_time(ev[-1]) / args.steps, 4)
            if graph["same_decisions_as_direct"]:
                per_step_graph = g_steps
                t_ms = graph["ms_per_step"] * args.steps
        seq.copy_(torch.from_numpy(seq_end.astype(np.int32)))
    # per-kernel-class device time from an instrumented pass (events between launches)
    model.set_timing(True)
    for j in range(args.steps):
        run(args.warmup + j)
    torch.cuda.synchronize()
    tim = model.timing()
    model.set_timing(False)
    clk = clocks.stop()
    trace = None
    if args.trace:  # device timeline of two more steps
        n_layers = shape["n_layers"]
        cap = 2 * (n_layers * (4 * 148 + 2 * 148) + 2 * 148)
        recs = torch.zeros((cap, 16), dtype=torch.int64, device="cuda")
        model.set_trace(recs)
        for j in range(2):
            run(args.warmup + args.steps + j)
        torch.cuda.synchronize()
        launches = model.trace_launches()
        model.set_trace(None)
        raw = recs.cpu().numpy().view(np.uint64)
        trace = trace_summary(raw, launches, n_layers)
        if args.trace_out:
            np.savez_compressed(args.trace_out, records=raw, launches=np.array([l[:2] for l in launches]),
                                kinds=np.array([l[2] for l in launches]))
    per_step = [ev[j].elapsed_time(ev[j + 1]) for j in range(args.steps)]
    if graph is not None and graph.get("same_decisions_as_direct"):
        per_step = per_step_graph
    else:
        t_ms = ev[0].elapsed_time(ev[-1])
    tokens = float((seq_end - seq_start).sum())  # accepted drafts + 1 per request per step
    value, t_max = aggregate(tokens, t_ms, world)
    if rank != 0:
        return None
    peak, peak_kind = measured_peaks()
    per_layer, wbytes, kv_row = step_bytes(shape)
    wscale = {"f32": 2.0, "bf16": 1.0, "w12": 0.75}[kind]
    kv_bytes = kv_row * (1.0 if kind != "f32" else 2.0)
    M = int(np.sum(np.asarray(lens) + 1))
    ctx_mean = (seq_start + seq_end) / 2.0
    step_alg = wbytes * wscale + kv_bytes * float(np.sum(ctx_mean + np.asarray(lens) + 1)) + kv_bytes * M
    ms_step = t_max / args.steps
    return {
        "metric": METRIC, "workload": wl, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "dtype": {"f32": "f32", "bf16": "bf16", "w12": "bf16 (W12 weights)"}[kind],
        "data": "synthetic (random weights, random N(0,1) KV context, " + (
            "greedy-mix drafts: the engine's greedy token w.p. 0.8^(i+1), else uniform)" if wl == "tiny"
            else "uniform random drafts)"),
        "config": {"workload": WORKLOADS[wl], "batch": B, "gamma": gamma, "M": M, "layers": shape["n_layers"]},
        "verify_us": {"median": round(1e3 * statistics.median(per_step), 1),
                      "p90": round(1e3 * float(np.percentile(per_step, 90)), 1)},
        "tokens_per_step": round(tokens / args.steps, 3),
        "hbm": {"bytes_per_step": step_alg, "gbs": round(step_alg / (ms_step * 1e-3) / 1e9, 1),
                "frac_of_peak": round(step_alg / (ms_step * 1e-3) / 1e9 / peak, 4), "peak_gbs": peak,
                "peak_kind": peak_kind, "bound_ms": round(step_alg / (peak * 1e9) * 1e3, 4)},
        "kernel_ms_per_step": {k: round(v[0] / args.steps, 4) for k, v in tim.items()},
        "clocks": clk,
        "launch": "CUDA graph replay" if graph is not None and graph.get("same_decisions_as_direct")
        else "direct launches",
        **({"graph": graph} if graph else {}),
        **({"trace": trace} if trace else {}),
    }


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.sweep == "gemm":
        res = run_sweep(args, local)
    elif args.sweep == "step":
        res = run_sweep_step(args, local)
    elif args.sweep == "schedule":
        res = run_sweep_schedule(args, local)
    elif args.workload != "8b" and args.impl == "ours":
        res = run_workload(args, world, rank, local)
    elif args.impl == "reference":
        res = run_reference(args, world, rank, local)
    else:
        res = run_ours(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
