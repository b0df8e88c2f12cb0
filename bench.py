"""Benchmark of one DDTree verification round (build + tree attention + tree GDN + walk +
commit) on the batched workload: 32 requests, drafter depth 15, vocabulary 151936,
budget 64, prefixes ~ U[1024, 32768], 16 full-attention layers (Hq 24, Hkv 4, d 256) and
48 GDN layers (Hk 16, Hv 48, dk = dv = 128), bf16 data, fp32 state.

Prints ONE JSON line (rank 0).  `value` = drafted tree nodes verified per second over
the whole job (all ranks), with every input resident in HBM; `e2e` is the same metric
with each round's inputs copied from pinned host memory and its emitted tokens copied
back inside the timed region.  `--impl reference` times the plain CPU oracle instead.

Multi-GPU: requests are independent, so N ranks run N independent replicas of the
workload (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "verified tree nodes/sec per round at 1 GB300; achieved HBM GB/s vs peak"
UNIT = "nodes/s"
WORKLOAD = 5
KERNELS = ("build", "attn", "gdn", "walk", "commit")


# ---------------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def all_max(x, world, dev):
    if world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def all_sum(x, world, dev):
    if world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken during the timed region."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, path):
        self.path = path
        self.proc = None

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader",
                                          "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, uuid):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10 or (uuid and f[1] != uuid):
                continue
            try:
                sm.append(float(f[2].split()[0]))
                mx.append(float(f[3].split()[0]))
            except ValueError:
                continue
            for n, v in zip(names, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_uuid():
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        return None


# ------------------------------------------------------------------- accounting
def attn_flops_bytes(r):
    """Algorithmic work of one ddt_tree_attn launch: 4*d flops per (query row, visible
    key); bytes = prefix K/V once per (layer, request, kv head) + tree K/V + q + o."""
    c = r.cfg
    depth = r.tree["depth"].cpu().numpy()
    nn = r.tree["n_nodes"].cpu().numpy()
    P = r.prefix0.cpu().numpy().astype(np.float64)
    keys = 0.0
    for b in range(len(nn)):
        keys += float(nn[b]) * P[b] + float((depth[b, :nn[b]] + 1).sum())
    flops = 4.0 * c["d"] * c["Hq"] * r.Lf * keys
    esz = 2 if c["dtype"] == torch.bfloat16 else 4
    bytes_ = r.Lf * c["Hkv"] * c["d"] * esz * 2 * float(P.sum())
    bytes_ += r.Lf * float(nn.sum()) * c["d"] * esz * (2 * c["Hkv"] + c["Hq"] + c["Hq"])
    return flops, bytes_


def round_bytes(r):
    """Algorithmic HBM bytes of the whole round (read + write once)."""
    c = r.cfg
    esz = 2 if c["dtype"] == torch.bfloat16 else 4
    B, D, V, N = c["B"], c["D"], c["V"], r.N
    total = B * D * V * esz + B * N * V * esz                     # drafter + target logits
    if r.Lf:
        total += attn_flops_bytes(r)[1]
        total += 2 * r.Lf * B * (D + 1) * c["Hkv"] * c["d"] * esz  # commit: copied KV rows (upper bound)
    if r.Lg:
        C = 2 * c["Hk"] * c["dk"] + c["Hv"] * c["dv"]
        S = r.Lg * B * c["Hv"] * c["dk"] * c["dv"] * 4
        total += S + r.Lg * B * N * C * esz + r.Lg * B * N * c["Hv"] * c["dv"] * esz  # tree GDN
        total += 2 * S                                                             # commit of the state
    return float(total)


# DRAM bytes (read + write) of one k_attn_tc launch, from an ncu capture of the bench's
# own timed launch (dram__bytes_read.sum + dram__bytes_write.sum, one pass, full size),
# keyed by the SHA-256 of the kernel's sources: once they change, the figure is stale
# and the bench reports null until it is captured again.
ATTN_TRAFFIC = {
    # ncu, batched round, mean of the three timed launches of one capture:
    # dram__bytes_read.sum 40,355,763,541 B + dram__bytes_write.sum 400,794,795 B
    "bfdc4160d21e99d36f74f45bb592cfea7ca3e4b2aade0e9bd2f1fe0da592e0a8": {"workload": 5, "bytes": 40756558336.0},
}
ATTN_SOURCES = ("attn_tc.cu", "tc.cuh")


def attn_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in ATTN_SOURCES:
        with open(os.path.join(ROOT, "tree_speculative_decoding_02_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def attn_traffic(workload):
    rec = ATTN_TRAFFIC.get(attn_source_hash())
    if rec is None or rec["workload"] != workload:
        return None
    return rec["bytes"]


def workload_desc(c):
    parts = [c["name"] + ":", f"B={c['B']}, D={c['D']}, V={c['V']}, budget {c['budget']}, top-k {c['top_k']}"]
    if "P_lo" in c:
        parts.append(f"P~U[{c['P_lo']},{c['P_hi']}]")
    elif c.get("P"):
        parts.append(f"P={c['P']}")
    if c.get("Lf"):
        parts.append(f"{c['Lf']} attn layers Hq{c['Hq']}/Hkv{c['Hkv']}/d{c['d']}")
    if c.get("Lg"):
        parts.append(f"{c['Lg']} GDN layers Hk{c['Hk']}/Hv{c['Hv']}/dk=dv={c['dk']}")
    return ", ".join(parts)


def arm_config(cfg, prefix_total, nodes_per_round, world):
    """The `config` object both arms print."""
    return {"workload": workload_desc(cfg), "B": cfg["B"], "budget": cfg["budget"],
            "nodes_per_round": nodes_per_round, "prefix_total": prefix_total,
            "l2": "inputs larger than L2 (tens of GB per round)", "parallelism": f"replicas x{world}"}


# --------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local):
    from tree_speculative_decoding_02_gb300 import ddt, synth
    from tree_speculative_decoding_02_gb300.round import Round

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    ddt.load()
    cfg = dict(synth.WORKLOADS[args.workload])
    if "budget" not in cfg:          # the build-and-walk workload lists budgets: time the largest
        cfg["budget"] = max(cfg["budgets"])
    if args.kv_page:
        cfg["page"] = args.kv_page
    cfg["flat"] = args.flat
    r = Round(cfg, device=dev, workload=args.workload)
    st = torch.cuda.current_stream()
    ev = {k: [] for k in KERNELS}

    # the five calls, each bracketed by events on the launching stream; a workload
    # without attention (or GDN) layers has no such call in its round
    def step(timed):
        r.restore_prefix()
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(6)] if timed else None
        if timed:
            marks[0].record(st)
        c = r.cfg
        ddt.ddt_build_tree(r.draft_logits, r.root_token, r.prefix_len, c["top_k"], c["budget"], out=r.tree,
                           workspace=r.build_ws)
        if timed:
            marks[1].record(st)
        kw = {}
        if r.Lf and r.page:
            a = r.attn
            ddt.ddt_tree_attn_paged(a.q, a.k_tree, a.v_tree, r.k_pages, r.v_pages, r.block_table, r.prefix_len,
                                    r.tree["n_nodes"], r.tree["anc"], scale=1.0 / math.sqrt(c["d"]), out=r.attn_o,
                                    status=r.attn_status, workspace=r.attn_ws)
        elif r.Lf:
            a = r.attn
            ddt.ddt_tree_attn(a.q, a.k_tree, a.v_tree, a.k_cache, a.v_cache, r.prefix_len, r.tree["n_nodes"],
                              r.tree["anc"], scale=1.0 / math.sqrt(c["d"]), out=r.attn_o, status=r.attn_status,
                              workspace=r.attn_ws)
            kw.update(k_tree=a.k_tree, v_tree=a.v_tree, k_cache=a.k_cache, v_cache=a.v_cache)
        if timed:
            marks[2].record(st)
        if r.Lg:
            g = r.gdn
            ddt.ddt_tree_gdn(g.x, g.conv_w, g.conv_state, g.beta, g.decay, g.S, r.tree["parent"],
                             r.tree["n_nodes"], Hk=c["Hk"], out=r.gdn_o, status=r.gdn_status)
            kw.update(x=g.x, conv_w=g.conv_w, beta=g.beta, decay=g.decay, S=g.S, conv_state=g.conv_state,
                      Hk=c["Hk"])
        if timed:
            marks[3].record(st)
        ddt.ddt_walk_accept(r.tree["token"], r.tree["parent"], r.tree["n_nodes"], r.A - 1,
                            target_logits=r.target_logits, out=r.walk, workspace=r.walk_ws, flat=args.flat)
        if timed:
            marks[4].record(st)
        if not (r.Lf or r.Lg):
            pass                       # nothing is cached: the round ends with the walk
        elif r.Lf and r.page:
            ddt.ddt_commit_paged(r.walk["acc_nodes"], r.walk["acc_len"], r.prefix_len, r.block_table,
                                 k_tree=r.attn.k_tree, v_tree=r.attn.v_tree, k_pages=r.k_pages, v_pages=r.v_pages,
                                 out=r.commit, **kw)
        else:
            ddt.ddt_commit(r.walk["acc_nodes"], r.walk["acc_len"], r.prefix_len, out=r.commit, **kw)
        if timed:
            marks[5].record(st)
            for i, k in enumerate(KERNELS):
                ev[k].append((marks[i], marks[i + 1]))

    accepted = None
    if args.planted:
        # the tree is a function of the drafter logits: build it once, then boost the
        # target logit of the child token along a path of each request, with lengths drawn
        # from a geometric distribution of mean `planted` (capped at the drafter depth)
        c = r.cfg
        ddt.ddt_build_tree(r.draft_logits, r.root_token, r.prefix_len, c["top_k"], c["budget"], out=r.tree,
                           workspace=r.build_ws)
        torch.cuda.synchronize()
        rng = np.random.default_rng(7)
        lens = np.minimum(rng.geometric(1.0 / (1.0 + args.planted), c["B"]) - 1, c["D"])
        synth.plant_path(r.target_logits, r.tree["token"].cpu().numpy(), r.tree["parent"].cpu().numpy(),
                         r.tree["n_nodes"].cpu().numpy(), lens)
    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    if args.planted:
        accepted = float(r.walk["acc_len"].float().mean())
    nodes_per_step = r.drafted_nodes()
    for k in ("status",):
        bad = int((r.tree[k] != 0).sum())
        if bad:
            raise RuntimeError(f"build reported {bad} request errors")

    # nvidia-smi samples during the timed region; the raw CSV goes to $DDT_CLOCKS_CSV when
    # set, else to a temporary file, and its summary into the JSON line
    clocks = None
    if rank == 0:
        import tempfile
        path = os.environ.get("DDT_CLOCKS_CSV") or os.path.join(tempfile.gettempdir(), f"ddt_clocks_{os.getpid()}.csv")
        clocks = ClockSampler(path)
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = ddt.ddt_launch_count()
    t0.record(st)
    for _ in range(args.steps):
        step(True)
    t1.record(st)
    launches = ddt.ddt_launch_count() - launches0
    torch.cuda.synchronize()
    barrier(world)
    ms = t0.elapsed_time(t1)
    clk = clocks.stop(gpu_uuid()) if clocks else None
    ms_max = all_max(ms, world, dev)
    nodes_total = all_sum(nodes_per_step * args.steps, world, dev)
    value = nodes_total / (ms_max / 1e3)
    per_kernel = {k: statistics.mean(a.elapsed_time(b) for a, b in ev[k]) for k in KERNELS}

    # end to end through the public API: each round's inputs are copied from pinned host
    # memory and its emitted tokens copied back, inside the timed region.  The inputs are
    # double-buffered: round i+1's copy runs on a copy stream while round i computes, the
    # way a serving loop overlaps them.  Each copy is split by the call that first reads
    # it (drafter logits, then q / tree K,V, then x and gates, then target logits), and a
    # call waits only for its own group, so even the first round's compute starts early.
    slots = [r.round_inputs()]
    slots.append({k: torch.empty_like(v) for k, v in slots[0].items()})
    host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in slots[0].items()}
    for k, v in slots[0].items():
        host[k].copy_(v)
    outs = r.round_outputs()
    host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    cs = torch.cuda.Stream(device=dev)
    groups = r.input_groups()
    copied = [{n: torch.cuda.Event() for n in groups} for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def copy_in(slot):
        with torch.cuda.stream(cs):
            cs.wait_event(free[slot])
            for n, names in groups.items():
                for k in names:
                    slots[slot][k].copy_(host[k], non_blocking=True)
                copied[slot][n].record(cs)

    def e2e_run(n):
        for sl in range(2):
            free[sl].record(st)
        copy_in(0)
        for i in range(n):
            sl = i % 2
            if i + 1 < n:
                copy_in(1 - sl)
            r.bind_inputs(slots[sl])
            r.restore_prefix()
            r.step(wait=lambda name, sl=sl: st.wait_event(copied[sl][name]))
            free[sl].record(st)
            for k, v in outs.items():
                host_out[k].copy_(v, non_blocking=True)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n_e2e = max(2, args.steps)
    e0.record(st)
    e2e_run(n_e2e)
    e1.record(st)
    torch.cuda.synchronize()
    barrier(world)
    r.bind_inputs(slots[0])
    e_ms = all_max(e0.elapsed_time(e1), world, dev)
    e2e_value = all_sum(nodes_per_step * n_e2e, world, dev) / (e_ms / 1e3)

    peaks = {}
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk_path):
        peaks = json.load(open(pk_path))
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    tc_peak = float(peaks.get("bf16_tflops_sustained", 1700.0))
    fl, by = attn_flops_bytes(r) if r.Lf else (0.0, 0.0)
    attn_ms = per_kernel["attn"]
    tflops = fl / (attn_ms / 1e3) / 1e12 if r.Lf else 0.0
    rb = round_bytes(r)
    step_ms = ms / args.steps
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": arm_config(cfg, int(r.prefix0.sum()), nodes_per_step, world),
        "hbm_gbs_round": rb / (step_ms / 1e3) / 1e9,
        "hbm_frac_round": rb / (step_ms / 1e3) / 1e9 / hbm_peak,
        "per_kernel_ms": per_kernel,
        "roofline": {"bound": "tensor", "kernel": "ddt_tree_attn", "achieved": tflops, "peak": tc_peak,
                     "unit": "TFLOP/s", "frac": tflops / tc_peak, "traffic": attn_traffic(args.workload),
                     "algorithmic_flops": fl, "algorithmic_bytes": by, "peak_note": "of measured (sustained)"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "inputs": "pinned host, double-buffered: round i+1 copied on a copy stream during round i; "
                          "each call waits for its own input group"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if args.flat:
        out["config"]["walk"] = "flat-commit safe mode (first children only)"
    if args.planted:
        out["config"]["acceptance"] = (f"planted paths, geometric lengths of mean {args.planted}; "
                                       f"mean accepted drafted nodes {accepted:.2f}")
    if args.kv_page:
        out["config"]["kv"] = f"paged: {args.kv_page} rows a page, shuffled block table"
        out["roofline"]["traffic"] = None   # the recorded capture is of the contiguous layout
    if rank == 0 and world == 1 and not args.no_cpu_baseline and r.Lf and r.Lg and not args.kv_page:
        out["cpu_baseline"] = cpu_baseline(r, seconds=args.cpu_seconds)
    return out


# ------------------------------------------------------------- oracle (CPU) timing
def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def request_from_round(r, b):
    """One request's inputs of a GPU Round, as fp64 host arrays for the oracle."""
    P = int(r.prefix0[b])
    a, g = r.attn, r.gdn
    return {"P": P, "draft_logits": _f64(r.draft_logits[b:b + 1]), "root": r.root_token[b:b + 1].cpu().numpy(),
            "target_logits": _f64(r.target_logits[b:b + 1]), "q": _f64(a.q[:, b:b + 1]),
            "k_tree": _f64(a.k_tree[:, b:b + 1]), "v_tree": _f64(a.v_tree[:, b:b + 1]),
            "k_cache": _f64(a.k_cache[:, b:b + 1, :, :P]), "v_cache": _f64(a.v_cache[:, b:b + 1, :, :P]),
            "x": _f64(g.x[:, b:b + 1]), "conv_w": _f64(g.conv_w), "conv_state": _f64(g.conv_state[:, b:b + 1]),
            "beta": _f64(g.beta[:, b:b + 1]), "decay": _f64(g.decay[:, b:b + 1]),
            "S": np.swapaxes(_f64(g.S[:, b:b + 1]), -1, -2)}


def workload_prefixes(cfg, workload):
    """The committed prefix lengths of the workload's requests (as the GPU round draws them)."""
    from tree_speculative_decoding_02_gb300 import synth

    if "P" in cfg:
        return np.full(cfg["B"], cfg["P"], np.int64)
    return synth.prefix_lengths(cfg["B"], cfg["P_lo"], cfg["P_hi"], g=synth.gen(workload, 2)).numpy().astype(np.int64)


def request_synth(cfg, b, workload, Lf=None, Lg=None):
    """One request of the workload drawn directly with the synth module (B = 1), for the
    reference arm, which must not touch the CUDA library.  Lf / Lg: how many attention /
    GDN layers to draw (default: all)."""
    from tree_speculative_decoding_02_gb300 import synth

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = 100 * workload + b
    P = int(workload_prefixes(cfg, workload)[b])
    N = cfg["budget"] + 1
    dt = cfg["dtype"]
    a = synth.attn_inputs(Lf or cfg["Lf"], 1, N, cfg["Hq"], cfg["Hkv"], cfg["d"], P, [P], workload=wl, dtype=dt,
                          device=dev, poison=False)
    g = synth.gdn_inputs(Lg or cfg["Lg"], 1, N, cfg["Hk"], cfg["Hv"], cfg["dk"], cfg["dv"], cfg["conv_k"],
                         workload=wl, dtype=dt, device=dev)
    return {"P": P, "draft_logits": _f64(synth.draft_logits(1, cfg["D"], cfg["V"], std=cfg["logit_std"],
                                                           boost=cfg["boost"], g=synth.gen(wl, 1), dtype=dt)),
            "root": np.array([b], np.int32),
            "target_logits": _f64(synth.target_logits(1, N, cfg["V"], g=synth.gen(wl, 30), dtype=dt)),
            "q": _f64(a.q), "k_tree": _f64(a.k_tree), "v_tree": _f64(a.v_tree), "k_cache": _f64(a.k_cache),
            "v_cache": _f64(a.v_cache), "x": _f64(g.x), "conv_w": _f64(g.conv_w), "conv_state": _f64(g.conv_state),
            "beta": _f64(g.beta), "decay": _f64(g.decay), "S": _f64(g.S)}


def oracle_round(cfg, q):
    """One request's round (build, attention, GDN, walk, commit) through the plain oracle
    on the layers present in `q`; the attention and GDN stages and the commit are scaled
    to the workload's full layer counts (the work is the same for every layer).  Returns
    (drafted nodes, seconds)."""
    import oracle

    P = q["P"]
    sa = cfg["Lf"] / q["q"].shape[0]
    sg = cfg["Lg"] / q["x"].shape[0]
    t0 = time.perf_counter()
    tree = oracle.build_tree(q["draft_logits"], q["root"], [P], cfg["top_k"], cfg["budget"])
    t1 = time.perf_counter()
    oracle.tree_attn(q["q"], q["k_tree"], q["v_tree"], q["k_cache"], q["v_cache"], [P], tree["n_nodes"],
                     tree["anc"], 1.0 / math.sqrt(cfg["d"]))
    t2 = time.perf_counter()
    oracle.tree_gdn(q["x"], q["conv_w"], q["conv_state"], q["beta"], q["decay"], q["S"], tree["parent"],
                    tree["n_nodes"], cfg["Hk"])
    t3 = time.perf_counter()
    wk = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], cfg["D"], target_logits=q["target_logits"])
    t4 = time.perf_counter()
    pad = ((0, 0), (0, 0), (0, 0), (0, cfg["D"] + 1), (0, 0))
    kc, vc = np.pad(q["k_cache"], pad), np.pad(q["v_cache"], pad)
    t5 = time.perf_counter()
    oracle.commit(wk["acc_nodes"], wk["acc_len"], [P], k_tree=q["k_tree"], v_tree=q["v_tree"], k_cache=kc,
                  v_cache=vc, x=q["x"], conv_w=q["conv_w"], beta=q["beta"], decay=q["decay"], S=q["S"],
                  conv_state=q["conv_state"], Hk=cfg["Hk"])
    t6 = time.perf_counter()
    el = (t1 - t0) + sa * (t2 - t1) + sg * (t3 - t2) + (t4 - t3) + max(sa, sg) * (t6 - t5)
    return int(tree["n_nodes"][0]) - 1, el


def cpu_baseline(r, seconds=15.0, max_requests=8):
    import oracle

    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    oracle.build()
    nodes, t_oracle, done = 0, 0.0, []
    for b in range(min(max_requests, r.cfg["B"])):
        n, t = oracle_round(r.cfg, request_from_round(r, b))
        nodes += n
        t_oracle += t
        done.append(b)
        if t_oracle >= seconds:
            break
    return {"value": nodes / t_oracle, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"full round (build, 16-layer tree attention, 48-layer tree GDN, walk, commit) of "
                      f"requests {done} of the batched workload, fp64, {t_oracle:.1f} s of oracle time"}


def run_reference(args, rank, world):
    """The reference arm: the plain CPU oracle.  Each step is one request's round on a
    quarter of the attention and GDN layers, scaled to the full layer counts."""
    if rank != 0:
        return None
    import oracle
    from tree_speculative_decoding_02_gb300 import synth

    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    oracle.build()
    cfg = dict(synth.WORKLOADS[args.workload])
    lf, lg = max(1, cfg.get("Lf", 0) // 4), max(1, cfg.get("Lg", 0) // 4)

    def one(i):
        return oracle_round(cfg, request_synth(cfg, i % cfg["B"], args.workload, Lf=lf, Lg=lg))

    for i in range(args.warmup):
        one(i)
    nodes, el = 0, 0.0
    for i in range(args.steps):
        n, t = one(args.warmup + i)
        nodes += n
        el += t
    v = nodes / el
    sample = (f"per step one request's round (budget {cfg['budget']}), build and walk in full, {lf} of "
              f"{cfg['Lf']} attention and {lg} of {cfg['Lg']} GDN layers timed and scaled to all layers; "
              f"fp64 oracle time only")
    prefix = workload_prefixes(cfg, args.workload)
    return {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": arm_config(cfg, int(prefix.sum()), cfg["B"] * cfg["budget"], world),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flat", action="store_true", help="flat-commit safe mode: walk first children only")
    ap.add_argument("--planted", type=float, default=0.0,
                    help="plant accepted paths with this mean length (0: random targets, little accepted)")
    ap.add_argument("--kv-page", type=int, default=0,
                    help="paged prefix caches with this many rows a page (0: contiguous)")
    args = ap.parse_args()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
