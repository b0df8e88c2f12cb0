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


def attn_issued_flops(r):
    """FLOPs the pair attention kernel issues to the tensor cores in one launch (head sizes
    128 and 256, no prefix split): every 256-row pair tile of a (layer, request, kv head)
    multiplies every 128-key tile, as one Q K^T and two P V passes (the two bf16 parts of P);
    padding rows and masked keys included."""
    c = r.cfg
    nn = r.tree["n_nodes"].cpu().numpy()
    P = r.prefix0.cpu().numpy()
    G = c["Hq"] // c["Hkv"]
    tiles = 0
    for b in range(len(nn)):
        pairs = -(-(r.N * G) // 256)
        keys = -(-int(P[b]) // 128) + -(-int(nn[b]) // 128)
        tiles += pairs * keys
    return float(tiles) * r.Lf * c["Hkv"] * 2.0 * 3 * 256 * 128 * c["d"]


def call_work(r):
    """Algorithmic work of each call of one round: {call: (bytes, flops)}; bytes are read +
    written once, flops are the attention contraction's (4 d per query row and visible key)."""
    c = r.cfg
    esz = 2 if c["dtype"] == torch.bfloat16 else 4
    B, D, V, N = c["B"], c["D"], c["V"], r.N
    acc = r.walk["acc_len"].cpu().numpy().astype(np.float64) + 1.0     # committed rows per request
    work = {"build": (float(B * D * V * esz), 0.0), "walk": (float(B * N * V * esz), 0.0)}
    commit = 0.0
    if r.Lf:
        fl, by = attn_flops_bytes(r)
        work["attn"] = (by, fl)
        commit += 2.0 * r.Lf * c["Hkv"] * c["d"] * esz * 2.0 * float(acc.sum())   # K and V rows: read + write
    if r.Lg:
        C = 2 * c["Hk"] * c["dk"] + c["Hv"] * c["dv"]
        S = float(r.Lg * B * c["Hv"] * c["dk"] * c["dv"] * 4)
        oesz = r.gdn_o.element_size()
        x = float(r.Lg * B * N * C * esz)
        gates = float(r.Lg * B * N * c["Hv"] * 4 * 2)
        conv = float(r.Lg * C * c["conv_k"] * esz + r.Lg * B * (c["conv_k"] - 1) * C * esz)
        work["gdn"] = (S + x + gates + conv + float(r.Lg * B * N * c["Hv"] * c["dv"] * oesz), 0.0)
        # the state read and written once; the path's x rows and gates; the conv state
        commit += 2.0 * S + float(r.Lg * C * esz) * float(acc.sum()) + 2.0 * r.Lg * (c["conv_k"] - 1) * C * esz * B
    if r.Lf or r.Lg:
        work["commit"] = (commit, 0.0)
    return work


def floors_ms(work, hbm_gbs, tc_tflops):
    """Roofline floor of each call: max(bytes / HBM rate, flops / tensor rate), in ms."""
    return {k: max(by / (hbm_gbs * 1e9), fl / (tc_tflops * 1e12)) * 1e3 for k, (by, fl) in work.items()}


def load_peaks():
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = json.load(open(pk_path)) if os.path.exists(pk_path) else {}
    src = "measured" if peaks else "fallback"
    return {"hbm_gbs": float(peaks.get("hbm_gbs", 6800.0)), "burst": float(peaks.get("bf16_tflops", 1900.0)),
            "sustained": float(peaks.get("bf16_tflops_sustained", 1700.0)),
            "sm_max_mhz": float(peaks.get("sm_max_mhz", 2070.0)), "source": src}


def tensor_peak(peaks, clk):
    """The bf16 peak that fits the run: the burst figure when the SM clock stayed at (or
    within 5 % of) its maximum under load, else the sustained (power-capped) figure."""
    at_max = clk is not None and clk.get("sm_mhz", 0.0) >= 0.95 * clk.get("sm_max_mhz", peaks["sm_max_mhz"])
    kind = "burst" if at_max else "sustained"
    return peaks[kind], kind


# DRAM traffic of one tree-attention launch, from a small capture: one launch of the
# tree-attn-bf16 workload (1 request, prefix 4096, 16 layers, Hkv 4, d 256: 268 MB of
# prefix K/V, more than L2), ncu dram__bytes_read.sum 286,167,552 B + dram__bytes_write.sum
# 13,430,784 B, against 298,254,336 algorithmic bytes.  Keyed by the attention sources;
# another workload's traffic is this per-algorithmic-byte figure times its own algorithmic
# bytes (each (layer, request, KV head) streams its prefix K/V once, which is almost all of
# the bytes, so traffic grows with sum_b P_b * Lf * Hkv * d).
ATTN_TRAFFIC = {
    "9f69801ee58a5d530efdd885aa6f477e949e50882f7fce1e099c55ccdd8448ff": {
        "workload": 3, "bytes": 299598336.0, "algorithmic_bytes": 298254336.0},
}
ATTN_SOURCES = ("attn_tc.cu", "tc.cuh")


def attn_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in ATTN_SOURCES:
        with open(os.path.join(ROOT, "tree_speculative_decoding_02_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def attn_traffic(algorithmic_bytes):
    """DRAM bytes of one attention launch with these algorithmic bytes, scaled from the
    recorded capture; None when the attention sources have changed since."""
    rec = ATTN_TRAFFIC.get(attn_source_hash())
    if rec is None:
        return None
    return rec["bytes"] * algorithmic_bytes / rec["algorithmic_bytes"]


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


L2_BYTES = 129e6          # the GB300's L2
FLUSH_BYTES = 512 << 20   # written between timed rounds when a round's inputs fit in L2


def round_input_bytes(cfg, prefix_total):
    """Bytes of the inputs one round reads at least once: drafter and target logits, the
    committed prefix K/V, and the committed GDN state."""
    esz = 2 if cfg["dtype"] == torch.bfloat16 else 4
    n = cfg["budget"] + 1
    by = cfg["B"] * (cfg["D"] + n) * cfg["V"] * esz
    if cfg.get("Lf"):
        by += 2 * cfg["Lf"] * cfg["Hkv"] * cfg["d"] * esz * prefix_total
    if cfg.get("Lg"):
        by += cfg["Lg"] * cfg["B"] * cfg["Hv"] * cfg["dk"] * cfg["dv"] * 4
    return float(by)


def needs_flush(cfg, prefix_total):
    """A round whose inputs are under twice the L2 would find them cached on the next
    round: those are timed with an L2 flush between rounds, outside the timed spans."""
    return round_input_bytes(cfg, prefix_total) < 2 * L2_BYTES


def arm_config(cfg, prefix_total, nodes_per_round, world):
    """The `config` object both arms print."""
    by = round_input_bytes(cfg, prefix_total)
    if needs_flush(cfg, prefix_total):
        l2 = (f"L2 flushed between timed rounds ({FLUSH_BYTES >> 20} MB written outside the timed spans); "
              f"inputs {by / 1e6:.1f} MB a round")
    else:
        l2 = f"inputs larger than L2 ({by / 1e9:.2f} GB read a round)"
    return {"workload": workload_desc(cfg), "B": cfg["B"], "budget": cfg["budget"],
            "nodes_per_round": nodes_per_round, "prefix_total": prefix_total,
            "l2": l2, "parallelism": f"replicas x{world}"}


# --------------------------------------------------------------------- our arm
def make_step(r, flat, ev):
    """One round of `r` through the public calls; with timed=True each call is bracketed by
    CUDA events on the launching stream (appended to ev[call]).  A workload without
    attention (or GDN) layers has no such call in its round."""
    from tree_speculative_decoding_02_gb300 import ddt

    st = torch.cuda.current_stream()
    c = r.cfg

    def step(timed):
        r.restore_prefix()
        marks = {}

        def mark(k):
            if timed:
                e = torch.cuda.Event(enable_timing=True)
                e.record(st)
                marks[k] = e

        mark("t0")
        ddt.ddt_build_tree(r.draft_logits, r.root_token, r.prefix_len, c["top_k"], c["budget"], out=r.tree,
                           workspace=r.build_ws)
        mark("build")
        kw = {}
        if r.Lf:
            r.attention()   # (with rotary embedding: the keys' in-place rotation, then the fused call)
            if not r.page:
                a = r.attn
                kw.update(k_tree=a.k_tree, v_tree=a.v_tree, k_cache=a.k_cache, v_cache=a.v_cache)
            mark("attn")
        if r.Lg:
            g = r.gdn
            ddt.ddt_tree_gdn(g.x, g.conv_w, g.conv_state, g.beta, g.decay, g.S, r.tree["parent"],
                             r.tree["n_nodes"], Hk=c["Hk"], out=r.gdn_o, status=r.gdn_status)
            kw.update(x=g.x, conv_w=g.conv_w, beta=g.beta, decay=g.decay, S=g.S, conv_state=g.conv_state,
                      Hk=c["Hk"])
            mark("gdn")
        r.walk_step()     # greedy, flat, or rejection sampling at the round's temperature
        mark("walk")
        if r.Lf and r.page:
            ddt.ddt_commit_paged(r.walk["acc_nodes"], r.walk["acc_len"], r.prefix_len, r.block_table,
                                 k_tree=r.attn.k_tree, v_tree=r.attn.v_tree, k_pages=r.k_pages, v_pages=r.v_pages,
                                 out=r.commit, **kw)
            mark("commit")
        elif r.Lf or r.Lg:
            ddt.ddt_commit(r.walk["acc_nodes"], r.walk["acc_len"], r.prefix_len, out=r.commit, **kw)
            mark("commit")
        if timed:
            names = list(marks)
            for a_, b_ in zip(names[:-1], names[1:]):
                ev.setdefault(b_, []).append((marks[a_], marks[b_]))
            spans.append((marks[names[0]], marks[names[-1]]))

    spans = ev.setdefault("_rounds", [])
    return step


def measure(r, steps, warmup, flat=False, clocks=None, world=1):
    """Times `steps` rounds after `warmup` untimed ones: CUDA events on the launching stream
    around the whole timed region (barrier + synchronize on both sides), around each round
    and around each call.  When the round's inputs fit in L2, a flush buffer is written
    between rounds and the total is the sum of the rounds' own spans.  Returns the total
    ms, mean ms per call, and the library's launch count."""
    from tree_speculative_decoding_02_gb300 import ddt

    st = torch.cuda.current_stream()
    ev = {}
    step = make_step(r, flat, ev)
    flush = flush_buffer(r)
    for _ in range(warmup):
        step(False)
    torch.cuda.synchronize()
    bad = int((r.tree["status"] != 0).sum())
    if bad:
        raise RuntimeError(f"build reported {bad} request errors")
    if clocks:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = ddt.ddt_launch_count()
    t0.record(st)
    for _ in range(steps):
        step(True)
        if flush is not None:
            flush.zero_()
    t1.record(st)
    launches = ddt.ddt_launch_count() - launches0
    torch.cuda.synchronize()
    barrier(world)
    rounds = ev.pop("_rounds")
    per_call = {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in ev.items()}
    # with flushes in between, the rounds' own spans; otherwise the whole region
    ms = sum(a.elapsed_time(b) for a, b in rounds) if flush is not None else t0.elapsed_time(t1)
    return {"ms": ms, "per_call_ms": per_call, "launches": launches}


def flush_buffer(r):
    """The buffer written between timed rounds when the round's inputs fit in L2, else None."""
    if not needs_flush(r.cfg, int(r.prefix0.sum())):
        return None
    return torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=r.prefix0.device)


def measure_graph(r, steps, warmup):
    """The same round captured once into a CUDA graph and replayed: `steps` replays after
    `warmup`, each bracketed by CUDA events on the replaying stream (with the L2 flushed
    between replays when the round's inputs fit in it).  Returns the ms per round and the
    library launches the graph holds."""
    from tree_speculative_decoding_02_gb300 import ddt

    step = make_step(r, False, {})
    cur = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(cur)
    with torch.cuda.stream(side):
        for _ in range(2):
            step(False)
    cur.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    n0 = ddt.ddt_launch_count()
    with torch.cuda.graph(g):
        step(False)
    captured = ddt.ddt_launch_count() - n0
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    flush = flush_buffer(r)
    marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in marks:
        a.record(cur)
        g.replay()
        b.record(cur)
        if flush is not None:
            flush.zero_()
    torch.cuda.synchronize()
    if flush is None:
        ms = marks[0][0].elapsed_time(marks[-1][1]) / steps
    else:
        ms = sum(a.elapsed_time(b) for a, b in marks) / steps
    del g
    return ms, captured


def roofline_of(call, work, ms, peaks, tc_peak, tc_kind, traffic=None):
    """The roofline object of one call: tensor-bound for the attention contraction, HBM-bound
    for the rest; `achieved` from the algorithmic work and the call's CUDA-event time."""
    by, fl = work[call]
    if fl > 0:
        ach = fl / (ms / 1e3) / 1e12
        return {"bound": "tensor", "kernel": KERNEL_OF[call], "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": ach / tc_peak, "traffic": traffic, "algorithmic_flops": fl, "algorithmic_bytes": by,
                "peak_note": f"of {peaks['source']} ({tc_kind} bf16)"}
    ach = by / (ms / 1e3) / 1e9
    return {"bound": "hbm", "kernel": KERNEL_OF[call], "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": ach / peaks["hbm_gbs"], "traffic": traffic, "algorithmic_bytes": by,
            "peak_note": f"of {peaks['source']} (HBM copy)"}


KERNEL_OF = {"build": "ddt_build_tree", "attn": "ddt_tree_attn", "gdn": "ddt_tree_gdn", "walk": "ddt_walk_accept",
             "commit": "ddt_commit"}


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
    if args.rope and cfg.get("Lf"):
        cfg["rope"] = cfg["d"]
    cfg["flat"] = args.flat
    if args.batch:
        cfg["B"] = args.batch
    if args.temperature > 0:
        cfg["temperature"] = args.temperature
    r = Round(cfg, device=dev, workload=args.workload)
    st = torch.cuda.current_stream()

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

    # nvidia-smi samples during the timed region; the raw CSV goes to $DDT_CLOCKS_CSV when
    # set, else to a temporary file, and its summary into the JSON line
    clocks = None
    if rank == 0:
        import tempfile
        path = os.environ.get("DDT_CLOCKS_CSV") or os.path.join(tempfile.gettempdir(), f"ddt_clocks_{os.getpid()}.csv")
        clocks = ClockSampler(path)
    m = measure(r, args.steps, args.warmup, flat=args.flat, clocks=clocks, world=world)
    ms = m["ms"]
    clk = clocks.stop(gpu_uuid()) if clocks else None
    if args.planted:
        accepted = float(r.walk["acc_len"].float().mean())
    nodes_per_step = r.drafted_nodes()
    ms_max = all_max(ms, world, dev)
    nodes_total = all_sum(nodes_per_step * args.steps, world, dev)
    value = nodes_total / (ms_max / 1e3)
    per_call = m["per_call_ms"]

    graph_ms, graph_launches = measure_graph(r, args.steps, args.warmup)
    e2e = e2e_measure(r, args.steps, world, dev)
    e2e["value"] = all_sum(nodes_per_step * e2e.pop("rounds"), world, dev) / (all_max(e2e.pop("ms"), world, dev) / 1e3)

    peaks = load_peaks()
    tc_peak, tc_kind = tensor_peak(peaks, clk)
    work = call_work(r)
    floors = floors_ms(work, peaks["hbm_gbs"], tc_peak)
    step_ms = ms / args.steps
    rb = sum(by for by, _ in work.values())
    dom = max(per_call, key=per_call.get)
    traffic = attn_traffic(work["attn"][0]) if dom == "attn" and not args.kv_page else None
    roof = roofline_of(dom, work, per_call[dom], peaks, tc_peak, tc_kind, traffic)
    if roof["bound"] == "tensor":
        roof["frac_sustained"] = roof["achieved"] / peaks["sustained"]
        roof["frac_burst"] = roof["achieved"] / peaks["burst"]
        if cfg["d"] in (128, 256) and cfg["dtype"] == torch.bfloat16:
            iss = attn_issued_flops(r)
            roof["issued"] = {"flops": iss, "tflops": iss / (per_call[dom] / 1e3) / 1e12,
                              "note": "MMA work the kernel issues: 256-row pair tiles x 128-key tiles, "
                                      "Q K^T plus two P V passes"}
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg["dtype"] == torch.bfloat16 else "f32", "data": "synthetic",
        "config": arm_config(cfg, int(r.prefix0.sum()), nodes_per_step, world),
        "hbm_gbs_round": rb / (step_ms / 1e3) / 1e9,
        "hbm_frac_round": rb / (step_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
        "round_frac": sum(floors.values()) / step_ms,
        "per_kernel_ms": per_call,
        "floor_ms": floors,
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": m["launches"],
        "clocks": clk,
        "graph": {"ms_per_step": graph_ms, "value": nodes_per_step / (graph_ms / 1e3),
                  "launches_per_step": graph_launches,
                  "note": "the same round captured once into a CUDA graph and replayed (rank 0's replays)"},
    }
    if args.flat:
        out["config"]["walk"] = "flat-commit safe mode (first children only)"
    if args.planted:
        out["config"]["acceptance"] = (f"planted paths, geometric lengths of mean {args.planted}; "
                                       f"mean accepted drafted nodes {accepted:.2f}")
    if args.temperature > 0:
        out["config"]["walk"] = (f"tree-walk rejection sampling at temperature {args.temperature} "
                                 "(ddt_walk_accept_sample, seeded uniforms)")
    if args.kv_page:
        out["config"]["kv"] = f"paged: {args.kv_page} rows a page, shuffled block table"
    if args.rope:
        out["config"]["rope"] = ("rotary embedding by depth: tree keys rotated in place, q rotated inside the "
                                 "fused attention call (inputs taken before rotation)")
    if rank == 0 and world == 1 and not args.no_cpu_baseline and r.Lf and r.Lg and not (
            args.kv_page or args.rope or args.temperature or args.batch):
        out["cpu_baseline"] = cpu_baseline(r, seconds=args.cpu_seconds)
    if rank == 0 and world == 1 and args.per_config and args.workload == WORKLOAD and not (
            args.kv_page or args.flat or args.planted or args.rope or args.temperature or args.batch):
        del r
        torch.cuda.empty_cache()
        out["per_config"] = [config_line(w, dev, peaks, tc_peak, tc_kind, not args.no_cpu_baseline)
                             for w in (1, 2, 3, 4)]
    return out


def e2e_measure(r, steps, world, dev):
    """End to end through the public API: each round's inputs are copied from pinned host
    memory and its emitted tokens copied back, inside the timed region.  The inputs are
    double-buffered: round i+1's copy runs on a copy stream while round i computes, the
    way a serving loop overlaps them.  Each copy is split by the call that first reads it
    (drafter logits, then q / tree K,V, then x and gates, then target logits), and a call
    waits only for its own group, so even the first round's compute starts early.  The
    copy stream's own time per round, and the host-to-device rate of the same copies
    with the GPU otherwise idle, are reported beside the rate."""
    st = torch.cuda.current_stream()
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
    copy_ev = []

    def copy_in(slot, timed):
        with torch.cuda.stream(cs):
            cs.wait_event(free[slot])
            if timed:
                a = torch.cuda.Event(enable_timing=True)
                a.record(cs)
            for n, names in groups.items():
                for k in names:
                    slots[slot][k].copy_(host[k], non_blocking=True)
                copied[slot][n].record(cs)
            if timed:
                b = torch.cuda.Event(enable_timing=True)
                b.record(cs)
                copy_ev.append((a, b))

    def run(n, timed):
        for sl in range(2):
            free[sl].record(st)
        copy_in(0, timed)
        for i in range(n):
            sl = i % 2
            if i + 1 < n:
                copy_in(1 - sl, timed)
            r.bind_inputs(slots[sl])
            r.restore_prefix()
            r.step(wait=lambda name, sl=sl: st.wait_event(copied[sl][name]))
            free[sl].record(st)
            for k, v in outs.items():
                host_out[k].copy_(v, non_blocking=True)

    run(2, False)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n = max(2, steps)
    e0.record(st)
    run(n, True)
    e1.record(st)
    torch.cuda.synchronize()
    barrier(world)
    e_ms = e0.elapsed_time(e1)
    h2d_ms = statistics.mean(a.elapsed_time(b) for a, b in copy_ev)
    # the same copies with nothing else on the GPU: the host link's own rate
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cs):
        a.record(cs)
        for k in host:
            slots[1][k].copy_(host[k], non_blocking=True)
        b.record(cs)
    torch.cuda.synchronize()
    alone_ms = a.elapsed_time(b)
    r.bind_inputs(slots[0])
    return {"ms": e_ms, "rounds": n, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_ms_per_step": h2d_ms, "h2d_gbs_during_rounds": h2d / (h2d_ms / 1e3) / 1e9,
            "h2d_gbs_alone": h2d / (alone_ms / 1e3) / 1e9, "ms_per_step": e_ms / n,
            "inputs": "pinned host, double-buffered: round i+1 copied on a copy stream during round i; "
                      "each call waits for its own input group"}


def config_line(w, dev, peaks, tc_peak, tc_kind, with_cpu):
    """One smaller workload measured the same way (a few rounds), with its dominant call's
    roofline and the oracle timed on one host thread and on all of them."""
    from tree_speculative_decoding_02_gb300 import synth
    from tree_speculative_decoding_02_gb300.round import Round

    cfg = dict(synth.WORKLOADS[w])
    if "budget" not in cfg:
        cfg["budget"] = max(cfg["budgets"])
    r = Round(cfg, device=dev, workload=w)
    m = measure(r, 10, 3)
    step_ms = m["ms"] / 10
    nodes = r.drafted_nodes()
    work = call_work(r)
    floors = floors_ms(work, peaks["hbm_gbs"], tc_peak)
    per = m["per_call_ms"]
    dom = max(per, key=per.get)
    line = {"workload": workload_desc(cfg), "dtype": "bf16" if cfg["dtype"] == torch.bfloat16 else "f32",
            "value": nodes / (step_ms / 1e3), "unit": UNIT, "ms_per_step": step_ms, "steps": 10, "warmup": 3,
            "per_kernel_ms": per, "floor_ms": floors, "round_frac": sum(floors.values()) / step_ms,
            "roofline": roofline_of(dom, work, per[dom], peaks, tc_peak, tc_kind,
                                    attn_traffic(work["attn"][0]) if dom == "attn" else None),
            "gpu_launches": m["launches"]}
    gms, glaunch = measure_graph(r, 10, 3)
    line["graph"] = {"ms_per_step": gms, "value": nodes / (gms / 1e3), "launches_per_step": glaunch}
    if with_cpu:
        line["cpu_baseline"] = config_cpu_baseline(r, w)
    del r
    torch.cuda.empty_cache()
    return line


# ------------------------------------------------------------- oracle (CPU) timing
def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def request_from_round(r, b):
    """One request's inputs of a GPU Round, as fp64 host arrays for the oracle (the parts of
    the round's layer stack that the workload has)."""
    P = int(r.prefix0[b])
    q = {"P": P, "draft_logits": _f64(r.draft_logits[b:b + 1]), "root": r.root_token[b:b + 1].cpu().numpy(),
         "target_logits": _f64(r.target_logits[b:b + 1])}
    if r.Lf:
        a = r.attn
        q.update(q=_f64(a.q[:, b:b + 1]), k_tree=_f64(a.k_tree[:, b:b + 1]), v_tree=_f64(a.v_tree[:, b:b + 1]),
                 k_cache=_f64(a.k_cache[:, b:b + 1, :, :P]), v_cache=_f64(a.v_cache[:, b:b + 1, :, :P]))
    if r.Lg:
        g = r.gdn
        q.update(x=_f64(g.x[:, b:b + 1]), conv_w=_f64(g.conv_w), conv_state=_f64(g.conv_state[:, b:b + 1]),
                 beta=_f64(g.beta[:, b:b + 1]), decay=_f64(g.decay[:, b:b + 1]),
                 S=np.swapaxes(_f64(g.S[:, b:b + 1]), -1, -2))
    return q


def subset_layers(q, lf, lg):
    """The first lf attention and lg GDN layers of a request's inputs (a bounded sample)."""
    out = dict(q)
    for k in ("q", "k_tree", "v_tree", "k_cache", "v_cache"):
        if k in out:
            out[k] = np.ascontiguousarray(out[k][:lf])
    for k in ("x", "conv_w", "conv_state", "beta", "decay", "S"):
        if k in out:
            out[k] = np.ascontiguousarray(out[k][:lg])
    return out


def workload_prefixes(cfg, workload):
    """The committed prefix lengths of the workload's requests (as the GPU round draws them)."""
    from tree_speculative_decoding_02_gb300 import synth

    if "P_lo" not in cfg:
        return np.full(cfg["B"], cfg.get("P", 0), np.int64)
    return synth.prefix_lengths(cfg["B"], cfg["P_lo"], cfg["P_hi"], g=synth.gen(workload, 2)).numpy().astype(np.int64)


def typical_order(prefix):
    """Request indices ordered by how close their prefix is to the workload's mean prefix, so
    that a sample of the first few is representative of the whole batch."""
    mean = float(np.mean(prefix))
    return sorted(range(len(prefix)), key=lambda b: (abs(float(prefix[b]) - mean), b))


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
    q = {"P": P, "draft_logits": _f64(synth.draft_logits(1, cfg["D"], cfg["V"], std=cfg["logit_std"],
                                                        boost=cfg["boost"], g=synth.gen(wl, 1), dtype=dt)),
         "root": np.array([b], np.int32),
         "target_logits": _f64(synth.target_logits(1, N, cfg["V"], g=synth.gen(wl, 30), dtype=dt))}
    if cfg.get("Lf"):
        a = synth.attn_inputs(Lf or cfg["Lf"], 1, N, cfg["Hq"], cfg["Hkv"], cfg["d"], P, [P], workload=wl, dtype=dt,
                              device=dev, poison=False)
        q.update(q=_f64(a.q), k_tree=_f64(a.k_tree), v_tree=_f64(a.v_tree), k_cache=_f64(a.k_cache),
                 v_cache=_f64(a.v_cache))
    if cfg.get("Lg"):
        g = synth.gdn_inputs(Lg or cfg["Lg"], 1, N, cfg["Hk"], cfg["Hv"], cfg["dk"], cfg["dv"], cfg["conv_k"],
                             workload=wl, dtype=dt, device=dev)
        q.update(x=_f64(g.x), conv_w=_f64(g.conv_w), conv_state=_f64(g.conv_state), beta=_f64(g.beta),
                 decay=_f64(g.decay), S=_f64(g.S))
    return q


def oracle_round(cfg, q):
    """One request's round (build, attention, GDN, walk, commit) through the plain oracle
    on the layers present in `q`; the attention and GDN stages and the commit are scaled
    to the workload's full layer counts (the work is the same for every layer).  Returns
    (drafted nodes, seconds, layer scale factors)."""
    import oracle

    P = q["P"]
    sa = cfg.get("Lf", 0) / q["q"].shape[0] if "q" in q else 0.0
    sg = cfg.get("Lg", 0) / q["x"].shape[0] if "x" in q else 0.0
    t0 = time.perf_counter()
    tree = oracle.build_tree(q["draft_logits"], q["root"], [P], cfg["top_k"], cfg["budget"])
    t1 = time.perf_counter()
    if "q" in q:
        oracle.tree_attn(q["q"], q["k_tree"], q["v_tree"], q["k_cache"], q["v_cache"], [P], tree["n_nodes"],
                         tree["anc"], 1.0 / math.sqrt(cfg["d"]))
    t2 = time.perf_counter()
    if "x" in q:
        oracle.tree_gdn(q["x"], q["conv_w"], q["conv_state"], q["beta"], q["decay"], q["S"], tree["parent"],
                        tree["n_nodes"], cfg["Hk"])
    t3 = time.perf_counter()
    wk = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], cfg["D"], target_logits=q["target_logits"])
    t4 = time.perf_counter()
    kw = {}
    if "q" in q:
        pad = ((0, 0), (0, 0), (0, 0), (0, cfg["D"] + 1), (0, 0))
        kw.update(k_tree=q["k_tree"], v_tree=q["v_tree"], k_cache=np.pad(q["k_cache"], pad),
                  v_cache=np.pad(q["v_cache"], pad))
    if "x" in q:
        kw.update(x=q["x"], conv_w=q["conv_w"], beta=q["beta"], decay=q["decay"], S=q["S"],
                  conv_state=q["conv_state"], Hk=cfg["Hk"])
    t5 = time.perf_counter()
    if kw:
        oracle.commit(wk["acc_nodes"], wk["acc_len"], [P], **kw)
    t6 = time.perf_counter()
    el = (t1 - t0) + sa * (t2 - t1) + sg * (t3 - t2) + (t4 - t3) + max(sa, sg, 1.0 if kw else 0.0) * (t6 - t5)
    return int(tree["n_nodes"][0]) - 1, el, {"attn": sa, "gdn": sg}


def cpu_baseline(r, seconds=15.0, max_requests=8):
    """The oracle, as it stands, on all host cores: whole rounds of single requests of the
    batched workload, taken in order of closeness to the mean prefix length."""
    import oracle

    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    oracle.build()
    prefix = r.prefix0.cpu().numpy()
    nodes, t_oracle, done = 0, 0.0, []
    for b in typical_order(prefix)[:max_requests]:
        n, t, _ = oracle_round(r.cfg, request_from_round(r, b))
        nodes += n
        t_oracle += t
        done.append(b)
        if t_oracle >= seconds:
            break
    return {"value": nodes / t_oracle, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"full round (build, 16-layer tree attention, 48-layer tree GDN, walk, commit) of requests "
                      f"{done} (prefixes {[int(prefix[b]) for b in done]}; the workload's mean is "
                      f"{float(prefix.mean()):.0f}), fp64, {t_oracle:.1f} s of oracle time"}


# bounded samples for the smaller workloads' oracle timings: (attention layers, GDN layers)
# on one thread and on all host cores; the rest of each round runs in full
CPU_SAMPLE = {1: ((1, 1), (1, 1)), 2: ((0, 0), (0, 0)), 3: ((1, 0), (16, 0)), 4: ((0, 4), (0, 48))}


def config_cpu_baseline(r, w):
    import oracle

    oracle.build()
    cores = len(os.sched_getaffinity(0))
    q = request_from_round(r, 0)
    res = {"unit": UNIT, "kind": "oracle"}
    for label, threads, (lf, lg) in (("single_thread", 1, CPU_SAMPLE[w][0]), ("all_cores", cores, CPU_SAMPLE[w][1])):
        oracle.set_threads(threads)
        n, t, sc = oracle_round(r.cfg, subset_layers(q, lf, lg))
        res[label] = {"value": n / t, "cores": threads, "seconds": t,
                      "sample": "one request's round" + (f", {lf} of {r.Lf} attention layers timed" if r.Lf else "")
                      + (f", {lg} of {r.Lg} GDN layers timed" if r.Lg else "")
                      + (" and scaled to all layers" if (r.Lf and lf < r.Lf) or (r.Lg and lg < r.Lg) else "")}
    oracle.set_threads(cores)
    res["value"], res["cores"], res["sample"] = res["all_cores"]["value"], cores, res["all_cores"]["sample"]
    return res


def run_reference(args, rank, world):
    """The reference arm: the plain CPU oracle.  Each step is one request's round on a
    quarter of the attention and GDN layers; the value is that sample's time scaled to the
    full layer counts (the per-layer work is the same), and ms_per_step is the time the
    sample itself took."""
    if rank != 0:
        return None
    import oracle
    from tree_speculative_decoding_02_gb300 import synth

    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    oracle.build()
    cfg = dict(synth.WORKLOADS[args.workload])
    if "budget" not in cfg:
        cfg["budget"] = max(cfg["budgets"])
    lf, lg = max(1, cfg.get("Lf", 0) // 4), max(1, cfg.get("Lg", 0) // 4)
    order = typical_order(workload_prefixes(cfg, args.workload))

    def one(i):
        q = request_synth(cfg, order[i % len(order)], args.workload, Lf=lf, Lg=lg)
        w0 = time.perf_counter()
        n, t, _ = oracle_round(cfg, q)
        return n, t, time.perf_counter() - w0

    for i in range(args.warmup):
        one(i)
    nodes, el, wall = 0, 0.0, 0.0
    for i in range(args.steps):
        n, t, wt = one(args.warmup + i)
        nodes += n
        el += t
        wall += wt
    v = nodes / el
    sample = (f"per step one request's round (budget {cfg['budget']}; requests nearest the mean prefix first), "
              f"build and walk in full, {lf} of {cfg.get('Lf', 0)} attention and {lg} of {cfg.get('Lg', 0)} GDN "
              f"layers timed and scaled to all layers; fp64 oracle time only")
    prefix = workload_prefixes(cfg, args.workload)
    return {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": wall * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "extrapolated": {"timed_attention_layers": lf, "timed_gdn_layers": lg,
                             "round_s_scaled_to_all_layers": el / args.steps,
                             "note": "value = drafted nodes / the sample's oracle time scaled to every layer; "
                                     "ms_per_step = the sample's own wall time"},
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
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the per-workload lines of the smaller configurations")
    ap.add_argument("--flat", action="store_true", help="flat-commit safe mode: walk first children only")
    ap.add_argument("--batch", type=int, default=0,
                    help="> 0: run the workload with this many requests instead of its own B")
    ap.add_argument("--temperature", type=float, default=0.0,
                    help="> 0: verify by tree-walk rejection sampling at this temperature")
    ap.add_argument("--planted", type=float, default=0.0,
                    help="plant accepted paths with this mean length (0: random targets, little accepted)")
    ap.add_argument("--rope", action="store_true",
                    help="rotary embedding by depth: keys rotated in place, q inside the fused attention call")
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
