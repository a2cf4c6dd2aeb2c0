#!/usr/bin/env python3
"""Draft-verify cycles/s of the EAGLE-2 dynamic draft-tree cycle on GB300.

One step = one whole cycle over one batch: tree init, D expand steps, rerank,
tree emission, tree attention (one layer), verification and KV compaction of
every layer, all in libeagle's kernels. Inputs (draft and target logits, Q,
KV cache) are synthetic and resident in HBM before the timed region; input
sets larger than L2 in total are rotated between steps. The cycle of each set
is captured once in a CUDA graph and replayed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

The JSON line's headline is the Llama-3.1-8B batch-1 cycle (lossless). The
same run then measures, with the same K and W, the other configurations of
the workload table (8B batch 64 greedy, as stated and with planted drafts and aligned targets,
70B batch 8 lossless, 13B batch 1 lossless, 8B batch 1 greedy) into the
line's `configs` block (skip with --no-configs). The oracle is timed on the
host cores: one core, and one process per core on independent cycles.

Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
sequences of a batch are independent: no collective on the data path);
ranks meet at a barrier, the max time over ranks is taken and rank 0 prints
one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
METRIC = "draft-verify cycles/s at Llama-8B shape; HBM GB/s & % roofline per kernel"
POLICIES = {"dynamic": 0, "confidence": 1, "no_rerank": 2, "static": 3}

# The configurations measured beside the headline: (label, workload, overrides, variant flags).
EXTRA_CONFIGS = [
    ("llama8b_b64_greedy", "llama8b_b64", {}, {}),
    ("llama8b_b64_greedy_planted_aligned", "llama8b_b64", {}, {"aligned": True, "planted": True}),
    ("llama70b_b8_lossless", "llama70b_b8", {}, {}),
    ("vicuna13b_b1_lossless", "vicuna13b_b1", {}, {}),
    ("llama8b_b1_greedy", "llama8b_b1", {"verify": "greedy"}, {}),
]


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b_b1")
    ap.add_argument("--sharpness", type=float, default=None)
    ap.add_argument("--verify", default=None, choices=[None, "greedy", "lossless"])
    ap.add_argument("--planted", action="store_true", help="sharp draft rows (deep chains)")
    ap.add_argument("--aligned", action="store_true",
                    help="target rows favour each slot's first kept child (deep acceptance; compaction moves KV)")
    ap.add_argument("--sets", type=int, default=0, help="rotating input sets (0 = enough to exceed L2)")
    ap.add_argument("--seed", type=int, default=42)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="measure the headline workload only")
    ap.add_argument("--cpu-seconds", type=float, default=8.0, help="oracle time per CPU-baseline leg")
    ap.add_argument("--kernel-reps", type=int, default=100)
    ap.add_argument("--layers", type=int, default=None, help="KV layers moved by compaction (memory cap)")
    ap.add_argument("--lmhead", action="store_true",
                    help="each draft step's rows come from the LM head (bf16 tensor-core GEMM of synthetic hidden "
                         "states against a resident random [V, H] weight)")
    ap.add_argument("--fused-head", action="store_true",
                    help="with the LM head: stage 1 in its epilogue (eagle_lmhead_topk, then eagle_expand_topk); "
                         "the logits are never written")
    ap.add_argument("--policy", default="dynamic", choices=list(POLICIES),
                    help="tree policy: EAGLE-2, confidence-ranked frontier, no rerank or static shape (ablations)")
    a = ap.parse_args(argv)
    if a.fused_head:
        a.lmhead = True
    return a


# ------------------------------------------------------------- helpers ---

def align_targets(target: np.ndarray, tokens: np.ndarray, parent: np.ndarray, n_tree: np.ndarray, value: float):
    """Aligned-target variant: in the target row of every tree slot, the token of
    the slot's first kept child gets the logit `value` (about 0.9 of the row's
    mass), so verification accepts along first children and compaction has KV
    to move. Input construction only; changes `target` in place."""
    B = target.shape[0]
    bits = np.uint16(np.float32(value).view(np.uint32) >> 16) if target.dtype == np.uint16 else np.float32(value)
    for b in range(B):
        n = int(n_tree[b])
        first = {}
        for c in range(1, n):
            p = int(parent[b, c])
            if p >= 0 and p not in first:
                first[p] = c
        for t, c in first.items():
            target[b, t, int(tokens[b, c])] = bits


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's replica: ranks draw different (independent) sequences."""
    return seed + 7919 * rank


def max_over_ranks(ms: float, device=None) -> float:
    """Largest timing over the ranks of the default process group (identity when
    there is none); the slowest replica sets the whole-job time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, steps: int, ms: float) -> float:
    """Cycles per second of the whole job: every rank ran `steps` cycles in at most `ms`."""
    return world * steps / (ms / 1e3)


def workload(args):
    from synth import workloads as WL
    w = WL.WORKLOADS[args.workload]
    kw = {}
    if args.sharpness is not None:
        kw["sharpness"] = args.sharpness
    if args.verify is not None:
        kw["verify"] = args.verify
    if args.layers is not None:
        kw["layers"] = args.layers
    return w.with_(**kw) if kw else w


def start_clocks(idx: int):
    path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
    q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    try:
        f = open(path, "w")
        p = subprocess.Popen(["nvidia-smi", "-i", str(idx), f"--query-gpu={q}", "--format=csv,noheader,nounits",
                              "-lms", "50"], stdout=f, stderr=subprocess.DEVNULL)
        return p, f, path
    except Exception:
        return None, None, path


def wait_first_sample(h, timeout_s: float = 3.0) -> None:
    """Block until the clock sampler has written its first line (its start-up
    takes longer than a short timed region)."""
    p, f, path = h
    if p is None:
        return
    t0 = time.time()
    while time.time() - t0 < timeout_s:
        f.flush()
        if os.path.getsize(path) > 0:
            return
        time.sleep(0.02)


def stop_clocks(h) -> dict | None:
    p, f, path = h
    if p is None:
        return None
    p.terminate()
    try:
        p.wait(timeout=5)
    except Exception:
        p.kill()
    f.close()
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in open(path):
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    os.unlink(path)
    if not sm:
        return None
    return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
            "samples": len(sm)}


CSRC = os.path.join(ROOT, "speculative_decoding_dynamic_gb300", "csrc")
# translation unit(s) of each profiled kernel (attention: the per-item kernel
# and the persistent pipeline, either may run depending on the shape)
KERNEL_TU = {"expand_kernel": "k_rows.cu", "verify_kernel": ("k_rows.cu", "k_draft.cu"),
             "attention": ("k_attn_tc.cu", "k_attn_pipe.cu"), "lmhead_kernel": "k_lmhead.cu",
             "lmhead_topk_kernel": "k_lmhead.cu", "kv_compact_kernel": "k_compact.cu"}


def _toolchain_id() -> bytes:
    """The compile flags of the library build and the nvcc release: a change of
    either changes the generated code."""
    from speculative_decoding_dynamic_gb300 import build as Bld
    try:
        ver = subprocess.run([Bld._nvcc(), "--version"], capture_output=True, text=True).stdout
        ver = " ".join(re.findall(r"release [0-9.]+, V[0-9.]+", ver))
    except Exception:
        ver = "unknown"
    flags = [f for f in Bld.NVCC_FLAGS if not os.path.isabs(f)]
    return (" ".join(Bld.ARCH + flags) + " | " + ver).encode()


def _src_hash(roots) -> str:
    """Hash of the csrc files `roots`, the csrc headers they include
    (transitively, in name order) and the toolchain (flags, nvcc release)."""
    h = hashlib.sha256()
    todo = list(roots)
    used = set()
    while todo:
        f = todo.pop()
        if f in used or not os.path.exists(os.path.join(CSRC, f)):
            continue
        used.add(f)
        for inc in re.findall(r'^\s*#\s*include\s+"([^"/]+)"', open(os.path.join(CSRC, f)).read(), re.M):
            todo.append(inc)
    for f in sorted(used):
        h.update(open(os.path.join(CSRC, f), "rb").read())
    h.update(_toolchain_id())
    return h.hexdigest()[:16]


def kernel_src_hash() -> str:
    """Hash of the sources the library is compiled from: every .cu file of csrc
    and the headers they include, with the toolchain."""
    return _src_hash(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def tu_src_hash(kernel: str) -> str:
    """Hash of the sources one profiled kernel is compiled from (its .cu file
    and the headers it includes, with the toolchain)."""
    tu = KERNEL_TU[kernel]
    return _src_hash([tu] if isinstance(tu, str) else list(tu))


def ncu_traffic(kernel: str, workload_name: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was
    taken on the current sources of that kernel's translation unit; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
    except Exception:
        return None
    e = d.get(workload_name, {}).get(kernel)
    if not e or kernel not in KERNEL_TU or e.get("src_hash") != tu_src_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        m = re.search(r"^Model name:\s*(.+)$", out, re.M)
        if m:
            return m.group(1).strip()
    except Exception:
        pass
    try:
        m = re.search(r"^model name\s*:\s*(.+)$", open("/proc/cpuinfo").read(), re.M)
        if m:
            return m.group(1).strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------ the cycle ---

def to_dev(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).cuda()
    return torch.from_numpy(a).cuda()


def pinned(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    elif a.dtype == np.uint32:
        t = torch.from_numpy(a.view(np.int32))
    else:
        t = torch.from_numpy(a)
    return t.pin_memory()


def rotation_sets(w, seed: int, sets: int = 0) -> tuple[int, int, int]:
    """(R, bytes per set, attention bytes per set): enough rotating input sets that
    one pass over them exceeds 1.5x L2 (one set when a single set already does)."""
    per_set = (w.depth * w.batch * w.top_k + w.batch * w.T) * w.vocab * w.esize
    attn_bytes = int(sum(int(L) + w.T for L in w.prefix_lengths(seed))) * w.n_kv_heads * w.head_dim * 2 * w.esize
    R = sets or max(1, int(np.ceil(1.5 * L2_BYTES / (per_set + attn_bytes))))
    return min(R, w.layers), per_set, attn_bytes


def config_of(w, args, variant: dict, R: int, per_set: int, attn_bytes: int) -> dict:
    """The workload description printed by both arms."""
    return {"workload": w.name, "batch": w.batch, "vocab": w.vocab, "depth": w.depth, "top_k": w.top_k,
            "node_budget": w.node_budget, "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads,
            "head_dim": w.head_dim, "prefix": list(w.prefix) if isinstance(w.prefix, tuple) else w.prefix,
            "sharpness": list(w.sharpness) if isinstance(w.sharpness, tuple) else w.sharpness,
            "verify": w.verify, "compact_layers": w.layers, "planted": bool(variant.get("planted", False)),
            "aligned": bool(variant.get("aligned", False)), "policy": args.policy, "lmhead": args.lmhead,
            "fused_head": args.fused_head, "hidden_size": w.hidden_size if args.lmhead else None,
            "l2": f"{R} rotating input set(s), {round(R * (per_set + attn_bytes) / 2**20)} MiB > 129 MB L2",
            "graph": "one CUDA graph per input set, replayed"}


def algorithmic_bytes(w, prefix_len, accept_len, layers):
    """Bytes each stage must move per cycle (reads + writes of its operands)."""
    es = w.esize
    B, D, k, V, T = w.batch, w.depth, w.top_k, w.vocab, w.T
    rows_per_seq = 1 + (D - 1) * k
    expand = B * rows_per_seq * V * es
    expand_step = B * k * V * es  # one step with a full frontier
    verify = B * T * V * es
    kv_read = int(sum(int(L) + T for L in prefix_len)) * w.n_kv_heads * w.head_dim * 2 * es
    qo = 2 * B * T * w.n_q_heads * w.head_dim * es
    attention = kv_read + qo
    compact = int(2 * sum(int(a) for a in accept_len) * layers * 2 * w.n_kv_heads * w.head_dim * es)
    return dict(expand=expand, expand_step=expand_step, verify=verify, attention=attention, compact=compact)


# ------------------------------------------------------------ the oracle ---

def oracle_cycle(w, s, prefix_len, root, kh, vh, geo, mode, tree_region, head_stride=1, policy=0):
    """One whole cycle in the CPU oracle (the bench's CPU baseline / reference arm).

    Returns the estimated cycle time in seconds: every stage is run in full
    except that, with head_stride m > 1, tree attention runs on every m-th query
    head only and its measured time is multiplied by m (attention is ~95% of
    the oracle's cycle)."""
    import oracle
    t0 = time.perf_counter()
    cfg = oracle.TreeCfg(w.batch, w.vocab, w.top_k, w.depth, w.node_budget, w.threshold, policy)
    t = oracle.Tree(cfg)
    for st in range(w.depth):
        t.expand(st, s["draft"][st])
    t.rerank()
    tr = t.build_tree(prefix_len, root)
    t1 = time.perf_counter()
    pos_stride = w.n_kv_heads * w.head_dim
    if head_stride == 1:
        oracle.attention(s["q"], kh, vh, geo["max_len"] * pos_stride, pos_stride, prefix_len, tr["mask"],
                         tr["n_tree"], w.n_kv_heads)
    else:
        rows = np.array([(b, i, h) for b in range(w.batch) for i in range(w.T)
                         for h in range(0, w.n_q_heads, head_stride)], np.int32)
        oracle.attention_rows(rows, s["q"], kh, vh, geo["max_len"] * pos_stride, pos_stride, prefix_len,
                              tr["mask"], tr["n_tree"], w.n_kv_heads)
    t2 = time.perf_counter()
    if mode == "greedy":
        a, sl, _, _ = oracle.verify_greedy(s["target"], tr["tokens"], tr["parent"], tr["n_tree"], w.depth)
    else:
        a, sl, _ = oracle.verify_lossless(s["target"], tr["tokens"], tr["parent"], tr["n_tree"], s["uniforms"],
                                          w.depth, np.float32(1.0 / w.temperature))
    reg = tree_region.copy()
    L = reg.shape[1]
    oracle.kv_compact(reg.reshape(-1), w.batch, L, w.n_kv_heads, w.head_dim, L * 2 * w.T * pos_stride,
                      2 * w.T * pos_stride, w.T * pos_stride, pos_stride, np.zeros(w.batch, np.int32), a, sl)
    t3 = time.perf_counter()
    return (t1 - t0) + head_stride * (t2 - t1) + (t3 - t2)


def host_attention_layer(w, geo, prefix_len, seed, layer):
    from synth import workloads as WL
    npdt = np.float32 if w.esize == 4 else np.uint16
    shape = (w.batch, geo["max_len"], w.n_kv_heads, w.head_dim)
    K = np.zeros(shape, npdt)
    Vv = np.zeros(shape, npdt)
    for b in range(w.batch):
        for which, arr in ((0, K), (1, Vv)):
            WL.kv_fill(arr, w, geo, b, layer, which, 0, int(prefix_len[b]) + w.T, seed,
                       offset=b * geo["seq_stride"] + layer * geo["layer_stride"] + which * geo["kv_stride"]
                       - b * geo["max_len"] * geo["pos_stride"])
    return K, Vv


def host_tree_region(w, geo, prefix_len, seed, layers):
    from synth import workloads as WL
    npdt = np.float32 if w.esize == 4 else np.uint16
    out = np.zeros((w.batch, layers, 2, w.T, w.n_kv_heads, w.head_dim), npdt)
    for b in range(w.batch):
        L = int(prefix_len[b])
        for layer in range(layers):
            for which in range(2):
                sub = np.zeros(w.T * geo["pos_stride"], npdt)
                base = b * geo["seq_stride"] + layer * geo["layer_stride"] + which * geo["kv_stride"]
                WL.kv_fill(sub, w, geo, b, layer, which, L, L + w.T, seed, offset=base + L * geo["pos_stride"])
                out[b, layer, which] = sub.reshape(w.T, w.n_kv_heads, w.head_dim)
    return out


class OracleInputs:
    """Host inputs of one oracle cycle of a workload (input set `set_index` of `seed`)."""

    def __init__(self, w, seed: int, set_index: int = 0, planted: bool = False):
        from synth import workloads as WL
        sd = seed + 1000 * set_index
        self.w = w
        self.s = dict(draft=WL.draft_logits(w, sd, planted=planted), target=WL.target_logits(w, sd),
                      q=WL.queries(w, sd), uniforms=WL.uniforms(w, sd, set_index))
        self.prefix_len = w.prefix_lengths(seed)
        self.root = WL.root_tokens(w, seed)
        self.geo = WL.kv_geometry(w, seed, w.layers)
        self.kh, self.vh = host_attention_layer(w, self.geo, self.prefix_len, seed, 0)
        self.region = host_tree_region(w, self.geo, self.prefix_len, seed, w.layers)

    def cycle(self, head_stride=1, policy=0) -> float:
        return oracle_cycle(self.w, self.s, self.prefix_len, self.root, self.kh, self.vh, self.geo, self.w.verify,
                            self.region, head_stride=head_stride, policy=policy)


def _oracle_worker_init():
    # one core per process: the input generator's OpenMP loops stay single-threaded
    os.environ["OMP_NUM_THREADS"] = "1"


def _oracle_worker(job):
    """One process of the all-cores CPU baseline: builds its own input set, waits
    for the common start time, then runs oracle cycles for `seconds` (or exactly
    `cycles` when given). Returns (cycles run, wall seconds, summed cycle estimates)."""
    name, kw, seed, set_index, policy, head_stride, seconds, cycles, start_at = job
    from synth import workloads as WL
    w = WL.WORKLOADS[name].with_(**kw)
    inp = OracleInputs(w, seed, set_index)
    inp.cycle(head_stride, policy)  # warm (first touch of the inputs, library load)
    while time.time() < start_at:
        time.sleep(0.005)
    t0 = time.perf_counter()
    n, est = 0, 0.0
    while (cycles and n < cycles) or (not cycles and (n < 1 or time.perf_counter() - t0 < seconds)):
        est += inp.cycle(head_stride, policy)
        n += 1
    return n, time.perf_counter() - t0, est


class OraclePool:
    """One spawned process per host core, for the oracle on all cores (started
    with `spawn` so that it is independent of any CUDA state of this process)."""

    def __init__(self, n: int):
        import multiprocessing as mp
        self.n = n
        self.pool = mp.get_context("spawn").Pool(n, initializer=_oracle_worker_init)

    def run(self, w, seed, policy, head_stride=1, seconds=8.0, cycles=0, lead=None):
        """All processes run independent cycles (input set i in process i) from a
        common start; returns (total cycles, wall seconds of the slowest, estimates)."""
        kw = {k: getattr(w, k) for k in ("sharpness", "verify", "layers", "prefix", "batch")}
        if lead is None:  # input generation and one warm cycle before the common start
            lead = 15.0 + 3e-8 * (w.depth * w.top_k + w.T) * w.batch * w.vocab
        start_at = time.time() + lead
        jobs = [(w.name, kw, seed, i, policy, head_stride, seconds, cycles, start_at) for i in range(self.n)]
        res = self.pool.map(_oracle_worker, jobs, chunksize=1)
        return sum(r[0] for r in res), max(r[1] for r in res), sum(r[2] for r in res)

    def close(self):
        self.pool.terminate()
        self.pool.join()


def cpu_baseline(w, args, seed, pool, lmhead_extra=None):
    """The oracle as it stands on the host: one core (in this process), and
    every core (one process per core, independent cycles)."""
    import oracle
    oracle.build()
    inp = OracleInputs(w, seed, 0, planted=args.planted)
    n, tot = 0, 0.0
    t0 = time.perf_counter()
    while n < 1 or (time.perf_counter() - t0 < args.cpu_seconds and n < 50):
        tot += inp.cycle(policy=POLICIES[args.policy])
        n += 1
    per_cycle = tot / n
    extra = lmhead_extra(inp) if lmhead_extra else (0.0, "")
    single = {"value": round(1.0 / (per_cycle + extra[0]), 6), "unit": "cycles/s", "cores": 1,
              "sample": f"{n} whole oracle cycles of {w.name} (every stage, all attention rows) on one core"
                        + extra[1]}
    out = dict(single, kind="oracle", cpu_model=cpu_model(), host_cores=host_cores(), single_core=single)
    if pool is not None and pool.n > 1:
        cyc, wall, _ = pool.run(w, seed, POLICIES[args.policy], seconds=args.cpu_seconds)
        v = cyc / wall
        if extra[0] > 0:  # the LM head leg is timed on one core and scaled: add it per cycle
            v = 1.0 / (1.0 / v + extra[0] / pool.n)
        out.update({"value": round(v, 6), "cores": pool.n,
                    "sample": f"{cyc} whole oracle cycles of {w.name} (every stage, all attention rows) in "
                              f"{wall:.1f} s, one process per core ({pool.n} processes), independent input sets"
                              + extra[1]})
    return out


# ------------------------------------------------------------ our arm ---

def run_workload(args, w, variant: dict, seed: int, ws_: int, rank: int, local: int, with_e2e: bool,
                 fill_all_regions: bool = True) -> dict:
    """Measure one configuration: returns the fields of a bench line (no CPU baseline).

    fill_all_regions: write generator values into every layer's tree region
    (else only the attention layers are generated; the other layers' regions,
    which only compaction touches, stay zero: the same bytes are moved)."""
    import torch
    from synth import workloads as WL
    from speculative_decoding_dynamic_gb300 import cycle as C
    from speculative_decoding_dynamic_gb300 import eagle as E

    planted, aligned = bool(variant.get("planted", False)), bool(variant.get("aligned", False))
    prefix_len = w.prefix_lengths(seed)
    geo = WL.kv_geometry(w, seed, w.layers)
    R, per_set, attn_bytes = rotation_sets(w, seed, args.sets)
    host_sets = []
    for r in range(R):
        sd = seed + 1000 * r
        host_sets.append(dict(draft=WL.draft_logits(w, sd, planted=planted), target=WL.target_logits(w, sd),
                              q=WL.queries(w, sd)))
    weight_d = lm_out = weight_h = None
    if args.lmhead:
        for r in range(R):
            host_sets[r]["hidden"] = WL.hidden_states(w, seed + 1000 * r)
        weight_h = WL.lmhead_weight(w, seed)
        weight_d = to_dev(weight_h)
    dev_sets = [{k: to_dev(v) for k, v in s.items()} for s in host_sets]
    root = WL.root_tokens(w, seed)
    prefix_d = to_dev(prefix_len)
    root_d = to_dev(root)

    # KV cache: attention layers 0..R-1 filled over [0, L+T), the other layers' tree regions.
    npdt = np.float32 if w.esize == 4 else np.uint16
    cache = torch.zeros(w.batch * geo["seq_stride"], dtype=C.torch_dtype(w.dtype), device="cuda")
    for b in range(w.batch):
        L = int(prefix_len[b])
        for layer in range(w.layers if fill_all_regions else R):
            for which in range(2):
                p0 = 0 if layer < R else L
                host = np.zeros((L + w.T - p0) * geo["pos_stride"], npdt)
                base = b * geo["seq_stride"] + layer * geo["layer_stride"] + which * geo["kv_stride"]
                WL.kv_fill(host, w, geo, b, layer, which, p0, L + w.T, seed, offset=base + p0 * geo["pos_stride"])
                lo = base + p0 * geo["pos_stride"]
                cache[lo:lo + host.size].copy_(to_dev(host).view(-1))

    cfg = E.TreeCfg(w.batch, w.vocab, w.top_k, w.depth, w.node_budget, w.threshold, w.dtype,
                    POLICIES[args.policy])
    kv = E.KvCfg(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.layers, geo["max_len"], w.dtype,
                 geo["seq_stride"], geo["layer_stride"], geo["kv_stride"], geo["pos_stride"])
    dc = C.DeviceCycle(cfg, kv, fused_head=args.fused_head)
    mode = E.GREEDY if w.verify == "greedy" else E.LOSSLESS
    if args.lmhead and not args.fused_head:  # the draft rows are an intermediate written by the LM head every step
        lm_out = torch.empty(w.depth, w.batch, w.top_k, w.vocab, dtype=C.torch_dtype(w.dtype), device="cuda")

    def cycle(r, stream=None):
        s = dev_sets[r]
        if args.lmhead:
            dc.run(lm_out, prefix_d, root_d, s["q"], cache, r, s["target"], seed + 1000 * r, r, mode, w.temperature,
                   compact=True, stream=stream, head=(weight_d, s["hidden"]))
        else:
            dc.run(s["draft"], prefix_d, root_d, s["q"], cache, r, s["target"], seed + 1000 * r, r, mode,
                   w.temperature, compact=True, stream=stream)

    # warm-up outside capture (sets kernel attributes), then one graph per set
    for r in range(R):
        cycle(r)
        if aligned:  # the tree depends on the draft rows only: align this set's targets to it
            torch.cuda.synchronize()
            align_targets(host_sets[r]["target"], dc.tokens.cpu().numpy(), dc.parent.cpu().numpy(),
                          dc.n_tree.cpu().numpy(), WL.plant_value(w, float(np.mean(w.sharpness_per_seq(seed)))))
            dev_sets[r]["target"].copy_(to_dev(host_sets[r]["target"]).view(dev_sets[r]["target"].shape))
            cycle(r)
    torch.cuda.synchronize()
    assert dc.status() == 0, "device status after warm-up"
    graphs = []
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    n0 = E.eagle_kernel_launches()
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            cycle(r)
        graphs.append(g)
    launches_per_cycle = (E.eagle_kernel_launches() - n0) // R
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    # clocks are sampled from before the warm-up to the end of the per-kernel
    # timings (the timed region alone can be shorter than one sample period)
    clk = start_clocks(local) if rank == 0 else None
    if clk:
        wait_first_sample(clk)
    for i in range(args.warmup):
        graphs[i % R].replay()
    torch.cuda.synchronize()
    if ws_ > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        graphs[i % R].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), device="cuda")
    if ws_ > 1:
        import torch.distributed as dist
        dist.barrier()
    ms_per_step = ms / args.steps
    value = job_throughput(ws_, args.steps, ms)

    # accepted lengths of every input set (lossless acceptance differs between sets)
    accs = []
    for r in range(R):
        graphs[r].replay()
        torch.cuda.synchronize()
        accs.append(dc.accept_len.cpu().numpy())
    acc_all = np.stack(accs)               # [R, B]
    # summed path value of the kept nodes (the tree's expected accepted length), averaged over sets
    vsum = torch.empty(w.batch, dtype=torch.float32, device="cuda")
    vals = []
    for r in range(R):
        graphs[r].replay()
        E.eagle_tree_value(cfg, dc.ws, vsum)
        torch.cuda.synchronize()
        vals.append(vsum.cpu().numpy())
    acc = acc_all.mean(axis=0)             # per sequence, averaged over the sets
    n_tree = dc.n_tree.cpu().numpy()
    depth_h = dc.depth.cpu().numpy()
    # attention FLOPs actually computed: QK^T and PV over every live slot's keys
    # (the prefix plus its ancestors-or-self), 2 FLOP per multiply-add
    attn_flop = 0
    for b in range(w.batch):
        nb = int(n_tree[b])
        anc = int(sum(int(depth_h[b, i]) + 1 for i in range(nb)))
        attn_flop += 4 * w.n_q_heads * w.head_dim * (nb * int(prefix_len[b]) + anc)

    # ---- per-kernel timing: each stage call alone, same launch configuration ----
    flush = None

    def time_call(fn, reps, flush_l2=False):
        """Average device time of one stage call: `reps` calls on rotating inputs
        captured in a CUDA graph, replayed once untimed and once timed. With
        flush_l2, every call is preceded by a write of a buffer larger than L2
        and the time of the writes alone is subtracted (for a stage whose
        inputs do not rotate, such as compaction of the same cache rows)."""
        nonlocal flush
        if flush_l2 and flush is None:
            flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device="cuda")
        for i in range(3):
            fn(i % R)
        torch.cuda.synchronize()

        def timed(with_fn):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(reps):
                    if flush_l2:
                        flush.fill_(i)
                    if with_fn:
                        fn(i % R)
            g.replay()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps

        t = timed(True)
        return max(t - timed(False), 0.0) if flush_l2 else t

    reps = args.kernel_reps
    # state for standalone stage calls: a completed cycle on set 0
    cycle(0)
    torch.cuda.synchronize()
    kt = {}
    if args.fused_head:
        kt["lmhead"] = time_call(lambda r: dc.head_topk(weight_d, dev_sets[r]["hidden"][1]), reps)
        cycle(0)
        kt["expand_step"] = time_call(lambda r: E.eagle_expand_topk(cfg, dc.ws, min(1, w.depth - 1), dc.lm_ids,
                                                                    dc.lm_vals, dc.lm_lse, dc.row_lse, dc.ftok,
                                                                    dc.fcount), reps)
    else:
        if args.lmhead:
            kt["lmhead"] = time_call(lambda r: E.eagle_lmhead(cfg, dc.ws, w.hidden_size, dev_sets[r]["hidden"][1],
                                                              weight_d, lm_out[1]), reps)
            cycle(0)
        kt["expand_step"] = time_call(lambda r: E.eagle_expand(cfg, dc.ws, min(1, w.depth - 1), dev_sets[r]["draft"][
            min(1, w.depth - 1)], None, dc.row_lse, dc.ftok, dc.fcount), reps)
    cycle(0)
    kt["rerank"] = time_call(lambda r: E.eagle_rerank(cfg, dc.ws), reps)
    kt["build_tree"] = time_call(lambda r: dc.build(prefix_d, root_d), reps)
    kt["attention"] = time_call(lambda r: dc.attention(dev_sets[r]["q"], cache, r, prefix_d), reps)
    kt["verify"] = time_call(lambda r: dc.verify(mode, w.temperature, dev_sets[r]["target"], seed + 1000 * r, r), reps)
    cycle(0)
    torch.cuda.synchronize()
    acc_compact = dc.accept_len.cpu().numpy()  # the accepted lengths the timed compaction calls move
    kt["compact"] = time_call(lambda r: dc.compact(cache, prefix_d), reps, flush_l2=True)
    torch.cuda.synchronize()
    clocks = stop_clocks(clk) if clk else None
    if clocks:
        clocks["window"] = "warm-up, timed region and per-kernel timings"
    alg = algorithmic_bytes(w, prefix_len, acc, w.layers)
    peak = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else None
    hbm_peak = peak["hbm_gbs"] if peak else 6800.0
    peak_src = "measured" if peak else "fallback"
    tensor_peak = peak["bf16_tflops"] if peak else 1900.0
    # LM head of one step: the weight, the hidden rows, the logits written
    # (fused: the merged lse and top-k ids and logits instead of the logits)
    lm_flop = 2 * w.batch * w.top_k * w.vocab * w.hidden_size
    rows_ = w.batch * w.top_k
    lm_bytes = (w.vocab + rows_) * w.hidden_size * 2 + (
        rows_ * (4 + 8 * w.top_k) if args.fused_head else rows_ * w.vocab * w.esize)
    if args.fused_head:  # stage 2 from the merged top-k: ids, logits and lse of the step's rows
        alg = dict(alg, expand_step=rows_ * (4 + 8 * w.top_k))
    per_kernel = {}
    for name, ms_k in kt.items():
        byt = {"expand_step": alg["expand_step"], "attention": alg["attention"], "verify": alg["verify"],
               "lmhead": lm_bytes,
               "compact": algorithmic_bytes(w, prefix_len, acc_compact, w.layers)["compact"]}.get(name)
        e = {"ms": round(ms_k, 5)}
        if byt is not None and ms_k > 0:  # (a flushed timing of a tiny call can come out as 0)
            e["bytes"] = int(byt)
            e["GB_s"] = round(byt / (ms_k * 1e-3) / 1e9, 1)
            e["frac_hbm"] = round(byt / (ms_k * 1e-3) / 1e9 / hbm_peak, 4)
        flop = {"attention": attn_flop, "lmhead": lm_flop}.get(name)
        if flop is not None and ms_k > 0:
            e["tflops"] = round(flop / (ms_k * 1e-3) / 1e12, 1)
            if peak:
                e["frac_tensor"] = round(flop / (ms_k * 1e-3) / 1e12 / peak["bf16_tflops"], 4)
        per_kernel[name] = e
    per_kernel["compact"]["accept_len_moved"] = round(float(np.mean(acc_compact)), 3)
    cyc_share = {"expand_step": kt["expand_step"] * (w.depth - 1), "attention": kt["attention"],
                 "verify": kt["verify"]}
    if args.lmhead:
        cyc_share["lmhead"] = kt["lmhead"] * w.depth
    dom = max(cyc_share, key=cyc_share.get)
    dom_bytes = {"expand_step": alg["expand_step"], "attention": alg["attention"], "verify": alg["verify"],
                 "lmhead": lm_bytes}[dom]
    achieved = dom_bytes / (kt[dom] * 1e-3) / 1e9
    kname = {"expand_step": "expand_kernel", "attention": "attention", "verify": "verify_kernel",
             "lmhead": "lmhead_topk_kernel" if args.fused_head else "lmhead_kernel"}[dom]
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": ncu_traffic(kname, w.name), "kernel": kname,
                "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                "bytes_per_launch": int(dom_bytes)}
    dom_flop = {"attention": attn_flop, "lmhead": lm_flop}.get(dom, 0)
    if dom_flop / (tensor_peak * 1e12) > dom_bytes / (hbm_peak * 1e9):
        # a compute-bound contraction: its roofline is the tensor pipe (bf16 dense)
        ach_t = dom_flop / (kt[dom] * 1e-3) / 1e12
        roofline.update({"bound": "tensor", "achieved": round(ach_t, 1), "peak": tensor_peak, "unit": "TFLOP/s",
                         "frac": round(ach_t / tensor_peak, 4),
                         "peak_source": f"{peak_src} bf16_tflops (burst cuBLAS GEMM)",
                         "flop_per_launch": int(dom_flop)})

    # ---- end to end through host buffers ----
    e2e = None
    if with_e2e:
        # with the LM head on, the draft rows are not an input (the hidden states are)
        pin = [{k: pinned(v) for k, v in s.items() if not (args.lmhead and k == "draft")} for s in host_sets]
        out_a = torch.empty(w.batch, dtype=torch.int32).pin_memory()
        out_t = torch.empty(w.batch, w.depth + 1, dtype=torch.int32).pin_memory()
        out_n = torch.empty(w.batch, dtype=torch.int32).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in pin[0].values())
        d2h = (out_a.numel() + out_t.numel() + out_n.numel()) * 4

        def e2e_step(i):
            r = i % R
            for k_, v in pin[r].items():
                dev_sets[r][k_].copy_(v, non_blocking=True)
            cycle(r)
            out_a.copy_(dc.accept_len, non_blocking=True)
            out_t.copy_(dc.out_tokens, non_blocking=True)
            out_n.copy_(dc.new_len, non_blocking=True)

        for i in range(min(args.warmup, 3)):
            e2e_step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            e2e_step(i)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        e2e = {"value": round(ws_ * args.steps / dt, 2), "unit": "cycles/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h),
               "note": "pinned host inputs copied in, C-ABI calls issued per step (no graph), results copied out"}
        del pin

    res = {
        "value": round(value, 2), "ms_per_step": round(ms_per_step, 5),
        "config": config_of(w, args, variant, R, per_set, attn_bytes),
        "tokens_of_tree_per_s": round(value * float(np.mean(n_tree)) * w.batch, 1),
        "accepted_tokens_per_s": round(value * float(np.mean(acc + 1)) * w.batch, 1),
        "mean_accept_len": round(float(np.mean(acc)), 3),
        "mean_tree_value": round(float(np.mean(vals)), 3),
        "roofline": roofline, "kernels": per_kernel, "e2e": e2e,
        "gpu_launches": int(launches_per_cycle * args.steps), "launches_per_cycle": int(launches_per_cycle),
        "clocks": clocks, "dtype": "bf16" if w.dtype == E.EAGLE_BF16 else "f32",
        "_host": {"weight_h": weight_h, "host_sets": host_sets},
    }
    # release the device buffers of this configuration before the next one
    del graphs, dev_sets, cache, dc, flush, weight_d, lm_out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def config_summary(r: dict) -> dict:
    """The compact record of one extra configuration in the `configs` block."""
    keep = ("value", "ms_per_step", "e2e", "kernels", "roofline", "mean_accept_len", "mean_tree_value",
            "tokens_of_tree_per_s", "accepted_tokens_per_s", "launches_per_cycle", "clocks", "config")
    out = {k: r[k] for k in keep}
    out["unit"] = "cycles/s"
    if out["e2e"]:
        out["e2e"] = {k: v for k, v in out["e2e"].items() if k != "note"}
    return out


# ------------------------------------------------------ the reference arm ---

def run_reference(args, w):
    """The oracle as it stands, timed on the host cores: the bench's reference arm.

    Each step runs one oracle cycle of the workload in every process of a pool
    (one process per host core, independent input sets, common start); the
    value is the cycles of all processes over the time of the slowest. When the
    steps would take more than ~150 s, tree attention (the dominant stage) is
    sampled on every m-th query head and its time scaled by m."""
    import oracle
    oracle.build()
    seed = args.seed
    cores = host_cores()
    pool = OraclePool(cores) if cores > 1 else None
    probe_inp = OracleInputs(w, seed, 0)
    probe = probe_inp.cycle(head_stride=w.n_q_heads, policy=POLICIES[args.policy])
    m = 1
    while m < w.n_q_heads and (args.steps + args.warmup) * probe / m > 150.0:
        m *= 2
    while w.n_q_heads % m:
        m //= 2
    if pool is None:
        for _ in range(args.warmup):
            probe_inp.cycle(m, POLICIES[args.policy])
        tot = sum(probe_inp.cycle(m, POLICIES[args.policy]) for _ in range(args.steps))
        v = args.steps / tot
        ms_step = 1e3 * tot / args.steps
        n_proc = 1
    else:
        # warm-up cycles run inside the workers before the common start; then K cycles each
        cyc, wall, est = pool.run(w, seed, POLICIES[args.policy], head_stride=m, cycles=args.steps)
        # with attention sampled the estimates scale each cycle back to a full one
        scale = max(1.0, (est / max(cyc, 1)) / (wall / args.steps))
        v = cyc / (wall * scale)
        ms_step = 1e3 * wall * scale / args.steps
        n_proc = pool.n
        pool.close()
    unit = "cycles/s"
    sample = (f"{args.steps} oracle cycles of {w.name} in each of {n_proc} process(es) (one per host core, "
              f"independent input sets): every stage in full"
              + ("" if m == 1 else f" except tree attention on every {m}-th query head, its time scaled by {m}"))
    R, per_set, attn_bytes = rotation_sets(w, seed, args.sets)
    variant = {"planted": args.planted, "aligned": args.aligned}
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, args, variant, R, per_set, attn_bytes),
            "cpu_baseline": {"value": v, "unit": unit, "cores": n_proc, "kind": "oracle", "sample": sample,
                             "cpu_model": cpu_model()},
            "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main ---

def main():
    args = parse()
    ws_, rank, local = dist_env()
    w = workload(args)
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w)
        return

    # the all-cores oracle pool is spawned before this process touches the GPU
    pool = None
    if rank == 0 and ws_ == 1 and not args.no_cpu_baseline and host_cores() > 1:
        pool = OraclePool(host_cores())

    import torch
    torch.cuda.set_device(local)
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from synth import workloads as WL
    from speculative_decoding_dynamic_gb300 import build as Bld
    Bld.build()
    from speculative_decoding_dynamic_gb300 import eagle as E  # noqa: F401  (loads libeagle.so)

    seed = rank_seed(args.seed, rank)
    variant = {"planted": args.planted, "aligned": args.aligned}
    head = run_workload(args, w, variant, seed, ws_, rank, local, with_e2e=not args.no_e2e)
    hostd = head.pop("_host")

    configs = None
    if not args.no_configs and ws_ == 1:
        configs = {}
        for label, name, kw, var in EXTRA_CONFIGS:
            wc = WL.WORKLOADS[name].with_(**kw) if kw else WL.WORKLOADS[name]
            if wc.name == w.name and wc.verify == w.verify and var.get("aligned", False) == args.aligned:
                continue  # the headline itself
            r = run_workload(args, wc, var, seed, ws_, rank, local, with_e2e=not args.no_e2e,
                             fill_all_regions=False)
            r.pop("_host")
            configs[label] = config_summary(r)

    cpu = None
    if rank == 0 and ws_ == 1 and not args.no_cpu_baseline:
        lm_extra = None
        if args.lmhead:
            def lm_extra(inp):
                # the oracle's LM head on one row against 2048 vocabulary rows, scaled
                # to every row of every step and the whole vocabulary
                import oracle
                nv = min(w.vocab, 2048)
                t1 = time.perf_counter()
                oracle.lmhead_logits(np.ascontiguousarray(hostd["host_sets"][0]["hidden"][0, :1]),
                                     hostd["weight_h"][:nv])
                t_lm = time.perf_counter() - t1
                return (t_lm * w.depth * w.batch * w.top_k * (w.vocab / nv),
                        f"; plus the oracle LM head timed on 1 row x {nv} vocabulary rows x {w.hidden_size} and "
                        f"scaled to {w.depth} steps x {w.batch * w.top_k} rows x {w.vocab} entries")
        cpu = cpu_baseline(w, args, seed, pool, lm_extra)
    if pool is not None:
        pool.close()

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "cycles/s", "n_gpus": ws_, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
            "config": head["config"],
            "tokens_of_tree_per_s": head["tokens_of_tree_per_s"],
            "accepted_tokens_per_s": head["accepted_tokens_per_s"],
            "mean_accept_len": head["mean_accept_len"], "mean_tree_value": head["mean_tree_value"],
            "roofline": head["roofline"], "kernels": head["kernels"], "cpu_baseline": cpu, "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"], "launches_per_cycle": head["launches_per_cycle"],
            "clocks": head["clocks"], "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if ws_ > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
