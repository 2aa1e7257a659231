#!/usr/bin/env python3
"""Benchmark of the hot path of one continuous-batching iteration on GB300.

A step is one pass of the whole path over one batch: paged decode/verify attention
(plan + split-KV attention + LSE merge) followed by spec_verify for the batch's verify
sequences.  Default workload: the 70B-shape stress batch (512 sequences, 64/8 heads,
d=128, bf16, page 32; 448 decode + 64 verify with k=4; vocab 128256).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is algorithmic bytes per step / device time per
step (GB/s) with every input resident in HBM; `e2e` is the same metric through the C ABI
with the step's inputs copied from pinned host memory and its results read back inside
the timed region (the KV page pool is the cache itself and stays resident).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn achieved HBM GB/s (% of GB300 peak); spec-verify seqs/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stress70b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-call timing of the small batches")
    ap.add_argument("--config-reps", type=int, default=200)
    ap.add_argument("--max-seqs", type=int, default=0,
                    help="profiling only: keep the first N sequences of the workload")
    return ap.parse_args()


def measured_peak(key="hbm_gbs"):
    """A denominator from MEASURED_PEAKS.json (`hbm_gbs` or `bf16_tflops`), else the
    fallback figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return (FALLBACK_HBM_GBS if key == "hbm_gbs" else FALLBACK_BF16_TFLOPS), "fallback"


# ---------------------------------------------------------------------------------
# Algorithmic bytes (each KV element read once per KV head, Q in, out + lse out, the
# block-table entries used; spec_verify: the row(s) it must read plus scalars).
# ---------------------------------------------------------------------------------
def attn_bytes(seq_lens, query_lens, Hq, Hkv, D, P, elem, kv_elem=None):
    """elem: bytes of a q / out element; kv_elem: of a K/V element (default elem).  A
    pool of 1-byte codes also reads one fp32 scale per token and KV head for K and V."""
    L = np.asarray(seq_lens, dtype=np.int64)
    ql = np.asarray(query_lens, dtype=np.int64)
    kv_elem = elem if kv_elem is None else kv_elem
    kv = int((L * Hkv * (D * 2 * kv_elem + (8 if kv_elem == 1 else 0))).sum())
    qo = int((ql * Hq * D * 2 * elem).sum())
    bt = int(((L + P - 1) // P * 4).sum())
    lse = int((ql * Hq * 4).sum())
    return kv + qo + bt + lse


def unique_kv_bytes(block_table, seq_lens, Hkv, D, P, kv_elem):
    """KV bytes of the distinct pages the batch reads (pages shared by several block
    tables counted once, each with the most slots any of them uses)."""
    bt = np.asarray(block_table)
    L = np.asarray(seq_lens, dtype=np.int64)
    used = {}
    for i, l in enumerate(L):
        for j in range(int((l + P - 1) // P)):
            pg = int(bt[i, j])
            used[pg] = max(used.get(pg, 0), int(min(P, l - j * P)))
    per_tok = Hkv * (D * 2 * kv_elem + (8 if kv_elem == 1 else 0))
    return int(sum(used.values())) * per_tok


def attn_flops(seq_lens, query_lens, Hq, D):
    """Algorithmic flops: query row (token j, head h) of sequence i attends positions
    0 .. L_i - ql_i + j, two products of 2 D flops per position."""
    L = np.asarray(seq_lens, dtype=np.int64)
    ql = np.asarray(query_lens, dtype=np.int64)
    # sum over j < ql of (L - ql + j + 1) = ql (L - ql) + ql (ql + 1) / 2
    pos = ql * (L - ql) + ql * (ql + 1) // 2
    return int(pos.sum()) * Hq * 4 * D


def verify_bytes(accepted_len, k, V):
    acc = np.asarray(accepted_len)
    rows = np.where(acc < k, 2, 1)  # residual needs p_j and q_j; the bonus needs p_k
    scalars = k * 4 + k * 8 + (k + 1) * 4 + 4
    return int((rows * V * 4).sum() + len(acc) * scalars)


def elem_sizes(kv_dtype):
    """(bytes of a q / out element, bytes of a K/V element) of a storage type."""
    from verify_attention_spec_gb300 import workloads as wl
    if kv_dtype in wl.QUANTIZED:
        return 2, 1
    return (2, 2) if kv_dtype == wl.BF16 else (4, 4)


def acceptance_stats(accepted_len, k, p=None, q=None):
    """Per-token acceptance of the drafts: accepted / ratio tests run (a sequence that
    accepts a drafts ran min(a + 1, k) tests), and, given the rows, the expected rate
    alpha = mean over (sequence, position) of sum_x min(p_i(x), q_i(x))."""
    acc = np.asarray(accepted_len, dtype=np.int64)
    tests = np.minimum(acc + 1, k)
    out = {"mean_accepted": float(acc.mean()),
           "per_token_acceptance": float(acc.sum() / max(int(tests.sum()), 1))}
    if p is not None and q is not None and k > 0:
        out["alpha_sum_min_pq"] = float(np.mean([np.minimum(p[b, :k], q[b]).sum(-1).mean()
                                                 for b in range(p.shape[0])]))
    return out


def tree_verify_bytes(accepted_len, path, parents, V):
    """As verify_bytes for draft trees: the walk ends at node u (the last accepted node,
    or the root); with children, its p and q rows (the residual), else its p row."""
    rows = 0
    n = parents.shape[1]
    for b, acc in enumerate(np.asarray(accepted_len)):
        u = int(path[b, acc - 1]) if acc > 0 else 0
        rows += 2 if np.any(parents[b] == u) else 1
    return int(rows * V * 4 + len(accepted_len) * (n * 4 * 3 + n * 8 + (n + 1) * 4 + 4))


def workload_desc(name):
    from verify_attention_spec_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    return (f"{name}: {w.num_seqs} seqs ({w.num_seqs - w.num_verify} decode + {w.num_verify} "
            f"verify {'trees of ' if w.tree else ''}k={w.k}), Hq/Hkv {w.num_q_heads}/{w.num_kv_heads}, d {w.head_dim}, "
            f"{w.kv_dtype}, page {w.page_size}, lengths {w.length_law}{w.length_args or w.fixed_lens}; "
            f"spec_verify vocab {w.vocab}")


# ---------------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.15)
        except Exception:  # no nvidia-smi: the line says the clocks were unavailable
            self.proc = None
            if getattr(self, "f", None) is not None:
                self.f.close()
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------
# ncu evidence (committed summary): DRAM traffic per launch of the attention kernel,
# valid only while the kernel source is unchanged.
# ---------------------------------------------------------------------------------
KERNEL_SOURCES = {"paged_attn": ["paged_attn.cu", "device_util.cuh"],
                  "spec_verify": ["spec_verify.cu", "device_util.cuh", "philox.cuh"],
                  "spec_verify_tree": ["spec_verify_tree.cu", "device_util.cuh", "philox.cuh"]}


def kernel_source_hash(kernel="paged_attn"):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "verify_attention_spec_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel="paged_attn"):
    """DRAM bytes per full-size launch of `kernel` on `workload` from its committed ncu
    summary, or None when there is none or the kernel has changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_ncu.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(kernel):
        return None
    return float(m_bytes.group(1))


# ---------------------------------------------------------------------------------
# The oracle on the host cores (CPU baseline and reference arm)
# ---------------------------------------------------------------------------------
def oracle_sample(a, seqs, parents=None):
    """Host copy of the chosen sequences with a compact pool (oracle input); parents:
    the batch's draft trees (per query row), sliced to the chosen rows."""
    import torch
    from verify_attention_spec_gb300 import workloads as wl
    bt = a.block_table.cpu().numpy()
    lens = a.seq_lens.cpu().numpy()
    qlens = a.query_lens.cpu().numpy()
    row0 = np.concatenate([[0], np.cumsum(qlens)])
    P = a.page_size
    ids, rows, nbt = [], [], []
    for i in seqs:
        n = (lens[i] + P - 1) // P
        base = sum(len(x) for x in ids)
        ids.append(bt[i, :n])
        nbt.append(np.arange(base, base + n, dtype=np.int32))
        rows.append(np.arange(row0[i], row0[i + 1]))
    idx = torch.from_numpy(np.concatenate(ids).astype(np.int64)).to(a.k_pages.device)
    maxp = max(len(x) for x in nbt)
    btn = np.full((len(seqs), maxp), -1, dtype=np.int32)
    for r, x in enumerate(nbt):
        btn[r, :len(x)] = x
    r = torch.from_numpy(np.concatenate(rows)).to(a.q.device)
    par = None if parents is None else np.asarray(parents)[np.concatenate(rows)]
    if a.kv_dtype in wl.QUANTIZED:
        np_ = lambda t: t.detach().cpu().contiguous().numpy()
        return dict(q=wl.bf16_bits(a.q[r].cpu()), k=np_(a.k_pages[idx]), v=np_(a.v_pages[idx]),
                    ks=np_(a.k_scale[idx]), vs=np_(a.v_scale[idx]), bt=btn, lens=lens[seqs],
                    qlens=qlens[seqs], parents=par)
    st = lambda t: wl.storage_for_oracle(t, a.kv_dtype)
    return dict(q=st(a.q[r]), k=st(a.k_pages[idx]), v=st(a.v_pages[idx]), bt=btn,
                lens=lens[seqs], qlens=qlens[seqs], parents=par)


def run_oracle_attention(sample, kv_dtype):
    import oracle
    from verify_attention_spec_gb300 import workloads as wl
    if kv_dtype in wl.QUANTIZED:
        fmt = oracle.Q_E4M3 if kv_dtype == wl.FP8 else oracle.Q_INT8
        return oracle.paged_attn_quant(sample["q"], sample["k"], sample["v"], sample["ks"],
                                       sample["vs"], sample["bt"], sample["lens"], sample["qlens"],
                                       fmt=fmt, parents=sample["parents"])
    code = oracle.BF16 if kv_dtype == wl.BF16 else oracle.F32
    return oracle.paged_attn(sample["q"], sample["k"], sample["v"], sample["bt"], sample["lens"],
                             sample["qlens"], dtype_code=code, parents=sample["parents"])


def run_oracle_verify(v, rows=None):
    """The oracle's verification of v (its first `rows` sequences): the tree walk when v
    holds trees, else the plain rule."""
    import oracle
    sl = slice(None) if rows is None else slice(0, rows)
    if v.parents is not None:
        return oracle.spec_verify_tree(v.p[sl], v.q[sl], v.draft[sl], v.parents[sl], v.seed)
    return oracle.spec_verify(v.p[sl], v.q[sl], v.draft[sl], v.seed)


def time_oracle_attention(sample, kv_dtype):
    t0 = time.perf_counter()
    run_oracle_attention(sample, kv_dtype)
    return time.perf_counter() - t0


def choose_oracle_sample(a, target_s, rng_seed=0, parents=None):
    """Grow a seeded random sample of sequences (doubling) until the oracle takes at
    least target_s seconds on it, or the batch is exhausted."""
    order = np.random.default_rng(rng_seed).permutation(a.num_seqs)
    n = 4
    while True:
        seqs = sorted(order[:n].tolist())
        smp = oracle_sample(a, seqs, parents)
        dt = time_oracle_attention(smp, a.kv_dtype)
        if dt >= target_s or n >= a.num_seqs:
            return seqs, smp, dt
        n = min(a.num_seqs, max(n * 2, int(n * target_s / max(dt, 1e-3) * 1.1)))


def cpu_baseline(a, v, name, parents=None):
    import oracle
    w = a
    seqs, smp, dt = choose_oracle_sample(a, 10.0, parents=parents)
    runs = 1
    if dt < 10.0:  # the whole batch takes less than the target: run it again
        extra = int(np.ceil(10.0 / max(dt, 1e-3))) - 1
        for _ in range(extra):
            dt += time_oracle_attention(smp, a.kv_dtype)
        runs += extra
    by = attn_bytes(smp["lens"], smp["qlens"], w.num_q_heads, w.num_kv_heads, w.head_dim,
                    w.page_size, *elem_sizes(w.kv_dtype)) * runs
    out = {"value": by / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"paged attention on {len(seqs)} of {a.num_seqs} sequences of {name}, "
                     f"{runs} run(s) ({by / 1e9:.3f} GB algorithmic, {dt:.1f} s)"}
    if v is not None:
        t0 = time.perf_counter()
        run_oracle_verify(v)
        tv = time.perf_counter() - t0
        out["spec_verify_seqs_per_s"] = v.B / tv
        out["sample"] += f"; spec_verify on all {v.B} verify sequences ({tv:.2f} s)"
    out["single_thread"] = single_thread_oracle()
    return out


def single_thread_oracle(names=("tiny", "decode64")):
    """The oracle on one host thread over the whole of each small batch (GB/s of
    algorithmic bytes; the tiny case also its spec_verify)."""
    import oracle
    from verify_attention_spec_gb300 import workloads as wl
    n0 = oracle.num_threads()
    res = {}
    oracle.set_num_threads(1)
    try:
        for nm in names:
            a = wl.workload_attention(nm)
            smp = oracle_sample(a, list(range(a.num_seqs)))
            runs, dt = 0, 0.0
            while dt < 1.0:
                dt += time_oracle_attention(smp, a.kv_dtype)
                runs += 1
            by = attn_bytes(smp["lens"], smp["qlens"], a.num_q_heads, a.num_kv_heads,
                            a.head_dim, a.page_size, *elem_sizes(a.kv_dtype)) * runs
            res[nm] = {"gbs": by / dt / 1e9, "runs": runs, "seconds": dt}
            v = wl.workload_verify(nm)
            if v is not None:
                t0 = time.perf_counter()
                run_oracle_verify(v)
                res[nm]["spec_verify_seqs_per_s"] = v.B / (time.perf_counter() - t0)
    finally:
        oracle.set_num_threads(n0)
    return res


# ---------------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------------
def dist_setup(args, backend="nccl"):
    """One process per GPU (torchrun's RANK / LOCAL_RANK / WORLD_SIZE).  The path has no
    data exchange: torch.distributed carries only the barrier and the max-over-ranks time."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
        else:
            dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The slowest rank's time (every rank returns it)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(bytes_per_rank_step, world, ms_per_step):
    """Weak scaling: every rank streams its own batch, so the job moves world times the
    per-rank bytes in the slowest rank's step time (GB/s)."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


SMALL_CONFIGS = ["decode64", "verify32", "mixed272"]
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2


class L2Flush:
    """Evicts the L2 between timed reps: writes one buffer larger than L2, then reads
    another, so that the lines left behind are clean (dirty lines would be written back
    while the next timed kernel reads)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def time_small_config(name, dev, reps, peak):
    """One of the small batches (0.27-0.45 GB of KV per call, launch- and latency-scale):
    `reps` calls of paged_attn_fwd then spec_verify, each preceded by a write of a
    buffer larger than L2 and timed alone with CUDA events on the launching stream.
    Returns median and best per call, with GB/s and the fraction of `peak` taken from
    the median."""
    import torch
    from verify_attention_spec_gb300 import binding as vas
    from verify_attention_spec_gb300 import workloads as wl
    a = wl.workload_attention(name)
    mv = lambda t: None if t is None else t.to(dev).contiguous()
    a = wl.AttentionInputs(*(mv(t) for t in (a.q, a.k_pages, a.v_pages, a.block_table,
                                             a.seq_lens, a.query_lens)),
                           a.num_q_heads, a.num_kv_heads, a.head_dim, a.page_size, a.kv_dtype)
    v = wl.workload_verify(name)
    dims = vas.attn_dims(a.q, a.k_pages, a.block_table, a.seq_lens)
    ws = vas.alloc_workspace(dims, device=dev)
    out = torch.empty_like(a.q)
    lse = torch.empty(a.q.shape[0], a.q.shape[1], dtype=torch.float32, device=dev)
    if v is not None:
        p_d, q_d, x_d = (torch.from_numpy(x).to(dev) for x in (v.p, v.q, v.draft))
        acc_d = torch.empty(v.B, dtype=torch.int32, device=dev)
        tok_d = torch.empty(v.B, v.k + 1, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)

    def call():
        vas.paged_attn_fwd(a.q, a.k_pages, a.v_pages, a.block_table, a.seq_lens, a.query_lens,
                           out, lse, ws, dims=dims)

    def verify():
        vas.spec_verify(p_d, q_d, x_d, v.seed, acc_d, tok_d)

    for _ in range(5):
        call()
        if v is not None:
            verify()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    for e in ev:
        flush()
        e[0].record()
        call()
        e[1].record()
        if v is not None:
            verify()
        e[2].record()
    torch.cuda.synchronize()
    at = np.array([e[0].elapsed_time(e[1]) for e in ev]) * 1e3
    by = attn_bytes(a.seq_lens.cpu().numpy(), a.query_lens.cpu().numpy(), a.num_q_heads,
                    a.num_kv_heads, a.head_dim, a.page_size, *elem_sizes(a.kv_dtype))
    med = float(np.median(at))
    res = {"workload": workload_desc(name), "reps": reps,
           "l2": f"before every rep a {L2_FLUSH_BYTES >> 20} MiB buffer written and another read",
           "paged_attn": {"us_median": med, "us_best": float(at.min()), "algorithmic_bytes": by,
                          "gbs": by / (med * 1e-6) / 1e9,
                          "frac_of_measured_peak": by / (med * 1e-6) / 1e9 / peak,
                          "frac_of_nominal_8tbs": by / (med * 1e-6) / 1e9 / NOMINAL_HBM_GBS}}
    if v is not None:
        vt = np.array([e[1].elapsed_time(e[2]) for e in ev]) * 1e3
        vb = verify_bytes(acc_d.cpu().numpy(), v.k, v.V)
        vmed = float(np.median(vt))
        res["spec_verify"] = {"us_median": vmed, "us_best": float(vt.min()),
                              "seqs_per_s": v.B / (vmed * 1e-6), "algorithmic_bytes": vb,
                              "gbs": vb / (vmed * 1e-6) / 1e9,
                              "frac_of_measured_peak": vb / (vmed * 1e-6) / 1e9 / peak,
                              **acceptance_stats(acc_d.cpu().numpy(), v.k, v.p, v.q)}
    del flush
    return res


def run_ours(args):
    import torch
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    from verify_attention_spec_gb300 import binding as vas
    from verify_attention_spec_gb300 import workloads as wl

    name = args.workload
    w = wl.WORKLOADS[name]
    if args.max_seqs:
        lens = wl.sample_lengths(w)[:args.max_seqs]
        qlens = wl.query_lengths(w)[:args.max_seqs]
        a = wl.attention_inputs(lens, qlens, num_q_heads=w.num_q_heads,
                                num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                                page_size=w.page_size, kv_dtype=w.kv_dtype, seed=w.seed,
                                pool_device=dev)
    else:
        a = wl.workload_attention(name, pool_device=dev)
    mv = lambda t: None if t is None else t.to(dev).contiguous()
    a = wl.AttentionInputs(*(mv(t) for t in (a.q, a.k_pages, a.v_pages, a.block_table,
                                             a.seq_lens, a.query_lens)),
                           a.num_q_heads, a.num_kv_heads, a.head_dim, a.page_size, a.kv_dtype,
                           mv(a.k_scale), mv(a.v_scale))
    quant = a.kv_dtype if a.kv_dtype in wl.QUANTIZED else None
    # Draft trees (tree workloads): one random tree per verify window, its ancestor
    # masks for the attention and its nodes for the verification.
    tree_masks = None
    attn_parents = None
    if w.tree:
        qlens_all = a.query_lens.cpu().numpy()
        attn_parents = wl.draft_tree_parents(qlens_all, seed=w.seed)
        tree_masks = torch.from_numpy(wl.ancestor_bits(attn_parents, qlens_all).view(np.int64)).to(dev)
    v = wl.workload_verify(name, attn_parents=attn_parents) if not args.max_seqs or not w.tree else None
    if args.max_seqs and v is not None:
        nv = max(1, int((qlens > 1).sum()))
        v = wl.VerifyInputs(v.p[:nv], v.q[:nv], v.draft[:nv], v.seed,
                            None if v.parents is None else v.parents[:nv])
    dims = vas.attn_dims(a.q, a.k_pages, a.block_table, a.seq_lens, quant=quant)
    ws = vas.alloc_workspace(dims, device=dev)

    def attn(q_, bt_, sl_, ql_, out_, lse_):
        """One attention call through the C ABI (quantised pools: paged_attn_fwd_quant;
        draft trees: paged_attn_fwd_tree)."""
        if quant:
            vas.paged_attn_fwd_quant(q_, a.k_pages, a.v_pages, a.k_scale, a.v_scale, bt_, sl_, ql_,
                                     out_, lse_, ws, quant=quant, tree_mask=tree_masks, dims=dims)
        elif tree_masks is not None:
            vas.paged_attn_fwd_tree(q_, a.k_pages, a.v_pages, bt_, sl_, ql_, tree_masks, out_,
                                    lse_, ws, dims=dims)
        else:
            vas.paged_attn_fwd(q_, a.k_pages, a.v_pages, bt_, sl_, ql_, out_, lse_, ws, dims=dims)

    out = torch.empty_like(a.q)
    lse = torch.empty(a.q.shape[0], a.q.shape[1], dtype=torch.float32, device=dev)
    if v is not None:
        p_d = torch.from_numpy(v.p).to(dev)
        q_d = torch.from_numpy(v.q).to(dev)
        x_d = torch.from_numpy(v.draft).to(dev)
        acc_d = torch.empty(v.B, dtype=torch.int32, device=dev)
        tok_d = torch.empty(v.B, v.k + 1, dtype=torch.int32, device=dev)
        par_d = torch.from_numpy(v.parents).to(dev) if v.parents is not None else None
        path_d = torch.empty(v.B, v.k, dtype=torch.int32, device=dev)

    def verify(p_, q_, x_, acc_, tok_):
        """One verification call through the C ABI (draft trees: spec_verify_tree)."""
        if par_d is not None:
            vas.spec_verify_tree(p_, q_, x_, par_d, v.seed, acc_, tok_, path_d)
        else:
            vas.spec_verify(p_, q_, x_, v.seed, acc_, tok_)

    def step():
        attn(a.q, a.block_table, a.seq_lens, a.query_lens, out, lse)
        if v is not None:
            verify(p_d, q_d, x_d, acc_d, tok_d)

    elem, kv_elem = elem_sizes(a.kv_dtype)
    a_bytes = attn_bytes(a.seq_lens.cpu().numpy(), a.query_lens.cpu().numpy(), a.num_q_heads,
                         a.num_kv_heads, a.head_dim, a.page_size, elem, kv_elem)
    # Prefix sharing: the KV bytes of distinct pages (what HBM must deliver at least)
    # against the per-sequence count in a_bytes.
    kv_logical = attn_bytes(a.seq_lens.cpu().numpy(), np.zeros(a.num_seqs), 0, a.num_kv_heads,
                            a.head_dim, a.page_size, elem, kv_elem) - \
        int(((a.seq_lens.cpu().numpy().astype(np.int64) + a.page_size - 1) // a.page_size * 4).sum())
    kv_unique = unique_kv_bytes(a.block_table.cpu().numpy(), a.seq_lens.cpu().numpy(),
                                a.num_kv_heads, a.head_dim, a.page_size, kv_elem)
    a_bytes_unique = a_bytes - kv_logical + kv_unique
    step()
    torch.cuda.synchronize()
    if v is None:
        v_bytes = 0
    elif v.parents is not None:
        v_bytes = tree_verify_bytes(acc_d.cpu().numpy(), path_d.cpu().numpy(), v.parents, v.V)
    else:
        v_bytes = verify_bytes(acc_d.cpu().numpy(), v.k, v.V)
    step_bytes = a_bytes + v_bytes

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start.record()
    for i in range(K):
        ev[i][0].record()
        attn(a.q, a.block_table, a.seq_lens, a.query_lens, out, lse)
        ev[i][1].record()
        if v is not None:
            verify(p_d, q_d, x_d, acc_d, tok_d)
        ev[i][2].record()
    t_end.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    attn_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    ver_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev])) if v is not None else 0.0
    ms_per_step = total_ms / K
    launches_per_step = 2 + (1 if v is not None else 0)  # plan + attention (+ spec_verify)

    # e2e: the same step through the C ABI from pinned host buffers, as a serving loop
    # runs it: every step's inputs are copied from pinned host memory and its results
    # read back, on one copy stream per direction, double-buffered so that the copies of
    # steps i + 1 and i - 1 overlap the compute of step i (the KV page pool is the cache:
    # it stays).
    e2e = None
    if not args.no_e2e:
        host_in = [t.cpu().pin_memory() for t in (a.q, a.block_table, a.seq_lens, a.query_lens)]
        host_v = ([torch.from_numpy(x).pin_memory() for x in (v.p, v.q, v.draft)]
                  if v is not None else [])
        res_like = [out, lse] + ([acc_d, tok_d] if v is not None else [])
        cs = torch.cuda.current_stream()
        xs = torch.cuda.Stream()  # host-to-device copies
        ds = torch.cuda.Stream()  # device-to-host copies: the other direction's engine
        slots = []
        for _ in range(2):
            slots.append(dict(
                din=[torch.empty_like(t, device=dev) for t in host_in],
                dv=[torch.empty_like(t, device=dev) for t in host_v],
                dout=[torch.empty_like(t) for t in res_like],
                hout=[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in res_like],
                up=torch.cuda.Event(), comp=torch.cuda.Event(), down=torch.cuda.Event()))
        h2d = sum(t.numel() * t.element_size() for t in host_in + host_v)
        d2h = sum(t.numel() * t.element_size() for t in slots[0]["hout"])

        def upload(sl):
            with torch.cuda.stream(xs):
                xs.wait_event(sl["comp"])  # the step that last read these inputs is done
                for hsrc, dd in zip(host_in + host_v, sl["din"] + sl["dv"]):
                    dd.copy_(hsrc, non_blocking=True)
                sl["up"].record(xs)

        def compute(sl):
            cs.wait_event(sl["up"])
            cs.wait_event(sl["down"])  # this slot's previous results have been read back
            q_, bt_, sl_, ql_ = sl["din"]
            attn(q_, bt_, sl_, ql_, sl["dout"][0], sl["dout"][1])
            if v is not None:
                verify(sl["dv"][0], sl["dv"][1], sl["dv"][2], sl["dout"][2], sl["dout"][3])
            sl["comp"].record(cs)

        def download(sl):
            with torch.cuda.stream(ds):
                ds.wait_event(sl["comp"])
                for dd, hdst in zip(sl["dout"], sl["hout"]):
                    hdst.copy_(dd, non_blocking=True)
                sl["down"].record(ds)

        def e2e_run(n, t0=None, t1=None):
            if t0 is not None:
                t0.record(xs)
            upload(slots[0])
            for i in range(n):
                if i + 1 < n:
                    upload(slots[(i + 1) % 2])
                compute(slots[i % 2])
                download(slots[i % 2])
            if t1 is not None:
                xs.wait_stream(ds)  # the last results are read back
                t1.record(xs)

        e2e_run(max(args.warmup, 2))
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e2e_run(K, e0, e1)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / K
        # The results read back by the last step are those of the resident run (the
        # kernels are deterministic): a pipelining mistake would not pass silently.
        last = slots[(K - 1) % 2]["hout"]
        if not all(torch.equal(h, r.cpu()) for h, r in zip(last, res_like)):
            raise RuntimeError("e2e results differ from the resident run")
        e2e = {"value": whole_job_rate(step_bytes, world, e2e_ms), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms}

    peak, peak_src = measured_peak()
    attn_gbs = a_bytes / (attn_ms * 1e-3) / 1e9
    a_flops = attn_flops(a.seq_lens.cpu().numpy(), a.query_lens.cpu().numpy(), a.num_q_heads,
                         a.head_dim)
    attn_tflops = a_flops / (attn_ms * 1e-3) / 1e12
    tpeak, tpeak_src = measured_peak("bf16_tflops")
    # Above the ridge (peak flops / peak bytes) the call is bound by the tensor cores
    # (chunked prefill); below it by HBM (decode and verify).
    tensor_bound = a_flops / max(a_bytes, 1) > tpeak * 1e12 / (peak * 1e9)
    value = whole_job_rate(step_bytes, world, ms_per_step)
    res = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": a.kv_dtype,
        "data": "synthetic",
        "config": {"workload": workload_desc(name) + (f" (first {args.max_seqs} sequences only)"
                                                       if args.max_seqs else ""),
                   "l2": "inputs larger than L2 (KV pool %.1f GB per step)"
                         % ((a.k_pages.numel() + a.v_pages.numel()) * kv_elem / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "paged_attn": {"gbs": attn_gbs, "ms": attn_ms, "algorithmic_bytes": a_bytes,
                       "distinct_page_bytes": a_bytes_unique,
                       "distinct_page_gbs": a_bytes_unique / (attn_ms * 1e-3) / 1e9,
                       "algorithmic_flops": a_flops, "tflops": attn_tflops,
                       "frac_of_measured_peak": attn_gbs / peak,
                       "frac_of_nominal_8tbs": attn_gbs / NOMINAL_HBM_GBS},
        "roofline": ({"bound": "tensor", "achieved": attn_tflops, "peak": tpeak,
                      "unit": "TFLOP/s", "frac": attn_tflops / tpeak, "traffic": ncu_traffic(name),
                      "peak_source": tpeak_src + " (bf16, burst)",
                      "kernel": "paged_attn_fwd (plan + attention with the fused LSE merge)"}
                     if tensor_bound else
                     {"bound": "hbm", "achieved": attn_gbs, "peak": peak, "unit": "GB/s",
                      "frac": attn_gbs / peak, "traffic": ncu_traffic(name),
                      "peak_source": peak_src,
                      "kernel": "paged_attn_fwd (plan + attention with the fused LSE merge)"}),
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
    }
    attn_steps = np.array([e[0].elapsed_time(e[1]) for e in ev]) * 1e3
    res["paged_attn"]["us_median"] = float(np.median(attn_steps))
    res["paged_attn"]["us_best"] = float(attn_steps.min())
    if v is not None:
        acc = acc_d.cpu().numpy()
        ver_steps = np.array([e[1].elapsed_time(e[2]) for e in ev]) * 1e3
        ver_gbs = v_bytes / (ver_ms * 1e-3) / 1e9
        res["spec_verify"] = {"seqs_per_s": v.B / (ver_ms * 1e-3), "ms": ver_ms,
                              "us_median": float(np.median(ver_steps)),
                              "us_best": float(ver_steps.min()),
                              "gbs": ver_gbs, "algorithmic_bytes": v_bytes,
                              "frac_of_measured_peak": ver_gbs / peak,
                              "frac_of_nominal_8tbs": ver_gbs / NOMINAL_HBM_GBS,
                              "traffic": ncu_traffic(name, "spec_verify" if v.parents is None
                                                     else "spec_verify_tree"),
                              **(acceptance_stats(acc, v.k, v.p, v.q) if v.parents is None
                                 else acceptance_stats(acc, v.k))}
    if e2e is not None:
        res["e2e"] = e2e
    if not args.no_configs and not args.max_seqs and name == "stress70b":
        res["configs"] = {c: time_small_config(c, dev, max(args.config_reps, 100), peak)
                          for c in SMALL_CONFIGS}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(a, v, name, attn_parents)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------------
# Reference arm: the oracle as it stands, on the host cores
# ---------------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from verify_attention_spec_gb300 import workloads as wl
    name = args.workload
    w = wl.WORKLOADS[name]
    # the inputs: the same workload, its pool drawn on the host (no GPU on this leg)
    lens, qlens = wl.sample_lengths(w) + w.prefix_tokens, wl.query_lengths(w)
    parents_all = wl.draft_tree_parents(qlens, seed=w.seed) if w.tree else None
    order = np.random.default_rng(0).permutation(len(lens))
    # a bounded sample: sequences in seeded order up to ~64 MB of KV
    elem, kv_elem = elem_sizes(w.kv_dtype)
    per_tok = w.num_kv_heads * w.head_dim * 2 * kv_elem
    seqs, tot = [], 0
    for i in order:
        if seqs and tot + lens[i] * per_tok > 64e6:
            break
        seqs.append(int(i))
        tot += lens[i] * per_tok
    seqs.sort()
    a = wl.attention_inputs(lens[seqs], qlens[seqs], num_q_heads=w.num_q_heads,
                            num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                            page_size=w.page_size, kv_dtype=w.kv_dtype, seed=w.seed)
    v = wl.workload_verify(name, attn_parents=parents_all)
    par = None
    if parents_all is not None:
        row0 = np.concatenate([[0], np.cumsum(qlens)])
        par = np.concatenate([parents_all[row0[i]:row0[i + 1]] for i in seqs])
    smp = oracle_sample(a, list(range(len(seqs))), par)
    by = attn_bytes(smp["lens"], smp["qlens"], w.num_q_heads, w.num_kv_heads, w.head_dim,
                    w.page_size, elem, kv_elem)

    def step():
        run_oracle_attention(smp, w.kv_dtype)
        if v is not None:
            run_oracle_verify(v, rows=8)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    vb = verify_bytes(np.zeros(8, np.int32), v.k, v.V) if v is not None else 0
    value = (by + vb) / dt / 1e9
    sample = (f"per step: paged attention on {len(seqs)} of {w.num_seqs} sequences of {name} "
              f"({by / 1e9:.3f} GB algorithmic)" + (f" + spec_verify on 8 of {v.B} verify sequences"
                                                    if v is not None else ""))
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": workload_desc(name)},
           "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
