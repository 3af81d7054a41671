"""Benchmark of the MSA decode hot path (score -> pool -> top-k -> attend).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--workloads all|NAME,NAME,...]

One step = one msa_decode call over one batch of synthetic input (the whole
path, every stage).  Prints ONE JSON line on rank 0: the headline workload
(default: the FP8 decode batch, 32 sequences of 16K-32K tokens) as the line's
value, and every workload of the set under "workloads" (FP8 decode, long
context, NVFP4 speculative verify, tiny BF16, prefill chunk), each timed the
same way.  Under torchrun with N > 1 every rank runs its own replica of the
workload (decode batches are independent problems: weak scaling, no
collective on the data path).
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MSA decode queries/s and HBM GB/s (% of GB300 peak), score+topk+attend"
WORKLOAD_TEXT = {
    "fp8_decode": "FP8 E4M3 decode: 32 seqs, context ~U[16K,32K] (seeded), 1 query token each, 16 q / 4 KV heads, "
                  "dim 128, index dim 128, top-16 of 128-token blocks, K/V/index keys E4M3 + fp32 per-token scales, "
                  "bf16 queries, shuffled physical block table",
    "fp8_long": "Long-context FP8 decode: 4 seqs x 512K tokens (4096 blocks), 1 query token, 16 q / 4 KV heads, "
                "dim 128, top-16, FP8 E4M3 K/V/index keys + per-token scales, bf16 queries",
    "nvfp4_verify": "NVFP4 speculative verify: 8 seqs x 128K, 8 query tokens each, NVFP4 K/V/index keys, E4M3 queries",
    "tiny_bf16": "Tiny BF16 decode: 1 seq x 4096 tokens, 1 query, BF16 everything",
    "fp8_prefill": "Prefill chunk: 8192 new tokens on a 64K-token FP8 E4M3 context (1 seq), bf16 queries, "
                   "per-query top-16, causal",
}
ALL_WORKLOADS = ("fp8_decode", "fp8_long", "nvfp4_verify", "tiny_bf16", "fp8_prefill")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="fp8_decode", choices=sorted(WORKLOAD_TEXT),
                    help="the workload the line's value is quoted on")
    ap.add_argument("--workloads", default="all",
                    help="workloads timed under 'workloads' ('all', 'none' or a comma list)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


def load_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, kind) from the driver's measurement, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernels_per_step(w) -> int:
    """Launches of one msa_decode (see the launch chains in msa_api.cu)."""
    r = w.num_q_heads // w.num_kv_heads
    if w.q_per_seq > 8 and w.kv_dtype == "fp8" and r in (1, 2, 4, 8):
        return 7  # tcgen05 indexer, warp top-k, count, scan, fill, key-block-major attend, combine
    return 3      # indexer, top-k, attend


def indexer_flops(w):
    """Algorithmic FLOPs of the index scores: every visible key x groups x index dim x 2."""
    tot = 0
    for T in w.seq_lens:
        first = T - w.q_per_seq + 1  # keys visible to the first new token
        tot += w.q_per_seq * first + w.q_per_seq * (w.q_per_seq - 1) // 2
    return 2.0 * tot * w.num_kv_heads * w.index_dim


def attend_flops(w, sel):
    """Algorithmic FLOPs of the attend: per (token, q head) 2 x 2 x D per visible selected key."""
    Q, G, r = w.q_per_seq, w.num_kv_heads, w.num_q_heads // w.num_kv_heads
    keys = 0
    for s, T in enumerate(w.seq_lens):
        for i in range(Q):
            pos = T - Q + i
            for g in range(G):
                for b in sel[s * Q + i, g]:
                    if b >= 0:
                        keys += max(0, min(128, pos + 1 - 128 * int(b)))
    return 4.0 * keys * r * w.head_dim


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def replica_seed(base_seed: int, rank: int) -> int:
    """Each rank runs its own, independent replica of the workload."""
    return base_seed + 1000 * rank


def max_over_ranks(values, world: int, dist=None, device=None):
    """Element-wise max of per-rank timings (the slowest rank defines the step)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def algorithmic_bytes(w, sel_union_blocks):
    """Bytes the pages' decode model reads per step: whole-context index keys +
    K/V of the selected blocks (union over a sequence's query tokens, per KV head)."""
    from block_sparse_attention_03_gb300 import roofline as R
    idx = sum(w.seq_lens) * R.index_bytes_per_token(w.index_dtype)
    kv_tok = R.kv_bytes_per_token(w.kv_dtype, 1)  # per KV head
    kv = 0.0
    for s, T in enumerate(w.seq_lens):
        for g, blocks in enumerate(sel_union_blocks[s]):
            for b in blocks:
                kv += min(128, T - 128 * b) * kv_tok
    sc_idx, sc_kv = R.scale_bytes_per_token(w.kv_dtype, w.index_dtype, 1)
    actual = idx + kv + sum(w.seq_lens) * sc_idx
    for s, T in enumerate(w.seq_lens):
        for blocks in sel_union_blocks[s]:
            actual += sum(min(128, T - 128 * b) for b in blocks) * sc_kv
    return idx, kv, actual


# ---------------------------------------------------------------- CPU oracle on the host cores

def sample_rows(q_per_seq: int):
    """Query rows of a sequence the CPU sample covers: all of them, or the last 8
    (one verify-sized chunk) of a prefill chunk, which would take minutes."""
    return None if q_per_seq <= 8 else list(range(q_per_seq - 8, q_per_seq))


def _oracle_job(name: str, seq_len: int, seed: int):
    """One worker task: regenerate one sequence of the workload on the host
    (same shape and value distribution) and time the oracle's whole path on it
    (generation excluded).  Returns (seconds, query rows)."""
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    import numpy as np
    import msa_synth as ms
    from oracle import msa_oracle as O
    w = ms.make_workload(name, seq_lens=(seq_len,), seed=seed)
    h = ms.case_to_host(ms.make_case(w, device="cpu"))
    rows = sample_rows(w.q_per_seq)
    t0 = time.perf_counter()
    if rows is None:
        O.run_path(h)
        n = w.q_per_seq
    else:
        Q = w.q_per_seq
        pooled = O.pooled_scores(h, 0, w.index_dim ** -0.5, rows=rows)
        pos = O.positions(seq_len, Q)
        sel = np.full((Q, w.num_kv_heads, w.topk), -1, dtype=np.int32)
        for k, i in enumerate(rows):
            for g in range(w.num_kv_heads):
                sel[i, g] = O.select_blocks(pooled[k, g], int(pos[i]), w.topk)
        O.attend_rows(h, 0, sel, w.head_dim ** -0.5, rows=rows)
        n = len(rows)
    return time.perf_counter() - t0, n


class OraclePool:
    """A spawn-started process pool on the host cores (started before any GPU
    call), one single-threaded oracle per worker."""

    def __init__(self):
        import multiprocessing as mp
        self.cores = max(1, min(os.cpu_count() or 1, 64))
        os.environ["OMP_NUM_THREADS"] = "1"
        os.environ["OPENBLAS_NUM_THREADS"] = "1"
        os.environ["MKL_NUM_THREADS"] = "1"
        self.pool = mp.get_context("spawn").Pool(self.cores)

    def sample(self, name: str, seqs, seed: int):
        """Run the oracle on the given sequence lengths, one task each, all at once:
        (queries/s over the wall time of the slowest task, queries, tasks)."""
        jobs = [self.pool.apply_async(_oracle_job, (name, int(T), seed + 17 * i)) for i, T in enumerate(seqs)]
        res = [j.get() for j in jobs]
        busy = [0.0] * self.cores
        for k, (dt, _) in enumerate(res):  # tasks spread round-robin over the workers
            busy[k % self.cores] += dt
        wall = max(busy)
        n = sum(q for _, q in res)
        return n / wall, n, len(res)

    def close(self):
        self.pool.terminate()


def cpu_sample_plan(w):
    """Sequences the CPU sample covers (about 10-30 s of single-core oracle work)."""
    if w.name == "fp8_long":
        return [w.seq_lens[0]] * 4, "all 4 sequences of 512K tokens, each regenerated on the host"
    if w.name == "fp8_prefill":
        return [w.seq_lens[0]] * 2, "the last 8 query tokens of the 8,192-token chunk, twice"
    if w.name == "nvfp4_verify":
        return list(w.seq_lens), "all 8 sequences x 8 verify tokens, each regenerated on the host"
    return list(w.seq_lens), f"all {w.num_seqs} sequences, each regenerated on the host"


def run_reference(args):
    """Reference arm: the CPU oracle on the host cores, a bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import msa_synth as ms
    pool = OraclePool()
    w = ms.make_workload(args.workload)
    per_step = w.seq_lens[:min(len(w.seq_lens), pool.cores)]
    times, nq = [], 0
    for it in range(args.warmup + args.steps):
        qps, n, _ = pool.sample(w.name, per_step, w.seed + 31 * it)
        if it >= args.warmup:
            times.append(n / qps)
            nq = n
    pool.close()
    mean = sum(times) / len(times)
    qps = nq / mean
    sample = (f"{len(per_step)} sequences of the workload per step, one per host core, whole path "
              f"(score, pool, top-k, attend) in fp64" +
              (", the last 8 query tokens of each" if w.q_per_seq > 8 else ""))
    line = {"metric": METRIC, "value": qps, "unit": "queries/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload], "sample": sample},
            "cpu_baseline": {"value": qps, "unit": "queries/s", "cores": pool.cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": qps, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU measurement

class Bench:
    def __init__(self, dev, stream, flush_bytes=256 << 20):
        import torch
        self.torch = torch
        self.dev = dev
        self.stream = stream
        # L2 flush between timed steps: write 256 MB (> 129 MB L2), then read 512 MB so
        # that the written lines are already back in HBM and L2 holds only clean data
        self.flush_w = torch.empty(flush_bytes, dtype=torch.uint8, device=dev)
        self.flush_r = torch.ones(2 * flush_bytes // 4, dtype=torch.float32, device=dev)
        self.flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def flush(self):
        self.flush_w.zero_()
        self.torch.sum(self.flush_r, dim=0, out=self.flush_out)

    def time(self, fn, steps, warmup=0):
        """Mean ms of fn over `steps` runs, each after an L2 flush, CUDA events on the stream."""
        torch = self.torch
        for _ in range(warmup):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for i in range(steps):
            self.flush()
            evs[i][0].record(self.stream)
            fn()
            evs[i][1].record(self.stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / steps


def setup_workload(msa, ms, name, seed, dev):
    import torch
    w = ms.make_workload(name, seed=seed)
    case = ms.make_case(w, device=dev)
    cache = msa.PagedCache(kv_dtype=w.kv_dtype, index_dtype=w.index_dtype, num_blocks=case["num_blocks"],
                           num_kv_heads=w.num_kv_heads, k=case["k"], v=case["v"], idx=case["idx"],
                           k_sf=case.get("k_sf"), v_sf=case.get("v_sf"), k_scale=case.get("k_scale"),
                           v_scale=case.get("v_scale"), idx_sf=case.get("idx_sf"),
                           idx_scale=case.get("idx_scale"), k_global=case.get("k_global", 0.0),
                           v_global=case.get("v_global", 0.0), idx_global=case.get("idx_global", 0.0))
    batch = msa.Batch(case["seq_lens"], case["block_table"], w.q_per_seq)
    cfg = msa.default_config(w.topk)
    iq = msa.Query(case["index_q"], w.q_dtype, case["index_q_scale"])
    q = msa.Query(case["q"], w.q_dtype, case["q_scale"])
    ws = torch.empty(msa.msa_workspace_size(cache, batch, cfg, w.num_q_heads), dtype=torch.uint8, device=dev)
    msa.msa_workspace_init(ws)
    rows = w.num_seqs * w.q_per_seq
    topk = torch.empty((rows, w.num_kv_heads, w.topk), dtype=torch.int32, device=dev)
    out = torch.empty((rows, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((rows, w.num_q_heads), dtype=torch.float32, device=dev)
    return dict(w=w, case=case, cache=cache, batch=batch, cfg=cfg, iq=iq, q=q, ws=ws, topk=topk, out=out,
                lse=lse, rows=rows)


def measure_workload(msa, B, st, steps, warmup, peak_gbs, peak_tf_e4m3):
    """Time one workload: the whole msa_decode step and each stage alone (its own
    entry point, same launch shapes); byte model and fractions of the roofline."""
    import numpy as np
    import torch
    w, stream = st["w"], B.stream

    def step():
        msa.msa_decode(st["cache"], st["batch"], st["cfg"], st["iq"], st["q"], w.num_q_heads, st["topk"],
                       st["out"], st["lse"], st["ws"], stream)

    ms_step = B.time(step, steps, warmup=max(3, warmup))
    s_, flags = msa.msa_read_device_status(st["ws"])
    if s_ != 0:
        raise RuntimeError(f"{w.name}: device status {msa.msa_status_string(s_)} flags {flags}")

    # the stages alone, through the staged entry points
    pooled = torch.empty((st["rows"], w.num_kv_heads, w.max_blocks), dtype=torch.float32, device=B.dev)
    topk2 = torch.empty_like(st["topk"])
    out2 = torch.empty_like(st["out"])
    n_alone = max(5, min(steps, 20))
    idx_ms = B.time(lambda: msa.msa_indexer_score(st["cache"], st["batch"], st["cfg"], st["iq"], pooled, st["ws"],
                                                  stream), n_alone, warmup=3)
    topk_ms = B.time(lambda: msa.msa_topk_blocks(st["batch"], st["cfg"], w.num_kv_heads, pooled, topk2, None,
                                                 st["ws"], stream), n_alone, warmup=3)
    att_ms = B.time(lambda: msa.msa_sparse_attend(st["cache"], st["batch"], st["cfg"], st["q"], w.num_q_heads,
                                                  topk2, out2, None, st["ws"], stream), n_alone, warmup=3)
    s_, flags = msa.msa_read_device_status(st["ws"])
    if s_ != 0:
        raise RuntimeError(f"{w.name} (stages): device status {msa.msa_status_string(s_)} flags {flags}")

    sel = st["topk"].cpu().numpy()
    Q = w.q_per_seq
    unions = []
    for s in range(w.num_seqs):
        per_g = []
        for g in range(w.num_kv_heads):
            blocks = set(int(b) for b in sel[s * Q:(s + 1) * Q, g].ravel() if b >= 0)
            per_g.append(sorted(blocks))
        unions.append(per_g)
    idx_bytes, kv_bytes, actual_bytes = algorithmic_bytes(w, unions)
    step_bytes = idx_bytes + kv_bytes
    res = {
        "workload": WORKLOAD_TEXT[w.name], "ms_per_step": ms_step, "queries_per_s": st["rows"] / (ms_step * 1e-3),
        "bytes_per_step": {"algorithmic": step_bytes, "index": idx_bytes, "kv_selected": kv_bytes,
                           "with_fp32_scales": actual_bytes},
        "path_hbm_gbs": step_bytes / (ms_step * 1e-3) / 1e9,
        "path_frac_of_peak": step_bytes / (ms_step * 1e-3) / 1e9 / peak_gbs,
        "stages_alone_us": {"indexer": 1e3 * idx_ms, "topk": 1e3 * topk_ms, "attend": 1e3 * att_ms},
        "launches_per_step": kernels_per_step(w),
    }
    if Q > 8:
        # a prefill chunk: the contraction is dense, so the roofline is the tensor pipe (e4m3)
        fi, fa = indexer_flops(w), attend_flops(w, sel)
        res["flops_per_step"] = {"indexer": fi, "attend": fa}
        res["stage_roofline"] = {
            "indexer": {"bound": "tensor", "achieved": fi / (idx_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                        "frac": fi / (idx_ms * 1e-3) / 1e12 / peak_tf_e4m3},
            "attend": {"bound": "tensor", "achieved": fa / (att_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "frac": fa / (att_ms * 1e-3) / 1e12 / peak_tf_e4m3},
        }
        res["path_tflops"] = (fi + fa) / (ms_step * 1e-3) / 1e12
        # the same step with the selection made in the indexer's epilogue (no pooled scores)
        cfg2 = dataclasses.replace(st["cfg"], prefill_select="indexer")
        n2 = msa.msa_workspace_size(st["cache"], st["batch"], cfg2, w.num_q_heads)
        ws2 = torch.empty(n2, dtype=torch.uint8, device=B.dev)
        msa.msa_workspace_init(ws2)
        topk3 = torch.empty_like(st["topk"])
        ms_sel = B.time(lambda: msa.msa_decode(st["cache"], st["batch"], cfg2, st["iq"], st["q"], w.num_q_heads,
                                               topk3, out2, None, ws2, stream), n_alone, warmup=3)
        s_, flags = msa.msa_read_device_status(ws2)
        if s_ != 0:
            raise RuntimeError(f"{w.name} (indexer selection): device status {msa.msa_status_string(s_)} flags {flags}")
        res["prefill_select_indexer"] = {
            "ms_per_step": ms_sel, "workspace_mib": n2 / 2**20, "workspace_mib_topk": st["ws"].numel() / 2**20,
            "same_selection": bool(torch.equal(topk3, st["topk"]))}
        del ws2
    else:
        res["stage_roofline"] = {
            "indexer": {"bound": "hbm", "achieved": idx_bytes / (idx_ms * 1e-3) / 1e9, "unit": "GB/s",
                        "frac": idx_bytes / (idx_ms * 1e-3) / 1e9 / peak_gbs},
            "attend": {"bound": "hbm", "achieved": kv_bytes / (att_ms * 1e-3) / 1e9, "unit": "GB/s",
                       "frac": kv_bytes / (att_ms * 1e-3) / 1e9 / peak_gbs},
        }
    return res


def measure_insert(msa, ms, B, peak_gbs, kv="fp8", tokens=65536):
    """The cache insert of a prefill chunk's new tokens (bf16 K, V, index keys in;
    the caches' formats out) timed alone: HBM-bound, algorithmic bytes = the bf16
    rows read + the quantized rows and scales written."""
    import torch
    from block_sparse_attention_03_gb300 import roofline as R
    H = 4
    nblk = tokens // 128 + 8
    w = ms.make_workload("tiny_bf16", seq_lens=(128,), kv_dtype=kv, index_dtype=kv, seed=5)
    dev = B.dev
    z8 = lambda *sh: torch.zeros(sh, dtype=torch.uint8, device=dev)
    z32 = lambda *sh: torch.zeros(sh, dtype=torch.float32, device=dev)
    if kv == "fp8":
        cache = msa.PagedCache(kv_dtype=kv, index_dtype=kv, num_blocks=nblk, num_kv_heads=H, k=z8(nblk, H, 128, 128),
                               v=z8(nblk, H, 128, 128), idx=z8(nblk, 128, 128), k_scale=z32(nblk, H, 128),
                               v_scale=z32(nblk, H, 128), idx_scale=z32(nblk, 128))
    else:
        cache = msa.PagedCache(kv_dtype=kv, index_dtype=kv, num_blocks=nblk, num_kv_heads=H, k=z8(nblk, H, 128, 64),
                               v=z8(nblk, H, 128, 64), idx=z8(nblk, 128, 64), k_sf=z8(nblk, H, 128, 8),
                               v_sf=z8(nblk, H, 128, 8), idx_sf=z8(nblk, 128, 8), k_global=2.0 ** -10,
                               v_global=2.0 ** -10, idx_global=2.0 ** -10)
    gen = torch.Generator(device=dev)
    gen.manual_seed(6)
    k = (torch.randn((tokens, H, 128), generator=gen, device=dev) * 0.1).bfloat16()
    v = (torch.randn((tokens, H, 128), generator=gen, device=dev) * 0.1).bfloat16()
    ik = (torch.randn((tokens, 128), generator=gen, device=dev) * 0.1).bfloat16()
    # a prefill chunk's mapping: consecutive tokens fill consecutive rows of
    # blocks taken from the pool in shuffled order
    blocks = torch.randperm(nblk, generator=gen, device=dev)[:tokens // 128]
    slots = (blocks[:, None] * 128 + torch.arange(128, device=dev)[None, :]).reshape(-1).int()
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    ms_ = B.time(lambda: msa.msa_cache_insert(cache, slots, k, v, ik, ws, B.stream), 20, warmup=3)
    st, flags = msa.msa_read_device_status(ws)
    if st != 0:
        raise RuntimeError(f"insert: device status {flags}")
    read = tokens * (2 * H * 128 * 2 + 128 * 2) + tokens * 4
    written = tokens * (R.kv_bytes_per_token(kv, H) + R.index_bytes_per_token(kv))
    written += tokens * (2 * H + 1) * 4 if kv == "fp8" else 0
    gbs = (read + written) / (ms_ * 1e-3) / 1e9
    del w
    return {"kernel": "insert_kernel", "tokens": tokens, "cache": kv, "us": ms_ * 1e3,
            "bytes": read + written, "achieved_gbs": gbs, "frac": gbs / peak_gbs,
            "note": "bf16 rows read + quantized rows and their scales written; consecutive tokens to consecutive "
                    "rows of shuffled blocks"}


def dominant_roofline(res, peak_gbs, peak_tf, peak_kind):
    """The roofline of the stage that takes the most time alone (the top-k is
    bound by neither HBM nor the tensor pipe and never dominates)."""
    st_us = res["stages_alone_us"]
    name = "indexer" if st_us["indexer"] >= st_us["attend"] else "attend"
    r = res["stage_roofline"][name]
    kernels = {"indexer": "indexer_kernel (score + block max-pool)",
               "attend": "attend_kernel (split-K sparse attend + split merge), with its union prologue"}
    if "flops_per_step" in res:
        kernels = {"indexer": "pindexer_kernel (tcgen05 score + block max-pool)",
                   "attend": "selection lists + k2q_attend_kernel + k2q_combine_kernel"}
    return {"bound": r["bound"], "kernel": kernels[name], "achieved": r["achieved"],
            "peak": peak_tf if r["bound"] == "tensor" else peak_gbs, "unit": r["unit"], "frac": r["frac"],
            "traffic": None,
            "launch_us": st_us[name],
            "peak_kind": peak_kind if r["bound"] == "hbm" else peak_kind + " (bf16 burst x 2 for e4m3, the nominal ratio)",
            "other_stage": {k: v for k, v in res["stage_roofline"].items() if k != name}}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pool = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool = OraclePool()  # before the first GPU call

    import torch
    import torch.distributed as dist

    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_03_gb300 as msa
    import msa_synth as ms

    peak, bf16_tflops, peak_kind = load_peaks()
    peak_tf = 2.0 * bf16_tflops
    stream = torch.cuda.current_stream(dev)
    B = Bench(dev, stream)

    base = ms.make_workload(args.workload)
    st = setup_workload(msa, ms, args.workload, replica_seed(base.seed, rank), dev)
    w = st["w"]

    def step():
        msa.msa_decode(st["cache"], st["batch"], st["cfg"], st["iq"], st["q"], w.num_q_heads, st["topk"],
                       st["out"], st["lse"], st["ws"], stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    s_, flags = msa.msa_read_device_status(st["ws"])
    if s_ != 0:
        raise RuntimeError(f"device status {msa.msa_status_string(s_)} flags {flags}")

    # ---------------- timed region: K steps, L2 flushed before each, events around each step
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        B.flush()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_step = sum(a.elapsed_time(b) for a, b in evs) / args.steps

    # ---------------- end to end through the public API with host buffers.  A
    # step's inputs (index queries, queries, sequence lengths, block table) travel
    # in one pinned host buffer and one copy, its results (output, selection) in
    # one device buffer and one copy back, as a serving loop packs them; the
    # library reads and writes views of those device buffers.
    case = st["case"]

    def packed(tensors):
        offs, o = [], 0
        for t in tensors:
            offs.append(o)
            o += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, o

    def view(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    ins = [case["index_q"], case["q"], case["seq_lens"], case["block_table"]]
    in_offs, in_bytes = packed(ins)
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    for t, o in zip(ins, in_offs):
        view(h_in, o, t).copy_(t.cpu())
    e_iq, e_q, e_lens, e_bt = (view(d_in, o, t) for t, o in zip(ins, in_offs))
    e_batch = msa.Batch(e_lens, e_bt, w.q_per_seq)
    e_iqq = msa.Query(e_iq, w.q_dtype, case["index_q_scale"])
    e_qq = msa.Query(e_q, w.q_dtype, case["q_scale"])
    res_t = [st["out"], st["topk"]]
    res_offs, res_bytes = packed(res_t)
    d_res = torch.empty(res_bytes, dtype=torch.uint8, device=dev)
    h_res = torch.empty(res_bytes, dtype=torch.uint8).pin_memory()
    e_out, e_topk = (view(d_res, o, t) for t, o in zip(res_t, res_offs))

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        msa.msa_decode(st["cache"], e_batch, st["cfg"], e_iqq, e_qq, w.num_q_heads, e_topk, e_out, None, st["ws"],
                       stream)
        h_res.copy_(d_res, non_blocking=True)

    e2e_ms = B.time(e2e_step, args.steps, warmup=2)
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in res_t)
    if not torch.equal(view(h_res, res_offs[1], st["topk"]), st["topk"].cpu()):
        raise RuntimeError("the end-to-end selection differs from the device-timed one")
    s_, flags = msa.msa_read_device_status(st["ws"])
    if s_ != 0:
        raise RuntimeError(f"device status {msa.msa_status_string(s_)} flags {flags}")

    # ---------------- the headline workload's stages and byte model, then every other workload
    head = measure_workload(msa, B, st, min(args.steps, 20), 3, peak, peak_tf)
    ms_step, e2e_ms = max_over_ranks([ms_step, e2e_ms], world, dist, dev)
    head["ms_per_step"] = ms_step
    head["queries_per_s"] = st["rows"] * world / (ms_step * 1e-3)
    step_bytes = head["bytes_per_step"]["algorithmic"]
    head["path_hbm_gbs"] = step_bytes / (ms_step * 1e-3) / 1e9
    head["path_frac_of_peak"] = head["path_hbm_gbs"] / peak
    del st, case, d_in, d_res
    torch.cuda.empty_cache()

    workloads = {args.workload: head}
    names = ALL_WORKLOADS if args.workloads == "all" else ([] if args.workloads == "none"
                                                            else args.workloads.split(","))
    if rank == 0 and world == 1:
        for name in names:
            if name in workloads:
                continue
            wb = ms.make_workload(name)
            sw = setup_workload(msa, ms, name, wb.seed, dev)
            workloads[name] = measure_workload(msa, B, sw, 10, 3, peak, peak_tf)
            del sw
            torch.cuda.empty_cache()

    insert = None
    if rank == 0 and world == 1:
        insert = {kv: measure_insert(msa, ms, B, peak, kv) for kv in ("fp8", "nvfp4")}
        torch.cuda.empty_cache()

    cpu_base = None
    if pool is not None:
        plan, what = cpu_sample_plan(w)
        qps_cpu, nq, ntask = pool.sample(w.name, plan, w.seed + 5)
        pool.close()
        cpu_base = {"value": qps_cpu, "unit": "queries/s", "cores": min(pool.cores, ntask), "kind": "oracle",
                    "sample": f"{nq} query tokens: {what}; whole path (score, pool, top-k, attend) in fp64, "
                              f"one single-threaded oracle per host core, throughput over the slowest core"}

    if rank == 0:
        rows_all = head["queries_per_s"] * ms_step * 1e-3  # query tokens of all ranks in one step
        e2e_qps = rows_all / (e2e_ms * 1e-3)
        line = {
            "metric": METRIC, "value": head["queries_per_s"], "unit": "queries/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 MMA, fp32 accumulate" if w.kv_dtype == "fp8" else w.kv_dtype,
            "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload],
                       "l2": "flushed before every timed step (256 MB write, then 512 MB read)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
            "path_hbm_gbs": head["path_hbm_gbs"], "path_frac_of_peak": head["path_frac_of_peak"],
            "bytes_per_step": head["bytes_per_step"],
            "stages_alone_us": head["stages_alone_us"],
            "roofline": dominant_roofline(head, peak, peak_tf, peak_kind),
            "cpu_baseline": cpu_base,
            "e2e": {"value": e2e_qps, "unit": "queries/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": head["launches_per_step"] * args.steps,
            "clocks": clocks,
            "workloads": workloads,
            "cache_insert": insert,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
