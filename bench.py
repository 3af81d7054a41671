"""Benchmark of the MSA decode hot path (score -> pool -> top-k -> attend).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one msa_decode call over one batch of synthetic input (the whole
path, every stage).  Prints ONE JSON line on rank 0.  Under torchrun with
N > 1 every rank runs its own replica of the workload (decode batches are
independent problems: weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
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

def kernels_per_step(w) -> int:
    """Launches of one msa_decode: indexer, top-k, attend; a prefill chunk (more
    than 8 new tokens) over an FP8 cache with 1, 2, 4 or 8 q heads a group runs
    the key-block-major attend instead: count, scan, fill, attend, combine."""
    r = w.num_q_heads // w.num_kv_heads
    if w.q_per_seq > 8 and w.kv_dtype == "fp8" and r in (1, 2, 4, 8):
        return 7
    return 3


def ncu_traffic(workload: str, kernel: str = "indexer"):
    """DRAM bytes (read + write) of one launch of the kernel from the committed
    ncu summary of this workload (profiles/<kernel>_<workload>.md), or None
    when there is none."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    total = 0.0
    for name in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
        for line in text.splitlines():
            cells = [c.strip() for c in line.split("|")]
            if len(cells) > 2 and cells[1] == name:
                val, _, unit = cells[2].partition(" ")
                total += float(val) * scale.get(unit.strip(), 1.0)
                break
        else:
            return None
    return total


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="fp8_decode", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def load_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, kind) from the driver's measurement, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def indexer_flops(w):
    """Algorithmic FLOPs of the index scores: every visible key x groups x index dim x 2."""
    tot = 0
    for T in w.seq_lens:
        first = T - w.q_per_seq + 1  # keys visible to the first new token
        tot += w.q_per_seq * first + w.q_per_seq * (w.q_per_seq - 1) // 2
    return 2.0 * tot * w.num_kv_heads * w.index_dim


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


def sample_rows(w):
    """Query rows of a sequence the CPU sample covers: all of them, or the last 8
    (one verify-sized chunk) of a prefill chunk, which would take minutes."""
    return None if w.q_per_seq <= 8 else list(range(w.q_per_seq - 8, w.q_per_seq))


def cpu_oracle_sample(w, case_host, seqs):
    """Time the oracle (as it stands) on the whole path (score, pool, select,
    attend) for the given sequences and their sample rows; returns (seconds, rows)."""
    import numpy as np
    from oracle import msa_oracle as O
    rows = sample_rows(w)
    t0 = time.perf_counter()
    if rows is None:
        O.run_path(case_host, seqs=seqs)
        n = len(seqs) * w.q_per_seq
    else:
        Q = w.q_per_seq
        for s in seqs:
            pooled = O.pooled_scores(case_host, s, w.index_dim ** -0.5, rows=rows)
            pos = O.positions(int(case_host["seq_lens"][s]), Q)
            sel = np.full((w.num_seqs * Q, w.num_kv_heads, w.topk), -1, dtype=np.int32)
            for k, i in enumerate(rows):
                for g in range(w.num_kv_heads):
                    sel[s * Q + i, g] = O.select_blocks(pooled[k, g], int(pos[i]), w.topk)
            O.attend_rows(case_host, s, sel, w.head_dim ** -0.5, rows=rows)
        n = len(seqs) * len(rows)
    return time.perf_counter() - t0, n


def run_reference(args):
    """Reference arm: the CPU oracle on host cores, bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import msa_synth as ms
    w = ms.make_workload(args.workload)
    case = ms.make_case(w, device="cpu") if args.workload != "fp8_long" else None
    if case is None:  # 512K-token contexts: generate one sequence's worth on the host
        w = ms.make_workload(args.workload, seq_lens=(w.seq_lens[0],))
        case = ms.make_case(w, device="cpu")
    h = ms.case_to_host(case)
    times, nq = [], 0
    for it in range(args.warmup + args.steps):
        s = it % w.num_seqs
        dt, n = cpu_oracle_sample(w, h, [s])
        if it >= args.warmup:
            times.append(dt)
            nq = n
    mean = sum(times) / len(times)
    qps = nq / mean
    line = {"metric": METRIC, "value": qps, "unit": "queries/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload],
                       "sample": f"one sequence of the workload per step ({nq} of its {w.q_per_seq} query tokens)"},
            "cpu_baseline": {"value": qps, "unit": "queries/s", "cores": 1, "kind": "oracle",
                             "sample": "one sequence per step, whole path (score, pool, top-k, attend) in fp64"},
            "e2e": {"value": qps, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_attention_03_gb300 as msa
    import msa_synth as ms

    base = ms.make_workload(args.workload)
    w = ms.make_workload(args.workload, seed=replica_seed(base.seed, rank))
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
    # L2 flush between timed steps: write 256 MB (> 129 MB L2), then read 512 MB so
    # that the written lines are already back in HBM and L2 holds only clean data
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(128 << 20, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_out)

    def step():
        msa.msa_decode(cache, batch, cfg, iq, q, w.num_q_heads, topk, out, lse, ws, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st, flags = msa.msa_read_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {msa.msa_status_string(st)} flags {flags}")

    # ---------------- timed region: K steps, L2 flushed before each, events around each step
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms_step = sum(step_ms) / len(step_ms)

    # dominant kernel (the indexer scan) timed alone on the same stream, same launch shape
    pooled = torch.empty((rows, w.num_kv_heads, w.max_blocks), dtype=torch.float32, device=dev)
    ievs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for _ in range(3):
        msa.msa_indexer_score(cache, batch, cfg, iq, pooled, ws, stream)
    for i in range(args.steps):
        flush()
        ievs[i][0].record(stream)
        msa.msa_indexer_score(cache, batch, cfg, iq, pooled, ws, stream)
        ievs[i][1].record(stream)
    torch.cuda.synchronize()
    idx_ms = sum(a.elapsed_time(b) for a, b in ievs) / args.steps

    # the other stages alone (through their own entry points), for the breakdown
    def time_stage(fn, n=10):
        evs_ = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        fn()
        for i in range(n):
            flush()
            evs_[i][0].record(stream)
            fn()
            evs_[i][1].record(stream)
        torch.cuda.synchronize()
        return 1e3 * sum(a.elapsed_time(b) for a, b in evs_) / n

    topk2 = torch.empty_like(topk)
    out2 = torch.empty_like(out)
    stages_us = {
        "indexer": 1e3 * idx_ms,
        "topk": time_stage(lambda: msa.msa_topk_blocks(batch, cfg, w.num_kv_heads, pooled, topk2, None, ws, stream)),
        "union+attend": time_stage(lambda: msa.msa_sparse_attend(cache, batch, cfg, q, w.num_q_heads, topk2, out2,
                                                                 None, ws, stream)),
    }
    clocks = sampler.stop()

    # ---------------- end to end through the public API with host buffers.  A
    # step's inputs (index queries, queries, sequence lengths, block table) travel
    # in one pinned host buffer and one copy, its results (output, selection) in
    # one device buffer and one copy back, as a serving loop packs them; the
    # library reads and writes views of those device buffers.
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
    res = [out, topk]
    res_offs, res_bytes = packed(res)
    d_res = torch.empty(res_bytes, dtype=torch.uint8, device=dev)
    h_res = torch.empty(res_bytes, dtype=torch.uint8).pin_memory()
    e_out, e_topk = (view(d_res, o, t) for t, o in zip(res, res_offs))
    e2e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush()
        e2e_evs[i][0].record(stream)
        d_in.copy_(h_in, non_blocking=True)
        msa.msa_decode(cache, e_batch, cfg, e_iqq, e_qq, w.num_q_heads, e_topk, e_out, None, ws, stream)
        h_res.copy_(d_res, non_blocking=True)
        e2e_evs[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_evs) / args.steps
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in res)
    if not torch.equal(view(h_res, res_offs[1], topk), topk.cpu()):
        raise RuntimeError("the end-to-end selection differs from the device-timed one")
    st, flags = msa.msa_read_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {msa.msa_status_string(st)} flags {flags}")

    # ---------------- byte model from this step's selection
    sel = topk.cpu().numpy()
    unions = []
    for s in range(w.num_seqs):
        per_g = []
        for g in range(w.num_kv_heads):
            blocks = set(int(b) for b in sel[s * w.q_per_seq:(s + 1) * w.q_per_seq, g].ravel() if b >= 0)
            per_g.append(sorted(blocks))
        unions.append(per_g)
    idx_bytes, kv_bytes, actual_bytes = algorithmic_bytes(w, unions)
    step_bytes = idx_bytes + kv_bytes
    peak, bf16_tflops, peak_kind = load_peaks()

    # max over ranks
    ms_step, idx_ms, e2e_ms = max_over_ranks([ms_step, idx_ms, e2e_ms], world, dist, dev)
    queries = rows * world
    qps = queries / (ms_step * 1e-3)
    e2e_qps = queries / (e2e_ms * 1e-3)

    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        h = ms.case_to_host(case) if args.workload != "fp8_long" else None
        if h is not None:
            nseq = min(2, w.num_seqs)
            dt, nq = cpu_oracle_sample(w, h, list(range(nseq)))
            cpu_base = {"value": nq / dt, "unit": "queries/s", "cores": 1, "kind": "oracle",
                        "sample": f"{nq} query tokens of the first {nseq} of the {w.num_seqs} sequences, "
                                  "whole path in fp64 (numpy)"}
        else:
            ws1 = ms.make_workload(args.workload, seq_lens=(w.seq_lens[0],))
            h1 = ms.case_to_host(ms.make_case(ws1, device="cpu"))
            dt, nq = cpu_oracle_sample(ws1, h1, [0])
            cpu_base = {"value": nq / dt, "unit": "queries/s", "cores": 1, "kind": "oracle",
                        "sample": "one 512K-token sequence regenerated on the host, whole path in fp64"}

    if rank == 0:
        idx_gbs = idx_bytes / (idx_ms * 1e-3) / 1e9
        path_gbs = step_bytes / (ms_step * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": qps, "unit": "queries/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3 MMA, fp32 accumulate" if w.kv_dtype == "fp8" else w.kv_dtype,
            "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload], "l2": "flushed before every timed step (256 MB write, then 512 MB read)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
            "path_hbm_gbs": path_gbs, "path_frac_of_peak": path_gbs / peak,
            "stages_us_alone": stages_us,
            "bytes_per_step": {"algorithmic": step_bytes, "index": idx_bytes, "kv_selected": kv_bytes,
                               "with_fp32_scales": actual_bytes},
            "roofline": ({"bound": "hbm", "kernel": "indexer_kernel (score + block max-pool)", "achieved": idx_gbs,
                          "peak": peak, "unit": "GB/s", "frac": idx_gbs / peak,
                          "traffic": ncu_traffic(args.workload),
                          "peak_kind": peak_kind} if w.q_per_seq <= 8 else
                         {"bound": "tensor", "kernel": "pindexer_kernel (tcgen05 score + block max-pool)",
                          "achieved": indexer_flops(w) / (idx_ms * 1e-3) / 1e12,
                          "peak": 2.0 * bf16_tflops, "unit": "TFLOP/s",
                          "frac": indexer_flops(w) / (idx_ms * 1e-3) / 1e12 / (2.0 * bf16_tflops),
                          "traffic": ncu_traffic(args.workload, "pindexer"),
                          "peak_kind": peak_kind + " (bf16 burst x 2 for e4m3, the nominal ratio)"}),
            "cpu_baseline": cpu_base,
            "e2e": {"value": e2e_qps, "unit": "queries/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": kernels_per_step(w) * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
