"""Shared test helpers: bind a generated case to the library's argument
objects, run the CUDA path, and apply the parity tolerances.

Tolerances (the pages give none; these are the stated targets):
* dequantized cache values: bit-exact in fp32;
* pooled indexer scores: |gpu - ref| <= 1e-3 * max(|ref|, 1e-2 * max_b |ref|)
  per (query, group) row, and identical -inf positions;
* selections: identical, except that blocks whose oracle scores lie within
  that tolerance of the k-th free score may trade places;
* attention output: max-abs <= 2e-2 and mean-abs <= 2e-3 against the oracle
  run on the GPU's own selection.
"""

from __future__ import annotations

import numpy as np
import torch

import block_sparse_attention_03_gb300 as msa
import msa_synth as ms
from oracle import msa_oracle as O

POOL_RTOL = 1e-3
POOL_FLOOR = 1e-2
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3


def bind(case: dict):
    """(PagedCache, Batch, index Query, Query) for a case generated on the GPU."""
    w = case["workload"]
    cache = msa.PagedCache(
        kv_dtype=w.kv_dtype, index_dtype=w.index_dtype, num_blocks=case["num_blocks"],
        num_kv_heads=w.num_kv_heads, k=case["k"], v=case["v"], idx=case["idx"],
        k_sf=case.get("k_sf"), v_sf=case.get("v_sf"), k_scale=case.get("k_scale"),
        v_scale=case.get("v_scale"), idx_sf=case.get("idx_sf"), idx_scale=case.get("idx_scale"),
        k_global=case.get("k_global", 0.0), v_global=case.get("v_global", 0.0),
        idx_global=case.get("idx_global", 0.0), nvfp4_mode=case.get("nvfp4_mode", "exact"))
    batch = msa.Batch(case["seq_lens"], case["block_table"], w.q_per_seq)
    iq = msa.Query(case["index_q"], w.q_dtype, case["index_q_scale"])
    q = msa.Query(case["q"], w.q_dtype, case["q_scale"])
    return cache, batch, iq, q


def workspace(cache, batch, cfg, hq):
    n = msa.msa_workspace_size(cache, batch, cfg, hq)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    msa.msa_workspace_init(ws)
    return ws


def gpu_path(case: dict, cfg=None, fused: bool = True):
    """Run the whole path on the GPU; returns host arrays pooled (or None), topk, out, lse."""
    w = case["workload"]
    cfg = cfg or msa.default_config(w.topk)
    cache, batch, iq, q = bind(case)
    ws = workspace(cache, batch, cfg, w.num_q_heads)
    rows = w.num_seqs * w.q_per_seq
    topk = torch.full((rows, w.num_kv_heads, cfg.topk), -7, dtype=torch.int32, device="cuda")
    out = torch.zeros((rows, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((rows, w.num_q_heads), dtype=torch.float32, device="cuda")
    pooled = None
    if fused:
        msa.msa_decode(cache, batch, cfg, iq, q, w.num_q_heads, topk, out, lse, ws)
    else:
        pooled = torch.full((rows, w.num_kv_heads, w.max_blocks), 7.0, dtype=torch.float32, device="cuda")
        msa.msa_indexer_score(cache, batch, cfg, iq, pooled, ws)
        msa.msa_topk_blocks(batch, cfg, w.num_kv_heads, pooled, topk, None, ws)
        msa.msa_sparse_attend(cache, batch, cfg, q, w.num_q_heads, topk, out, lse, ws)
    st, flags = msa.msa_read_device_status(ws)
    assert st == 0, (msa.msa_status_string(st), flags)
    return dict(pooled=None if pooled is None else pooled.cpu().numpy(), topk=topk.cpu().numpy(),
                out=out.float().cpu().numpy(), lse=lse.cpu().numpy())


def check_pooled(gpu: np.ndarray, ref: np.ndarray, rows=None):
    rows = range(gpu.shape[0]) if rows is None else rows
    worst = 0.0
    for r in rows:
        for g in range(gpu.shape[1]):
            a, b = gpu[r, g], ref[r, g]
            inf_ref = np.isneginf(b)
            assert np.array_equal(np.isneginf(a), inf_ref), (r, g)
            fin = ~inf_ref
            if not fin.any():
                continue
            scale = np.maximum(np.abs(b[fin]), POOL_FLOOR * np.abs(b[fin]).max())
            err = np.abs(a[fin] - b[fin]) / scale
            worst = max(worst, float(err.max()))
    assert worst <= POOL_RTOL, worst
    return worst


def check_selection(sel: np.ndarray, ref_pooled: np.ndarray, seq_lens, q_per_seq: int, topk: int,
                    init_blocks: int = 0, local_blocks: int = 0, rows=None):
    """GPU selection must be a valid top-k of the oracle's pooled scores,
    allowing swaps only among near-ties (within the pooled tolerance)."""
    rows = range(sel.shape[0]) if rows is None else rows
    n_exact = 0
    for r in rows:
        s, i = divmod(r, q_per_seq)
        pos = int(seq_lens[s]) - q_per_seq + i
        for g in range(sel.shape[1]):
            want = O.select_blocks(ref_pooled[r, g], pos, topk, init_blocks, local_blocks)
            got = sel[r, g]
            if np.array_equal(got, want):
                n_exact += 1
                continue
            ids = got[got >= 0]
            assert np.all(np.diff(ids) > 0), (r, g, got)
            forced = set(O.forced_blocks(pos, init_blocks, local_blocks))
            assert forced.issubset(set(ids)), (r, g, got)
            assert len(ids) == (want >= 0).sum(), (r, g, got, want)
            p = ref_pooled[r, g]
            free_ref = [b for b in want if b >= 0 and b not in forced]
            kth = min(p[b] for b in free_ref)
            tol = POOL_RTOL * max(abs(kth), POOL_FLOOR * np.abs(p[np.isfinite(p)]).max())
            for b in set(ids) - set(want):
                assert p[b] >= kth - tol, (r, g, b, p[b], kth)
            for b in set(want) - set(ids):
                assert p[b] <= kth + tol, (r, g, b, p[b], kth)
    return n_exact


def check_out(gpu_out: np.ndarray, ref_out: np.ndarray):
    err = np.abs(gpu_out - ref_out)
    assert err.max() <= OUT_MAX_ABS, err.max()
    assert err.mean() <= OUT_MEAN_ABS, err.mean()
    return float(err.max()), float(err.mean())


def small(name: str, **over):
    return ms.make_workload(name, **over)
