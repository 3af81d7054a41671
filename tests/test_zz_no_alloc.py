"""The allocation-free decode entry point, for callers that cannot allocate
device memory (code inside another framework's memory pool, plugins that may
not call cudaMalloc on their hot path).  It runs the same kernels as
msa_decode on a fixed scratch array inside the library, so its results must
match msa_decode's; two calls in a row check that the shared scratch carries
nothing stale from one call into the next.  This file is collected last."""

import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import block_sparse_attention_03_gb300 as msa
import msa_synth as ms

from _helpers import OUT_MAX_ABS, OUT_MEAN_ABS, bind, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_sparse_attention_03_gb300 import _build
    _build.build()


def _with_workspace(case, **cfg_over):
    w = case["workload"]
    cache, batch, iq, q = bind(case)
    cfg = dataclasses.replace(msa.default_config(w.topk), **cfg_over)
    ws = workspace(cache, batch, cfg, w.num_q_heads)
    rows = w.num_seqs * w.q_per_seq
    topk = torch.empty((rows, w.num_kv_heads, w.topk), dtype=torch.int32, device="cuda")
    out = torch.empty((rows, w.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((rows, w.num_q_heads), dtype=torch.float32, device="cuda")
    msa.msa_decode(cache, batch, cfg, iq, q, w.num_q_heads, topk, out, lse, ws)
    assert msa.msa_read_device_status(ws)[0] == 0
    return topk.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()


def _without_workspace(case, **cfg_over):
    w = case["workload"]
    cache, batch, iq, q = bind(case)
    cfg = dataclasses.replace(msa.default_config(w.topk), **cfg_over)
    rows = w.num_seqs * w.q_per_seq
    topk = torch.full((rows, w.num_kv_heads, w.topk), -5, dtype=torch.int32, device="cuda")
    out = torch.full((rows, w.num_q_heads, 128), 9.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((rows, w.num_q_heads), dtype=torch.float32, device="cuda")
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    msa.msa_decode_noalloc(cache, batch, cfg, iq, q, w.num_q_heads, topk, out, lse, status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    return topk.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    # different problems back to back through the same scratch: one-token
    # decode, speculative verify over NVFP4, and a small prefill chunk over FP8
    # (the selection-list chain msa_decode runs for it)
    cases = [ms.make_case(ms.make_workload("fp8_decode", seq_lens=(9000, 3000, 700), seed=91), device="cuda"),
             ms.make_case(ms.make_workload("nvfp4_verify", seq_lens=(4000, 2100), seed=92), device="cuda"),
             ms.make_case(ms.make_workload("fp8_prefill", seq_lens=(1300,), q_per_seq=24, seed=94), device="cuda")]
    for case in cases:
        t_ref, o_ref, l_ref = _with_workspace(case)
        t, o, l = _without_workspace(case)
        assert np.array_equal(t, t_ref)
        err = np.abs(o - o_ref)
        assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS
        assert np.abs(l - l_ref).max() <= 1e-3


@pytest.mark.parametrize("seq_len,lists_fit", [(1300, True), (40000, False)])
def test_noalloc_prefill_with_selection_in_the_indexer(seq_len, lists_fit):
    # prefill_select="indexer": where the candidate lists fit the scratch the
    # chain uses them; where they do not (one query tile over 157 units, one list
    # slot per CTA) but the pooled scores do, it falls back to the top-k launch.
    # Either way the results equal msa_decode's with its default selection.
    w = ms.make_workload("fp8_prefill", seq_lens=(seq_len,), q_per_seq=24, seed=95)
    case = ms.make_case(w, device="cuda")
    cache, batch, _, _ = bind(case)
    sel = dataclasses.replace(msa.default_config(w.topk), prefill_select="indexer")
    assert (msa.msa_workspace_size(cache, batch, sel, w.num_q_heads) <= 8 << 20) == lists_fit
    assert msa.msa_workspace_size(cache, batch, msa.default_config(w.topk), w.num_q_heads) <= 8 << 20
    t_ref, o_ref, l_ref = _with_workspace(case)
    t, o, l = _without_workspace(case, prefill_select="indexer")
    assert np.array_equal(t, t_ref)
    err = np.abs(o - o_ref)
    assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS
    assert np.abs(l - l_ref).max() <= 1e-3


def test_noalloc_rejects_problems_beyond_the_scratch():
    # 256 sequences with 8 new tokens each: the workspace (pooled scores, the
    # selection union, split partials) is larger than the scratch
    w = ms.make_workload("fp8_decode", seq_lens=(2048,) * 256, q_per_seq=8, seed=93)
    case = ms.make_case(w, device="cuda")
    cache, batch, iq, q = bind(case)
    cfg = msa.default_config()
    assert msa.msa_workspace_size(cache, batch, cfg, 16) > 8 << 20
    topk = torch.empty((256 * 8, 4, 16), dtype=torch.int32, device="cuda")
    out = torch.empty((256 * 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(msa.MsaError) as e:
        msa.msa_decode_noalloc(cache, batch, cfg, iq, q, 16, topk, out, None)
    assert e.value.status == 3
