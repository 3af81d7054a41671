"""msa_decode for one new token over FP8 index and K/V caches against the
oracle, through the C ABI, on the shapes and inputs the schedule of the path
depends on: the number and lengths of the sequences (indexer units per warp,
lengths of 1 token and exact block multiples, many short sequences), the
groups (1, 2, 4, 8 index columns) and q heads per group (1, 2, 4), k, forced
blocks, E4M3 queries, bad input (a block-table entry outside the pool, a
malformed sequence length), and back-to-back calls of different sizes on one
workspace.
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_03_gb300 as msa
import msa_synth as ms
from oracle import msa_oracle as O

from _helpers import bind, check_out, check_selection, gpu_path, workspace

pytestmark = pytest.mark.gpu


def _check_against_oracle(w, c, g, cfg=None):
    h = ms.case_to_host(c)
    init = cfg.init_blocks if cfg else 0
    local = cfg.local_blocks if cfg else 0
    ref = O.run_path(h, topk=w.topk, init_blocks=init, local_blocks=local)
    check_selection(g["topk"], ref["pooled"], w.seq_lens, 1, w.topk, init, local)
    out = np.zeros_like(ref["out"])
    lse = np.zeros_like(ref["lse"])
    for s in range(w.num_seqs):
        o, l = O.attend_rows(h, s, g["topk"], w.head_dim ** -0.5)
        out[s], lse[s] = o[0], l[0]
    check_out(g["out"], out)
    assert np.abs(g["lse"] - lse).max() < 1e-3


CASES = [
    dict(seq_lens=(1000, 2500, 3333, 777)),
    dict(seq_lens=(1, 127, 128, 129, 4096, 4097)),                   # one token, exact block multiples
    dict(seq_lens=(20000, 300, 9000), num_kv_heads=1, num_q_heads=4),   # one group, 4 heads
    dict(seq_lens=(7000, 5000), num_kv_heads=2, num_q_heads=8),          # two groups
    dict(seq_lens=(6000, 3000), num_kv_heads=8, num_q_heads=32),         # eight index columns
    dict(seq_lens=(5000, 2100), num_q_heads=4),                          # one q head a group
    dict(seq_lens=(5000, 2100), num_q_heads=8),                          # two q heads a group
    dict(seq_lens=(9000, 4000), topk=4),
    dict(seq_lens=(9000, 4000), topk=32),
    dict(seq_lens=(4500, 2000), q_dtype="fp8"),                          # E4M3 queries: one MMA term
]


@pytest.mark.parametrize("over", CASES)
def test_decode_matches_oracle(over):
    w = ms.make_workload("fp8_decode", seed=101, **over)
    c = ms.make_case(w, device="cuda")
    g = gpu_path(c)
    _check_against_oracle(w, c, g)


def test_decode_forced_blocks():
    w = ms.make_workload("fp8_decode", seed=102, seq_lens=(6000, 2000, 900))
    c = ms.make_case(w, device="cuda")
    cfg = msa.Config(topk=16, init_blocks=2, local_blocks=3)
    g = gpu_path(c, cfg=cfg)
    _check_against_oracle(w, c, g, cfg)


def test_decode_many_sequences():
    # 300 sequences of 1-3,000 tokens: the indexer warps' runs cross many
    # sequences, and the attend walks many splits per CTA
    rng = np.random.default_rng(103)
    lens = rng.integers(1, 3000, size=300)
    w = ms.make_workload("fp8_decode", seq_lens=lens, seed=103)
    c = ms.make_case(w, device="cuda")
    g = gpu_path(c)
    h = ms.case_to_host(c)
    for s in [0, 1, 150, 298, 299] + [int(x) for x in rng.choice(300, 5, replace=False)]:
        pooled = O.pooled_scores(h, s, w.index_dim ** -0.5)
        full = np.full((w.num_seqs, w.num_kv_heads, w.max_blocks), -np.inf)
        full[s] = pooled[0]
        check_selection(g["topk"], full, w.seq_lens, 1, w.topk, rows=[s])
        o, _ = O.attend_rows(h, s, g["topk"], w.head_dim ** -0.5)
        check_out(g["out"][[s]], o)


def test_decode_back_to_back_calls_of_different_sizes():
    # one workspace, calls of different batch sizes in a row: nothing a call
    # leaves in the workspace changes the next one
    ws = None
    for seed, lens in [(104, (3000, 2000, 1000)), (105, (9000,) * 12), (106, (500, 70000)), (107, (3000, 2000, 1000))]:
        w = ms.make_workload("fp8_decode", seq_lens=lens, seed=seed)
        c = ms.make_case(w, device="cuda")
        cache, batch, iq, q = bind(c)
        cfg = msa.default_config()
        need = msa.msa_workspace_size(cache, batch, cfg, 16)
        if ws is None or ws.numel() < need:
            ws = torch.empty(max(need, 64 << 20), dtype=torch.uint8, device="cuda")
            msa.msa_workspace_init(ws)
        topk = torch.full((w.num_seqs, 4, 16), -7, dtype=torch.int32, device="cuda")
        out = torch.zeros((w.num_seqs, 16, 128), dtype=torch.bfloat16, device="cuda")
        for _ in range(2):
            msa.msa_decode(cache, batch, cfg, iq, q, 16, topk, out, None, ws)
        assert msa.msa_read_device_status(ws)[0] == 0
        ref = gpu_path(c, fused=False)
        assert np.array_equal(topk.cpu().numpy(), ref["topk"])
        assert np.array_equal(out.float().cpu().numpy(), ref["out"])


def test_decode_bad_block_table_entry_flags_and_ends():
    w = ms.make_workload("fp8_decode", seed=108, seq_lens=(3000, 2000))
    c = ms.make_case(w, device="cuda")
    c["block_table"][1, 5] = c["num_blocks"] + 3
    cache, batch, iq, q = bind(c)
    cfg = msa.default_config()
    ws = workspace(cache, batch, cfg, 16)
    topk = torch.empty((2, 4, 16), dtype=torch.int32, device="cuda")
    out = torch.full((2, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    msa.msa_decode(cache, batch, cfg, iq, q, 16, topk, out, None, ws)
    st, flags = msa.msa_read_device_status(ws)
    assert st == 5 and flags & 1 and not flags & 8
    assert torch.isfinite(out.float()).all()
    # the first sequence is untouched by the bad entry
    h = ms.case_to_host(c)
    pooled = O.pooled_scores(h, 0, w.index_dim ** -0.5)
    full = np.full((2, 4, w.max_blocks), -np.inf)
    full[0] = pooled[0]
    check_selection(topk.cpu().numpy(), full, w.seq_lens, 1, 16, rows=[0])


def test_decode_malformed_sequence_length():
    # a sequence length beyond its block-table row: flagged, its rows left as
    # documented (no selection, zero output, -inf LSE), the others exact
    w = ms.make_workload("fp8_decode", seed=109, seq_lens=(3000, 2000, 2500))
    c = ms.make_case(w, device="cuda")
    c["seq_lens"][1] = w.max_blocks * 128 + 1
    cache, batch, iq, q = bind(c)
    cfg = msa.default_config()
    ws = workspace(cache, batch, cfg, 16)
    topk = torch.empty((3, 4, 16), dtype=torch.int32, device="cuda")
    out = torch.full((3, 16, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((3, 16), dtype=torch.float32, device="cuda")
    msa.msa_decode(cache, batch, cfg, iq, q, 16, topk, out, lse, ws)
    st, flags = msa.msa_read_device_status(ws)
    assert st == 5 and flags & 2 and not flags & 8
    assert (topk[1] == -1).all()
    assert (out[1].float() == 0).all() and torch.isneginf(lse[1]).all()
    h = ms.case_to_host(c)
    for s in (0, 2):
        o, _ = O.attend_rows(h, s, topk.cpu().numpy(), w.head_dim ** -0.5)
        check_out(out[[s]].float().cpu().numpy(), o)
