"""The indexer of prefill chunks (more than 8 new tokens per sequence, FP8
index cache), which runs on the tcgen05 tensor cores with the query tokens
as the MMA's M side, against the oracle's pooled scores (vLLM Day-0 blog,
sections "MSA 入门" and "NVIDIA Blackwell 优化的 MSA 内核", which names an MSA indexer prefill
kernel).  The cases cover one and several 128-row query tiles, ragged last
tiles, several sequences of different lengths, e4m3 index queries (one MMA
term instead of the bf16 hi + lo pair), 1 / 2 / 4 / 8 groups (128, 64, 32, 16
tokens a tile) and a bad block-table entry.
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_03_gb300 as msa
import msa_synth as ms
from oracle import msa_oracle as O

from _helpers import bind, check_pooled, workspace

pytestmark = pytest.mark.gpu


def _pooled(c, w):
    cfg = msa.default_config(w.topk)
    cache, batch, iq, _ = bind(c)
    ws = workspace(cache, batch, cfg, w.num_q_heads)
    pooled = torch.full((w.num_seqs * w.q_per_seq, w.num_kv_heads, w.max_blocks), 7.0, dtype=torch.float32,
                        device="cuda")
    msa.msa_indexer_score(cache, batch, cfg, iq, pooled, ws)
    st, flags = msa.msa_read_device_status(ws)
    return pooled.cpu().numpy(), st, flags


def _oracle(c, w):
    h = ms.case_to_host(c)
    return np.concatenate([O.pooled_scores(h, s, w.index_dim ** -0.5) for s in range(w.num_seqs)])


CASES = [
    dict(seq_lens=(2000 + 64,), q_per_seq=64),
    dict(seq_lens=(1500, 900), q_per_seq=24),
    dict(seq_lens=(5000, 130, 4000), q_per_seq=100),
    dict(seq_lens=(3000,), q_per_seq=40, q_dtype="fp8"),
    dict(seq_lens=(2500,), q_per_seq=48, num_kv_heads=8),
    dict(seq_lens=(2500,), q_per_seq=80, num_kv_heads=2),
    dict(seq_lens=(1200,), q_per_seq=128, num_kv_heads=1),
]


@pytest.mark.parametrize("over", CASES)
def test_prefill_indexer_matches_oracle(over):
    w = ms.make_workload("fp8_prefill", seed=81, **over)
    c = ms.make_case(w, device="cuda")
    got, st, flags = _pooled(c, w)
    assert st == 0, (msa.msa_status_string(st), flags)
    check_pooled(got, _oracle(c, w))


def test_prefill_indexer_bad_block_flags_and_skips():
    w = ms.make_workload("fp8_prefill", seed=82, seq_lens=(1000,), q_per_seq=32)
    c = ms.make_case(w, device="cuda")
    ref = _oracle(c, w)
    c["block_table"][0, 2] = c["num_blocks"] + 5
    got, st, flags = _pooled(c, w)
    assert st != 0 and flags & 1  # a block-table entry outside the pool
    assert np.isneginf(got[:, :, 2]).all()
    keep = [b for b in range(w.max_blocks) if b != 2]
    check_pooled(got[:, :, keep], ref[:, :, keep])


@pytest.mark.parametrize("over", [dict(seq_lens=(3000, 1700), q_per_seq=40, num_kv_heads=8),
                                  dict(seq_lens=(2600,), q_per_seq=72, num_kv_heads=2),
                                  dict(seq_lens=(2200,), q_per_seq=48, q_dtype="fp8")])
def test_prefill_whole_path_matches_oracle(over):
    # msa_decode end to end on a prefill chunk: tcgen05 indexer, top-k, per-token attend
    from _helpers import check_out, check_selection, gpu_path
    w = ms.make_workload("fp8_prefill", seed=83, **over)
    c = ms.make_case(w, device="cuda")
    g = gpu_path(c)
    h = ms.case_to_host(c)
    ref = _oracle(c, w)
    check_selection(g["topk"], ref, w.seq_lens, w.q_per_seq, w.topk)
    out = np.zeros_like(g["out"])
    for s in range(w.num_seqs):
        o, _ = O.attend_rows(h, s, g["topk"], w.head_dim ** -0.5)
        out[s * w.q_per_seq:(s + 1) * w.q_per_seq] = o
    check_out(g["out"], out)


def test_prefill_indexer_bad_seq_len_flags_and_fills():
    # a sequence shorter than its new tokens: flagged, its rows stay -inf, the other is scored
    w = ms.make_workload("fp8_prefill", seed=84, seq_lens=(900, 700), q_per_seq=32)
    c = ms.make_case(w, device="cuda")
    ref = _oracle(c, w)
    c["seq_lens"][1] = 20
    got, st, flags = _pooled(c, w)
    assert st != 0 and flags & 2
    assert np.isneginf(got[32:]).all()
    check_pooled(got[:32], ref[:32])


@pytest.mark.parametrize("mode", ["topk", "indexer"])
def test_prefill_selection_of_a_bad_sequence(mode):
    # a sequence shorter than its new tokens next to a good one: its rows are
    # all -1 and the status says so, whichever way the chunk is selected; the
    # good sequence's rows equal the staged top-k's
    w = ms.make_workload("fp8_prefill", seed=88, seq_lens=(3000, 2000), q_per_seq=40)
    c = ms.make_case(w, device="cuda")
    c["seq_lens"][1] = 30
    cfg = msa.Config(topk=16, prefill_select=mode)
    cache, batch, iq, q = bind(c)
    ws = workspace(cache, batch, cfg, w.num_q_heads)
    rows, G = w.num_seqs * w.q_per_seq, w.num_kv_heads
    topk = torch.full((rows, G, 16), -7, dtype=torch.int32, device="cuda")
    out = torch.empty((rows, w.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    msa.msa_decode(cache, batch, cfg, iq, q, w.num_q_heads, topk, out, None, ws)
    st, flags = msa.msa_read_device_status(ws)
    assert st != 0 and flags & 2
    assert (topk[40:] == -1).all()
    pooled = torch.empty((rows, G, w.max_blocks), dtype=torch.float32, device="cuda")
    msa.msa_indexer_score(cache, batch, cfg, iq, pooled, ws)
    ref = torch.full_like(topk, -9)
    msa.msa_topk_blocks(batch, cfg, G, pooled, ref, None, ws)
    assert torch.equal(topk[:40], ref[:40])


def test_prefill_bad_block_flags_and_leaves_it_out():
    # a block-table entry outside the pool in a prefill chunk: the status word
    # says so, and the attend leaves the block out (finite outputs, no stale partials)
    from _helpers import gpu_path
    w = ms.make_workload("fp8_prefill", seed=85, seq_lens=(1500,), q_per_seq=40)
    c = ms.make_case(w, device="cuda")
    c["block_table"][0, 3] = c["num_blocks"] + 9
    cache, batch, iq, q = bind(c)
    cfg = msa.default_config(w.topk)
    ws = workspace(cache, batch, cfg, w.num_q_heads)
    rows = w.num_seqs * w.q_per_seq
    topk = torch.empty((rows, w.num_kv_heads, w.topk), dtype=torch.int32, device="cuda")
    out = torch.full((rows, w.num_q_heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    msa.msa_decode(cache, batch, cfg, iq, q, w.num_q_heads, topk, out, None, ws)
    st, flags = msa.msa_read_device_status(ws)
    assert st != 0 and flags & 1
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("mode,zero_idx,init,local,k,over", [
    ("topk", False, 0, 0, 16, None),
    ("topk", True, 0, 0, 16, None),
    ("topk", False, 2, 3, 16, None),
    ("topk", False, 8, 7, 16, None),        # the forced blocks fill every slot (kfree = 0)
    ("indexer", False, 0, 0, 16, None),
    ("indexer", True, 0, 0, 16, None),
    ("indexer", False, 2, 3, 16, None),
    ("indexer", False, 8, 7, 16, None),
    ("indexer", False, 0, 0, 4, None),
    ("indexer", True, 1, 1, 8, None),
    # every query tile scored by several CTAs (about 17 units a CTA, 79 a tile)
    ("indexer", False, 0, 0, 16, dict(seq_lens=(20000,), q_per_seq=1024)),
    # more CTAs a tile than the merge holds in registers
    ("indexer", False, 0, 1, 16, dict(seq_lens=(128 * 300,), q_per_seq=256)),
    # a tile split between two CTAs, as in the full-size chunk (~200 units a CTA, 235 a tile)
    ("indexer", False, 1, 2, 16, dict(seq_lens=(60000,), q_per_seq=4096)),
    ("indexer", True, 0, 0, 16, dict(seq_lens=(60000,), q_per_seq=4096)),
])
def test_prefill_selection_equals_block_topk(mode, zero_idx, init, local, k, over):
    # msa_decode of a prefill chunk selects either with one warp per row over
    # the pooled scores ("topk") or in the tcgen05 indexer's epilogue
    # ("indexer": per-thread running top-16 lists, merged a warp per row); the
    # staged msa_indexer_score + msa_topk_blocks (a CTA per row on the pooled
    # scores, checked against the oracle in test_topk_gpu.py) must give the same
    # rows, ties included (a zero index cache ties every block).  The small case
    # has more CTAs than units, so a tile's CTAs include some without units.
    over = over or dict(seq_lens=(128 * 40 + 5, 3000), q_per_seq=48)
    w = ms.make_workload("fp8_prefill", seed=86, **over)
    c = ms.make_case(w, device="cuda")
    if zero_idx:
        c["idx"].zero_()
    cfg = msa.Config(topk=k, init_blocks=init, local_blocks=local, prefill_select=mode)
    cache, batch, iq, q = bind(c)
    ws = workspace(cache, batch, cfg, w.num_q_heads)
    rows, G = w.num_seqs * w.q_per_seq, w.num_kv_heads
    topk = torch.full((rows, G, k), -7, dtype=torch.int32, device="cuda")
    out = torch.empty((rows, w.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    msa.msa_decode(cache, batch, cfg, iq, q, w.num_q_heads, topk, out, None, ws)
    pooled = torch.empty((rows, G, w.max_blocks), dtype=torch.float32, device="cuda")
    msa.msa_indexer_score(cache, batch, cfg, iq, pooled, ws)
    ref = torch.full_like(topk, -9)
    msa.msa_topk_blocks(batch, cfg, G, pooled, ref, None, ws)
    assert msa.msa_read_device_status(ws)[0] == 0
    assert torch.equal(topk, ref)


@pytest.mark.parametrize("over,cfg", [
    (dict(seq_lens=(1800,), q_per_seq=24, num_q_heads=4), None),           # 1 q head a group: 8 tokens a tile
    (dict(seq_lens=(2500, 1300), q_per_seq=16, topk=32), None),             # 32 slots a token
    (dict(seq_lens=(3000,), q_per_seq=20), dict(init_blocks=1, local_blocks=2)),
    (dict(seq_lens=(2100,), q_per_seq=40, num_q_heads=32), None),           # 8 q heads a group: 16 tokens an item
    (dict(seq_lens=(2900,), q_per_seq=24, num_q_heads=32, topk=32), None),  # 8 heads a group and 32 slots a token
    (dict(seq_lens=(1900, 700), q_per_seq=24, num_q_heads=8, q_dtype="fp8"), None),  # 2 a group, e4m3 query
    (dict(seq_lens=(6000,), q_per_seq=300), None),                           # lists of several items
])
def test_prefill_key_block_major_variants(over, cfg):
    from _helpers import check_out, check_selection, gpu_path
    w = ms.make_workload("fp8_prefill", seed=87, **over)
    c = ms.make_case(w, device="cuda")
    conf = msa.Config(topk=w.topk, **(cfg or {}))
    g = gpu_path(c, cfg=conf)
    h = ms.case_to_host(c)
    ref = _oracle(c, w)
    init, local = (cfg or {}).get("init_blocks", 0), (cfg or {}).get("local_blocks", 0)
    check_selection(g["topk"], ref, w.seq_lens, w.q_per_seq, w.topk, init, local)
    out = np.zeros_like(g["out"])
    lse = np.zeros_like(g["lse"])
    for s in range(w.num_seqs):
        o, l = O.attend_rows(h, s, g["topk"], w.head_dim ** -0.5)
        out[s * w.q_per_seq:(s + 1) * w.q_per_seq] = o
        lse[s * w.q_per_seq:(s + 1) * w.q_per_seq] = l
    check_out(g["out"], out)
    # the combine's log-sum-exp of the token's slots
    assert np.abs(g["lse"] - lse).max() < 1e-3


@pytest.mark.parametrize("name,over", [
    ("fp8_prefill", dict(seq_lens=(1700,), q_per_seq=24)),   # key-block-major lists
    ("fp8_decode", dict(seq_lens=(2600, 1900))),              # per-token union
])
def test_repeated_selected_block_attended_once_and_flagged(name, over):
    # a caller's selection naming one block twice in a row: the softmax runs over
    # the selected key set with each key once, and the status word says so
    from _helpers import check_out, gpu_path
    w = ms.make_workload(name, seed=90, **over)
    c = ms.make_case(w, device="cuda")
    g = gpu_path(c)
    h = ms.case_to_host(c)
    cache, batch, iq, q = bind(c)
    cfg = msa.default_config(w.topk)
    ws = workspace(cache, batch, cfg, w.num_q_heads)
    bad = g["topk"].copy()
    rows = w.num_seqs * w.q_per_seq
    for r in range(0, rows, 3):
        bad[r, r % w.num_kv_heads, 1] = bad[r, r % w.num_kv_heads, 3]  # slot 1 repeats slot 3
    out = torch.full((rows, w.num_q_heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((rows, w.num_q_heads), dtype=torch.float32, device="cuda")
    msa.msa_sparse_attend(cache, batch, cfg, q, w.num_q_heads, torch.from_numpy(bad).cuda(), out, lse, ws)
    st, flags = msa.msa_read_device_status(ws)
    assert st != 0 and flags & 4
    dedup = bad.copy()
    for r in range(0, rows, 3):
        dedup[r, r % w.num_kv_heads, 1] = -1
    ref = np.zeros((rows, w.num_q_heads, 128))
    ref_lse = np.zeros((rows, w.num_q_heads))
    for s in range(w.num_seqs):
        o, l = O.attend_rows(h, s, dedup, w.head_dim ** -0.5)
        ref[s * w.q_per_seq:(s + 1) * w.q_per_seq] = o
        ref_lse[s * w.q_per_seq:(s + 1) * w.q_per_seq] = l
    check_out(out.float().cpu().numpy(), ref)
    assert np.abs(lse.cpu().numpy() - ref_lse).max() < 1e-3


def test_prefill_bf16_cache_per_token_path():
    # BF16 keys / index keys: the decode indexer over 8-token virtual sequences
    # and the per-token attend (the key-block-major path is FP8 only)
    from _helpers import check_out, check_selection, check_pooled, gpu_path
    w = ms.make_workload("fp8_prefill", seed=88, seq_lens=(2200, 900), q_per_seq=24,
                         kv_dtype="bf16", index_dtype="bf16")
    c = ms.make_case(w, device="cuda")
    h = ms.case_to_host(c)
    ref = _oracle(c, w)
    got, st, flags = _pooled(c, w)
    assert st == 0, (msa.msa_status_string(st), flags)
    check_pooled(got, ref)
    g = gpu_path(c)
    check_selection(g["topk"], ref, w.seq_lens, w.q_per_seq, w.topk)
    out = np.zeros_like(g["out"])
    for s in range(w.num_seqs):
        o, _ = O.attend_rows(h, s, g["topk"], w.head_dim ** -0.5)
        out[s * w.q_per_seq:(s + 1) * w.q_per_seq] = o
    check_out(g["out"], out)


def test_prefill_invisible_selection_flags_and_is_left_out():
    # a caller's selection naming a block the token cannot see (the staged
    # msa_sparse_attend): the status word says so and the output stays finite
    w = ms.make_workload("fp8_prefill", seed=89, seq_lens=(1300,), q_per_seq=24)
    c = ms.make_case(w, device="cuda")
    cache, batch, iq, q = bind(c)
    cfg = msa.default_config(w.topk)
    ws = workspace(cache, batch, cfg, w.num_q_heads)
    rows = w.num_seqs * w.q_per_seq
    topk = torch.empty((rows, w.num_kv_heads, w.topk), dtype=torch.int32, device="cuda")
    out = torch.empty((rows, w.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    msa.msa_decode(cache, batch, cfg, iq, q, w.num_q_heads, topk, out, None, ws)
    assert msa.msa_read_device_status(ws)[0] == 0
    bad = topk.clone()
    bad[0, 0, 1] = (w.seq_lens[0] - 1) // 128  # token 0 sits in an earlier block: this one is invisible to it
    out2 = torch.full_like(out, float("nan"))
    msa.msa_sparse_attend(cache, batch, cfg, q, w.num_q_heads, bad, out2, None, ws)
    st, flags = msa.msa_read_device_status(ws)
    assert st != 0 and flags & 4
    assert torch.isfinite(out2.float()).all()


def test_prefill_partials_with_large_v_scales():
    # V per-token scales near 3e4 put |v| near 1e7, far above the fp16 range of
    # the key-block-major partials (o / l <= max |v|): a power-of-two scale per
    # partial must keep them finite.  Scaling every V scale by c scales the
    # output by c, so the comparison is made on out / c.
    from _helpers import check_out, gpu_path
    w = ms.make_workload("fp8_prefill", seed=91, seq_lens=(1700,), q_per_seq=24)
    c = ms.make_case(w, device="cuda")
    mult = 1.0e7
    c["v_scale"] *= mult
    g = gpu_path(c)
    assert np.isfinite(g["out"]).all()
    h = ms.case_to_host(c)
    o, lse = O.attend_rows(h, 0, g["topk"], w.head_dim ** -0.5)
    check_out(g["out"] / mult, o / mult)
    assert np.abs(g["lse"] - lse).max() < 1e-3
