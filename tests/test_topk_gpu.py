"""Block selection alone: msa_topk_blocks on given pooled scores against the
oracle's selection rule (vLLM Day-0 blog, section "MSA 入门"; the model
page's top-k buffer, `MiniMaxM3Model`).

Both sides see the same fp32 scores, so the selections must be identical,
ties included (equal scores keep the smaller block id).  The cases reach
every branch of the kernel: the threshold + rank test, its fall-back to the
radix select when thousands of candidates tie at the threshold, rows longer
than the keys a thread holds in registers, and the forced init / local
blocks.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import block_sparse_attention_03_gb300 as msa
from oracle import msa_oracle as O

pytestmark = pytest.mark.gpu

G = 4


def _run(seq_lens, q_per_seq, max_blocks, scores, cfg):
    S = len(seq_lens)
    lens = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    table = torch.zeros((S, max_blocks), dtype=torch.int32, device="cuda")
    batch = msa.Batch(lens, table, q_per_seq)
    pooled = torch.from_numpy(scores.astype(np.float32)).cuda()
    topk = torch.full((S * q_per_seq, G, cfg.topk), -7, dtype=torch.int32, device="cuda")
    score_out = torch.empty((S * q_per_seq, G, cfg.topk), dtype=torch.float32, device="cuda")
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    msa.msa_workspace_init(ws)
    msa.msa_topk_blocks(batch, cfg, G, pooled, topk, score_out, ws)
    st, flags = msa.msa_read_device_status(ws)
    assert st == 0, (msa.msa_status_string(st), flags)
    return topk.cpu().numpy(), score_out.cpu().numpy()


def _check(seq_lens, q_per_seq, max_blocks, scores, cfg):
    got, got_sc = _run(seq_lens, q_per_seq, max_blocks, scores, cfg)
    for s, T in enumerate(seq_lens):
        for i in range(q_per_seq):
            row = s * q_per_seq + i
            pos = T - q_per_seq + i
            for g in range(G):
                ref = O.select_blocks(scores[row, g].astype(np.float64), pos, cfg.topk,
                                      cfg.init_blocks, cfg.local_blocks)
                assert np.array_equal(got[row, g], ref), (s, i, g, got[row, g], ref)
                real = ref >= 0
                assert np.array_equal(got_sc[row, g][real], scores[row, g][ref[real]].astype(np.float32))


def _scores(rng, rows, max_blocks, kind):
    shape = (rows, G, max_blocks)
    if kind == "normal":
        return rng.standard_normal(shape).astype(np.float32)
    if kind == "ties":  # four distinct values: hundreds tie at the threshold
        return rng.integers(0, 4, size=shape).astype(np.float32)
    if kind == "ties2":  # two values: thousands tie at the threshold (the radix fall-back)
        return rng.integers(0, 2, size=shape).astype(np.float32)
    if kind == "equal":
        return np.full(shape, 0.25, dtype=np.float32)
    if kind == "signed_zero":  # +0 and -0 compare equal: ties between them keep the smaller id
        x = rng.standard_normal(shape).astype(np.float32) * np.float32(0.1) - np.float32(1.0)
        z = rng.random(shape) < 0.5
        x[z] = np.where(rng.random(z.sum()) < 0.5, np.float32(0.0), np.float32(-0.0))
        return x
    if kind == "neg_inf":  # masked scores mixed in
        x = rng.standard_normal(shape).astype(np.float32)
        x[rng.random(shape) < 0.7] = -np.inf
        return x
    if kind == "near_ties":  # every third score within 40 ulps of 1.0, the rest far below
        x = rng.standard_normal(shape).astype(np.float32) * np.float32(1e-3)
        ulps = rng.integers(0, 40, size=shape).astype(np.int32)
        one = np.float32(1.0).view(np.int32)
        x[:, :, ::3] = (one + ulps[:, :, ::3]).astype(np.int32).view(np.float32)
        return x
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["normal", "ties", "equal", "neg_inf", "near_ties", "signed_zero"])
def test_topk_short_rows(kind):
    rng = np.random.default_rng(100 + len(kind))
    seq_lens = [1, 128, 129, 700, 2049, 5000, 40000, 128 * 1000]
    mb = 1000
    _check(seq_lens, 1, mb, _scores(rng, len(seq_lens), mb, kind), msa.Config(topk=16))


@pytest.mark.parametrize("kind", ["normal", "ties", "ties2", "equal", "neg_inf"])
def test_topk_long_rows(kind):
    # up to 4096 blocks per row: 256 threads x 16 keys in registers
    rng = np.random.default_rng(200 + len(kind))
    seq_lens = [128 * 1025 + 3, 524288, 300]
    mb = 4096
    _check(seq_lens, 1, mb, _scores(rng, len(seq_lens), mb, kind), msa.Config(topk=16))


@pytest.mark.parametrize("kind", ["normal", "ties2"])
def test_topk_wide_rows(kind):
    # 4097 .. 8192 blocks per row: the 1024-thread variant, 8 keys each in registers
    rng = np.random.default_rng(250 + len(kind))
    seq_lens = [128 * 6000, 128 * 4097 + 1, 128 * 50]
    mb = 6000
    _check(seq_lens, 1, mb, _scores(rng, len(seq_lens), mb, kind), msa.Config(topk=16))


def test_topk_rows_beyond_registers():
    # 9000 blocks: more than 1024 threads x 8 keys, the radix select re-reads the row
    rng = np.random.default_rng(300)
    seq_lens = [128 * 9000, 128 * 8193 + 1]
    mb = 9000
    _check(seq_lens, 1, mb, _scores(rng, len(seq_lens), mb, "normal"), msa.Config(topk=32))


@pytest.mark.parametrize("topk,init,local", [(4, 0, 0), (8, 1, 2), (32, 0, 0), (32, 4, 8), (16, 15, 0)])
def test_topk_config_and_forced_blocks(topk, init, local):
    rng = np.random.default_rng(400 + topk + 10 * init + local)
    seq_lens = [100, 128 * 20, 3000, 128 * 700 + 5]
    mb = 720
    _check(seq_lens, 1, mb, _scores(rng, len(seq_lens), mb, "normal"),
           msa.Config(topk=topk, init_blocks=init, local_blocks=local))


def test_topk_multi_token_rows():
    # 8 query tokens per sequence: each row sees its own causal prefix of blocks
    rng = np.random.default_rng(500)
    seq_lens = [130, 128 * 64, 128 * 64 + 7, 9000]
    mb = 80
    _check(seq_lens, 8, mb, _scores(rng, len(seq_lens) * 8, mb, "ties"),
           msa.Config(topk=16, init_blocks=1, local_blocks=1))
