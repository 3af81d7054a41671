"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Every case generates its inputs once on the GPU (seeded), runs the library,
copies the inputs to the host and runs the oracle on the same bytes.
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_03_gb300 as msa
import msa_synth as ms
from oracle import msa_oracle as O

from _helpers import bind, check_out, check_pooled, check_selection, gpu_path, workspace

pytestmark = pytest.mark.gpu

KV = ["bf16", "fp8", "nvfp4"]


def _case(name, **over):
    w = ms.make_workload(name, **over)
    c = ms.make_case(w, device="cuda")
    return w, c, ms.case_to_host(c)


# ---------------------------------------------------------------- a1: decode of stored elements

@pytest.mark.parametrize("kv", KV)
def test_dequant_bit_exact(kv):
    w, c, h = _case("tiny_bf16", seq_lens=(700, 300), kv_dtype=kv, index_dtype=kv)
    cache, _, _, _ = bind(c)
    phys = torch.tensor(list(range(c["num_blocks"])) + [-1, c["num_blocks"]], dtype=torch.int32, device="cuda")
    n = phys.numel()
    for which in (0, 1, 2):
        heads = 1 if which == 2 else w.num_kv_heads
        out = torch.empty((n, heads, 128, 128), dtype=torch.float32, device="cuda")
        msa.msa_dequant_debug(cache, which, phys, out)
        got = out.cpu().numpy()
        for i in range(c["num_blocks"]):
            ref = O.dequant_index_tile(h, i)[None] if which == 2 else O.dequant_kv_tile(h, "kv"[which], i)
            assert np.array_equal(got[i].view(np.uint32), ref.astype(np.float32).view(np.uint32)), (kv, which, i)
        assert np.isnan(got[-2:]).all()


# ---------------------------------------------------------------- a2-a6 staged, a9 fused

STAGED_CASES = [
    ("tiny_bf16", {}),
    ("tiny_bf16", dict(topk=32)),
    ("fp8_decode", dict(seq_lens=(1000, 2500, 3333, 777), seed=11)),
    ("fp8_decode", dict(seq_lens=(4096, 129, 128, 1), seed=12)),
    ("nvfp4_verify", dict(seq_lens=(5000, 3000), seed=13)),
    ("nvfp4_verify", dict(seq_lens=(1029, 1024 + 3), seed=14)),  # 8 verify tokens straddle a block edge
    ("fp8_long", dict(seq_lens=(20000, 9000), seed=15)),
    ("fp8_decode", dict(seq_lens=(3000, 2000), q_per_seq=4, seed=16)),  # bf16 q, multi-token FP8
    ("tiny_bf16", dict(seq_lens=(2000, 1500), kv_dtype="fp8", index_dtype="nvfp4", seed=17)),
    ("tiny_bf16", dict(seq_lens=(2000,), kv_dtype="nvfp4", index_dtype="bf16", q_dtype="fp8", seed=18)),
    # prefill chunks: more than 8 new tokens are split into 8/4/2/1-token virtual sequences
    ("fp8_prefill", dict(seq_lens=(2000 + 64,), q_per_seq=64, seed=19)),
    ("fp8_prefill", dict(seq_lens=(1500, 900), q_per_seq=24, seed=20)),
    ("fp8_decode", dict(seq_lens=(700, 900), q_per_seq=12, seed=22)),
    ("tiny_bf16", dict(seq_lens=(1000,), q_per_seq=33, kv_dtype="nvfp4", index_dtype="nvfp4", q_dtype="fp8",
                       seed=23)),
]


@pytest.mark.parametrize("name,over", STAGED_CASES)
def test_staged_path_matches_oracle(name, over):
    w, c, h = _case(name, **over)
    g = gpu_path(c, fused=False)
    ref = O.run_path(h, topk=w.topk)
    check_pooled(g["pooled"], ref["pooled"])
    check_selection(g["topk"], ref["pooled"], w.seq_lens, w.q_per_seq, w.topk)
    out = np.zeros_like(ref["out"])
    for s in range(w.num_seqs):  # the oracle's attend on the GPU's own selection
        o, _ = O.attend_rows(h, s, g["topk"], w.head_dim ** -0.5)
        out[s * w.q_per_seq:(s + 1) * w.q_per_seq] = o
    check_out(g["out"], out)


@pytest.mark.parametrize("name,over", STAGED_CASES[:7])
def test_fused_decode_matches_staged(name, over):
    w, c, h = _case(name, **over)
    a = gpu_path(c, fused=False)
    b = gpu_path(c, fused=True)
    assert np.array_equal(a["topk"], b["topk"])
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["lse"], b["lse"])


def test_lse_matches_oracle():
    w, c, h = _case("fp8_decode", seq_lens=(3000, 1111), seed=21)
    g = gpu_path(c)
    for s in range(w.num_seqs):
        o, lse = O.attend_rows(h, s, g["topk"], w.head_dim ** -0.5)
        assert np.abs(g["lse"][s] - lse[0]).max() < 1e-3


def test_topk32_equals_dense_attention():
    # with k >= number of blocks the path is dense causal attention
    w, c, h = _case("tiny_bf16", topk=32)
    g = gpu_path(c)
    assert np.array_equal(g["topk"][0, 0], np.arange(32))
    T = w.seq_lens[0]
    K = np.concatenate([O.dequant_kv_tile(h, "k", int(h["block_table"][0, b])) for b in range(32)], axis=1)
    V = np.concatenate([O.dequant_kv_tile(h, "v", int(h["block_table"][0, b])) for b in range(32)], axis=1)
    q = O.query_values(h["q"], "bf16", 1.0)[0]
    ref = np.stack([O.attend(q[hh], K[hh // 4, :T], V[hh // 4, :T], 128 ** -0.5)[0] for hh in range(16)])
    check_out(g["out"][0], ref)


@pytest.mark.parametrize("topk", [4, 8, 32])
def test_other_topk(topk):
    w, c, h = _case("fp8_decode", seq_lens=(5000, 300), topk=topk, seed=30 + topk)
    g = gpu_path(c, fused=False)
    ref = O.run_path(h, topk=topk)
    check_pooled(g["pooled"], ref["pooled"])
    check_selection(g["topk"], ref["pooled"], w.seq_lens, 1, topk)


def test_init_and_local_blocks():
    w, c, h = _case("fp8_decode", seq_lens=(6000, 2000), seed=40)
    cfg = msa.Config(topk=16, init_blocks=2, local_blocks=3)
    g = gpu_path(c, cfg=cfg, fused=False)
    ref = O.run_path(h, topk=16, init_blocks=2, local_blocks=3)
    check_selection(g["topk"], ref["pooled"], w.seq_lens, 1, 16, 2, 3)


def test_planted_hot_blocks_selected():
    w, c, h = _case("fp8_decode", seq_lens=(12000, 9000, 7000), seed=41)
    g = gpu_path(c)
    for s in range(w.num_seqs):
        for grp in range(w.num_kv_heads):
            assert set(h["hot"][s, grp]).issubset(set(g["topk"][s, grp]))


def test_bad_block_table_sets_status_not_trap():
    w, c, h = _case("fp8_decode", seq_lens=(2000, 2000), seed=42)
    c["block_table"][1, 3] = c["num_blocks"] + 5
    cache, batch, iq, q = bind(c)
    cfg = msa.default_config()
    ws = workspace(cache, batch, cfg, 16)
    topk = torch.empty((2, 4, 16), dtype=torch.int32, device="cuda")
    out = torch.empty((2, 16, 128), dtype=torch.bfloat16, device="cuda")
    msa.msa_decode(cache, batch, cfg, iq, q, 16, topk, out, None, ws)
    st, flags = msa.msa_read_device_status(ws)
    assert st == 5 and flags & 1
    # the context stays usable and the status word was cleared
    msa.msa_decode(cache, batch, cfg, iq, q, 16, topk, out, None, ws)
    torch.cuda.synchronize()
    st2, _ = msa.msa_read_device_status(ws)
    assert st2 == 5  # still bad data -> flagged again


def test_host_errors_launch_nothing():
    w, c, h = _case("fp8_decode", seq_lens=(2000,), seed=43)
    cache, batch, iq, q = bind(c)
    cfg = msa.default_config()
    ws = workspace(cache, batch, cfg, 16)
    topk = torch.empty((1, 4, 16), dtype=torch.int32, device="cuda")
    out = torch.empty((1, 16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(msa.MsaError) as e:
        msa.msa_decode(cache, batch, msa.Config(topk=12), iq, q, 16, topk, out, None, ws)
    assert e.value.status == 2
    with pytest.raises(msa.MsaError) as e:
        msa.msa_decode(cache, batch, cfg, iq, q, 16, topk, out, None, ws[:1000])
    assert e.value.status == 3
    with pytest.raises(msa.MsaError) as e:
        msa.msa_decode(cache, batch, cfg, iq, q, 15, topk, out, None, ws)
    assert e.value.status == 1


# ---------------------------------------------------------------- full-size workloads, sampled

@pytest.mark.parametrize("name,seqs", [("tiny_bf16", [0]), ("fp8_decode", [0, 17, 31]),
                                       ("fp8_long", [2]), ("nvfp4_verify", [5])])
def test_full_size_sampled(name, seqs):
    w = ms.make_workload(name)
    c = ms.make_case(w, device="cuda")
    g = gpu_path(c)
    # the pooled scores of the full-size launch too (the staged indexer entry point)
    cache, batch, iq, _ = bind(c)
    cfg = msa.default_config(w.topk)
    ws = workspace(cache, batch, cfg, w.num_q_heads)
    pooled_gpu = torch.empty((w.num_seqs * w.q_per_seq, w.num_kv_heads, w.max_blocks), dtype=torch.float32,
                             device="cuda")
    msa.msa_indexer_score(cache, batch, cfg, iq, pooled_gpu, ws)
    assert msa.msa_read_device_status(ws)[0] == 0
    pooled_gpu = pooled_gpu.cpu().numpy()
    h = ms.case_to_host(c)
    del c, ws
    torch.cuda.empty_cache()
    Q = w.q_per_seq
    for s in seqs:
        pooled = O.pooled_scores(h, s, w.index_dim ** -0.5)
        rows = list(range(s * Q, (s + 1) * Q))
        check_pooled(pooled_gpu[rows], pooled)
        full = np.full((w.num_seqs * Q, w.num_kv_heads, w.max_blocks), -np.inf)
        full[rows] = pooled
        check_selection(g["topk"], full, w.seq_lens, Q, w.topk, rows=rows)
        o, _ = O.attend_rows(h, s, g["topk"], w.head_dim ** -0.5)
        check_out(g["out"][rows], o)


def test_many_short_sequences():
    # 2,600 sequences of 1..700 tokens: more (sequence, group) units than the attend
    # has CTAs by far, so every CTA walks dozens of splits in several batches
    rng = np.random.default_rng(77)
    lens = rng.integers(1, 700, size=2600)
    w = ms.make_workload("fp8_decode", seq_lens=lens, seed=77)
    c = ms.make_case(w, device="cuda")
    g = gpu_path(c)
    h = ms.case_to_host(c)
    del c
    for s in [0, 1, 2, 777, 1500, 2599] + [int(x) for x in rng.choice(2600, 6, replace=False)]:
        pooled = O.pooled_scores(h, s, w.index_dim ** -0.5)
        full = np.full((w.num_seqs, w.num_kv_heads, w.max_blocks), -np.inf)
        full[s] = pooled[0]
        check_selection(g["topk"], full, w.seq_lens, 1, w.topk, rows=[s])
        o, _ = O.attend_rows(h, s, g["topk"], w.head_dim ** -0.5)
        check_out(g["out"][[s]], o)


@pytest.mark.parametrize("mode", ["topk", "indexer"])
def test_full_size_prefill_sampled(mode):
    # 8,192 new tokens on a 64K-token FP8 context: sampled query rows against the
    # oracle, with the selection by the top-k launch or in the indexer's epilogue
    w = ms.make_workload("fp8_prefill")
    c = ms.make_case(w, device="cuda")
    g = gpu_path(c, cfg=msa.Config(topk=w.topk, prefill_select=mode))
    h = ms.case_to_host(c)
    del c
    torch.cuda.empty_cache()
    rows = [0, 1, 7, 8, 2047, 4096, 8190, 8191]
    pooled = O.pooled_scores(h, 0, w.index_dim ** -0.5, rows=rows)
    full = np.full((w.q_per_seq, w.num_kv_heads, w.max_blocks), -np.inf)
    full[rows] = pooled
    check_selection(g["topk"], full, w.seq_lens, w.q_per_seq, w.topk, rows=rows)
    o, _ = O.attend_rows(h, 0, g["topk"], w.head_dim ** -0.5, rows=rows)
    check_out(g["out"][rows], o)


def test_indexer_warps_with_more_than_32_blocks():
    # 64 sequences of 128K tokens = 65,536 blocks over the persistent indexer's
    # warps: each warp owns more than 32 blocks, so its window of 32 + 32 block
    # facts slides during its run.  Only the index cache is built (1 GB of FP8
    # keys); pooled scores of sampled sequences are checked against the oracle.
    S, T = 64, 131072
    nb = T // 128
    gen = torch.Generator(device="cuda")
    gen.manual_seed(61)
    nblk = S * nb + 3
    idx = torch.randint(0, 256, (nblk, 128, 128), dtype=torch.uint8, device="cuda", generator=gen)
    idx[(idx & 0x7F) == 0x7F] = 0  # no NaN codes
    idx_scale = torch.rand((nblk, 128), device="cuda", generator=gen) * 1e-3 + 1e-4
    perm = torch.randperm(nblk, device="cuda", generator=gen)[: S * nb].int().reshape(S, nb)
    lens = torch.full((S,), T, dtype=torch.int32, device="cuda")
    lens[::3] -= 77  # ragged last blocks
    iq = (torch.randn((S, 4, 128), device="cuda", generator=gen) / 11.3).bfloat16()
    cache = msa.PagedCache(kv_dtype="fp8", index_dtype="fp8", num_blocks=nblk, num_kv_heads=4, k=idx, v=idx, idx=idx,
                           idx_scale=idx_scale)
    batch = msa.Batch(lens, perm, 1)
    cfg = msa.default_config()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    pooled = torch.empty((S, 4, nb), dtype=torch.float32, device="cuda")
    msa.msa_indexer_score(cache, batch, cfg, msa.Query(iq), pooled, ws)
    assert msa.msa_read_device_status(ws)[0] == 0
    got = pooled.cpu().numpy()
    w = ms.make_workload("fp8_long", seq_lens=tuple(int(x) for x in lens.cpu()), num_seqs=S)
    rows = [0, 13, 31, 47, 63]
    iq_host = iq.view(torch.int16).cpu().numpy().view(np.uint16)
    for s in rows:
        # the sequence's blocks gathered in logical order, under an identity table
        h = {"workload": w, "seq_lens": lens.cpu().numpy(), "index_q": iq_host, "index_q_scale": 1.0,
             "idx": idx[perm[s].long()].cpu().numpy(), "idx_scale": idx_scale[perm[s].long()].cpu().numpy(),
             "block_table": np.arange(nb, dtype=np.int32)[None].repeat(S, axis=0)}
        ref = O.pooled_scores(h, s, 128 ** -0.5)
        check_pooled(got[[s]], ref)
