"""Cache insert (msa_cache_insert) against the oracle's quantizers, byte for
byte, through the C ABI: BF16 copies, FP8 rows with their fp32 scales, NVFP4
rows with their E4M3 group scales, for the K / V caches and the index cache,
with padding slots, rows that are all zero, rows whose values sit on the
rounding ties of E4M3 and E2M1, and a slot outside the pool.  Then the path
itself runs over caches written by the insert (the step before the path,
vLLM Day-0 blog, section "QKV GEMM + norm + RoPE + KV 插入融合")."""

import numpy as np
import pytest
import torch

import block_sparse_attention_03_gb300 as msa
import msa_synth as ms
from oracle import msa_oracle as O

from _helpers import bind, check_out, check_selection, gpu_path

pytestmark = pytest.mark.gpu

ARRAYS = ("k", "v", "idx", "k_scale", "v_scale", "idx_scale", "k_sf", "v_sf", "idx_sf")


def _new_tokens(rng, n, H, gscale):
    """bf16 K, V, index keys of n new tokens, with crafted rows: token 0 all
    zero; token 1 with an element at 448 (FP8 scale 1: the bf16 values meet the
    E4M3 ties); token 2 on the E2M1 ties of an E4M3 group scale of 1/4 and a
    power-of-two per-tensor scale."""
    k = torch.randn((n, H, 128), generator=rng) * 0.1
    v = torch.randn((n, H, 128), generator=rng) * 0.1
    ik = torch.randn((n, 128), generator=rng) * 0.1
    for t in (k, v):
        t[0] = 0.0
        t[1] = (torch.rand((H, 128), generator=rng) * 896 - 448).round()
        t[1, :, 5] = 448.0
    ik[0] = 0.0
    ik[1] = (torch.rand(128, generator=rng) * 896 - 448).round()
    ik[1, 5] = 448.0
    # a group maximum of 6 x (1/4) x g makes the E4M3 group scale exactly 1/4
    ties = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -6.0])
    row = (ties * 0.25 * gscale).repeat(8)
    k[2] = row
    v[2] = row
    ik[2] = row
    return k.bfloat16().cuda(), v.bfloat16().cuda(), ik.bfloat16().cuda()


def _host(case):
    h = ms.case_to_host(case)
    out = {"kv_dtype": case["workload"].kv_dtype, "index_dtype": case["workload"].index_dtype}
    for name in ARRAYS:
        if name in h:
            out[name] = h[name].copy()
    for name in ("k_global", "v_global", "idx_global"):
        out[name] = case.get(name, 0.0)
    return out


@pytest.mark.parametrize("kv,idx", [("bf16", "bf16"), ("fp8", "fp8"), ("nvfp4", "nvfp4"), ("fp8", "nvfp4"),
                                    ("nvfp4", "bf16")])
def test_insert_matches_oracle_bytes(kv, idx):
    w = ms.make_workload("tiny_bf16", seq_lens=(1000, 700), kv_dtype=kv, index_dtype=idx, seed=120)
    case = ms.make_case(w, device="cuda")
    g = 2.0 ** -10
    for name in ("k_global", "v_global", "idx_global"):
        if name in case:
            case[name] = g
    cache, _, _, _ = bind(case)
    before = _host(case)
    rng = torch.Generator().manual_seed(121)
    n = 300
    k, v, ik = _new_tokens(rng, n, w.num_kv_heads, g)
    slots = torch.randperm(case["num_blocks"] * 128, generator=rng)[:n].int()
    slots[torch.arange(n) % 11 == 7] = -1
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    msa.msa_cache_insert(cache, slots.cuda(), k, v, ik, ws)
    st, flags = msa.msa_read_device_status(ws)
    assert st == 0, (st, flags)
    want = before
    O.insert_tokens(want, slots.numpy(), k.float().cpu().numpy(), v.float().cpu().numpy(),
                    ik.float().cpu().numpy())
    got = _host(case)
    for name in ARRAYS:
        if name in want:
            a, b = got[name], want[name]
            if a.dtype == np.float32:
                a, b = a.view(np.uint32), b.view(np.uint32)
            bad = np.argwhere(a != b)
            assert len(bad) == 0, (name, bad[:5], a[tuple(bad[0])], b[tuple(bad[0])])


def test_insert_slot_outside_the_pool_is_flagged_and_skipped():
    w = ms.make_workload("fp8_decode", seq_lens=(600,), seed=122)
    case = ms.make_case(w, device="cuda")
    cache, _, _, _ = bind(case)
    before = _host(case)
    rng = torch.Generator().manual_seed(123)
    k, v, ik = _new_tokens(rng, 3, 4, 1.0)
    slots = torch.tensor([3, case["num_blocks"] * 128 + 5, 130], dtype=torch.int32)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    msa.msa_cache_insert(cache, slots.cuda(), k, v, ik, ws)
    st, flags = msa.msa_read_device_status(ws)
    assert st == 5 and flags & 1
    want = before
    keep = slots.numpy().copy()
    keep[1] = -1
    O.insert_tokens(want, keep, k.float().cpu().numpy(), v.float().cpu().numpy(), ik.float().cpu().numpy())
    got = _host(case)
    for name in ARRAYS:
        if name in want:
            assert np.array_equal(got[name].view(np.uint8), want[name].view(np.uint8)), name


@pytest.mark.parametrize("kv", ["fp8", "nvfp4"])
def test_path_over_inserted_tokens(kv):
    # the last 200 tokens of every sequence are (re)written by the insert; the
    # whole path then runs over the caches it wrote, against the oracle
    q_dtype = "fp8" if kv == "nvfp4" else "bf16"
    w = ms.make_workload("fp8_decode", seq_lens=(5000, 3000), kv_dtype=kv, index_dtype=kv, q_dtype=q_dtype,
                         seed=124)
    case = ms.make_case(w, device="cuda")
    cache, _, _, _ = bind(case)
    rng = torch.Generator().manual_seed(125)
    slots = []
    bt = case["block_table"].cpu()
    for s, T in enumerate(w.seq_lens):
        for t in range(T - 200, T):
            slots.append(int(bt[s, t // 128]) * 128 + t % 128)
    slots = torch.tensor(slots, dtype=torch.int32)
    k = (torch.randn((len(slots), 4, 128), generator=rng) * 0.1).bfloat16().cuda()
    v = (torch.randn((len(slots), 4, 128), generator=rng) * 0.1).bfloat16().cuda()
    ik = (torch.randn((len(slots), 128), generator=rng) * 0.1).bfloat16().cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    msa.msa_cache_insert(cache, slots.cuda(), k, v, ik, ws)
    assert msa.msa_read_device_status(ws)[0] == 0
    g = gpu_path(case)
    h = ms.case_to_host(case)
    ref = O.run_path(h)
    check_selection(g["topk"], ref["pooled"], w.seq_lens, 1, w.topk)
    out = np.zeros_like(ref["out"])
    for s in range(w.num_seqs):
        out[s] = O.attend_rows(h, s, g["topk"], w.head_dim ** -0.5)[0][0]
    check_out(g["out"], out)
