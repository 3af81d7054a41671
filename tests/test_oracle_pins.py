"""Pins of the CPU oracle against facts fixed outside it.

Each test ties one oracle function to something other than itself: a format
definition's textbook values, a library routine (torch's fp8 cast, SDPA,
scipy's logsumexp), a closed form on a hand-built cache, brute force on tiny
inputs, or a figure the pages print (tests/golden/pages_figures.txt).
"""

import itertools
import math
import os

import numpy as np
import pytest
import torch

import msa_synth as ms
from oracle import msa_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_figures.txt")


def golden():
    vals = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (x.strip() for x in line.split("="))
            vals[k] = float(v)
    return vals


# ---------------------------------------------------------------- formats

def test_e4m3_textbook_values():
    # OCP 8-bit floating point spec, E4M3: bias 7, max normal 448, min normal
    # 2^-6, min subnormal 2^-9, S.1111.111 is NaN, no infinities.
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0,
             0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9)}
    for code, val in table.items():
        assert O.e4m3_value(code) == val, hex(code)
    assert np.isnan(O.e4m3_value(0x7F)) and np.isnan(O.e4m3_value(0xFF))


def test_e4m3_matches_torch_cast():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    mine = O.e4m3_value(codes).astype(np.float32)
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok].view(np.uint32), mine[ok].view(np.uint32))


def test_e2m1_textbook_values():
    # OCP MX spec, FP4 E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 = sign
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for code in range(16):
        want = (-1.0 if code & 8 else 1.0) * mags[code & 7]
        assert O.e2m1_value(code) == want


def test_bf16_widen_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # drop inf/nan patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(O.bf16_value(bits).view(np.uint32), ref.view(np.uint32))


def test_nvfp4_products_exact_in_fp32():
    # every e2m1 x e4m3 product is exact in fp32, so the dequant has one rounding
    for n in range(16):
        for sc in range(256):
            if (sc & 0x7F) == 0x7F:
                continue
            exact = O.nvfp4_product_exact(n, sc)
            f32 = np.float32(O.e2m1_value(n) * O.e4m3_value(sc))
            assert exact == float(f32)


def test_fp8_dequant_one_rounding_matches_torch():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 256, size=(3, 128), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0
    scale = rng.random(3).astype(np.float32) * 0.01
    mine = O._dequant("fp8", codes, scale=scale)
    ref = (torch.from_numpy(codes).view(torch.float8_e4m3fn).float()
           * torch.from_numpy(scale)[:, None]).numpy()
    assert np.array_equal(mine.view(np.uint32), ref.view(np.uint32))


def test_nvfp4_roundtrip_nibble_order_and_scale_index():
    # exactly representable input: x = e2m1 * e4m3_scale * global, with the
    # group amax equal to 6 * scale * global so the quantizer recovers the
    # same scale; the oracle must decode the generator's bytes back to x.
    rng = np.random.default_rng(2)
    gscale = 0.0078125
    sf_codes = rng.integers(0x20, 0x60, size=(2, 8), dtype=np.uint8)
    nib = rng.integers(0, 16, size=(2, 128), dtype=np.uint8)
    nib[:, ::16] = 7  # magnitude 6 in every group -> amax16 = 6 * scale
    x = O.e2m1_value(nib) * np.repeat(O.e4m3_value(sf_codes), 16, axis=-1) * gscale
    packed, sf, g = ms.quantize_nvfp4(torch.from_numpy(x).float(), global_scale=gscale)
    assert np.array_equal(sf.numpy(), sf_codes)
    deq = O._dequant("nvfp4", packed.numpy(), sf=sf.numpy(), gscale=g)
    assert np.array_equal(deq, x.astype(np.float32))
    # element 2j is the low nibble of byte j
    assert np.array_equal(packed.numpy()[0, 0] & 0xF, nib[0, 0] & 0xF)


# ---------------------------------------------------------------- layout / byte figures

def test_layout_bytes_match_pages():
    g = golden()
    w = ms.make_workload("tiny_bf16", seq_lens=(256,), kv_dtype="nvfp4", index_dtype="fp8",
                         q_dtype="bf16")
    c = ms.make_case(w)
    H, D = w.num_kv_heads, w.head_dim
    tokens = c["num_blocks"] * 128
    nvfp4_per_elem = (c["k"].numel() + c["k_sf"].numel()) / (tokens * H * D)
    assert nvfp4_per_elem == g["nvfp4_kv_bytes_per_token"] / g["fp8_kv_bytes_per_token"] == 9 / 16
    assert 1 - nvfp4_per_elem == g["nvfp4_saving"]
    # FP8 index keys: one shared head of 128 dims, 1 byte each
    assert c["idx"].numel() / tokens == g["index_bytes_per_token_fp8"]
    assert 2 * H * D == g["kv_bytes_per_token_fp8"]  # K + V, 4 heads x 128 dims, FP8
    assert g["index_bytes_per_token_fp8"] / g["kv_bytes_per_token_fp8"] == g["index_to_kv_ratio"]
    assert g["topk_blocks"] * g["block_size_tokens"] == g["max_keys_per_query"]


def test_traffic_model_long_context_limit():
    from block_sparse_attention_03_gb300 import roofline as R
    g = golden()
    dense = lambda T: g["kv_bytes_per_token_fp8"] * T
    for T, lo, hi in [(524288, 0.128, 0.130), (1 << 30, 0.12500, 0.12501)]:
        sparse = R.decode_bytes_per_query("fp8", "fp8", T, 16 * 128, 4, 128, 128)
        assert lo < sparse / dense(T) < hi
    assert abs(R.decode_bytes_per_query("fp8", "fp8", 1 << 40, 2048, 4, 128, 128) / dense(1 << 40)
               - g["long_context_traffic_ratio"]) < 1e-6


# ---------------------------------------------------------------- score / pool

def _onehot_keys(T, Di=128):
    keys = np.zeros((T, Di), dtype=np.float32)
    keys[np.arange(T), np.arange(T) % Di] = 1.0
    return keys


def test_index_score_closed_form():
    # key t = unit vector e_(t mod 128): score(g, t) = scale * iq[g][t mod 128]
    T, Q, G = 300, 2, 4
    rng = np.random.default_rng(3)
    iq = rng.standard_normal((Q, G, 128))
    pos = np.array([T - 2, T - 1])
    scale = 128 ** -0.5
    s = O.index_scores(_onehot_keys(T), iq, pos, scale)
    for q in range(Q):
        for g in range(G):
            for t in range(T):
                want = scale * iq[q, g, t % 128] if t <= pos[q] else -np.inf
                assert s[q, g, t] == pytest.approx(want, rel=1e-14, abs=0) if t <= pos[q] else s[q, g, t] == want


def test_pool_closed_form_with_causal_tail():
    # key t = (1 + t // 128) * e_(t mod 128): block b's scores are (b+1) * iq
    T, Q, G = 300, 3, 4
    rng = np.random.default_rng(4)
    iq = np.abs(rng.standard_normal((Q, G, 128)))
    keys = _onehot_keys(T) * (1 + np.arange(T) // 128)[:, None]
    pos = np.array([255, 256, 299])  # straddles the 2nd/3rd block boundary
    s = O.index_scores(keys, iq, pos, 1.0)
    P = O.pool_blocks(s, 4)
    for q in range(Q):
        for g in range(G):
            for b in range(4):
                n = min(128, pos[q] + 1 - b * 128, T - b * 128)
                want = (b + 1) * iq[q, g, :n].max() if n > 0 else -np.inf
                assert P[q, g, b] == want


def test_scale_applies_to_scores():
    T = 130
    iq = np.ones((1, 1, 128))
    s1 = O.index_scores(_onehot_keys(T), iq, np.array([T - 1]), 1.0)
    s2 = O.index_scores(_onehot_keys(T), iq, np.array([T - 1]), 128 ** -0.5)
    assert np.allclose(s2, s1 * 128 ** -0.5)


# ---------------------------------------------------------------- selection

def _brute_topk(pooled, recent, k):
    """Best (k-1)-subset of the blocks before `recent` by total score."""
    cand = list(range(recent))
    m = min(k - 1, len(cand))
    best = max(itertools.combinations(cand, m), key=lambda c: (sum(pooled[b] for b in c),))
    return sorted(list(best) + [recent])


def test_selection_matches_brute_force():
    rng = np.random.default_rng(5)
    for trial in range(300):
        nb = int(rng.integers(1, 10))
        k = int(rng.choice([2, 3, 4, 5]))
        pooled = rng.standard_normal(nb)  # distinct values
        pos = (nb - 1) * 128 + int(rng.integers(0, 128))
        got = O.select_blocks(pooled, pos, k)
        want = _brute_topk(pooled, nb - 1, k)
        assert list(got[: len(want)]) == want
        assert np.all(got[len(want):] == -1)


def test_selection_ties_prefer_smaller_id():
    pooled = np.array([1.0, 2.0, 2.0, 2.0, 0.5, 9.0])
    got = O.select_blocks(pooled, 5 * 128 + 3, 3)  # recent = 5 forced, 2 free slots
    assert list(got) == [1, 2, 5]


def test_selection_invariants():
    rng = np.random.default_rng(6)
    for _ in range(200):
        nb = int(rng.integers(1, 60))
        pooled = rng.standard_normal(nb)
        pos = (nb - 1) * 128 + int(rng.integers(0, 128))
        for k in (4, 8, 16, 32):
            sel = O.select_blocks(pooled, pos, k)
            ids = sel[sel >= 0]
            assert (nb - 1) in ids  # the most recent block is always kept
            assert len(ids) == min(k, nb)
            assert np.all(np.diff(ids) > 0)
            assert len(ids) * 128 <= 2048 or k == 32  # <= 2,048 keys for k = 16


def test_forced_init_and_local_blocks():
    pooled = np.arange(20, dtype=float)[::-1].copy()  # block 0 best
    sel = O.select_blocks(pooled, 19 * 128, 6, init_blocks=2, local_blocks=2)
    assert {0, 1, 17, 18, 19}.issubset(set(sel))
    assert len(set(sel)) == 6


# ---------------------------------------------------------------- attend

def _small_case(**kw):
    w = ms.make_workload("tiny_bf16", **kw)
    return w, ms.case_to_host(ms.make_case(w))


@pytest.mark.parametrize("kv", ["bf16", "fp8", "nvfp4"])
def test_full_topk_equals_dense_causal_sdpa(kv):
    # top-k >= number of blocks: MSA must equal dense causal attention
    w, c = _small_case(seq_lens=(1000, 700), q_per_seq=3, kv_dtype=kv, index_dtype=kv, topk=8)
    r = O.run_path(c)
    Q, G, Hq = w.q_per_seq, w.num_kv_heads, w.num_q_heads
    for s, T in enumerate(w.seq_lens):
        K = np.concatenate([O.dequant_kv_tile(c, "k", int(c["block_table"][s, b]))
                            for b in range((T + 127) // 128)], axis=1)[:, :T]
        V = np.concatenate([O.dequant_kv_tile(c, "v", int(c["block_table"][s, b]))
                            for b in range((T + 127) // 128)], axis=1)[:, :T]
        q = O.query_values(c["q"], w.q_dtype, c["q_scale"])[s * Q:(s + 1) * Q]
        qt = torch.from_numpy(q).permute(1, 0, 2)[None]  # [1, Hq, Q, D]
        kt = torch.from_numpy(K.astype(np.float64))[None]  # [1, G, T, D]
        vt = torch.from_numpy(V.astype(np.float64))[None]
        pos = torch.arange(T - Q, T)
        mask = torch.arange(T)[None, :] <= pos[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=mask, scale=w.head_dim ** -0.5, enable_gqa=True)
        ref = ref[0].permute(1, 0, 2).numpy()
        assert np.allclose(r["out"][s * Q:(s + 1) * Q], ref, rtol=0, atol=1e-12)


def test_lse_matches_scipy():
    from scipy.special import logsumexp
    rng = np.random.default_rng(7)
    q = rng.standard_normal(128)
    K = rng.standard_normal((300, 128))
    V = rng.standard_normal((300, 128))
    o, lse = O.attend(q, K, V, 0.1)
    assert lse == pytest.approx(logsumexp(0.1 * K @ q), rel=1e-13)
    w = np.exp(0.1 * K @ q - lse)
    assert np.allclose(o, w @ V, atol=1e-12)


def test_block_table_permutation_invariance():
    w, c = _small_case(seq_lens=(1500,), kv_dtype="fp8", index_dtype="fp8")
    r1 = O.run_path(c)
    rng = np.random.default_rng(8)
    perm = rng.permutation(c["num_blocks"])  # new physical slot of each block
    c2 = dict(c)
    for key in ("idx", "idx_scale", "k", "v", "k_scale", "v_scale"):
        arr = np.empty_like(c[key])
        arr[perm] = c[key]
        c2[key] = arr
    c2["block_table"] = perm[c["block_table"]].astype(np.int32)
    r2 = O.run_path(c2)
    assert np.array_equal(r1["topk"], r2["topk"])
    assert np.array_equal(r1["out"], r2["out"])
    assert np.array_equal(r1["pooled"], r2["pooled"])


def test_planted_hot_blocks_are_selected():
    for kv in ("bf16", "fp8", "nvfp4"):
        w, c = _small_case(seq_lens=(8192, 6000), kv_dtype=kv, index_dtype=kv)
        r = O.run_path(c)
        for s in range(w.num_seqs):
            for g in range(w.num_kv_heads):
                assert set(c["hot"][s, g]).issubset(set(r["topk"][s, g])), (kv, s, g)


def test_multi_token_causal_positions():
    # 8 verify tokens straddling a block boundary: each keeps its own block
    w, c = _small_case(seq_lens=(128 * 6 + 3,), q_per_seq=8)
    r = O.run_path(c)
    T = w.seq_lens[0]
    for i in range(8):
        pos = T - 8 + i
        for g in range(w.num_kv_heads):
            assert pos // 128 in r["topk"][i, g]
            assert np.all(np.isneginf(r["pooled"][i, g, pos // 128 + 1:]))


# ---------------------------------------------------------------- query and K/V scales, decoded independently

# OCP MX FP4 E2M1 magnitudes by code (bit 3 = sign), written out from the format
# definition for the independent decodes below
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _torch_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).float()


def _indep_fp8(codes, scale):
    """fp32 value of e4m3 codes times their per-row fp32 scale, through torch's cast."""
    return (_torch_e4m3(codes) * torch.from_numpy(np.asarray(scale, np.float32))[..., None]).numpy()


def _indep_nvfp4(packed, sf, gscale):
    """fp32 NVFP4 value: table-decoded nibbles (low nibble first) x torch-decoded
    e4m3 block scales, then x the per-tensor scale in fp32."""
    p = np.asarray(packed, np.uint8)
    nib = np.stack([p & 0xF, p >> 4], axis=-1).reshape(p.shape[:-1] + (2 * p.shape[-1],))
    vals = np.where(nib & 8, -1.0, 1.0) * _E2M1_MAG[nib & 7]
    sfv = np.repeat(_torch_e4m3(sf).numpy().astype(np.float64), 16, axis=-1)
    return (vals * sfv).astype(np.float32) * np.float32(gscale)


@pytest.mark.parametrize("scale", [0.0173, 3.25e-3, 1.0])
def test_fp8_query_values_match_torch_cast_times_scale(scale):
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]
    got = O.query_values(codes, "fp8", scale)
    ref = (_torch_e4m3(codes) * torch.tensor(scale, dtype=torch.float32)).double().numpy()
    assert np.array_equal(got, ref)


def test_generated_fp8_queries_decode_with_their_own_scales():
    # q and index_q of an E4M3-query case have different per-tensor scales; each
    # decodes as torch's cast times its own scale
    w, c = _small_case(seq_lens=(600,), q_per_seq=2, kv_dtype="nvfp4", index_dtype="nvfp4", q_dtype="fp8")
    assert c["q_scale"] != c["index_q_scale"] and c["q_scale"] != 1.0
    for key in ("q", "index_q"):
        got = O.query_values(c[key], "fp8", c[key + "_scale"])
        ref = (_torch_e4m3(c[key]) * torch.tensor(c[key + "_scale"], dtype=torch.float32)).double().numpy()
        assert np.array_equal(got, ref), key


@pytest.mark.parametrize("kv", ["fp8", "nvfp4"])
def test_kv_tiles_decode_with_their_own_scales(kv):
    # K and V differ in data and in scales; each tile must decode with its own
    w, c = _small_case(seq_lens=(300, 200), kv_dtype=kv, index_dtype=kv)
    for phys in range(c["num_blocks"]):
        for which in ("k", "v"):
            if kv == "fp8":
                ref = _indep_fp8(c[which][phys], c[which + "_scale"][phys])
            else:
                ref = _indep_nvfp4(c[which][phys], c[which + "_sf"][phys], c[which + "_global"])
            got = O.dequant_kv_tile(c, which, phys)
            assert np.array_equal(got.view(np.uint32), ref.astype(np.float32).view(np.uint32)), (which, phys)
    if kv == "fp8":
        assert not np.array_equal(c["k_scale"], c["v_scale"])
    else:
        assert c["k_global"] != c["v_global"]


@pytest.mark.parametrize("kv", ["fp8", "nvfp4"])
def test_kv_quantize_dequant_round_trip_within_format_bound(kv):
    # x -> generator's quantizer -> oracle decode lands within the format's
    # rounding bound of x, for K and V separately (distinct data, distinct scales)
    gen = torch.Generator().manual_seed(9)
    k = torch.randn((2, 4, 128, 128), generator=gen) / math.sqrt(128.0)
    v = 3.0 * torch.randn((2, 4, 128, 128), generator=gen) / math.sqrt(128.0)
    w = ms.make_workload("tiny_bf16", seq_lens=(256,), kv_dtype=kv, index_dtype=kv)
    case = {"workload": w}
    for name, x in (("k", k), ("v", v)):
        if kv == "fp8":
            codes, scale = ms.quantize_fp8_rows(x)
            case[name], case[name + "_scale"] = codes.numpy(), scale.numpy()
        else:
            packed, sf, g = ms.quantize_nvfp4(x)
            case[name], case[name + "_sf"], case[name + "_global"] = packed.numpy(), sf.numpy(), g
    for name, x in (("k", k), ("v", v)):
        xs = x.numpy().astype(np.float64)
        for phys in range(2):
            d = O.dequant_kv_tile(case, name, phys).astype(np.float64)
            if kv == "fp8":
                # E4M3 round to nearest: |err| <= 2^-4 |x| (normal range) or half the
                # subnormal step 2^-10, in units of the row scale
                sc = case[name + "_scale"][phys].astype(np.float64)[..., None]
                bound = np.maximum(np.abs(xs[phys]) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 1e-6)
            else:
                # E2M1 step within a 16-group is at most 2 (between 4 and 6) in units of
                # scale x global, half of it after rounding; the e4m3 scale itself carries
                # a relative error up to 2^-4, which moves the group's largest value by
                # at most 6 x 2^-4 units
                sfv = np.repeat(O.e4m3_value(case[name + "_sf"][phys]), 16, axis=-1) * case[name + "_global"]
                bound = sfv * (1.0 + 6 * 2.0 ** -4) * (1 + 1e-6) + 1e-30
            assert np.all(np.abs(d - xs[phys]) <= bound), (kv, name)
        # the scales differ between K and V (V is 3x wider), so a swap is visible
    if kv == "fp8":
        assert np.median(case["v_scale"]) > 2 * np.median(case["k_scale"])
    else:
        assert case["v_global"] > 2 * case["k_global"]


def test_full_topk_equals_dense_sdpa_with_fp8_queries_decoded_independently():
    # top-k >= blocks: equal to dense causal attention; the reference side decodes
    # q (E4M3 x its scale) and the FP8 K / V tiles (x their own per-token scales)
    # through torch's float8 cast, not through the oracle's helpers
    w, c = _small_case(seq_lens=(900,), q_per_seq=3, kv_dtype="fp8", index_dtype="fp8", q_dtype="fp8", topk=8)
    r = O.run_path(c)
    Q, T = w.q_per_seq, w.seq_lens[0]
    nb = (T + 127) // 128
    phys = [int(c["block_table"][0, b]) for b in range(nb)]
    K = np.concatenate([_indep_fp8(c["k"][p], c["k_scale"][p]) for p in phys], axis=1)[:, :T]
    V = np.concatenate([_indep_fp8(c["v"][p], c["v_scale"][p]) for p in phys], axis=1)[:, :T]
    q = (_torch_e4m3(c["q"]) * torch.tensor(c["q_scale"], dtype=torch.float32)).double()[:Q]
    qt = q.permute(1, 0, 2)[None]
    kt = torch.from_numpy(K.astype(np.float64))[None]
    vt = torch.from_numpy(V.astype(np.float64))[None]
    pos = torch.arange(T - Q, T)
    mask = torch.arange(T)[None, :] <= pos[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=mask, scale=w.head_dim ** -0.5, enable_gqa=True)[0].permute(1, 0, 2).numpy()
    assert np.allclose(r["out"][:Q], ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- cache insert quantizers

def test_e4m3_code_matches_torch_cast_in_range():
    # round to nearest even on the OCP E4M3 grid, normals and subnormals, ties included
    rng = np.random.default_rng(30)
    v = (rng.standard_normal(100000) * np.exp2(rng.integers(-14, 9, 100000))).astype(np.float32)
    mids = (O.e4m3_value(np.arange(0, 126, dtype=np.uint8)) + O.e4m3_value(np.arange(1, 127, dtype=np.uint8))) / 2
    v = np.concatenate([v, mids.astype(np.float32), -mids.astype(np.float32), np.float32([0.0, -0.0])])
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_code(v), ref)


def test_e4m3_code_saturates():
    big = np.float32([448.0, 449.0, 464.0, 1e6, np.float32(3e38)])
    assert np.all(O.e4m3_code(big) == 0x7E)
    assert np.all(O.e4m3_code(-big) == 0xFE)


def test_e2m1_code_is_the_nearest_magnitude_ties_to_even():
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    grid = np.arange(-7.0, 7.0, 1.0 / 64, dtype=np.float32)
    got = O.e2m1_code(grid)
    for x, c in zip(grid, got):
        a = min(abs(float(x)), 6.0)
        d = np.abs(a - mags)
        near = np.flatnonzero(d == d.min())
        want = near[0] if len(near) == 1 else [n for n in near if n % 2 == 0][0]
        if x < 0 and want > 0:
            want |= 8
        assert c == want, (x, c, want)
    # the tie points of the OCP FP4 grid by hand
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for x, c in ties.items():
        assert O.e2m1_code(np.float32(x)) == c and O.e2m1_code(np.float32(-x)) == (c | 8 if c else 0)


def test_fp8_row_quantizer_scale_and_bound():
    rng = np.random.default_rng(31)
    x = (rng.standard_normal(128) * 0.3).astype(np.float32)
    codes, scale = O.quantize_fp8_row(x)
    amax = np.abs(x).max()
    assert scale == np.float32(amax / np.float32(448.0))
    back = O.e4m3_value(codes) * np.float64(scale)
    assert np.all(np.abs(back - x) <= np.maximum(np.abs(x) * 2.0 ** -4, float(scale) * 2.0 ** -10) * (1 + 1e-6))
    assert O.e4m3_value(codes[np.argmax(np.abs(x))]) in (448.0, -448.0)
    codes0, scale0 = O.quantize_fp8_row(np.zeros(128, np.float32))
    assert scale0 == 1.0 and np.all(codes0 == 0)


def test_nvfp4_row_quantizer_recovers_representable_rows():
    # x = e2m1 * e4m3 scale * g with a 6 in every group of 16: the quantizer must
    # give back exactly these codes (nibble order: element 2j low)
    rng = np.random.default_rng(32)
    g = np.float32(0.0078125)
    sf_codes = rng.integers(0x20, 0x60, size=8, dtype=np.uint8)
    nib = rng.integers(0, 16, size=128, dtype=np.uint8)
    nib[::16] = 7
    nib[(nib & 7) == 0] = 0  # +0 only
    x = (O.e2m1_value(nib) * np.repeat(O.e4m3_value(sf_codes), 16) * float(g)).astype(np.float32)
    packed, sf = O.quantize_nvfp4_row(x, g)
    assert np.array_equal(sf, sf_codes)
    assert np.array_equal(packed & 0xF, nib[0::2]) and np.array_equal(packed >> 4, nib[1::2])


def test_insert_writes_only_the_mapped_slots():
    rng = np.random.default_rng(33)
    H, D, nblk = 2, 128, 3
    for kv in ("bf16", "fp8", "nvfp4"):
        c = {"kv_dtype": kv, "index_dtype": kv, "k_global": 0.01, "v_global": 0.02, "idx_global": 0.005}
        for name, shape in (("k", (nblk, H, 128)), ("v", (nblk, H, 128)), ("idx", (nblk, 128))):
            if kv == "bf16":
                c[name] = rng.integers(0, 1 << 16, size=shape + (D,), dtype=np.uint16)
            elif kv == "fp8":
                c[name] = rng.integers(0, 256, size=shape + (D,), dtype=np.uint8)
                c[name + "_scale"] = rng.random(shape).astype(np.float32)
            else:
                c[name] = rng.integers(0, 256, size=shape + (D // 2,), dtype=np.uint8)
                c[name + "_sf"] = rng.integers(0, 256, size=shape + (D // 16,), dtype=np.uint8)
        before = {k2: v2.copy() for k2, v2 in c.items() if isinstance(v2, np.ndarray)}
        slots = np.array([5, -1, 130, 383])
        k = (rng.standard_normal((4, H, D)) * 0.1).astype(np.float32)
        v = (rng.standard_normal((4, H, D)) * 0.1).astype(np.float32)
        ik = (rng.standard_normal((4, D)) * 0.1).astype(np.float32)
        k, v, ik = (torch.from_numpy(a).bfloat16().float().numpy() for a in (k, v, ik))
        O.insert_tokens(c, slots, k, v, ik)
        touched = {(0, 5), (1, 2), (2, 127)}
        for name in ("k", "v", "idx"):
            for blk in range(nblk):
                for off in range(128):
                    same = np.array_equal(c[name][blk, ..., off, :] if name == "idx" else c[name][blk, :, off],
                                          before[name][blk, ..., off, :] if name == "idx" else before[name][blk, :, off])
                    assert same == ((blk, off) not in touched), (kv, name, blk, off)
        # the inserted values decode back within the format's bound
        t, (blk, off) = 3, (2, 127)
        for name, ref in (("k", k[t]), ("v", v[t])):
            if kv == "bf16":
                got = O.bf16_value(c[name][blk, :, off])
            else:
                got = O._dequant(kv, c[name][blk, :, off], scale=c.get(name + "_scale", np.ones((3, 2, 128)))[blk, :, off],
                                 sf=c.get(name + "_sf", np.zeros((3, 2, 128, 8), np.uint8))[blk, :, off],
                                 gscale=c[name + "_global"])
            tol = 0 if kv == "bf16" else (0.07 if kv == "fp8" else 0.3)
            assert np.abs(got - ref).max() <= tol * np.abs(ref).max() + 1e-12, (kv, name)


# ---------------------------------------------------------------- NVFP4 E4M3-product mode
# The Blackwell kernels dequantize NVFP4 with the product e2m1 x e4m3 rounded to
# E4M3 (Day-0 blog, "NVIDIA Blackwell 优化的 MSA 内核"); the oracle's "e4m3" mode
# must equal torch's float8 cast of that exact product (clamped to +-448, the
# saturating conversion), times the fp32 per-tensor scale afterwards.

_E2M1_OCP = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def _all_products_tile():
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]  # every non-NaN scale code
    nib = np.arange(16, dtype=np.uint8)
    packed = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)  # element 2j in the low nibble
    data = np.tile(packed, (len(codes), 1))                   # [codes][8]
    sf = np.array(codes, dtype=np.uint8)[:, None]              # one scale per 16 elements
    return codes, data, sf


@pytest.mark.parametrize("g", [1.0, 0.75, 3.0e-3])
def test_nvfp4_e4m3_product_mode_equals_torch_cast(g):
    codes, data, sf = _all_products_tile()
    got = O._dequant("nvfp4", data, sf=sf, gscale=g, nvfp4_mode="e4m3")
    sc = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double()
    prod = sc[:, None] * torch.tensor(_E2M1_OCP, dtype=torch.float64)[None, :]   # exact
    rounded = prod.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).double()
    ref = (rounded.float() * torch.tensor(g, dtype=torch.float32)).numpy()
    assert np.array_equal(got.view(np.uint32), ref.astype(np.float32).view(np.uint32))


def test_nvfp4_modes_differ_only_where_the_product_is_not_an_e4m3_value():
    codes, data, sf = _all_products_tile()
    exact = O._dequant("nvfp4", data, sf=sf, gscale=1.0)
    rnd = O._dequant("nvfp4", data, sf=sf, gscale=1.0, nvfp4_mode="e4m3")
    sc = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double()
    prod = (sc[:, None] * torch.tensor(_E2M1_OCP, dtype=torch.float64)[None, :]).numpy()
    representable = prod.clip(-448, 448) == torch.tensor(prod.clip(-448, 448)).to(torch.float8_e4m3fn).double().numpy()
    representable &= np.abs(prod) <= 448
    assert np.array_equal(exact[representable], rnd[representable])
    assert (exact[~representable] != rnd[~representable]).all()
    assert (~representable).sum() > 100  # the mode changes many products (e.g. 1.5 x 1.125)
    with pytest.raises(ValueError):
        O._dequant("nvfp4", data, sf=sf, gscale=1.0, nvfp4_mode="e5m2")
