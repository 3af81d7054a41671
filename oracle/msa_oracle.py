"""Plain CPU oracle of the MiniMax Sparse Attention (MSA) decode hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code, table or constant
generator with the CUDA library; the only thing both sides share is the seeded
input generator (``msa_synth``), which holds none of the method's arithmetic.

What it computes, in fp64 unless a step fixes another precision:

1. Cache decode (``dequant_kv_tile``, ``dequant_index_tile``) -- the fp32 value
   of every stored element.  BF16 widens exactly; FP8 E4M3 (OCP "FN" format,
   the KV dtype of "[M3] Enable FP8 sparse GQA", section "功能与动机") times its
   per-token fp32 scale with ONE fp32 rounding; NVFP4 (e2m1 values, one e4m3
   scale per 16 elements, one fp32 per-tensor scale: vLLM Day-0 blog, section
   "MiniMax-M3.1 架构中的新特性") as fp32(e2m1 * e4m3) * global, where the inner
   product is exact in fp32, again one rounding.
2. Index score (``index_scores``) -- vLLM Day-0 blog, section "MSA 入门": one
   index query per GQA group against the single shared index-key head, for
   every key of the context.  The scale applied is the one the model passes to
   its indexer (model.py docs, ``MiniMaxM3SparseAttention.__init__``:
   ``scale=self.scaling`` = head_dim ** -0.5).  Key t is visible to the query
   at position p iff t <= p (causal).
3. Block max-pool (``pool_blocks``) -- same section: the per-key scores are
   max-pooled to one score per 128-token block (``score_type="max"`` in the
   indexer constructor).  A block with no visible key pools to -inf.
4. Top-k blocks (``select_blocks``) -- same section: keep the top 16 blocks per
   group, the most recent block always kept.  Readings (the pages are silent):
   the query's own block is forced and counts as one of the k; equal pooled
   scores prefer the smaller block id; fewer visible blocks than k -> all of
   them, padded with -1; output ascending.  ``init_blocks``/``local_blocks``
   (indexer constructor arguments, default 0) force the first blocks and the
   blocks just before the query's block (reading of their names; parity
   unpinned for nonzero values).
5. Sparse attend (``attend``) -- same section and Figure 1: exact softmax
   attention for every query head of the group over only the selected
   blocks' visible keys, logits scaled by head_dim ** -0.5 (model.py docs,
   ``self.scaling``).  Query head h belongs to group h // (H_q / H_kv)
   (contiguous GQA convention of the model's KV-head sharding).  Also returns
   the log-sum-exp of the scaled logits.

Query i (0-based) of the Q new tokens of a sequence of T tokens sits at
position T - Q + i: the new tokens' keys are already in the cache when
attention runs (model.py docs, ``forward``: the cache insert precedes
``_run_attention``).
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

BLOCK = 128


# ----------------------------------------------------------------------------
# element decoding (bit fields)
# ----------------------------------------------------------------------------

def e4m3_value(codes) -> np.ndarray:
    """Decode OCP FP8 E4M3 ("FN": bias 7, no infinities, S.1111.111 = NaN)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = sign * (1.0 + m / 8.0) * np.exp2(e - 7.0)
    subnormal = sign * (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, subnormal, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def e2m1_value(nibbles) -> np.ndarray:
    """Decode FP4 E2M1 (bias 1, no inf/NaN): magnitudes 0,.5,1,1.5,2,3,4,6."""
    n = np.asarray(nibbles, dtype=np.uint8).astype(np.int64) & 0xF
    sign = np.where(n & 0x8, -1.0, 1.0)
    e = (n >> 1) & 0x3
    m = n & 0x1
    normal = (1.0 + m / 2.0) * np.exp2(e - 1.0)
    subnormal = m * 0.5
    return sign * np.where(e == 0, subnormal, normal)


def bf16_value(bits) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def unpack_e2m1(packed) -> np.ndarray:
    """Split packed bytes into nibbles; element 2j is the low nibble of byte j."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def nvfp4_product_exact(nibble: int, scale_code: int) -> Fraction:
    """Exact rational value of e2m1(nibble) * e4m3(scale_code) (pins only)."""
    return Fraction(float(e2m1_value(nibble))) * Fraction(float(e4m3_value(scale_code)))


# ----------------------------------------------------------------------------
# cache decode to fp32 (the values the whole path works on)
# ----------------------------------------------------------------------------

def _dequant(dtype, data, scale=None, sf=None, gscale=None, nvfp4_mode="exact") -> np.ndarray:
    if dtype == "bf16":
        return bf16_value(data)
    if dtype == "fp8":
        v = e4m3_value(data).astype(np.float32)
        return (v * np.asarray(scale, np.float32)[..., None]).astype(np.float32)
    if dtype == "nvfp4":
        vals = e2m1_value(unpack_e2m1(data))  # [..., D]
        sfv = e4m3_value(sf)  # [..., D/16]
        prod = (vals * np.repeat(sfv, 16, axis=-1)).astype(np.float32)  # exact
        if nvfp4_mode == "e4m3":
            # the product rounded to E4M3 first (nearest even, saturating), as
            # the Blackwell kernels' NVFP4 -> FP8 dequant does (Day-0 blog,
            # "NVIDIA Blackwell 优化的 MSA 内核")
            prod = e4m3_value(e4m3_code(prod)).astype(np.float32)
        elif nvfp4_mode != "exact":
            raise ValueError(nvfp4_mode)
        return (prod * np.float32(gscale)).astype(np.float32)
    raise ValueError(dtype)


def dequant_kv_tile(case: dict, which: str, phys: int) -> np.ndarray:
    """fp32 [H_kv][128][D] of the K (which='k') or V ('v') tile of one physical block."""
    w = case["workload"]
    dt = w.kv_dtype
    return _dequant(dt, case[which][phys],
                    case[which + "_scale"][phys] if dt == "fp8" else None,
                    case[which + "_sf"][phys] if dt == "nvfp4" else None,
                    case.get(which + "_global"), case.get("nvfp4_mode", "exact"))


def dequant_index_tile(case: dict, phys: int) -> np.ndarray:
    """fp32 [128][D_i] index keys of one physical block."""
    dt = case["workload"].index_dtype
    return _dequant(dt, case["idx"][phys],
                    case["idx_scale"][phys] if dt == "fp8" else None,
                    case["idx_sf"][phys] if dt == "nvfp4" else None,
                    case.get("idx_global"), case.get("nvfp4_mode", "exact"))


def query_values(data, dtype: str, scale: float) -> np.ndarray:
    """fp64 value of a stored query tensor (bf16 bits, or e4m3 codes x fp32 scale)."""
    if dtype == "bf16":
        return bf16_value(data).astype(np.float64)
    if dtype == "fp8":
        return (e4m3_value(data).astype(np.float32) * np.float32(scale)).astype(np.float64)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------
# the method
# ----------------------------------------------------------------------------

def positions(seq_len: int, q_per_seq: int) -> np.ndarray:
    return np.arange(seq_len - q_per_seq, seq_len)


def index_scores(key_rows: np.ndarray, iq: np.ndarray, pos: np.ndarray, scale: float) -> np.ndarray:
    """Scores of one sequence's keys.

    key_rows: fp32/fp64 [T][D_i] dequantized index keys in logical order.
    iq: fp64 [Q][G][D_i] index queries.  pos: [Q] query positions.
    Returns fp64 [Q][G][T]; invisible keys (t > pos) are -inf.
    """
    T = key_rows.shape[0]
    s = scale * np.einsum("qgd,td->qgt", iq, key_rows.astype(np.float64))
    visible = np.arange(T)[None, :] <= pos[:, None]  # [Q][T]
    return np.where(visible[:, None, :], s, -np.inf)


def pool_blocks(scores: np.ndarray, num_blocks: int) -> np.ndarray:
    """Max over each 128-token block of [..., T] scores -> [..., num_blocks]."""
    T = scores.shape[-1]
    out = np.full(scores.shape[:-1] + (num_blocks,), -np.inf)
    for b in range(num_blocks):
        lo, hi = b * BLOCK, min((b + 1) * BLOCK, T)
        if lo < hi:
            out[..., b] = scores[..., lo:hi].max(axis=-1)
    return out


def forced_blocks(pos: int, init_blocks: int = 0, local_blocks: int = 0) -> list:
    recent = pos // BLOCK
    forced = {recent}
    forced.update(b for b in range(min(init_blocks, recent + 1)))
    forced.update(b for b in range(max(0, recent - local_blocks), recent))
    return sorted(forced)


def select_blocks(pooled: np.ndarray, pos: int, topk: int,
                  init_blocks: int = 0, local_blocks: int = 0) -> np.ndarray:
    """Top-k block ids of one (query, group) row, ascending, -1 padded.

    pooled: [nb] pooled scores.  Candidates are the blocks before the query's
    own block; the forced set comes first, the rest are the highest pooled
    scores (ties -> smaller id).
    """
    recent = pos // BLOCK
    forced = forced_blocks(pos, init_blocks, local_blocks)[:topk]
    rest = [b for b in range(recent) if b not in forced]
    order = sorted(rest, key=lambda b: (-pooled[b], b))
    chosen = sorted(forced + order[: max(0, topk - len(forced))])
    out = np.full(topk, -1, dtype=np.int32)
    out[: len(chosen)] = chosen
    return out


def attend(q: np.ndarray, keys: np.ndarray, values: np.ndarray, sm_scale: float):
    """Exact softmax attention of one query head over the given keys.

    q: [D]; keys, values: [n][D].  Returns (o [D], lse)."""
    logits = sm_scale * (keys.astype(np.float64) @ q)
    m = logits.max()
    p = np.exp(logits - m)
    l = p.sum()
    o = (p[:, None] * values.astype(np.float64)).sum(axis=0) / l
    return o, m + math.log(l)


# ----------------------------------------------------------------------------
# whole-path drivers over a generated case
# ----------------------------------------------------------------------------

def seq_index_keys(case: dict, s: int, upto: int | None = None) -> np.ndarray:
    """Logical-order dequantized index keys [T][D_i] of sequence s."""
    T = int(case["seq_lens"][s]) if upto is None else upto
    nb = (T + BLOCK - 1) // BLOCK
    bt = case["block_table"][s]
    rows = np.concatenate([dequant_index_tile(case, int(bt[b])) for b in range(nb)], axis=0)
    return rows[:T]


def pooled_scores(case: dict, s: int, index_scale: float, rows=None, chunk: int = 64) -> np.ndarray:
    """Pooled indexer scores of sequence s: fp64 [len(rows)][G][max_blocks], -inf beyond.

    Scores every visible key of the sequence (index_scores), then max-pools
    them per 128-token block (pool_blocks); queries go ``chunk`` at a time
    only to bound memory."""
    w = case["workload"]
    T = int(case["seq_lens"][s])
    Q = w.q_per_seq
    rows = np.arange(Q) if rows is None else np.asarray(rows)
    iq = query_values(case["index_q"], w.q_dtype, case["index_q_scale"])[s * Q:(s + 1) * Q]
    pos = positions(T, Q)
    keys = seq_index_keys(case, s)
    out = np.empty((len(rows), w.num_kv_heads, w.max_blocks))
    for c0 in range(0, len(rows), chunk):
        sel = rows[c0:c0 + chunk]
        sc = index_scores(keys, iq[sel], pos[sel], index_scale)
        out[c0:c0 + chunk] = pool_blocks(sc, w.max_blocks)
    return out


def select_all(case: dict, pooled_rows, topk: int, init_blocks: int = 0, local_blocks: int = 0) -> np.ndarray:
    """Selections [S*Q][G][topk] from pooled rows [S*Q][G][max_blocks]."""
    w = case["workload"]
    Q = w.q_per_seq
    out = np.full((w.num_seqs * Q, w.num_kv_heads, topk), -1, dtype=np.int32)
    for s in range(w.num_seqs):
        T = int(case["seq_lens"][s])
        for i, p in enumerate(positions(T, Q)):
            for g in range(w.num_kv_heads):
                out[s * Q + i, g] = select_blocks(pooled_rows[s * Q + i, g], int(p), topk,
                                                  init_blocks, local_blocks)
    return out


def attend_rows(case: dict, s: int, selection, sm_scale: float, rows=None):
    """Attention output of sequence s given a selection [S*Q][G][k].

    Returns (o fp64 [Q][H_q][D], lse fp64 [Q][H_q]) for the query indices in
    ``rows`` (default: all Q)."""
    w = case["workload"]
    T = int(case["seq_lens"][s])
    Q, G, Hq = w.q_per_seq, w.num_kv_heads, w.num_q_heads
    r = Hq // G
    qv = query_values(case["q"], w.q_dtype, case["q_scale"])[s * Q:(s + 1) * Q]
    pos = positions(T, Q)
    bt = case["block_table"][s]
    rows = range(Q) if rows is None else rows
    o = np.zeros((len(rows), Hq, w.head_dim))
    lse = np.zeros((len(rows), Hq))
    tiles = {}
    for ri, i in enumerate(rows):
        for g in range(G):
            blocks = [int(b) for b in selection[s * Q + i, g] if b >= 0]
            ks, vs = [], []
            for b in blocks:
                if b not in tiles:
                    phys = int(bt[b])
                    tiles[b] = (dequant_kv_tile(case, "k", phys), dequant_kv_tile(case, "v", phys))
                n = min(BLOCK, int(pos[i]) + 1 - b * BLOCK)  # visible keys of block b
                ks.append(tiles[b][0][g, :n])
                vs.append(tiles[b][1][g, :n])
            K = np.concatenate(ks, axis=0)
            V = np.concatenate(vs, axis=0)
            for h in range(g * r, (g + 1) * r):
                o[ri, h], lse[ri, h] = attend(qv[i, h], K, V, sm_scale)
    return o, lse


def run_path(case: dict, topk=None, index_scale=None, sm_scale=None,
             init_blocks=0, local_blocks=0, seqs=None):
    """Whole path for the sequences in ``seqs``: pooled, selection, out, lse."""
    w = case["workload"]
    topk = w.topk if topk is None else topk
    index_scale = w.index_dim ** -0.5 if index_scale is None else index_scale
    sm_scale = w.head_dim ** -0.5 if sm_scale is None else sm_scale
    seqs = range(w.num_seqs) if seqs is None else seqs
    Q = w.q_per_seq
    pooled = np.full((w.num_seqs * Q, w.num_kv_heads, w.max_blocks), -np.inf)
    for s in seqs:
        pooled[s * Q:(s + 1) * Q] = pooled_scores(case, s, index_scale)
    sel = np.full((w.num_seqs * Q, w.num_kv_heads, topk), -1, dtype=np.int32)
    for s in seqs:
        T = int(case["seq_lens"][s])
        for i, p in enumerate(positions(T, Q)):
            for g in range(w.num_kv_heads):
                sel[s * Q + i, g] = select_blocks(pooled[s * Q + i, g], int(p), topk,
                                                  init_blocks, local_blocks)
    out = np.zeros((w.num_seqs * Q, w.num_q_heads, w.head_dim))
    lse = np.zeros((w.num_seqs * Q, w.num_q_heads))
    for s in seqs:
        o, l = attend_rows(case, s, sel, sm_scale)
        out[s * Q:(s + 1) * Q], lse[s * Q:(s + 1) * Q] = o, l
    return dict(pooled=pooled, topk=sel, out=out, lse=lse)


# ----------------------------------------------------------------------------
# cache insert (the step before the path): quantization of new tokens
# ----------------------------------------------------------------------------
#
# vLLM Day-0 blog, section "QKV GEMM + norm + RoPE + KV 插入融合": the K, V and
# index key of each new token are quantized and written straight into their
# paged caches; "[M3] Enable FP8 sparse GQA" (items 1 and 4): the FP8 path
# stores quantized values through the slot mapping.  Readings (the pages give
# no formula): FP8 uses one fp32 scale per (token, head) row, amax / 448 (1 for
# an all-zero row), and the codes round x / scale to nearest even, saturating at
# +-448; NVFP4 uses the cache's fp32 per-tensor scale g (calibrated, given), an
# e4m3 scale per 16 elements rounding amax16 / (6 g) to nearest even, and e2m1
# codes rounding x / (scale * g) to nearest even, saturating at +-6, with a
# value that rounds to zero stored as +0.  Every division and product is one
# fp32 operation, as written.

E4M3_MAX = 448.0
E2M1_MAGS = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e4m3_code(v) -> np.ndarray:
    """OCP E4M3 code of fp32 values, round to nearest even, saturating at +-448.

    The grid: 3 fraction bits; exponent floor(log2 |v|) for normals (>= 2^-6),
    quantum 2^-9 below 2^-6 (subnormals).  The sign is kept (a negative value
    that rounds to zero gives 0x80).
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    quantum = np.exp2(e - 3.0)
    q = a / quantum                      # exact (power-of-two quantum)
    r = np.floor(q)
    frac = q - r
    r = np.where((frac > 0.5) | ((frac == 0.5) & (np.mod(r, 2) == 1)), r + 1, r)
    mag = np.minimum(r * quantum, E4M3_MAX)
    # bits of the rounded magnitude
    ee = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
    normal = mag >= 2.0 ** -6
    exp_field = np.where(normal, ee + 7, 0).astype(np.int64)
    man = np.where(normal, mag / np.exp2(ee) - 1.0, mag / 2.0 ** -9)
    man_field = np.where(normal, np.round(man * 8), np.round(man)).astype(np.int64)
    code = (exp_field << 3) | man_field
    code = np.where(mag == 0, 0, code)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def e2m1_code(v) -> np.ndarray:
    """FP4 E2M1 nibble of fp32 values: the nearest of 0, .5, 1, 1.5, 2, 3, 4, 6
    (equal distance: the even code), saturating at 6; zero is stored as +0."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), 6.0)
    mags = np.array(E2M1_MAGS)
    d = np.abs(a[..., None] - mags)                     # distance to every magnitude
    best = d.min(axis=-1, keepdims=True)
    tie = d == best
    # among the nearest codes take the even one (there are at most two)
    even = tie & (np.arange(8) % 2 == 0)
    code = np.where(even.any(axis=-1), even.argmax(axis=-1), tie.argmax(axis=-1))
    return (code | np.where((v < 0) & (code > 0), 8, 0)).astype(np.uint8)


def quantize_fp8_row(x):
    """(codes uint8 [D], fp32 scale) of one bf16/fp32 row: scale = amax / 448."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.abs(x).max())
    scale = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
    return e4m3_code((x / scale).astype(np.float32)), scale


def quantize_nvfp4_row(x, gscale: float):
    """(packed uint8 [D/2], e4m3 scale codes [D/16]) of one row with the given
    fp32 per-tensor scale; element 2j in the low nibble of byte j."""
    x = np.asarray(x, dtype=np.float32).reshape(-1, 16)
    g = np.float32(gscale)
    amax16 = np.abs(x).max(axis=1).astype(np.float32)
    six_g = np.float32(np.float32(6.0) * g)
    sf = e4m3_code((amax16 / six_g).astype(np.float32))
    sfv = e4m3_value(sf).astype(np.float32)
    denom = (sfv * g).astype(np.float32)
    safe = np.where(denom > 0, denom, np.float32(1.0))
    vals = np.where(denom[:, None] > 0, (x / safe[:, None]).astype(np.float32), np.float32(0.0))
    nib = e2m1_code(vals).reshape(-1)
    return (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8), sf


def insert_tokens(cache: dict, slots, k, v, index_k):
    """Apply the insert of new tokens to a host copy of the caches (in place).

    cache: dict with kv_dtype, index_dtype, and the arrays of the layout (k, v,
    k_scale / k_sf, ..., idx, idx_scale / idx_sf) plus k_global, v_global,
    idx_global.  slots[t] = physical block * 128 + offset (negative: skipped).
    k, v: float32 [T][H][D] (bf16 values); index_k: float32 [T][Di] or None."""
    for t, slot in enumerate(np.asarray(slots)):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), BLOCK)
        for name, rows in (("k", k), ("v", v)):
            dt = cache["kv_dtype"]
            for h in range(rows.shape[1]):
                _put_row(cache, name, dt, (blk, h, off), rows[t, h])
        if index_k is not None:
            _put_row(cache, "idx", cache["index_dtype"], (blk, off), index_k[t])


def _put_row(cache, name, dt, where, row):
    if dt == "bf16":
        cache[name][where] = (np.asarray(row, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    elif dt == "fp8":
        codes, scale = quantize_fp8_row(row)
        cache[name][where] = codes
        cache[name + "_scale"][where] = scale
    elif dt == "nvfp4":
        packed, sf = quantize_nvfp4_row(row, cache[name + "_global"])
        cache[name][where] = packed
        cache[name + "_sf"][where] = sf
    else:
        raise ValueError(dt)
