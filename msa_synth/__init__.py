"""Seeded synthetic inputs for the MSA decode hot path.

This module is shared by the tests, the benchmark and the oracle checks.  It
holds no step of the method itself (no scoring, pooling, selection or
attention): it only draws random values, plants "hot" blocks, quantizes the
draws into the paged-cache byte layout the library reads, and shuffles the
physical block table.

Workloads (names describe the shapes; see ``WORKLOADS``):

* ``tiny_bf16``      1 seq x 4,096 tokens, 1 query token, BF16 everything.
* ``fp8_decode``     32 seqs, context ~U{16K..32K}, 1 query token, FP8 E4M3
                     K/V/index keys with per-token fp32 scales, bf16 queries,
                     shuffled physical block table.
* ``nvfp4_verify``   8 seqs x 128K, 8 query tokens each (speculative verify),
                     NVFP4 K/V/index keys, E4M3 queries with per-tensor scale.
* ``fp8_long``       4 seqs x 512K (4,096 blocks), 1 query token, FP8.
* ``fp8_prefill``    1 seq, 8,192 new tokens on a 64K FP8 context, bf16 q.

All value tensors are N(0,1)/sqrt(128).  For every (sequence, group), 3
distinct blocks (never the last one) get their index keys shifted by +0.5
along the unit direction of that group's index query (the mean over the
sequence's query tokens, normalised).  Tokens of the last block beyond the
sequence length are filled with large garbage aligned with the index queries,
so a kernel that forgets to mask them produces visibly wrong scores.

Layouts (one physical block = 128 tokens):

* K, V       ``[num_blocks][H_kv][128][D]``  bf16 / e4m3 bytes, or
             ``[num_blocks][H_kv][128][D/2]`` packed e2m1 (element 2j in the
             low nibble of byte j) with e4m3 scales ``[num_blocks][H_kv][128][D/16]``
* FP8 scales ``[num_blocks][H_kv][128]`` fp32 (K and V), ``[num_blocks][128]`` (index)
* index keys ``[num_blocks][128][D_i]`` (one shared index-key head), same dtypes
* NVFP4 per-tensor fp32 scales for K, V and index keys.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BLOCK = 128
FP8_MAX = 448.0
E2M1_MAX = 6.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_seqs: int
    seq_lens: tuple  # total tokens per sequence, new query tokens included
    q_per_seq: int
    kv_dtype: str  # "bf16" | "fp8" | "nvfp4"
    index_dtype: str
    q_dtype: str  # "bf16" | "fp8"
    topk: int = 16
    num_q_heads: int = 16
    num_kv_heads: int = 4
    head_dim: int = 128
    index_dim: int = 128
    seed: int = 0
    hot_blocks: int = 3
    spare_blocks: int = 3  # unused physical blocks in the pool

    @property
    def max_blocks(self) -> int:
        return max((t + BLOCK - 1) // BLOCK for t in self.seq_lens)

    @property
    def num_blocks_used(self) -> int:
        return sum((t + BLOCK - 1) // BLOCK for t in self.seq_lens)


def _fp8_decode_lens(seed: int, n: int, lo: int, hi: int) -> tuple:
    rng = np.random.default_rng(seed + 1000)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=n))


def make_workload(name: str, **over) -> Workload:
    """Build one of the named workloads; keyword overrides shrink it for tests."""
    if name == "tiny_bf16":
        w = Workload(name, 1, (4096,), 1, "bf16", "bf16", "bf16", seed=0)
    elif name == "fp8_decode":
        w = Workload(name, 32, _fp8_decode_lens(1, 32, 16384, 32768), 1,
                     "fp8", "fp8", "bf16", seed=1)
    elif name == "nvfp4_verify":
        w = Workload(name, 8, (131072,) * 8, 8, "nvfp4", "nvfp4", "fp8", seed=2)
    elif name == "fp8_long":
        w = Workload(name, 4, (524288,) * 4, 1, "fp8", "fp8", "bf16", seed=3)
    elif name == "fp8_prefill":
        w = Workload(name, 1, (65536 + 8192,), 8192, "fp8", "fp8", "bf16", seed=4)
    else:
        raise KeyError(name)
    if over:
        if "seq_lens" in over:
            over["seq_lens"] = tuple(int(t) for t in over["seq_lens"])
            over.setdefault("num_seqs", len(over["seq_lens"]))
        w = dataclasses.replace(w, **over)
    assert len(w.seq_lens) == w.num_seqs
    assert all(t >= w.q_per_seq for t in w.seq_lens)
    return w


WORKLOADS = ("tiny_bf16", "fp8_decode", "nvfp4_verify", "fp8_long", "fp8_prefill")


# ----------------------------------------------------------------------------
# quantizers (input construction only)
# ----------------------------------------------------------------------------

def quantize_fp8_rows(x: torch.Tensor):
    """Per-row (last dim) E4M3 quantization: scale = amax/448, RN-even, clamped."""
    amax = x.abs().amax(dim=-1, keepdim=True).float()
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    codes = (x.float() / scale).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8), scale.squeeze(-1).contiguous()


def quantize_fp8_tensor(x: torch.Tensor):
    """Per-tensor E4M3 quantization: scale = amax/448."""
    amax = float(x.abs().max())
    scale = amax / FP8_MAX if amax > 0 else 1.0
    scale = float(np.float32(scale))
    codes = (x.float() / scale).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8), scale


def _e2m1_encode(v: torch.Tensor) -> torch.Tensor:
    """Round |v| to the nearest e2m1 magnitude (ties to the even code), add sign."""
    m = v.abs()
    code = torch.zeros(v.shape, dtype=torch.uint8, device=v.device)
    # thresholds between consecutive magnitudes {0,.5,1,1.5,2,3,4,6};
    # at a midpoint the even code wins, so for odd targets the bound is strict.
    bounds = [(0.25, False), (0.75, True), (1.25, False), (1.75, True),
              (2.5, False), (3.5, True), (5.0, False)]
    for b, inclusive in bounds:
        code += (m >= b).to(torch.uint8) if inclusive else (m > b).to(torch.uint8)
    sign = ((v < 0) & (code > 0)).to(torch.uint8) << 3
    return code | sign


def quantize_nvfp4(x: torch.Tensor, global_scale: Optional[float] = None):
    """NVFP4: fp32 per-tensor scale, e4m3 scale per 16 elements, e2m1 values.

    Returns (packed bytes [..., D/2], scale codes [..., D/16], global scale).
    """
    d = x.shape[-1]
    assert d % 16 == 0
    if global_scale is None:
        amax = float(x.abs().max())
        global_scale = amax / (E2M1_MAX * FP8_MAX) if amax > 0 else 1.0
    global_scale = float(np.float32(global_scale))
    g = x.float().reshape(*x.shape[:-1], d // 16, 16)
    amax16 = g.abs().amax(dim=-1)
    sf = (amax16 / (E2M1_MAX * global_scale)).clamp(0, FP8_MAX).to(torch.float8_e4m3fn)
    sf_val = sf.float()
    denom = (sf_val * global_scale).unsqueeze(-1)
    vals = torch.where(denom > 0, g / torch.where(denom > 0, denom, torch.ones_like(denom)),
                       torch.zeros_like(g))
    codes = _e2m1_encode(vals.clamp(-E2M1_MAX, E2M1_MAX)).reshape(*x.shape[:-1], d)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    return packed.contiguous(), sf.view(torch.uint8).contiguous(), global_scale


# ----------------------------------------------------------------------------
# the case generator
# ----------------------------------------------------------------------------

def _randn(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) / math.sqrt(128.0)


def make_case(w: Workload, device="cpu") -> dict:
    """Generate every input of one workload on ``device`` (seeded by ``w.seed``).

    Values come from a torch generator on ``device``; structure (block table,
    hot blocks) from numpy, so it is identical on every device.
    """
    device = torch.device(device)
    rng = np.random.default_rng(w.seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    S, Q, G, Hq = w.num_seqs, w.q_per_seq, w.num_kv_heads, w.num_q_heads
    D, Di = w.head_dim, w.index_dim
    nbs = [(t + BLOCK - 1) // BLOCK for t in w.seq_lens]
    max_nb = max(nbs)
    num_blocks = sum(nbs) + w.spare_blocks
    perm = rng.permutation(num_blocks)
    block_table = np.zeros((S, max_nb), dtype=np.int32)
    off = 0
    for s, nb in enumerate(nbs):
        block_table[s, :nb] = perm[off:off + nb]
        off += nb
    hot = np.full((S, G, w.hot_blocks), -1, dtype=np.int32)
    for s, nb in enumerate(nbs):
        cand = nb - 1
        for g in range(G):
            k = min(w.hot_blocks, cand)
            if k > 0:
                hot[s, g, :k] = np.sort(rng.choice(cand, size=k, replace=False))

    # queries
    iq = _randn((S * Q, G, Di), gen, device)
    q = _randn((S * Q, Hq, D), gen, device)

    # index keys, physical layout [num_blocks][B][Di]
    ik = _randn((num_blocks, BLOCK, Di), gen, device)
    iq_dir = iq.reshape(S, Q, G, Di).mean(dim=1)
    iq_dir = iq_dir / iq_dir.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    bt_dev = torch.from_numpy(block_table).to(device=device, dtype=torch.long)
    for s, nb in enumerate(nbs):
        for g in range(G):
            for b in hot[s, g]:
                if b >= 0:
                    ik[bt_dev[s, int(b)]] += 0.5 * iq_dir[s, g]
        tail = w.seq_lens[s] - (nb - 1) * BLOCK
        if tail < BLOCK:  # garbage past the end of the sequence
            ik[bt_dev[s, nb - 1], tail:] = 4.0 * iq_dir[s].sum(dim=0)
    k = _randn((num_blocks, G, BLOCK, D), gen, device)
    v = _randn((num_blocks, G, BLOCK, D), gen, device)
    for s, nb in enumerate(nbs):
        tail = w.seq_lens[s] - (nb - 1) * BLOCK
        if tail < BLOCK:
            k[bt_dev[s, nb - 1], :, tail:] *= 16.0
            v[bt_dev[s, nb - 1], :, tail:] = 30.0

    case = dict(workload=w, num_blocks=num_blocks,
                seq_lens=torch.tensor(w.seq_lens, dtype=torch.int32, device=device),
                block_table=torch.from_numpy(block_table).to(device),
                hot=hot)

    def put_cache(prefix, x):
        dt = w.index_dtype if prefix == "idx" else w.kv_dtype
        if dt == "bf16":
            case[prefix] = x.to(torch.bfloat16).contiguous()
        elif dt == "fp8":
            codes, scale = quantize_fp8_rows(x)
            case[prefix] = codes.contiguous()
            case[prefix + "_scale"] = scale
        elif dt == "nvfp4":
            packed, sf, gscale = quantize_nvfp4(x)
            case[prefix] = packed
            case[prefix + "_sf"] = sf
            case[prefix + "_global"] = gscale
        else:
            raise ValueError(dt)

    put_cache("idx", ik)
    del ik
    put_cache("k", k)
    del k
    put_cache("v", v)
    del v

    if w.q_dtype == "bf16":
        case["index_q"], case["index_q_scale"] = iq.to(torch.bfloat16).contiguous(), 1.0
        case["q"], case["q_scale"] = q.to(torch.bfloat16).contiguous(), 1.0
    elif w.q_dtype == "fp8":
        case["index_q"], case["index_q_scale"] = quantize_fp8_tensor(iq)
        case["q"], case["q_scale"] = quantize_fp8_tensor(q)
    else:
        raise ValueError(w.q_dtype)
    return case


def case_to_host(case: dict) -> dict:
    """Copy every tensor of a case to host numpy arrays (bf16 kept as uint16 bits)."""
    out = {}
    for key, val in case.items():
        if isinstance(val, torch.Tensor):
            t = val.detach().cpu()
            if t.dtype == torch.bfloat16:
                out[key] = t.view(torch.int16).numpy().view(np.uint16)
            else:
                out[key] = t.numpy()
        else:
            out[key] = val
    return out
