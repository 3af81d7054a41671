"""NVFP4 caches in the E4M3-product mode (MSA_NVFP4_E4M3_PRODUCT): every NVFP4
element is fp32(E4M3(e2m1 x e4m3 scale)) x the per-tensor scale, as the Blackwell
kernels' NVFP4 -> FP8 dequant computes it (vLLM Day-0 blog, "NVIDIA Blackwell 优化的
MSA 内核").  The CUDA path against the oracle run in the same mode, on the same
bytes.
"""

import numpy as np
import pytest
import torch

import block_sparse_attention_03_gb300 as msa
import msa_synth as ms
from oracle import msa_oracle as O

from _helpers import bind, check_out, check_pooled, check_selection, gpu_path

pytestmark = pytest.mark.gpu


def _case(name, mode, **over):
    w = ms.make_workload(name, **over)
    c = ms.make_case(w, device="cuda")
    c["nvfp4_mode"] = mode
    return w, c, ms.case_to_host(c)


def _dequant_all(c, w):
    cache, _, _, _ = bind(c)
    phys = torch.arange(c["num_blocks"], dtype=torch.int32, device="cuda")
    got = []
    for which in (0, 1, 2):
        heads = 1 if which == 2 else w.num_kv_heads
        out = torch.empty((c["num_blocks"], heads, 128, 128), dtype=torch.float32, device="cuda")
        msa.msa_dequant_debug(cache, which, phys, out)
        got.append(out.cpu().numpy())
    return got


def test_dequant_bit_exact_in_e4m3_mode():
    w, c, h = _case("tiny_bf16", "e4m3", seq_lens=(700, 300), kv_dtype="nvfp4", index_dtype="nvfp4", seed=31)
    got = _dequant_all(c, w)
    for which in (0, 1, 2):
        for i in range(c["num_blocks"]):
            ref = O.dequant_index_tile(h, i)[None] if which == 2 else O.dequant_kv_tile(h, "kv"[which], i)
            assert np.array_equal(got[which][i].view(np.uint32), ref.astype(np.float32).view(np.uint32)), (which, i)
    # the mode is in effect: the same bytes decode differently in the exact mode
    c["nvfp4_mode"] = "exact"
    exact = _dequant_all(c, w)
    assert any((exact[k] != got[k]).any() for k in range(3))


@pytest.mark.parametrize("name,over", [
    ("nvfp4_verify", dict(seq_lens=(5000, 3000), seed=32)),
    ("tiny_bf16", dict(seq_lens=(2000, 1500), kv_dtype="nvfp4", index_dtype="nvfp4", q_dtype="fp8", seed=33)),
])
@pytest.mark.parametrize("fused", [False, True])
def test_path_matches_oracle_in_e4m3_mode(name, over, fused):
    w, c, h = _case(name, "e4m3", **over)
    g = gpu_path(c, fused=fused)
    ref = O.run_path(h, topk=w.topk)
    if not fused:
        check_pooled(g["pooled"], ref["pooled"])
    check_selection(g["topk"], ref["pooled"], w.seq_lens, w.q_per_seq, w.topk)
    out = np.zeros_like(ref["out"])
    for s in range(w.num_seqs):  # the oracle's attend on the GPU's own selection
        o, _ = O.attend_rows(h, s, g["topk"], w.head_dim ** -0.5)
        out[s * w.q_per_seq:(s + 1) * w.q_per_seq] = o
    check_out(g["out"], out)
