"""Host-side checks of the C ABI library: it builds, loads, exports every
symbol include/msa.h declares, and rejects bad arguments before touching the
GPU (no compute call is made here)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_attention_03_gb300 import _build
    import block_sparse_attention_03_gb300 as msa
    _build.build()
    return msa.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "msa.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_path(lib):
    names = declared_functions()
    for want in ("msa_indexer_score", "msa_topk_blocks", "msa_sparse_attend", "msa_decode",
                 "msa_workspace_size", "msa_read_device_status", "msa_status_string", "msa_dequant_debug"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    import block_sparse_attention_03_gb300 as msa
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(msa.EXPORTS)


def test_status_strings(lib):
    import block_sparse_attention_03_gb300 as msa
    for code, name in msa.STATUS_NAMES.items():
        assert msa.msa_status_string(code) == name


def _structs(**over):
    import block_sparse_attention_03_gb300 as msa
    c = msa.MsaCacheT(1, 1, 100, 128, 4, 128, 128, 16, 32, None, None, 48, 64, 80, None, 96, 0, 0, 0)
    b = msa.MsaBatchT(2, 1, 50, 16, 32)
    f = msa.MsaConfigT(16, 0, 0, 128 ** -0.5, 128 ** -0.5, 0)
    for k, v in over.items():
        obj, field = k.split("__")
        setattr({"c": c, "b": b, "f": f}[obj], field, v)
    return c, b, f


def test_workspace_size_host_only(lib):
    c, b, f = _structs()
    n = lib.msa_workspace_size(ctypes.byref(c), ctypes.byref(b), ctypes.byref(f), 16)
    assert n > 0
    assert lib.msa_workspace_size(ctypes.byref(c), ctypes.byref(b), ctypes.byref(f), 15) == 0
    for over in ({"f__topk": 12}, {"f__score_type": 1}, {"f__score_type": -1}, {"c__block_size": 64}, {"c__head_dim": 64}, {"b__num_seqs": 0},
                 {"f__init_blocks": 16}, {"b__q_per_seq": 50 * 128 + 1}, {"c__num_kv_heads": 9},
                 {"c__nvfp4_mode": 2}, {"c__nvfp4_mode": -1}, {"f__prefill_select": 2},
                 {"f__prefill_select": -1}):
        c2, b2, f2 = _structs(**over)
        assert lib.msa_workspace_size(ctypes.byref(c2), ctypes.byref(b2), ctypes.byref(f2), 16) == 0, over
    # more sequences or blocks never shrink the workspace
    # both NVFP4 modes are valid descriptions
    c4, b4, f4 = _structs(c__nvfp4_mode=1)
    assert lib.msa_workspace_size(ctypes.byref(c4), ctypes.byref(b4), ctypes.byref(f4), 16) == n
    c3, b3, f3 = _structs(b__num_seqs=8, b__max_blocks_per_seq=500)
    assert lib.msa_workspace_size(ctypes.byref(c3), ctypes.byref(b3), ctypes.byref(f3), 16) > n


def test_bad_arguments_rejected_before_launch(lib):
    import block_sparse_attention_03_gb300 as msa
    c, b, f = _structs()
    q = msa.MsaQueryT(16, 0, 1.0)
    ws = ctypes.c_void_p(4096)
    # null pointers
    assert lib.msa_indexer_score(None, ctypes.byref(b), ctypes.byref(f), ctypes.byref(q), 16, ws, 1 << 20, None) == 1
    assert lib.msa_decode(ctypes.byref(c), ctypes.byref(b), ctypes.byref(f), ctypes.byref(q), ctypes.byref(q), 16,
                          None, 16, None, ws, 1 << 20, None) == 1
    assert lib.msa_workspace_init(None, 1024, None) == 1
    assert lib.msa_read_device_status(None, None, None) == 1
    assert lib.msa_dequant_debug(ctypes.byref(c), 5, 16, 1, 16, None) == 1
    # unsupported settings
    c2, b2, f2 = _structs(f__topk=12)
    assert lib.msa_topk_blocks(ctypes.byref(b2), ctypes.byref(f2), 4, 16, 16, None, ws, 1 << 20, None) == 2
    # misaligned base pointer
    c3, _, _ = _structs(c__k=17)
    assert lib.msa_sparse_attend(ctypes.byref(c3), ctypes.byref(b), ctypes.byref(f), ctypes.byref(q), 16, 16, 16,
                                 None, ws, 1 << 20, None) == 1
    # a workspace that is too small
    assert lib.msa_decode(ctypes.byref(c), ctypes.byref(b), ctypes.byref(f), ctypes.byref(q), ctypes.byref(q), 16,
                          16, 16, None, ws, 300, None) == 3
    # cache insert: null slot mapping, misaligned rows
    assert lib.msa_cache_insert(ctypes.byref(c), 4, None, 16, 32, None, ws, 1 << 20, None) == 1
    assert lib.msa_cache_insert(ctypes.byref(c), 4, 16, 17, 32, None, ws, 1 << 20, None) == 1
    assert lib.msa_cache_insert(ctypes.byref(c), 4, 16, 16, 32, None, ws, 100, None) == 3
    assert lib.msa_cache_insert(ctypes.byref(c), 0, None, None, None, None, ws, 1 << 20, None) == 0
    # e4m3 query without a scale
    qbad = msa.MsaQueryT(16, 1, 0.0)
    assert lib.msa_indexer_score(ctypes.byref(c), ctypes.byref(b), ctypes.byref(f), ctypes.byref(qbad), 16, ws,
                                 1 << 20, None) == 1


def test_prefill_workspace_holds_the_partials(lib):
    # a prefill chunk over an FP8 cache keeps one partial (fp16 o / l, fp32 m and l)
    # per (token, q head, selected block): 8,192 tokens x 16 heads x 16 -> >= 554 MB
    c, b, f = _structs(b__num_seqs=1, b__q_per_seq=8192, b__max_blocks_per_seq=576, c__num_blocks=600)
    n = lib.msa_workspace_size(ctypes.byref(c), ctypes.byref(b), ctypes.byref(f), 16)
    assert n >= 8192 * 16 * 16 * (128 * 2 + 2 * 4)
    # the same chunk over an NVFP4 cache attends per token: no such partials
    c2, b2, f2 = _structs(b__num_seqs=1, b__q_per_seq=8192, b__max_blocks_per_seq=576, c__num_blocks=600,
                          c__kv_dtype=2)
    assert 0 < lib.msa_workspace_size(ctypes.byref(c2), ctypes.byref(b2), ctypes.byref(f2), 16) < n


def test_prefill_select_in_indexer_needs_no_pooled_scores(lib):
    # a prefill chunk (2048 new tokens on 256K keys, FP8 caches): selecting in
    # the indexer's epilogue replaces the pooled scores (2048 x 4 groups x 2048
    # blocks x 4 B = 64 MiB) with candidate lists of a fixed size per query tile
    import block_sparse_attention_03_gb300 as msa
    big = dict(b__num_seqs=1, b__q_per_seq=2048, b__max_blocks_per_seq=2048, c__num_blocks=4096)
    c, b, f = _structs(**big)
    topk_ws = lib.msa_workspace_size(ctypes.byref(c), ctypes.byref(b), ctypes.byref(f), 16)
    c, b, f = _structs(f__prefill_select=1, **big)
    lists_ws = lib.msa_workspace_size(ctypes.byref(c), ctypes.byref(b), ctypes.byref(f), 16)
    # 64 MiB of pooled scores against (64 tiles + at most 148-152 CTAs) x 64 KiB of lists
    assert 0 < lists_ws <= topk_ws - (64 << 20) + 216 * (64 << 10)
    # topk 32 keeps the top-k launch (the lists hold 16 blocks a thread)
    c, b, f = _structs(f__prefill_select=1, f__topk=32, **big)
    c2, b2, f2 = _structs(f__topk=32, **big)
    assert lib.msa_workspace_size(ctypes.byref(c), ctypes.byref(b), ctypes.byref(f), 16) == \
        lib.msa_workspace_size(ctypes.byref(c2), ctypes.byref(b2), ctypes.byref(f2), 16)
    assert msa.Config(prefill_select="indexer").struct().prefill_select == 1
    assert msa.Config().struct().prefill_select == 0
    assert msa.Config(prefill_select="other").struct().prefill_select == -1


def test_score_type_other_than_max_is_unsupported(lib):
    # the pages define only the "max" block pooling (the indexer's default
    # score_type); any other value is refused before a launch
    import block_sparse_attention_03_gb300 as msa
    c, b, f = _structs(f__score_type=1)
    q = msa.MsaQueryT(16, 0, 1.0)
    ws = ctypes.c_void_p(4096)
    assert lib.msa_indexer_score(ctypes.byref(c), ctypes.byref(b), ctypes.byref(f), ctypes.byref(q), 16, ws,
                                 1 << 20, None) == 2
    assert lib.msa_decode(ctypes.byref(c), ctypes.byref(b), ctypes.byref(f), ctypes.byref(q), ctypes.byref(q), 16,
                          16, 16, None, ws, 1 << 20, None) == 2
    assert msa.Config(score_type="mean").struct().score_type == -1
    assert msa.Config().struct().score_type == 0
