"""GB300-native MiniMax Sparse Attention (MSA) decode hot path.

Thin Python binding over the C ABI of ``libmsa.so`` (declared in
``include/msa.h``): every function here only marshals arguments (torch tensors
-> device pointers, the current CUDA stream) and raises on a non-OK status.
All computation runs in the library's CUDA kernels; there is no fallback.
"""

from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

from . import roofline  # noqa: F401  (host-side byte model)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmsa.so")

MSA_OK = 0
STATUS_NAMES = {0: "MSA_OK", 1: "MSA_ERR_INVALID_ARGUMENT", 2: "MSA_ERR_UNSUPPORTED",
                3: "MSA_ERR_WORKSPACE_TOO_SMALL", 4: "MSA_ERR_CUDA", 5: "MSA_ERR_DEVICE_FAULT",
                6: "MSA_ERR_TIMEOUT"}
DTYPES = {"bf16": 0, "fp8": 1, "nvfp4": 2}

# every symbol include/msa.h declares
EXPORTS = ("msa_workspace_size", "msa_workspace_init", "msa_indexer_score", "msa_topk_blocks",
           "msa_sparse_attend", "msa_decode", "msa_read_device_status", "msa_status_string",
           "msa_dequant_debug", "msa_decode_noalloc", "msa_cache_insert")


class MsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class MsaCacheT(ctypes.Structure):
    _fields_ = [("kv_dtype", ctypes.c_int), ("index_dtype", ctypes.c_int),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("index_dim", ctypes.c_int32),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_sf", ctypes.c_void_p), ("v_sf", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("idx", ctypes.c_void_p), ("idx_sf", ctypes.c_void_p), ("idx_scale", ctypes.c_void_p),
                ("k_global", ctypes.c_float), ("v_global", ctypes.c_float), ("idx_global", ctypes.c_float),
                ("nvfp4_mode", ctypes.c_int32)]


class MsaBatchT(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("q_per_seq", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32),
                ("seq_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p)]


class MsaConfigT(ctypes.Structure):
    _fields_ = [("topk", ctypes.c_int32), ("init_blocks", ctypes.c_int32),
                ("local_blocks", ctypes.c_int32), ("index_scale", ctypes.c_float),
                ("sm_scale", ctypes.c_float), ("score_type", ctypes.c_int32), ("prefill_select", ctypes.c_int32)]


SCORE_TYPES = {"max": 0}  # msa_score_type_t: the block pooling of the index scores
# msa_nvfp4_mode_t: "exact" e2m1 x e4m3 products, or "e4m3": rounded to E4M3 first
NVFP4_MODES = {"exact": 0, "e4m3": 1}
# msa_prefill_select_t: a prefill chunk's selection by a top-k launch over the
# pooled scores, or in the tcgen05 indexer's epilogue (candidate lists)
PREFILL_SELECT = {"topk": 0, "indexer": 1}


class MsaQueryT(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int), ("scale", ctypes.c_float)]


_lib_handle = None


def lib() -> ctypes.CDLL:
    """Load libmsa.so (built in-tree by __graft_entry__.build()); raises if absent."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() first "
                               "(there is no non-CUDA implementation)")
        h = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        h.msa_workspace_size.restype = ctypes.c_size_t
        h.msa_workspace_size.argtypes = [P, P, P, ctypes.c_int32]
        h.msa_workspace_init.argtypes = [P, ctypes.c_size_t, P]
        h.msa_indexer_score.argtypes = [P, P, P, P, P, P, ctypes.c_size_t, P]
        h.msa_topk_blocks.argtypes = [P, P, ctypes.c_int32, P, P, P, P, ctypes.c_size_t, P]
        h.msa_sparse_attend.argtypes = [P, P, P, P, ctypes.c_int32, P, P, P, P, ctypes.c_size_t, P]
        h.msa_decode.argtypes = [P, P, P, P, P, ctypes.c_int32, P, P, P, P, ctypes.c_size_t, P]
        h.msa_read_device_status.argtypes = [P, P, P]
        h.msa_status_string.restype = ctypes.c_char_p
        h.msa_status_string.argtypes = [ctypes.c_int]
        h.msa_dequant_debug.argtypes = [P, ctypes.c_int32, P, ctypes.c_int32, P, P]
        h.msa_decode_noalloc.argtypes = [P, P, P, P, P, ctypes.c_int32, P, P, P, P, P]
        h.msa_cache_insert.argtypes = [P, ctypes.c_int32, P, P, P, P, P, ctypes.c_size_t, P]
        for name in EXPORTS:
            if name != "msa_workspace_size" and name != "msa_status_string":
                getattr(h, name).restype = ctypes.c_int
        _lib_handle = h
    return _lib_handle


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str) -> None:
    if status != MSA_OK:
        raise MsaError(status, where)


# ---------------------------------------------------------------- argument holders

@dataclasses.dataclass
class PagedCache:
    """Device tensors of one layer's paged K/V cache and index-key cache (layout in include/msa.h)."""
    kv_dtype: str
    index_dtype: str
    num_blocks: int
    num_kv_heads: int
    k: object
    v: object
    idx: object
    k_sf: object = None
    v_sf: object = None
    k_scale: object = None
    v_scale: object = None
    idx_sf: object = None
    idx_scale: object = None
    k_global: float = 0.0
    v_global: float = 0.0
    idx_global: float = 0.0
    head_dim: int = 128
    index_dim: int = 128
    nvfp4_mode: str = "exact"

    def struct(self) -> MsaCacheT:
        return MsaCacheT(DTYPES[self.kv_dtype], DTYPES[self.index_dtype], self.num_blocks, 128,
                         self.num_kv_heads, self.head_dim, self.index_dim,
                         _ptr(self.k), _ptr(self.v), _ptr(self.k_sf), _ptr(self.v_sf),
                         _ptr(self.k_scale), _ptr(self.v_scale), _ptr(self.idx), _ptr(self.idx_sf),
                         _ptr(self.idx_scale), self.k_global, self.v_global, self.idx_global,
                         NVFP4_MODES.get(self.nvfp4_mode, -1))


@dataclasses.dataclass
class Batch:
    seq_lens: object      # int32 [S] on the device
    block_table: object   # int32 [S][max_blocks] on the device
    q_per_seq: int = 1

    def struct(self) -> MsaBatchT:
        return MsaBatchT(self.seq_lens.shape[0], self.q_per_seq, self.block_table.shape[1],
                         _ptr(self.seq_lens), _ptr(self.block_table))


@dataclasses.dataclass
class Config:
    topk: int = 16
    init_blocks: int = 0
    local_blocks: int = 0
    index_scale: float = 128 ** -0.5
    sm_scale: float = 128 ** -0.5
    score_type: str = "max"
    prefill_select: str = "topk"

    def struct(self) -> MsaConfigT:
        # an unknown score type reaches the library as -1, which rejects it
        return MsaConfigT(self.topk, self.init_blocks, self.local_blocks, self.index_scale, self.sm_scale,
                          SCORE_TYPES.get(self.score_type, -1), PREFILL_SELECT.get(self.prefill_select, -1))


@dataclasses.dataclass
class Query:
    data: object          # bf16 tensor, or uint8 e4m3 codes
    dtype: str = "bf16"   # "bf16" | "fp8"
    scale: float = 1.0

    def struct(self) -> MsaQueryT:
        return MsaQueryT(_ptr(self.data), DTYPES[self.dtype], self.scale)


def _ref(x):
    return ctypes.byref(x)


# ---------------------------------------------------------------- entry points (same names as the C ABI)

def msa_workspace_size(cache: PagedCache, batch: Batch, cfg: Config, num_q_heads: int) -> int:
    c, b, f = cache.struct(), batch.struct(), cfg.struct()
    n = lib().msa_workspace_size(_ref(c), _ref(b), _ref(f), num_q_heads)
    if n == 0:
        raise MsaError(1, "msa_workspace_size")
    return int(n)


def msa_workspace_init(workspace, stream=None) -> None:
    _check(lib().msa_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream)), "msa_workspace_init")


def msa_indexer_score(cache, batch, cfg, index_q: Query, pooled, workspace, stream=None) -> None:
    c, b, f, q = cache.struct(), batch.struct(), cfg.struct(), index_q.struct()
    _check(lib().msa_indexer_score(_ref(c), _ref(b), _ref(f), _ref(q), _ptr(pooled), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "msa_indexer_score")


def msa_topk_blocks(batch, cfg, num_groups: int, pooled, topk_idx, topk_score, workspace, stream=None) -> None:
    b, f = batch.struct(), cfg.struct()
    _check(lib().msa_topk_blocks(_ref(b), _ref(f), num_groups, _ptr(pooled), _ptr(topk_idx), _ptr(topk_score),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)), "msa_topk_blocks")


def msa_sparse_attend(cache, batch, cfg, q: Query, num_q_heads: int, topk_idx, out, lse, workspace,
                      stream=None) -> None:
    c, b, f, qq = cache.struct(), batch.struct(), cfg.struct(), q.struct()
    _check(lib().msa_sparse_attend(_ref(c), _ref(b), _ref(f), _ref(qq), num_q_heads, _ptr(topk_idx), _ptr(out),
                                   _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)), "msa_sparse_attend")


def msa_decode(cache, batch, cfg, index_q: Query, q: Query, num_q_heads: int, topk_idx, out, lse, workspace,
               stream=None) -> None:
    c, b, f, iq, qq = cache.struct(), batch.struct(), cfg.struct(), index_q.struct(), q.struct()
    _check(lib().msa_decode(_ref(c), _ref(b), _ref(f), _ref(iq), _ref(qq), num_q_heads, _ptr(topk_idx),
                            _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                            _stream(stream)), "msa_decode")


def msa_read_device_status(workspace, stream=None):
    """Synchronise, read and clear the device status word: (status code, raw flags)."""
    detail = ctypes.c_int32(0)
    st = lib().msa_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(detail))
    return int(st), int(detail.value)


def msa_status_string(status: int) -> str:
    return lib().msa_status_string(status).decode()


def msa_dequant_debug(cache, which: int, phys_blocks, out, stream=None) -> None:
    c = cache.struct()
    _check(lib().msa_dequant_debug(_ref(c), which, _ptr(phys_blocks), phys_blocks.numel(), _ptr(out),
                                   _stream(stream)), "msa_dequant_debug")


def msa_decode_noalloc(cache, batch, cfg, index_q: Query, q: Query, num_q_heads: int, topk_idx, out, lse,
                       status_out=None, stream=None) -> None:
    """msa_decode without a caller workspace, for callers that cannot allocate
    device memory (e.g. code living inside another framework's memory pool):
    the library's own fixed scratch array is used instead.  Problems whose
    workspace exceeds the scratch size are rejected; calls must not overlap on
    the GPU because they share that scratch.  status_out: optional device
    int32[2] that receives the call's device status flags."""
    c, b, f, iq, qq = cache.struct(), batch.struct(), cfg.struct(), index_q.struct(), q.struct()
    _check(lib().msa_decode_noalloc(_ref(c), _ref(b), _ref(f), _ref(iq), _ref(qq), num_q_heads, _ptr(topk_idx),
                                    _ptr(out), _ptr(lse), _ptr(status_out), _stream(stream)),
           "msa_decode_noalloc")


def msa_cache_insert(cache, slot_mapping, k, v, index_k, workspace, stream=None) -> None:
    """Quantize and write new tokens' K, V (bf16 [T][H][128]) and index keys (bf16
    [T][128], or None) into the paged caches at slot_mapping (int32 [T])."""
    c = cache.struct()
    _check(lib().msa_cache_insert(_ref(c), int(slot_mapping.numel()), _ptr(slot_mapping), _ptr(k), _ptr(v),
                                  _ptr(index_k), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "msa_cache_insert")


def default_config(topk: int = 16, head_dim: int = 128, index_dim: int = 128) -> Config:
    """The model's settings: index and softmax scales head_dim ** -0.5."""
    return Config(topk=topk, index_scale=index_dim ** -0.5, sm_scale=head_dim ** -0.5)


__all__ = ["PagedCache", "Batch", "Config", "Query", "MsaError", "lib", "EXPORTS", "default_config",
           "msa_workspace_size", "msa_workspace_init", "msa_indexer_score", "msa_topk_blocks",
           "msa_sparse_attend", "msa_decode", "msa_read_device_status", "msa_status_string",
           "msa_dequant_debug", "msa_decode_noalloc", "msa_cache_insert", "roofline"]
