"""Algorithmic byte model of the MSA decode path (host-side arithmetic only).

Decode reads the whole context's index keys once per step, plus full K/V for
only the selected tokens (vLLM Day-0 blog, section "MSA 入门": 128 B/token of
FP8 index keys against 1,024 B/token of FP8 K/V for 4 KV heads x 128 dims).
The per-token fp32 scales of the FP8 layout are reported separately as
"actual" bytes; the algorithmic figure counts only element storage.
"""

from __future__ import annotations


def index_bytes_per_token(dtype: str, index_dim: int = 128) -> float:
    if dtype == "bf16":
        return 2.0 * index_dim
    if dtype == "fp8":
        return 1.0 * index_dim
    if dtype == "nvfp4":
        return index_dim / 2 + index_dim / 16
    raise ValueError(dtype)


def kv_bytes_per_token(dtype: str, num_kv_heads: int = 4, head_dim: int = 128) -> float:
    """K + V bytes of one token over all KV heads."""
    if dtype == "bf16":
        per = 2.0 * head_dim
    elif dtype == "fp8":
        per = 1.0 * head_dim
    elif dtype == "nvfp4":
        per = head_dim / 2 + head_dim / 16
    else:
        raise ValueError(dtype)
    return 2.0 * num_kv_heads * per


def scale_bytes_per_token(kv_dtype: str, index_dtype: str, num_kv_heads: int = 4) -> tuple:
    """(index, K/V) bytes of per-token fp32 scales (FP8 layout only)."""
    return (4.0 if index_dtype == "fp8" else 0.0,
            8.0 * num_kv_heads if kv_dtype == "fp8" else 0.0)


def decode_bytes_per_query(kv_dtype: str, index_dtype: str, context: int, selected_tokens: int,
                           num_kv_heads: int = 4, head_dim: int = 128, index_dim: int = 128) -> float:
    """Bytes one single-token decode query reads: whole-context index keys plus
    the K/V of its selected tokens."""
    return (context * index_bytes_per_token(index_dtype, index_dim)
            + selected_tokens * kv_bytes_per_token(kv_dtype, num_kv_heads, head_dim))
