"""Cache byte accounting: the bytes a compressed cache holds and a decode step reads.

"StreamingLLM + KIVI", "Storage layout" and "Cache-bytes table": per layer,
codes [B, H, T, D] plus fp16 kScales/kZeros [B, H, D] and vScales/vZeros
[B, H, T].  "Low-bit KV caches on MLX", section 4: with groups of 64
elements, the two fp16 values of each group cost an extra 0.5 bit per element.
"""
from __future__ import annotations


def bits_per_element(bits: int, group: int, meta_bits: int = 16, meta_per_group: int = 2) -> float:
    """Storage bits per cached element of a group-scalar format."""
    return bits + meta_per_group * meta_bits / group


def dense_cache_bytes(layers: int, heads: int, T: int, D: int, elem_bytes: int, batch: int = 1) -> int:
    """K + V bytes of an unquantised cache."""
    return 2 * layers * batch * heads * T * D * elem_bytes


def kivi_cache_bytes(layers: int, heads: int, T: int, D: int, code_bits: int, batch: int = 1) -> int:
    """K + V bytes of the KIVI layout: codes, per-channel K (scale, zero), per-token V (scale, zero).

    code_bits is the storage width of one code (8 for int8 storage, 4 when
    nibbles are packed).
    """
    codes = 2 * layers * batch * heads * T * D * code_bits // 8
    k_meta = 2 * layers * batch * heads * D * 2
    v_meta = 2 * layers * batch * heads * T * 2
    return codes + k_meta + v_meta


def side_bytes_per_token(fmt: str, bits: int, group: int, D: int) -> int:
    """Bytes one token of one (b, kv-head) occupies for K or V in a given format."""
    if fmt == "fp16":
        return 2 * D
    codes = D * bits // 8
    if fmt == "affine_token":
        return codes + 2 * 2 * (D // group)
    if fmt == "q4_0":
        return codes + 2 * (D // 32)
    if fmt == "kivi_chan":
        return codes
    raise ValueError(fmt)


def side_fixed_bytes(fmt: str, D: int) -> int:
    """Token-independent bytes per (b, kv-head): the per-channel fp16 scale and zero of KIVI keys."""
    return 2 * 2 * D if fmt == "kivi_chan" else 0


def decode_read_bytes(w_batch: int, hkv: int, hq: int, D: int, T: int,
                      k_fmt: str, k_bits: int, k_group: int,
                      v_fmt: str, v_bits: int, v_group: int, io_bytes: int) -> int:
    """Algorithmic bytes of one decode-attention call: cache codes + metadata + Q + O."""
    per_head = T * (side_bytes_per_token(k_fmt, k_bits, k_group, D)
                    + side_bytes_per_token(v_fmt, v_bits, v_group, D))
    per_head += side_fixed_bytes(k_fmt, D) + side_fixed_bytes(v_fmt, D)
    return w_batch * hkv * per_head + 2 * w_batch * hq * D * io_bytes
