// The row quantiser shared by the append kernels and the fused append of
// decode attention: one warp codes one token row of D = 32 * E channels
// with the formats' fp32 rules (kvq_internal.cuh), writes the codes and the
// per-token fp16 metadata, and can return the values the stored row
// dequantises to.  "StreamingLLM + KIVI", "Affine quantisation formula" and
// "Storage layout"; "Low-bit KV caches on MLX", section 1; "kv-cache:
// optional per-channel K-cache mean-centering for Q4_0", "The idea".
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

// Lane l of the warp holds channels [l*E, l*E + E).

template <int E>
__device__ __forceinline__ void store_bytes(uint8_t* dst, const uint8_t (&b)[E]) {
  if constexpr (E == 1) {
    dst[0] = b[0];
  } else if constexpr (E == 2) {
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(b[0] | (b[1] << 8));
  } else {
#pragma unroll
    for (int i = 0; i < E; i += 4) {
      *reinterpret_cast<uint32_t*>(dst + i) = (uint32_t)b[i] | ((uint32_t)b[i + 1] << 8) |
                                              ((uint32_t)b[i + 2] << 16) | ((uint32_t)b[i + 3] << 24);
    }
  }
}

// Writes the lane's E codes u (0..levels) in the side's storage encoding.
template <int E>
__device__ __forceinline__ void store_codes(uint8_t* row, int lane, int bits, const int (&u)[E]) {
  if (bits == 8) {
    uint8_t b[E];
#pragma unroll
    for (int i = 0; i < E; ++i) b[i] = (uint8_t)(u[i] ^ 0x80);   // signed level q = u - 128
    store_bytes<E>(row + lane * E, b);
  } else {  // 4-bit: channel 2j in the low nibble of byte j
    if constexpr (E == 1) {
      const int nb = __shfl_down_sync(0xffffffffu, u[0], 1);
      if ((lane & 1) == 0) row[lane >> 1] = (uint8_t)(u[0] | (nb << 4));
    } else {
      uint8_t b[E / 2];
#pragma unroll
      for (int i = 0; i < E / 2; ++i) b[i] = (uint8_t)(u[2 * i] | (u[2 * i + 1] << 4));
      store_bytes<E / 2>(row + lane * (E / 2), b);
    }
  }
}

// Max / min over the `width` lanes (a power of two) of the lane's group.
__device__ __forceinline__ float group_max(float x, int width) {
  for (int o = 1; o < width; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float group_min(float x, int width) {
  for (int o = 1; o < width; o <<= 1) x = fminf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Codes lane `lane`'s E channels x (already loaded as fp32) of one row.
// DQ: also leave in xh the value each channel dequantises to from what was
// stored, in fp32 with the stored fp16 metadata upcast: u * s + z (affine),
// (u - 8) * d (Q4_0), the fp16 value (fp16 rows), and for per-channel KIVI
// keys u * s without the channel's zero (decode attention drops that zero
// term, the same per-row constant for every key of a query, from all keys).
template <int E, bool DQ>
__device__ __forceinline__ void quantize_row_dq(const SideView& s, const float* __restrict__ bias, float (&x)[E],
                                                size_t bh, int cap_alloc, int slot, int lane, float (&xh)[E]) {
  uint8_t* row = s.codes + ((size_t)bh * cap_alloc + slot) * s.row_bytes;
  const size_t meta_row = ((size_t)bh * cap_alloc + slot) * s.n_groups;

  if (s.fmt == KVQ_FMT_FP16) {
    __half* dst = reinterpret_cast<__half*>(row) + lane * E;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const __half h = __float2half_rn(x[i]);
      dst[i] = h;
      if constexpr (DQ) xh[i] = __half2float(h);
    }
    return;
  }

  const float levels = (s.bits == 8) ? 255.0f : 15.0f;
  int u[E];

  if (s.fmt == KVQ_FMT_KIVI_CHAN) {
    const float* sc = s.ch_scale32 + bh * (32 * E) + lane * E;
    const float* zr = s.ch_zero32 + bh * (32 * E) + lane * E;
#pragma unroll
    for (int i = 0; i < E; ++i) u[i] = affine_code(x[i], sc[i], zr[i], levels);
    if constexpr (DQ) {   // read before the store below (which the compiler cannot move loads past)
      const __half* s16 = s.ch_scale + bh * (32 * E) + lane * E;
#pragma unroll
      for (int i = 0; i < E; ++i) xh[i] = (float)u[i] * __half2float(s16[i]);
    }
    store_codes<E>(row, lane, s.bits, u);
    return;
  }

  if (s.fmt == KVQ_FMT_AFFINE_TOKEN) {
    const int width = s.group / E;           // lanes per group
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int i = 1; i < E; ++i) {
      mn = fminf(mn, x[i]);
      mx = fmaxf(mx, x[i]);
    }
    mn = group_min(mn, width);
    mx = group_max(mx, width);
    const float sc = affine_scale(mn, mx, levels);
    const float inv = __frcp_rn(sc);
#pragma unroll
    for (int i = 0; i < E; ++i) u[i] = affine_code_inv(x[i], sc, inv, mn, levels);
    store_codes<E>(row, lane, s.bits, u);
    const __half s16 = __float2half_rn(sc), z16 = __float2half_rn(mn);
    if (lane % width == 0) {
      const int g = lane / width;
      s.tok_scale[meta_row + g] = s16;
      s.tok_zero[meta_row + g] = z16;
    }
    if constexpr (DQ) {
#pragma unroll
      for (int i = 0; i < E; ++i) xh[i] = fmaf((float)u[i], __half2float(s16), __half2float(z16));
    }
    return;
  }

  // KVQ_FMT_Q4_0: optional centering, then symmetric 32-channel blocks.
  if (bias != nullptr) {
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] = __fsub_rn(x[i], bias[lane * E + i]);
  }
  const int width = 32 / E;
  float a = fabsf(x[0]);
#pragma unroll
  for (int i = 1; i < E; ++i) a = fmaxf(a, fabsf(x[i]));
  a = group_max(a, width);
  const float d = __fdiv_rn(a, 7.0f);
  const float dinv = __frcp_rn(d);   // inf when d == 0 (q40_code_inv does not use it then)
#pragma unroll
  for (int i = 0; i < E; ++i) u[i] = q40_code_inv(x[i], d, dinv);
  store_codes<E>(row, lane, 4, u);
  const __half d16 = __float2half_rn(d);
  if (lane % width == 0) s.tok_scale[meta_row + lane / width] = d16;
  if constexpr (DQ) {
#pragma unroll
    for (int i = 0; i < E; ++i) xh[i] = (float)(u[i] - 8) * __half2float(d16);
  }
}

// Codes lane `lane`'s E channels x (already loaded as fp32) of one row.
template <int E>
__device__ __forceinline__ void quantize_row(const SideView& s, const float* __restrict__ bias, float (&x)[E],
                                             size_t bh, int cap_alloc, int slot, int lane) {
  float unused[E];
  quantize_row_dq<E, false>(s, bias, x, bh, cap_alloc, slot, lane, unused);
}

}  // namespace kvq
