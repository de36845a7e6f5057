// Decode attention on the tensor cores (mma.sync m16n8k16, fp16 operands, fp32
// accumulators) for head_dim 64 / 128 and bf16 / fp16 queries and outputs.
//
// Same split-KV structure, 64-token cp.async tiles and online-softmax merge as
// decode_kernel; the difference is where the two contractions run.  Per warp
// and 16-token block:
//   S[16 x 16] = Q[16 x D] . K_hat^T : M rows 0..7 hold fp16(q) of the (up to
//     8) query heads of the kv head, rows 8..15 the fp16 residual q - fp16(q),
//     so the score of head h is row h + row h + 8 and q enters exactly; B is
//     the dequantised key block, unpacked from the codes in registers.
//   O[16 x D] += P[16 x 16] . V_hat : the probabilities of the block as A (hi
//     / residual rows again), B the dequantised value block.
// Codes become fp16 exactly: a nibble n (or byte) placed in the mantissa of
// 1024.0 gives 1024 + n, one HSUB2 removes 1024 (nibbles in the high half of a
// byte give 1024 + 16n and one HFMA2 by 1/16, -64 recovers n).  Dequantisation
// is one HFMA2 with the token's fp16 (scale, zero), i.e. x_hat rounded to
// fp16; per-channel KIVI scales are folded into q instead (the zero term is
// dropped, a per-row constant the softmax does not see).
//
// Token order inside a 16-token block: mma k index j reads physical row
// tau(j), tau(2t + e) = t + 4e, tau(8 + 2t + e) = 8 + t + 4e, so that every
// fragment load of K and V from shared memory is free of bank conflicts.
// Channel order: thread t (lane % 4) owns channels [t*D/4, (t+1)*D/4) of a key
// row, thread g (lane / 4) owns channels [g*D/8, (g+1)*D/8) of a value row; the
// query fragment is gathered in the matching order.
#pragma once

#include "decode_impl.cuh"

namespace kvq {

__device__ __forceinline__ __half2 u2h(uint32_t x) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = x;
  return h;
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Eight nibbles of w (channel i in bits 4i..4i+3) as exact fp16 pairs:
// h[0] = (c0, c4), h[1] = (c1, c5), h[2] = (c2, c6), h[3] = (c3, c7).
__device__ __forceinline__ void nibbles_to_h2(uint32_t w, __half2 (&h)[4]) {
  const uint32_t M = 0x64006400u;
  const __half2 k1024 = u2h(0x64006400u);
  const __half2 k16th = u2h(0x2C002C00u);   // 1/16
  const __half2 km64 = u2h(0xD400D400u);    // -64
  const uint32_t w8 = w >> 8;
  h[0] = __hsub2(u2h((w & 0x000F000Fu) | M), k1024);
  h[1] = __hfma2(u2h((w & 0x00F000F0u) | M), k16th, km64);
  h[2] = __hsub2(u2h((w8 & 0x000F000Fu) | M), k1024);
  h[3] = __hfma2(u2h((w8 & 0x00F000F0u) | M), k16th, km64);
}

// Four unsigned bytes of x as exact fp16 pairs: lo = (b0, b1), hi = (b2, b3).
__device__ __forceinline__ void bytes_to_h2(uint32_t x, __half2& lo, __half2& hi) {
  const __half2 k1024 = u2h(0x64006400u);
  lo = __hsub2(u2h(__byte_perm(x, 0x64646464u, 0x5140u)), k1024);
  hi = __hsub2(u2h(__byte_perm(x, 0x64646464u, 0x7362u)), k1024);
}

// Logical k index j of a 16-token block -> physical row inside the block.
__device__ __forceinline__ int tau(int j) { return (j & 8) + ((j & 7) >> 1) + 4 * (j & 1); }

// Tile copy with zero fill: rows at or beyond `valid_rows` of the tile read as
// zero bytes (cp.async with a short source size), so codes and metadata of
// rows the split does not own never reach an MMA.
__device__ __forceinline__ void cp_async16_zfill(void* smem, const void* gmem, int src_bytes) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
}

__device__ __forceinline__ void copy_plane_rows(uint8_t* dst, const uint8_t* src, int row_bytes, int valid_rows) {
  const int n16 = kTileTokens * row_bytes / 16;
  const int valid = valid_rows * row_bytes;
  for (int i = threadIdx.x; i < n16; i += kDecodeThreads) {
    int nb = valid - 16 * i;
    nb = nb < 0 ? 0 : (nb > 16 ? 16 : nb);
    cp_async16_zfill(dst + 16 * i, src + 16 * i, nb);
  }
}

// Same, with the 16-byte chunk c of row r stored at chunk c ^ f(r), f(r) =
// (r / rows-per-128-byte-line) mod chunks-per-row: rows that would share a
// shared-memory bank line put the same logical chunk in different banks.
__device__ __forceinline__ int swz(int r, int row_bytes) {
  return (r / (128 / row_bytes)) & (row_bytes / 16 - 1);
}
__device__ __forceinline__ void copy_plane_rows_swz(uint8_t* dst, const uint8_t* src, int row_bytes, int valid_rows) {
  const int nch = row_bytes / 16;
  const int n16 = kTileTokens * nch;
  const int valid = valid_rows * row_bytes;
  for (int i = threadIdx.x; i < n16; i += kDecodeThreads) {
    const int r = i / nch, cc = i % nch;
    int nb = valid - 16 * i;
    nb = nb < 0 ? 0 : (nb > 16 ? 16 : nb);
    cp_async16_zfill(dst + r * row_bytes + 16 * (cc ^ swz(r, row_bytes)), src + 16 * i, nb);
  }
}

// Keys with per-token groups are multiplied exactly (codes in the MMA, scales
// applied to the fp32 block sums afterwards); they use the swizzled tile.
template <int KF> struct KGrouped { static constexpr bool v = (KF == F_AFF8 || KF == F_AFF4 || KF == F_Q40); };

template <int D, int KF, int VF>
__device__ __forceinline__ void issue_tile_zfill(uint8_t* st, const TileLayout& L, const CacheView& c, size_t bh,
                                                 int row0, int valid_rows) {
  constexpr int KROW = D * FmtBits<KF>::v / 8;
  constexpr int VROW = D * FmtBits<VF>::v / 8;
  constexpr bool K_AFF = (KF == F_AFF8 || KF == F_AFF4);
  constexpr bool K_Q40 = (KF == F_Q40);
  constexpr bool V_AFF = (VF == F_AFF8 || VF == F_AFF4);
  const size_t row = bh * c.cap_alloc + row0;
  if constexpr (KGrouped<KF>::v) copy_plane_rows_swz(st + L.kc, c.k.codes + row * KROW, KROW, valid_rows);
  else copy_plane_rows(st + L.kc, c.k.codes + row * KROW, KROW, valid_rows);
  copy_plane_rows(st + L.vc, c.v.codes + row * VROW, VROW, valid_rows);
  if constexpr (K_AFF || K_Q40) {
    const int mb = c.k.n_groups * 2;
    copy_plane_rows(st + L.ks, reinterpret_cast<const uint8_t*>(c.k.tok_scale) + row * mb, mb, valid_rows);
    if constexpr (K_AFF)
      copy_plane_rows(st + L.kz, reinterpret_cast<const uint8_t*>(c.k.tok_zero) + row * mb, mb, valid_rows);
  }
  if constexpr (V_AFF) {
    const int mb = c.v.n_groups * 2;
    copy_plane_rows(st + L.vs, reinterpret_cast<const uint8_t*>(c.v.tok_scale) + row * mb, mb, valid_rows);
    copy_plane_rows(st + L.vz, reinterpret_cast<const uint8_t*>(c.v.tok_zero) + row * mb, mb, valid_rows);
  }
}

// Loads NW consecutive 32-bit words from shared memory.
template <int NW>
__device__ __forceinline__ void lds_words(uint32_t (&w)[NW], const uint8_t* p) {
  static_assert(NW == 1 || NW == 2 || NW % 4 == 0, "word count");
  if constexpr (NW == 1) {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  } else if constexpr (NW == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < NW / 4; ++i) {
      const uint4 v = reinterpret_cast<const uint4*>(p)[i];
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  }
}

template <int D, int G, int KF, int VF>
__global__ void __launch_bounds__(kDecodeThreads) decode_tc_kernel(CacheView c, DecodeArgs a) {
  constexpr int NSTAGE = Stages<KF>::v;
  constexpr int KB = FmtBits<KF>::v;
  constexpr int VB = FmtBits<VF>::v;
  constexpr int KROW = D * KB / 8;
  constexpr int VROW = D * VB / 8;
  constexpr int KS = D / 16;       // k-steps of Q K^T
  constexpr int NT = D / 8;        // n-tiles of P V
  constexpr int KCH = D / 4;       // key channels owned by quad thread t
  constexpr int VCH = D / 8;       // value channels owned by thread g
  constexpr bool K_AFF = (KF == F_AFF8 || KF == F_AFF4);
  constexpr bool K_KIVI = (KF == F_KIVI8 || KF == F_KIVI4);
  constexpr bool K_Q40 = (KF == F_Q40);
  constexpr bool V_AFF = (VF == F_AFF8 || VF == F_AFF4);
  static_assert(G >= 1 && G <= 8, "up to 8 query heads per kv head");

  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float sm_m[kDecodeWarps][G];
  __shared__ float sm_l[kDecodeWarps][G];
  __shared__ __align__(16) float sm_acc[kDecodeWarps][G][D];
  __shared__ int s_T;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
  const size_t bh = (size_t)b * c.Hkv + kvh;
  const int kng = c.k.n_groups;
  const int vng = c.v.n_groups;
  const TileLayout TL = tile_layout<D, KF, VF>(kng, vng);

  if (threadIdx.x == 0) s_T = c.state->stored;
  __syncthreads();
  const int T = s_T;
  int per = (T + a.nsplit - 1) / a.nsplit;
  per = (per + kTileTokens - 1) / kTileTokens * kTileTokens;
  const int t0 = min(T, split * per);
  const int t1 = min(T, t0 + per);
  const int ntiles = (t1 - t0 + kTileTokens - 1) / kTileTokens;

#pragma unroll
  for (int s = 0; s < NSTAGE - 1; ++s) {
    if (s < ntiles) {
      const int row0 = t0 + s * kTileTokens;
      issue_tile_zfill<D, KF, VF>(smem + s * TL.bytes, TL, c, bh, row0, t1 - row0);
    }
    cp_async_commit();
  }

  // Query fragments: row g = fp16(q), row g + 8 = fp16(q - fp16(q)), in the
  // channel order the key fragments arrive in.
  // Grouped keys: quad thread t owns word t of every 16-byte chunk of a key row,
  // so k-step pair p (4-bit) or k-steps 2p, 2p + 1 (8-bit) cover exactly the
  // 32-channel block p; other keys: thread t owns the contiguous quarter row.
  constexpr bool KG = KGrouped<KF>::v;
  constexpr int NB = D / 32;
  uint32_t qa[KS][4];
  float qblk[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) qblk[i] = 0.0f;
  {
    const bool live = g < G;
    const size_t qo = ((size_t)b * a.Hq + (size_t)kvh * G + (live ? g : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      int ch[4];
      if constexpr (KB == 4) {
        const int base = (KG ? 32 * (ks >> 1) + 8 * t : t * KCH + 8 * (ks >> 1)) + (ks & 1);
        ch[0] = base; ch[1] = base + 4; ch[2] = base + 2; ch[3] = base + 6;
      } else {
        const int base = KG ? 16 * ks + 4 * t : t * KCH + 4 * ks;
        ch[0] = base; ch[1] = base + 1; ch[2] = base + 2; ch[3] = base + 3;
      }
      float qv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float x = live ? load_io(a.q, qo + ch[i], a.io_dtype) : 0.0f;
        if constexpr (K_KIVI) x *= __half2float(c.k.ch_scale[bh * D + ch[i]]);
        qv[i] = x;
      }
      if constexpr (KG) qblk[ks >> 1] += (qv[0] + qv[1]) + (qv[2] + qv[3]);
      const __half2 h01 = __floats2half2_rn(qv[0], qv[1]);
      const __half2 h23 = __floats2half2_rn(qv[2], qv[3]);
      const float2 f01 = __half22float2(h01);
      const float2 f23 = __half22float2(h23);
      qa[ks][0] = h2u(h01);
      qa[ks][1] = h2u(__floats2half2_rn(qv[0] - f01.x, qv[1] - f01.y));
      qa[ks][2] = h2u(h23);
      qa[ks][3] = h2u(__floats2half2_rn(qv[2] - f23.x, qv[3] - f23.y));
    }
  }
  if constexpr (KG) {
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      qblk[i] += __shfl_xor_sync(0xffffffffu, qblk[i], 1);
      qblk[i] += __shfl_xor_sync(0xffffffffu, qblk[i], 2);
    }
  }
  const int kbpg = K_AFF ? c.k.group / 32 : 1;          // 32-channel blocks per key group
  const int vgi = V_AFF ? (g * VCH) / c.v.group : 0;

  float m_run = neg_inf();
  float l_part = 0.0f;
  float oacc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) oacc[nt][0] = oacc[nt][1] = oacc[nt][2] = oacc[nt][3] = 0.0f;

  for (int it = 0; it < ntiles; ++it) {
    cp_async_wait<NSTAGE - 2>();
    __syncthreads();
    {
      const int nx = it + NSTAGE - 1;
      if (nx < ntiles) {
        const int row0 = t0 + nx * kTileTokens;
        issue_tile_zfill<D, KF, VF>(smem + (nx % NSTAGE) * TL.bytes, TL, c, bh, row0, t1 - row0);
      }
      cp_async_commit();
    }
    const uint8_t* st = smem + (it % NSTAGE) * TL.bytes;
    const int blk = warp * 16;                          // this warp's 16 rows of the tile
    const int tok0 = t0 + it * kTileTokens + blk;
    if (tok0 >= t1) continue;                           // warp-uniform

    // ---------------------------------------------------------- S = Q K^T
    // sc[2 nt + e]: head g, logical token 8 nt + 2t + e (row blk + 8 nt + t + 4e)
    float sc[4];
    const int rr[4] = {blk + t, blk + t + 4, blk + 8 + t, blk + 12 + t};
    if constexpr (KG) {
      // exact codes, one fp32 accumulator per 32-channel block, scales after
      float acc[NB][2][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) acc[nb][nt][0] = acc[nb][nt][1] = acc[nb][nt][2] = acc[nb][nt][3] = 0.0f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int r = blk + tau(nt * 8 + g);
        const uint8_t* krow = st + TL.kc + r * KROW + 4 * t;
        const int f = swz(r, KROW);
        if constexpr (KB == 4) {
#pragma unroll
          for (int p = 0; p < NB; ++p) {
            __half2 h[4];
            nibbles_to_h2(*reinterpret_cast<const uint32_t*>(krow + 16 * (p ^ f)), h);
            mma_f16(acc[p][nt], qa[2 * p][0], qa[2 * p][1], qa[2 * p][2], qa[2 * p][3], h2u(h[0]), h2u(h[2]));
            mma_f16(acc[p][nt], qa[2 * p + 1][0], qa[2 * p + 1][1], qa[2 * p + 1][2], qa[2 * p + 1][3], h2u(h[1]),
                    h2u(h[3]));
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            __half2 lo, hi;
            bytes_to_h2(*reinterpret_cast<const uint32_t*>(krow + 16 * (ks ^ f)) ^ 0x80808080u, lo, hi);
            mma_f16(acc[ks >> 1][nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], h2u(lo), h2u(hi));
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int nt = i >> 1, e = i & 1;
        const __half* srow = reinterpret_cast<const __half*>(st + TL.ks) + rr[i] * kng;
        float v = 0.0f;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const float x = acc[nb][nt][e] + acc[nb][nt][2 + e];
          const float sb = __half2float(srow[nb / kbpg]);
          if constexpr (K_AFF) {
            const float zb = __half2float(reinterpret_cast<const __half*>(st + TL.kz)[rr[i] * kng + nb / kbpg]);
            v = fmaf(sb, x, fmaf(zb, qblk[nb], v));
          } else {
            v = fmaf(sb, fmaf(-8.0f, qblk[nb], x), v);   // d (sum q u - 8 sum q)
          }
        }
        sc[i] = v * a.qscale;
      }
    } else {
    float sacc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.0f;
      const int r = blk + tau(nt * 8 + g);
      const __half2 s2 = u2h(0x3C003C00u), z2 = u2h(0u);   // unused: these keys carry no per-token scale
      const uint8_t* kp = st + TL.kc + r * KROW + t * (KROW / 4);
      if constexpr (KB == 4) {
        uint32_t w[KCH / 8];
        lds_words<KCH / 8>(w, kp);
#pragma unroll
        for (int wi = 0; wi < KCH / 8; ++wi) {
          __half2 h[4];
          nibbles_to_h2(w[wi], h);
          if constexpr (K_AFF || K_Q40) {
#pragma unroll
            for (int i = 0; i < 4; ++i) h[i] = __hfma2(h[i], s2, z2);
          }
          mma_f16(sacc[nt], qa[2 * wi][0], qa[2 * wi][1], qa[2 * wi][2], qa[2 * wi][3], h2u(h[0]), h2u(h[2]));
          mma_f16(sacc[nt], qa[2 * wi + 1][0], qa[2 * wi + 1][1], qa[2 * wi + 1][2], qa[2 * wi + 1][3], h2u(h[1]),
                  h2u(h[3]));
        }
      } else if constexpr (KB == 8) {
        uint32_t w[KCH / 4];
        lds_words<KCH / 4>(w, kp);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          __half2 lo, hi;
          bytes_to_h2(w[ks] ^ 0x80808080u, lo, hi);
          if constexpr (K_AFF) {
            lo = __hfma2(lo, s2, z2);
            hi = __hfma2(hi, s2, z2);
          }
          mma_f16(sacc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], h2u(lo), h2u(hi));
        }
      } else {
        uint32_t w[KCH / 2];
        lds_words<KCH / 2>(w, kp);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
          mma_f16(sacc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], w[2 * ks], w[2 * ks + 1]);
      }
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i] = (sacc[i >> 1][i & 1] + sacc[i >> 1][2 + (i & 1)]) * a.qscale;
    }

    // ------------------------------------------------- online softmax (log2)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (tok0 + rr[i] - blk >= t1) sc[i] = neg_inf();
    float mb = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const float mn = fmaxf(m_run, mb);                 // finite: row tok0 is valid
    if (mn > m_run) {
      const float alpha = exp2f(m_run - mn);
      l_part *= alpha;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        oacc[nt][0] *= alpha; oacc[nt][1] *= alpha; oacc[nt][2] *= alpha; oacc[nt][3] *= alpha;
      }
      m_run = mn;
    }
    float p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      p[i] = exp2f(sc[i] - mn);
      l_part += p[i];
    }
    const __half2 ph0 = __floats2half2_rn(p[0], p[1]);
    const __half2 ph1 = __floats2half2_rn(p[2], p[3]);
    const float2 pf0 = __half22float2(ph0);
    const float2 pf1 = __half22float2(ph1);
    const uint32_t pa0 = h2u(ph0);
    const uint32_t pa1 = h2u(__floats2half2_rn(p[0] - pf0.x, p[1] - pf0.y));
    const uint32_t pa2 = h2u(ph1);
    const uint32_t pa3 = h2u(__floats2half2_rn(p[2] - pf1.x, p[3] - pf1.y));

    // ------------------------------------------------------------ O += P V
    // rows of the four tokens this thread feeds: k = 2t, 2t+1 (b0), 2t+8, 2t+9 (b1)
    const int rA = blk + t, rB = blk + t + 4, rC = blk + 8 + t, rD = blk + 12 + t;
    __half2 sAB, zAB, sCD, zCD;
    if constexpr (V_AFF) {
      const __half* vs = reinterpret_cast<const __half*>(st + TL.vs);
      const __half* vz = reinterpret_cast<const __half*>(st + TL.vz);
      sAB = __halves2half2(vs[rA * vng + vgi], vs[rB * vng + vgi]);
      zAB = __halves2half2(vz[rA * vng + vgi], vz[rB * vng + vgi]);
      sCD = __halves2half2(vs[rC * vng + vgi], vs[rD * vng + vgi]);
      zCD = __halves2half2(vz[rC * vng + vgi], vz[rD * vng + vgi]);
    }
    const uint8_t* vbase = st + TL.vc + g * (VROW / 8);
    if constexpr (VB == 4) {
      constexpr int NW = VCH / 8;                      // words per token
      uint32_t A[NW], B[NW], C[NW], E[NW];
      lds_words<NW>(A, vbase + rA * VROW);
      lds_words<NW>(B, vbase + rB * VROW);
      lds_words<NW>(C, vbase + rC * VROW);
      lds_words<NW>(E, vbase + rD * VROW);
#pragma unroll
      for (int wi = 0; wi < NW; ++wi) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t sel = half ? 0x7632u : 0x5410u;
          __half2 h0[4], h1[4];
          nibbles_to_h2(__byte_perm(A[wi], B[wi], sel), h0);
          nibbles_to_h2(__byte_perm(C[wi], E[wi], sel), h1);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if constexpr (V_AFF) {
              h0[i] = __hfma2(h0[i], sAB, zAB);
              h1[i] = __hfma2(h1[i], sCD, zCD);
            }
            // channel pairs come out as (0,1,2,3) of the byte pair: h[0]=c0, h[1]=c1, h[2]=c2, h[3]=c3
            const int nt = 8 * wi + 4 * half + i;
            mma_f16(oacc[nt], pa0, pa1, pa2, pa3, h2u(h0[i]), h2u(h1[i]));
          }
        }
      }
    } else if constexpr (VB == 8) {
      constexpr int NW = VCH / 4;
      uint32_t A[NW], B[NW], C[NW], E[NW];
      lds_words<NW>(A, vbase + rA * VROW);
      lds_words<NW>(B, vbase + rB * VROW);
      lds_words<NW>(C, vbase + rC * VROW);
      lds_words<NW>(E, vbase + rD * VROW);
#pragma unroll
      for (int wi = 0; wi < NW; ++wi) {
        const uint32_t a_ = A[wi] ^ 0x80808080u, b_ = B[wi] ^ 0x80808080u;
        const uint32_t c_ = C[wi] ^ 0x80808080u, e_ = E[wi] ^ 0x80808080u;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t sel = half ? 0x7362u : 0x5140u;
          __half2 l0, h0, l1, h1;
          bytes_to_h2(__byte_perm(a_, b_, sel), l0, h0);
          bytes_to_h2(__byte_perm(c_, e_, sel), l1, h1);
          if constexpr (V_AFF) {
            l0 = __hfma2(l0, sAB, zAB); h0 = __hfma2(h0, sAB, zAB);
            l1 = __hfma2(l1, sCD, zCD); h1 = __hfma2(h1, sCD, zCD);
          }
          const int nt = 4 * wi + 2 * half;
          mma_f16(oacc[nt], pa0, pa1, pa2, pa3, h2u(l0), h2u(l1));
          mma_f16(oacc[nt + 1], pa0, pa1, pa2, pa3, h2u(h0), h2u(h1));
        }
      }
    } else {
      constexpr int NW = VCH / 2;
      uint32_t A[NW], B[NW], C[NW], E[NW];
      lds_words<NW>(A, vbase + rA * VROW);
      lds_words<NW>(B, vbase + rB * VROW);
      lds_words<NW>(C, vbase + rC * VROW);
      lds_words<NW>(E, vbase + rD * VROW);
#pragma unroll
      for (int wi = 0; wi < NW; ++wi) {
        mma_f16(oacc[2 * wi], pa0, pa1, pa2, pa3, __byte_perm(A[wi], B[wi], 0x5410u),
                __byte_perm(C[wi], E[wi], 0x5410u));
        mma_f16(oacc[2 * wi + 1], pa0, pa1, pa2, pa3, __byte_perm(A[wi], B[wi], 0x7632u),
                __byte_perm(C[wi], E[wi], 0x7632u));
      }
    }
  }
  cp_async_wait<0>();

  // Per-warp results to shared memory: head g, channels (2t + e) * VCH + nt.
  l_part += __shfl_xor_sync(0xffffffffu, l_part, 1);
  l_part += __shfl_xor_sync(0xffffffffu, l_part, 2);
  if (g < G) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      sm_acc[warp][g][(2 * t) * VCH + nt] = oacc[nt][0] + oacc[nt][2];
      sm_acc[warp][g][(2 * t + 1) * VCH + nt] = oacc[nt][1] + oacc[nt][3];
    }
    if (t == 0) {
      sm_m[warp][g] = m_run;
      sm_l[warp][g] = l_part;
    }
  }
  __syncthreads();
  merge_store<D, G>(c, a, b, kvh, split, sm_m, sm_l, sm_acc);
}

template <int D, int G, int KF, int VF>
cudaError_t launch_decode_tc_dg(const CacheView& c, const DecodeArgs& a, cudaStream_t st) {
  constexpr int NSTAGE = Stages<KF>::v;
  const TileLayout L = tile_layout<D, KF, VF>(c.k.n_groups, c.v.n_groups);
  const int smem = NSTAGE * L.bytes;
  if (a.nsplit > kMaxSplits) return cudaErrorInvalidValue;
  static int configured = 0;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<D, G, KF, VF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         NSTAGE * tile_layout<D, KF, VF>(D / 16, D / 16).bytes);
    if (e != cudaSuccess) return e;
    configured = 1;
  }
  const dim3 grid(a.nsplit, c.Hkv, c.B);
  decode_tc_kernel<D, G, KF, VF><<<grid, kDecodeThreads, smem, st>>>(c, a);
  note_launch();
  return cudaGetLastError();
}

template <int D, int KF, int VF>
cudaError_t launch_decode_tc_d(const CacheView& c, int G, const DecodeArgs& a, cudaStream_t st) {
  switch (G) {
    case 1: return launch_decode_tc_dg<D, 1, KF, VF>(c, a, st);
    case 2: return launch_decode_tc_dg<D, 2, KF, VF>(c, a, st);
    case 3: return launch_decode_tc_dg<D, 3, KF, VF>(c, a, st);
    case 4: return launch_decode_tc_dg<D, 4, KF, VF>(c, a, st);
    case 5: return launch_decode_tc_dg<D, 5, KF, VF>(c, a, st);
    case 6: return launch_decode_tc_dg<D, 6, KF, VF>(c, a, st);
    case 7: return launch_decode_tc_dg<D, 7, KF, VF>(c, a, st);
    case 8: return launch_decode_tc_dg<D, 8, KF, VF>(c, a, st);
    default: return cudaErrorNotSupported;
  }
}

// Tensor-core path when its preconditions hold (head_dim 64 / 128, 16-bit io,
// every thread's key and value channels inside one metadata group), the
// CUDA-core kernel otherwise (exact fp32 arithmetic, used for fp32 outputs).
template <int KF, int VF>
cudaError_t launch_decode(const CacheView& c, int G, const DecodeArgs& a, cudaStream_t st) {
  constexpr bool K_AFF = (KF == F_AFF8 || KF == F_AFF4);
  constexpr bool V_AFF = (VF == F_AFF8 || VF == F_AFF4);
  const bool groups_ok = (!K_AFF || c.k.group >= c.D / 4) && (!V_AFF || c.v.group >= c.D / 8);
  if ((c.D == 64 || c.D == 128) && a.io_dtype != KVQ_DTYPE_F32 && groups_ok) {
    if (c.D == 128) return launch_decode_tc_d<128, KF, VF>(c, G, a, st);
    return launch_decode_tc_d<64, KF, VF>(c, G, a, st);
  }
  return launch_decode_cc<KF, VF>(c, G, a, st);
}

}  // namespace kvq
