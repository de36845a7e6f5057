// Fragment, tile and TMA helpers of the tensor-core decode kernel (decode_tc.cuh).
//
// A pipeline stage holds one 64-token tile: the K and V code planes arrive by
// TMA tensor copies (one per plane) with the hardware 16-byte-chunk swizzle of
// the row length (32 / 64 / 128 bytes; 256-byte rows as [row][2][128]), the
// per-token metadata planes by bulk copies.  One thread issues them and arms
// the stage's mbarrier with the byte count; every thread waits on the mbarrier
// (bounded in time) before reading the stage.
#pragma once

#include "async_copy.cuh"
#include "decode_impl.cuh"

namespace kvq {

__device__ __forceinline__ __half2 u2h(uint32_t x) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = x;
  return h;
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Eight nibbles of w (channel i in bits 4i..4i+3) as exact fp16 pairs:
// h[0] = (c0, c4), h[1] = (c1, c5), h[2] = (c2, c6), h[3] = (c3, c7).
// This is the exponent-bias ("magic number") integer-to-fp16 conversion of
// weight-only quantised GEMM kernels (Kim et al., "Who Says Elephants Can't
// Run", 2022): an fp16 with exponent field 25 (bits 0x6400) has a mantissa
// step of exactly 1 over [1024, 2048), so ORing a small integer n into the
// mantissa gives the fp16 1024 + n, and 0x6400 | (n << 4) gives 1024 + 16 n;
// one subtraction (or fma by 1/16) leaves n exactly.  OFF = 8 gives the
// signed levels n - 8 (Q4_0) instead.
template <int OFF = 0>
__device__ __forceinline__ void nibbles_to_h2(uint32_t w, __half2 (&h)[4]) {
  static_assert(OFF == 0 || OFF == 8, "offset");
  const uint32_t M = 0x64006400u;
  const __half2 kLow = u2h(OFF ? 0x64086408u : 0x64006400u);    // 1024 + OFF
  const __half2 k16th = u2h(0x2C002C00u);                         // 1/16
  const __half2 kHigh = u2h(OFF ? 0xD480D480u : 0xD400D400u);    // -(64 + OFF)
  const uint32_t w8 = w >> 8;
  h[0] = __hsub2(u2h((w & 0x000F000Fu) | M), kLow);
  h[1] = __hfma2(u2h((w & 0x00F000F0u) | M), k16th, kHigh);
  h[2] = __hsub2(u2h((w8 & 0x000F000Fu) | M), kLow);
  h[3] = __hfma2(u2h((w8 & 0x00F000F0u) | M), k16th, kHigh);
}

// Transpose of an 8 x 8 fp16 matrix held as mma fragments: lane l holds
// elements (l / 4, 2 (l % 4)) and (l / 4, 2 (l % 4) + 1) of the input and
// receives the same elements of the transpose.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

// N consecutive fp16 values (N = 1, 2 or 4; 2N-byte aligned) as fp32.
template <int N>
__device__ __forceinline__ void load_halves(const uint8_t* p, float (&f)[N]) {
  static_assert(N == 1 || N == 2 || N == 4, "count");
  if constexpr (N == 1) {
    f[0] = __half2float(*reinterpret_cast<const __half*>(p));
  } else if constexpr (N == 2) {
    const float2 a = __half22float2(u2h(*reinterpret_cast<const uint32_t*>(p)));
    f[0] = a.x; f[1] = a.y;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __half22float2(u2h(u.x)), b = __half22float2(u2h(u.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  }
}

// Four unsigned bytes of x as exact fp16 pairs: lo = (b0, b1), hi = (b2, b3),
// by the same exponent-bias conversion (byte b in the mantissa of 1024).
__device__ __forceinline__ void bytes_to_h2(uint32_t x, __half2& lo, __half2& hi) {
  const __half2 k1024 = u2h(0x64006400u);
  lo = __hsub2(u2h(__byte_perm(x, 0x64646464u, 0x5140u)), k1024);
  hi = __hsub2(u2h(__byte_perm(x, 0x64646464u, 0x7362u)), k1024);
}

// The same pairs as fp16 1024 + b (exact), without the subtraction.
__device__ __forceinline__ void bytes_to_h2_1024(uint32_t x, __half2& lo, __half2& hi) {
  lo = u2h(__byte_perm(x, 0x64646464u, 0x5140u));
  hi = u2h(__byte_perm(x, 0x64646464u, 0x7362u));
}

// Logical k index j of a 16-token block -> physical row inside the block.
// The value fragments of quad thread t read rows tau(2t), tau(2t + 1),
// tau(2t + 8), tau(2t + 9); the order is chosen so those reads are free of
// bank conflicts for the value row length: 64-byte (and shorter) rows use
// tau(2t + e) = t + 4e, tau(8 + 2t + e) = 8 + t + 4e; 128-byte and longer rows
// the identity.  Key loads are conflict-free under either.
template <int VROW>
__device__ __forceinline__ int tau(int j) {
  if constexpr (VROW >= 128) return j;
  else return (j & 8) + ((j & 7) >> 1) + 4 * (j & 1);
}

// Shared-memory byte offset of byte `off` of tile row r of a code plane whose
// rows are ROWB bytes, as the TMA swizzle places it: the 16-byte chunk index
// is XORed with address bits 7.. of the row (bits 7-9 for 128-byte spans,
// 7-8 for 64, 7 for 32); a 256-byte row is two 128-byte rows.
template <int ROWB>
__device__ __forceinline__ int swz_off(int r, int off) {
  if constexpr (ROWB == 256) {
    const int half = off >> 7;
    return r * 256 + half * 128 + ((((off >> 4) & 7) ^ ((2 * r + half) & 7)) << 4) + (off & 15);
  } else if constexpr (ROWB == 128) {
    return r * 128 + ((((off >> 4) ^ r) & 7) << 4) + (off & 15);
  } else if constexpr (ROWB == 64) {
    return r * 64 + ((((off >> 4) ^ (r >> 1)) & 3) << 4) + (off & 15);
  } else {
    static_assert(ROWB == 32, "code rows of 32, 64, 128 or 256 bytes");
    return r * 32 + ((((off >> 4) ^ (r >> 2)) & 1) << 4) + (off & 15);
  }
}

// ------------------------------------------------------------------- TMA --

// 64 rows of a code plane starting at row y (TMA tensor copy, swizzled).
template <int ROWB>
__device__ __forceinline__ void tma_rows(void* dst, const CUtensorMap* map, int y, uint64_t* m) {
  if constexpr (ROWB == 256) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];\n" ::"r"(smem_u32(dst)),
        "l"(map), "r"(0), "r"(0), "r"(y), "r"(smem_u32(m))
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];\n" ::"r"(smem_u32(dst)),
        "l"(map), "r"(0), "r"(y), "r"(smem_u32(m))
        : "memory");
  }
}

// Shared-memory ring of NSTAGE tile stages, in one of two layouts.
// Plane-major (PM): the K codes of stage s at kc + s * KCT and the V codes at
// vc + s * VCT (tiles of 64 rows, each a multiple of 1024 bytes, where the
// 128-byte swizzle pattern repeats), then each per-token metadata plane as one
// array of NSTAGE * 64 ring rows of this cache's row size, so that the
// metadata of a split's first tiles (consecutive rows in global memory) lands
// with one copy per plane: one-wave grids, whose CTAs request a whole split at
// once and wait on every copy request the SM's copy engine serves in turn.
// Stage-major (!PM): stage s is one block of STAGE bytes holding its tile's
// planes at fixed offsets: multi-wave grids of short rings, where plane bases
// that are compile-time constants save instructions in the loop.  In both,
// every region is sized for the largest group counts the kernel accepts (key
// scale groups of 32 channels, value groups of D / 8), and KIVI_BLOCK keys
// add the (scale, zero) rows of each stage's block.
template <int D, int KF, int VF, int NSTAGE, bool PM>
struct TcRing {
  static constexpr bool K_AFF = (KF == F_AFF8 || KF == F_AFF4);
  static constexpr bool K_Q40 = (KF == F_Q40);
  static constexpr bool V_AFF = (VF == F_AFF8 || VF == F_AFF4);
  static constexpr bool K_KIVIB = (KF == F_KIVIB8 || KF == F_KIVIB4);
  static constexpr int KCT = kTileTokens * D * FmtBits<KF>::v / 8;
  static constexpr int VCT = kTileTokens * D * FmtBits<VF>::v / 8;
  static_assert(KCT % 1024 == 0 && VCT % 1024 == 0, "code tiles keep the swizzle alignment");
  static constexpr int KMR_MAX = (K_AFF || K_Q40) ? 2 * (D / 32) : 0;   // metadata bytes per row, at most
  static constexpr int VMR_MAX = V_AFF ? 2 * 8 : 0;
  // one stage's planes at their largest (stage-major offsets)
  static constexpr int S_KS = KCT + VCT;
  static constexpr int S_KZ = S_KS + kTileTokens * KMR_MAX;
  static constexpr int S_VS = S_KZ + (K_AFF ? kTileTokens * KMR_MAX : 0);
  static constexpr int S_VZ = S_VS + kTileTokens * VMR_MAX;
  static constexpr int S_KBS = S_VZ + kTileTokens * VMR_MAX;
  static constexpr int S_KBZ = S_KBS + (K_KIVIB ? D * 2 : 0);
  static constexpr int STAGE = (S_KBZ + (K_KIVIB ? D * 2 : 0) + 1023) / 1024 * 1024;
  // plane-major region bases
  static constexpr int P_VC = NSTAGE * KCT;
  static constexpr int P_KS = P_VC + NSTAGE * VCT;
  static constexpr int P_KZ = P_KS + NSTAGE * kTileTokens * KMR_MAX;
  static constexpr int P_VS = P_KZ + (K_AFF ? NSTAGE * kTileTokens * KMR_MAX : 0);
  static constexpr int P_VZ = P_VS + NSTAGE * kTileTokens * VMR_MAX;
  static constexpr int P_KBS = P_VZ + NSTAGE * kTileTokens * VMR_MAX;
  static constexpr int P_KBZ = P_KBS + (K_KIVIB ? NSTAGE * D * 2 : 0);
  static constexpr int bytes = PM ? P_KBZ + (K_KIVIB ? NSTAGE * D * 2 : 0) : NSTAGE * STAGE;
  int kmr, vmr;     // this cache's metadata bytes per row of the key and value planes
  int tx_codes;     // bytes one tile's code planes (and block rows) bring
  int tx_meta;      // bytes one tile's metadata planes bring

  __host__ __device__ __forceinline__ TcRing(int kng, int vng) {
    kmr = (K_AFF || K_Q40) ? 2 * kng : 0;
    vmr = V_AFF ? 2 * vng : 0;
    tx_codes = KCT + VCT + (K_KIVIB ? 2 * D * 2 : 0);
    tx_meta = kTileTokens * ((K_AFF ? 2 : 1) * kmr + 2 * vmr);
  }
  // byte offsets of stage s's planes; row r of a metadata plane follows at
  // r times the plane's row size
  __device__ __forceinline__ int kc(int s) const { return PM ? s * KCT : s * STAGE; }
  __device__ __forceinline__ int vc(int s) const { return PM ? P_VC + s * VCT : s * STAGE + KCT; }
  __device__ __forceinline__ int ks(int s) const { return PM ? P_KS + s * kTileTokens * kmr : s * STAGE + S_KS; }
  __device__ __forceinline__ int kz(int s) const { return PM ? P_KZ + s * kTileTokens * kmr : s * STAGE + S_KZ; }
  __device__ __forceinline__ int vs(int s) const { return PM ? P_VS + s * kTileTokens * vmr : s * STAGE + S_VS; }
  __device__ __forceinline__ int vz(int s) const { return PM ? P_VZ + s * kTileTokens * vmr : s * STAGE + S_VZ; }
  __device__ __forceinline__ int kbs(int s) const { return PM ? P_KBS + s * D * 2 : s * STAGE + S_KBS; }
  __device__ __forceinline__ int kbz(int s) const { return PM ? P_KBZ + s * D * 2 : s * STAGE + S_KBZ; }
};

// One thread: the code planes (and KIVI_BLOCK block rows) of tile rows
// [row0, row0 + 64) into stage s, completing on m (whose expected bytes the
// caller has armed).
template <int D, int KF, int VF, class Ring>
__device__ __forceinline__ void issue_codes(uint8_t* smem, const Ring& R, int s, const CacheView& c, size_t bh,
                                            int row0, uint64_t* m) {
  constexpr int KROW = D * FmtBits<KF>::v / 8;
  constexpr int VROW = D * FmtBits<VF>::v / 8;
  const size_t row = bh * c.cap_alloc + row0;
  tma_rows<KROW>(smem + R.kc(s), &c.kmap, (int)row, m);
  tma_rows<VROW>(smem + R.vc(s), &c.vmap, (int)row, m);
  if constexpr (KF == F_KIVIB8 || KF == F_KIVIB4) {
    // the per-channel scale and zero of the tile's block (a tile never spans two)
    const size_t mr = (bh * (c.cap_alloc / c.k.group) + row0 / c.k.group) * D;
    bulk_copy(smem + R.kbs(s), c.k.blk_scale + mr, D * 2, m);
    bulk_copy(smem + R.kbz(s), c.k.blk_zero + mr, D * 2, m);
  }
}

// One thread: the per-token metadata of nt consecutive tiles from row0 on
// into stages s0 .. s0 + nt - 1, completing on m: one copy per plane (nt > 1
// only in the plane-major layout, where those stages' rows are contiguous).
template <class Ring>
__device__ __forceinline__ void issue_meta(uint8_t* smem, const Ring& R, int s0, int nt, const CacheView& c,
                                           size_t bh, int row0, uint64_t* m) {
  const size_t row = bh * c.cap_alloc + row0;
  const uint32_t rows = (uint32_t)(nt * kTileTokens);
  if constexpr (Ring::K_AFF || Ring::K_Q40) {
    bulk_copy(smem + R.ks(s0), reinterpret_cast<const uint8_t*>(c.k.tok_scale) + row * R.kmr, rows * R.kmr, m);
    if constexpr (Ring::K_AFF)
      bulk_copy(smem + R.kz(s0), reinterpret_cast<const uint8_t*>(c.k.tok_zero) + row * R.kmr, rows * R.kmr, m);
  }
  if constexpr (Ring::V_AFF) {
    bulk_copy(smem + R.vs(s0), reinterpret_cast<const uint8_t*>(c.v.tok_scale) + row * R.vmr, rows * R.vmr, m);
    bulk_copy(smem + R.vz(s0), reinterpret_cast<const uint8_t*>(c.v.tok_zero) + row * R.vmr, rows * R.vmr, m);
  }
}

// 2^x with the hardware's approximate base-2 exponential (ex2.approx.ftz: a
// couple of ulp, results below 2^-126 flushed to zero).  Used for softmax
// weights 2^(s - max) in (0, 1], where that error is far below the
// tolerance and the flushed weights are negligible.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}


// A hint: bring the line at p into L2 (and its page translation into the TLBs).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}

// A hint: bring `bytes` bytes at p into L2 with one bulk request (p 16-byte
// aligned, bytes a multiple of 16).  L2 is the GPU's point of coherence, so
// a prefetch issued before a producer kernel has finished writing cannot
// leave a stale copy behind; it only wastes bandwidth if the data changes.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

// Key channel order: k-step ks, mma k index 2t + jj (jj in {0, 1}) and
// 2t + 8 + jj of quad thread t.  4-bit codes: thread t reads word t of chunk
// ks / 2 (channels 32 (ks / 2) + 8 t + 0..7), nibble pairs (c0, c4), (c2, c6)
// for even ks and (c1, c5), (c3, c7) for odd ks.  8-bit and fp16: thread t
// reads channels 16 ks + 4 t + 0..3.  Either way k-steps 2p, 2p + 1 cover the
// 32-channel block p exactly.
template <int KB>
__device__ __forceinline__ void key_channels(int ks, int t, int (&ch)[4]) {
  if constexpr (KB == 4) {
    const int base = 32 * (ks >> 1) + 8 * t + (ks & 1);
    ch[0] = base; ch[1] = base + 4; ch[2] = base + 2; ch[3] = base + 6;
  } else {
    const int base = 16 * ks + 4 * t;
    ch[0] = base; ch[1] = base + 1; ch[2] = base + 2; ch[3] = base + 3;
  }
}

// Query values of quad thread t at the channels key_channels gives for every
// k-step, as fp32, from a 16-bit (bf16 / fp16) query row starting at element
// qo; zeros when !live.  A 16-byte aligned row is read with one 16-byte load
// per 32-channel block (4-bit keys: k-steps 2p, 2p + 1 take channels 32 p +
// 8 t + 0..7) or one 8-byte load per k-step (channels 16 ks + 4 t + 0..3);
// any other row element by element.
template <int D, int KB>
__device__ __forceinline__ void load_query_channels(const void* q, size_t qo, int io_dtype, int t, bool live,
                                                    float (&x)[D / 16][4]) {
  constexpr int KS = D / 16;
  const uint16_t* row = static_cast<const uint16_t*>(q) + qo;
  const bool bf = io_dtype == KVQ_DTYPE_BF16;
  auto f = [bf](uint32_t h16) {
    return bf ? __uint_as_float(h16 << 16) : __half2float(__ushort_as_half((unsigned short)h16));
  };
  if (!live) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) x[ks][0] = x[ks][1] = x[ks][2] = x[ks][3] = 0.0f;
  } else if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
    if constexpr (KB == 4) {
#pragma unroll
      for (int p = 0; p < KS / 2; ++p) {
        const uint4 w = *reinterpret_cast<const uint4*>(row + 32 * p + 8 * t);
        const float c0 = f(w.x & 0xffffu), c1 = f(w.x >> 16), c2 = f(w.y & 0xffffu), c3 = f(w.y >> 16);
        const float c4 = f(w.z & 0xffffu), c5 = f(w.z >> 16), c6 = f(w.w & 0xffffu), c7 = f(w.w >> 16);
        x[2 * p][0] = c0; x[2 * p][1] = c4; x[2 * p][2] = c2; x[2 * p][3] = c6;
        x[2 * p + 1][0] = c1; x[2 * p + 1][1] = c5; x[2 * p + 1][2] = c3; x[2 * p + 1][3] = c7;
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint2 w = *reinterpret_cast<const uint2*>(row + 16 * ks + 4 * t);
        x[ks][0] = f(w.x & 0xffffu); x[ks][1] = f(w.x >> 16); x[ks][2] = f(w.y & 0xffffu); x[ks][3] = f(w.y >> 16);
      }
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      int ch[4];
      key_channels<KB>(ks, t, ch);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[ks][i] = load_io(q, qo + ch[i], io_dtype);
    }
  }
}

}  // namespace kvq
