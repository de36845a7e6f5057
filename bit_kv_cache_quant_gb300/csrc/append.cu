// Quantise-on-append kernels.
//
// "StreamingLLM + KIVI" page, "Affine quantisation formula" and "KIVI": keys
// per channel, values per token, scale = max(eps, (max - min)/(qMax - qMin)),
// zero = min, codes round((x - zero)/scale) clamped to the level range.
// "Low-bit KV caches on MLX", section 1: the same affine rule per token and
// per 64-channel group.  "kv-cache: optional per-channel K-cache
// mean-centering for Q4_0": subtract the per-(kv head, channel) bias, then
// code symmetric blocks (32 channels, one fp16 scale: the Q4_0 layout, which
// the page does not spell out).
#include "async_copy.cuh"
#include "quantize_row.cuh"

namespace kvq {

// ---------------------------------------------------------------------------
// Per-channel K calibration: min / max over the n tokens of one (b, kv head),
// then the fp32 scale / zero that codes are computed from and their fp16
// stored copies.  One CTA of 256 threads per (b, kv head).  Thread tid reads
// VE consecutive channels of a token per load (one 16-byte load when the
// input is 16-byte aligned, VE = 16 / sizeof(T); single elements otherwise):
// tpr = D / VE threads cover a token row, 256 / tpr rows per sweep, and the
// sweeps' per-thread ranges are combined per channel in shared memory.
// Token t of (b, kv head) bh is row bh * hstride + t of k.
constexpr int kCalibThreads = 256;

template <typename T, int VE>
__global__ void __launch_bounds__(kCalibThreads) calibrate_kivi_kernel(CacheView c, const T* __restrict__ k, int n,
                                                                       long long hstride) {
  __shared__ float smn[kCalibThreads * VE];
  __shared__ float smx[kCalibThreads * VE];
  const int D = c.D;
  const int bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int tpr = D / VE;                 // threads per token row (divides 256)
  const int rps = kCalibThreads / tpr;    // token rows per sweep
  const int col = tid % tpr;
  float mn[VE], mx[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) {
    mn[e] = __int_as_float(0x7f800000);   // +inf
    mx[e] = __int_as_float(0xff800000);   // -inf
  }
  const T* base = k + (size_t)bh * hstride * D + col * VE;
  auto take = [&](const T* p) {
    alignas(16) T t[VE];
    if constexpr (VE * sizeof(T) == 16) {
      *reinterpret_cast<uint4*>(t) = __ldg(reinterpret_cast<const uint4*>(p));
    } else {
      static_assert(VE == 1, "16-byte vectors or single elements");
      t[0] = p[0];
    }
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      const float x = In<T>::ld(&t[e]);
      mn[e] = fminf(mn[e], x);
      mx[e] = fmaxf(mx[e], x);
    }
  };
  int t = tid / tpr;
  for (; t + 3 * rps < n; t += 4 * rps) {   // four rows in flight per thread
#pragma unroll
    for (int j = 0; j < 4; ++j) take(base + (size_t)(t + j * rps) * D);
  }
  for (; t < n; t += rps) take(base + (size_t)t * D);
#pragma unroll
  for (int e = 0; e < VE; ++e) {
    smn[tid * VE + e] = mn[e];
    smx[tid * VE + e] = mx[e];
  }
  __syncthreads();
  // channel ch = col * VE + e sits at [r * tpr + col][e] for each sweep row r
  for (int ch = tid; ch < D; ch += kCalibThreads) {
    const int cc = ch / VE, e = ch % VE;
    float a = smn[cc * VE + e], z = smx[cc * VE + e];
    for (int r = 1; r < rps; ++r) {
      a = fminf(a, smn[(r * tpr + cc) * VE + e]);
      z = fmaxf(z, smx[(r * tpr + cc) * VE + e]);
    }
    const float levels = (c.k.bits == 8) ? 255.0f : 15.0f;
    const float sc = affine_scale(a, z, levels);
    const size_t o = (size_t)bh * D + ch;
    c.k.ch_scale32[o] = sc;
    c.k.ch_zero32[o] = a;
    c.k.ch_scale[o] = __float2half_rn(sc);
    c.k.ch_zero[o] = __float2half_rn(a);
  }
  if (blockIdx.x == 0 && tid == 0) c.state->k_calibrated = 1;
}

// ---------------------------------------------------------------------------
// Recompute-on-append of the per-channel K range ("StreamingLLM + KIVI",
// "KIVI" and "Caveats": any new token may shift a channel's min / max, so the
// whole K block is coded again, O(T D) per append).  One CTA of 256 threads
// per (b, kv head): the stored keys are dequantised in fp32 from the stored
// fp16 scale and zero (u * s, then + z, each rounded once), the range is
// taken over them and the n new keys, the new fp32 scale / zero and their
// fp16 copies are written, and every stored key is coded again against them
// (byte by byte, so a 4-bit byte's two nibbles stay with one thread).  The new
// tokens are then coded by append_kernel with the new scales.  An append that
// would overflow changes nothing here (append_kernel reports it).
template <typename T>
__global__ void __launch_bounds__(256) recompute_kivi_kernel(CacheView c, const T* __restrict__ k, int n,
                                                             long long hstride) {
  __shared__ float s_old[128], z_old[128], s_new[128], z_new[128];
  __shared__ float smn[256];
  __shared__ float smx[256];
  __shared__ int s_T, s_ok;
  const int D = c.D;
  const size_t bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int d = tid % D;
  const int tg = tid / D;
  const int ntg = blockDim.x / D;
  if (tid == 0) {
    s_T = c.state->stored;
    s_ok = c.layout != KVQ_LAYOUT_RING && s_T + n <= c.cap;
  }
  if (tid < D) {
    s_old[tid] = __half2float(c.k.ch_scale[bh * D + tid]);
    z_old[tid] = __half2float(c.k.ch_zero[bh * D + tid]);
  }
  __syncthreads();
  if (!s_ok) return;
  const int Tn = s_T;
  const int bits = c.k.bits;
  const int rb = c.k.row_bytes;
  const float levels = (bits == 8) ? 255.0f : 15.0f;
  uint8_t* codes = c.k.codes + bh * c.cap_alloc * rb;
  float mn = __int_as_float(0x7f800000);   // +inf
  float mx = __int_as_float(0xff800000);   // -inf
  for (int t = tg; t < Tn; t += ntg) {
    const uint8_t byte = codes[(size_t)t * rb + (bits == 8 ? d : d / 2)];
    const int u = bits == 8 ? (byte ^ 0x80) : ((byte >> (4 * (d & 1))) & 15);
    const float x = __fadd_rn(__fmul_rn((float)u, s_old[d]), z_old[d]);
    mn = fminf(mn, x);
    mx = fmaxf(mx, x);
  }
  const T* base = k + bh * hstride * D;
  for (int t = tg; t < n; t += ntg) {
    const float x = In<T>::ld(base + (size_t)t * D + d);
    mn = fminf(mn, x);
    mx = fmaxf(mx, x);
  }
  smn[tid] = mn;
  smx[tid] = mx;
  __syncthreads();
  if (tg == 0) {
    for (int i = 1; i < ntg; ++i) {
      mn = fminf(mn, smn[i * D + d]);
      mx = fmaxf(mx, smx[i * D + d]);
    }
    const float sc = affine_scale(mn, mx, levels);
    s_new[d] = sc;
    z_new[d] = mn;
    const size_t o = bh * D + d;
    c.k.ch_scale32[o] = sc;
    c.k.ch_zero32[o] = mn;
    c.k.ch_scale[o] = __float2half_rn(sc);
    c.k.ch_zero[o] = __float2half_rn(mn);
  }
  __syncthreads();
  for (int i = tid; i < Tn * rb; i += blockDim.x) {
    uint8_t* p = codes + i;
    const int j = i % rb;
    if (bits == 8) {
      const float x = __fadd_rn(__fmul_rn((float)(*p ^ 0x80), s_old[j]), z_old[j]);
      *p = (uint8_t)(affine_code(x, s_new[j], z_new[j], levels) ^ 0x80);
    } else {
      const int c0 = 2 * j, c1 = 2 * j + 1;
      const float x0 = __fadd_rn(__fmul_rn((float)(*p & 15), s_old[c0]), z_old[c0]);
      const float x1 = __fadd_rn(__fmul_rn((float)(*p >> 4), s_old[c1]), z_old[c1]);
      *p = (uint8_t)(affine_code(x0, s_new[c0], z_new[c0], levels) | (affine_code(x1, s_new[c1], z_new[c1], levels) << 4));
    }
  }
  if (blockIdx.x == 0 && tid == 0) c.state->k_calibrated = 1;
}

// Append counters as a CTA reads them, and the check that the append fits.
struct AppendCounters {
  long long pos;
  int stored;
  int ok;
};

// Thread 0 of each CTA: the counters before this append; the first CTA
// reports an overflow (nothing is written then).
__device__ __forceinline__ void read_append_counters(const CacheView& c, int n, AppendCounters& a) {
  a.pos = c.state->pos;
  a.stored = c.state->stored;
  const bool ok = (c.layout == KVQ_LAYOUT_RING) || ((long long)a.stored + n <= c.cap);
  a.ok = ok ? 1 : 0;
  if (!ok && blockIdx.x == 0) set_status(c.state, KVQ_DEV_OVERFLOW);
}

// The cache slot of token i of the append, or -1 when a later token of the
// same append lands in that ring slot (the earlier one is never written).
__device__ __forceinline__ int append_slot(const CacheView& c, const AppendCounters& a, int n, int i) {
  if (c.layout != KVQ_LAYOUT_RING) return a.stored + i;
  const long long p = a.pos + i;
  if (p < c.sink) return (int)p;
  if (p < a.pos + n - c.window) return -1;
  return c.sink + (int)((p - c.sink) % c.window);
}

// Thread 0 of each CTA, after the CTA's rows are written: with more than one
// CTA the last to arrive advances the counters, once every CTA has read
// them; a one-CTA append advances them directly.
__device__ __forceinline__ void finish_append(const CacheView& c, const AppendCounters& a, int n) {
  bool last = true;
  if (gridDim.x > 1) {
    __threadfence();
    last = atomicAdd(&c.state->append_arrive, 1u) == gridDim.x - 1;
  }
  if (!last) return;
  if (a.ok) {
    const long long np = a.pos + n;
    c.state->pos = np;
    if (c.layout == KVQ_LAYOUT_RING) {
      const long long w = (long long)c.sink + c.window;
      c.state->stored = (int)(np < w ? np : w);
    } else {
      c.state->stored = a.stored + n;
    }
  }
  if (gridDim.x > 1) {
    c.state->append_arrive = 0u;
    __threadfence();
  }
}

// One warp per (b, kv head, token) row of the append; 8 warps per CTA.  Used
// for short appends (fewer tokens per (b, kv head) than a bulk chunk holds).
constexpr int kAppendWarps = 8;
constexpr int kAppendCtasPerSm = 8;

template <typename T, int E>
__global__ void __launch_bounds__(32 * kAppendWarps) append_kernel(CacheView c, const T* __restrict__ k,
                                                                    const T* __restrict__ v, int n, long long rows,
                                                                    long long hstride) {
  __shared__ AppendCounters s_cnt;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * kAppendWarps;   // rows per sweep of the grid
  long long row = (long long)blockIdx.x * kAppendWarps + warp;
  // token row % n of (b, kv head) row / n sits at row (row / n) * hstride + row % n of the input;
  // rows < B * Hkv * cap_alloc < 2^31 (the layout refuses larger caches), so 32-bit division suffices
  auto load = [&](long long r, float (&xk)[E], float (&xv)[E]) {
    const unsigned q = (unsigned)r / (unsigned)n, i = (unsigned)r % (unsigned)n;
    const long long src = (long long)q * hstride + i;
    load_row_slice<T, E>(k + src * c.D + lane * E, xk);
    load_row_slice<T, E>(v + src * c.D + lane * E, xv);
  };
  // launched as a programmatic dependent: the inputs and counters may come
  // from the previous kernel; the next launch may start its prologue now
  grid_dependency_wait();
  grid_launch_dependents();
  float xk[E], xv[E];
  if (row < rows) load(row, xk, xv);
  if (threadIdx.x == 0) read_append_counters(c, n, s_cnt);
  __syncthreads();
  const AppendCounters a = s_cnt;
  // a warp codes rows row, row + stride, ...: the grid is capped at a few
  // CTAs per SM (one arrival each on the append counter), and each warp
  // requests its next row before coding the current one
  for (; a.ok && row < rows; row += stride) {
    float nk[E], nv[E];
    const bool more = row + stride < rows;
    if (more) load(row + stride, nk, nv);
    const int i = (int)((unsigned)row % (unsigned)n);
    const long long bh = (unsigned)row / (unsigned)n;
    const int kvh = (int)((unsigned)bh % (unsigned)c.Hkv);
    const int slot = append_slot(c, a, n, i);
    if (slot >= 0) {
      const float* bias = c.k_bias ? c.k_bias + (size_t)kvh * c.D : nullptr;
      quantize_row<E>(c.k, bias, xk, bh, c.cap_alloc, slot, lane);
      quantize_row<E>(c.v, nullptr, xv, bh, c.cap_alloc, slot, lane);
    }
    if (more) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        xk[e] = nk[e];
        xv[e] = nv[e];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) finish_append(c, a, n);
}

// ---------------------------------------------------------------------------
// Bulk append (kvq_convert, prefill-sized appends).  The input tokens of one
// (b, kv head) are consecutive rows, so the work is cut into chunks of
// 256 / (D / 32) = 8192 / D tokens of one (b, kv head).  CTA x takes chunks
// x, x + grid, ... (the grid is the resident CTA count); thread 0 copies each
// chunk's K rows and V rows into one of the shared-memory stages with two bulk
// copies on one mbarrier, one stage ahead of the chunk being coded.
//
// Thread t of the 256 codes channels [32 p, 32 p + 32) (its part p = t % (D /
// 32)) of token row t / (D / 32) of the chunk, first of K, then of V, with the
// formats' fp32 rules.  A part holds a whole Q4_0 block, two 16-channel affine
// groups, one 32-channel group, or half / a quarter of a 64 / 128-channel
// group, whose range the 2 / 4 lanes of the group then combine with
// shuffles; divisions and reciprocals are taken once per part.  Codes come
// from one reciprocal per group (per channel for KIVI keys); a quotient
// within 2^-13 of a rounding tie (rare) is taken again with the exact
// division (code_side states the bound), so the bytes equal the exact rule's.
// Parts are read from shared memory as 16-byte units, starting at unit
// `rot` and wrapping, so that the threads of a shared-memory wavefront hit
// distinct banks; each unit's codes are stored at the unit's own offset.
constexpr int kBulkThreads = 256;
constexpr int kBulkMinTokens = 32;   // shorter appends take append_kernel
constexpr int kPart = 32;   // channels per thread and side

template <typename T>
struct BulkShape {
  static constexpr int UE = 16 / (int)sizeof(T);     // elements per 16-byte unit
  static constexpr int NU = kPart / UE;              // units per part
  static constexpr int stages = 2;   // 64 KB per CTA for 16-bit inputs: three CTAs (24 warps) per SM
  static constexpr int stage_bytes = 2 * 8192 * (int)sizeof(T);   // K and V rows of one chunk
  static constexpr int smem = stages * stage_bytes;
};

// Per-chunk parameters of KIVI_CHAN keys staged in shared memory: the fp32
// scale, its reciprocal and the zero of each channel of the chunk's (b, kv head).
struct KiviParams {
  float sc[128];
  float inv[128];
  float zr[128];
};

// The Q4_0 centering bias of keys stored without centering.
__device__ __align__(16) const float kZeroBias[128] = {};

// How a side is coded by the bulk kernel (one code path each).
enum BulkKind { BK_FP16, BK_Q40, BK_KIVI8, BK_KIVI4, BK_AFF8, BK_AFF4, BK_AFF8_G16, BK_AFF4_G16 };

__device__ __forceinline__ int bulk_kind(const SideView& s) {
  switch (s.fmt) {
    case KVQ_FMT_FP16: return BK_FP16;
    case KVQ_FMT_Q4_0: return BK_Q40;
    case KVQ_FMT_KIVI_CHAN: return s.bits == 8 ? BK_KIVI8 : BK_KIVI4;
    default:
      if (s.group == 16) return s.bits == 8 ? BK_AFF8_G16 : BK_AFF4_G16;
      return s.bits == 8 ? BK_AFF8 : BK_AFF4;
  }
}

// Codes one side's part: the thread's 32 channels [32 part, 32 part + 32) of
// one staged row (x in register order: unit (jj + rot) % NU of the part in
// slots [jj UE, jj UE + UE)), with the formats' fp32 rules, and stores the
// codes (each unit's at its own offset) and the part's metadata.  Codes come
// from one reciprocal per group (per channel for KIVI_CHAN): the product is
// within 2^-15 of the exact quotient wherever the code depends on it, so a
// quotient further than 2^-13 from a rounding tie rounds as the exact one
// does; the few nearer a tie (a 16-byte unit is checked at once) are taken
// again with the exact division.
template <typename T, int KIND>
__device__ __forceinline__ void code_side(const SideView& sv, float (&x)[kPart], int rot, int part, int lane,
                                          size_t orow, const float* __restrict__ bias, const KiviParams& kp) {
  using S = BulkShape<T>;
  constexpr bool Q40 = KIND == BK_Q40;
  constexpr bool CHAN = KIND == BK_KIVI8 || KIND == BK_KIVI4;
  constexpr bool G16 = KIND == BK_AFF8_G16 || KIND == BK_AFF4_G16;
  constexpr int BITS = (KIND == BK_KIVI8 || KIND == BK_AFF8 || KIND == BK_AFF8_G16) ? 8 : 4;
  constexpr float LEVELS = BITS == 8 ? 255.0f : 15.0f;
  constexpr float LO = Q40 ? -8.0f : 0.0f, HI = Q40 ? 7.0f : LEVELS;
  uint8_t* out = sv.codes + orow * sv.row_bytes;
  const size_t meta = orow * sv.n_groups;
  if constexpr (KIND == BK_FP16) {
    __half* o = reinterpret_cast<__half*>(out) + part * kPart;
#pragma unroll
    for (int jj = 0; jj < S::NU; ++jj) {
      alignas(16) __half h[S::UE];
#pragma unroll
      for (int e = 0; e < S::UE; ++e) h[e] = __float2half_rn(x[jj * S::UE + e]);
      __half* dst = o + ((jj + rot) % S::NU) * S::UE;
      if constexpr (S::UE == 8) *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(h);
      else *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(h);
    }
    return;
  } else {
    // scale s, zero z and reciprocal i of the part's group(s): [0] the first
    // 16-channel half, [1] the second (the same group unless G16)
    float s0 = 0.0f, s1 = 0.0f, z0 = 0.0f, z1 = 0.0f, i0 = 0.0f, i1 = 0.0f;
    if constexpr (Q40) {   // centre (bias 0 without centering), then one symmetric block
      float m = 0.0f;
#pragma unroll
      for (int jj = 0; jj < S::NU; ++jj) {
        const int uu = (jj + rot) % S::NU;
#pragma unroll
        for (int q = 0; q < S::UE; q += 4) {
          const float4 b4 = __ldg(reinterpret_cast<const float4*>(bias + part * kPart + uu * S::UE + q));
          const float bq[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float& xe = x[jj * S::UE + q + e];
            xe = __fsub_rn(xe, bq[e]);
            m = fmaxf(m, fabsf(xe));
          }
        }
      }
      s0 = __fdiv_rn(m, 7.0f);
      i0 = __frcp_rn(s0);   // inf when s0 == 0 (the all-zero block is stored directly)
      sv.tok_scale[meta + part] = __float2half_rn(s0);
    } else if constexpr (!CHAN) {
      float mn0 = __int_as_float(0x7f800000), mx0 = __int_as_float(0xff800000);   // +inf, -inf
      float mn1 = mn0, mx1 = mx0;
#pragma unroll
      for (int jj = 0; jj < S::NU; ++jj) {
        const bool second = G16 && ((jj + rot) % S::NU) * S::UE >= 16;
#pragma unroll
        for (int e = 0; e < S::UE; ++e) {
          const float xe = x[jj * S::UE + e];
          if (G16) {
            mn0 = second ? mn0 : fminf(mn0, xe);
            mx0 = second ? mx0 : fmaxf(mx0, xe);
            mn1 = second ? fminf(mn1, xe) : mn1;
            mx1 = second ? fmaxf(mx1, xe) : mx1;
          } else {
            mn0 = fminf(mn0, xe);
            mx0 = fmaxf(mx0, xe);
          }
        }
      }
      if constexpr (G16) {
        s0 = affine_scale(mn0, mx0, LEVELS);
        s1 = affine_scale(mn1, mx1, LEVELS);
        z0 = mn0;
        z1 = mn1;
        sv.tok_scale[meta + 2 * part] = __float2half_rn(s0);
        sv.tok_zero[meta + 2 * part] = __float2half_rn(z0);
        sv.tok_scale[meta + 2 * part + 1] = __float2half_rn(s1);
        sv.tok_zero[meta + 2 * part + 1] = __float2half_rn(z1);
      } else {
        const int ppg = sv.group / kPart;   // lanes per group: 1, 2 or 4 (consecutive, one row)
        if (ppg > 1) {
          const unsigned mask = ((1u << ppg) - 1u) << (lane & ~(ppg - 1));
          for (int o = 1; o < ppg; o <<= 1) {
            mn0 = fminf(mn0, __shfl_xor_sync(mask, mn0, o));
            mx0 = fmaxf(mx0, __shfl_xor_sync(mask, mx0, o));
          }
        }
        s0 = s1 = affine_scale(mn0, mx0, LEVELS);
        z0 = z1 = mn0;
        if (part % ppg == 0) {
          sv.tok_scale[meta + part / ppg] = __float2half_rn(s0);
          sv.tok_zero[meta + part / ppg] = __float2half_rn(z0);
        }
      }
      i0 = __frcp_rn(s0);
      i1 = G16 ? __frcp_rn(s1) : i0;
    }
    const float* psc = kp.sc + part * kPart;
    const float* pinv = kp.inv + part * kPart;
    const float* pzr = kp.zr + part * kPart;
    // Rounding: adding MAGIC = 1.5 * 2^23 + OFF to a value v in [-2^21, 2^21]
    // rounds it to the nearest integer, ties to even, and leaves OFF + rint(v)
    // in the low bits of the sum; OFF = 8 gives the Q4_0 nibble u + 8, OFF =
    // -128 the int8 byte u ^ 0x80 (the signed level u - 128), OFF = 0 the
    // 4-bit code.  The quotient is first clamped to the level range where it
    // can leave it: per-channel KIVI scales come from a calibration that later
    // tokens may exceed; a per-token group's own range bounds its quotients to
    // [0, levels (1 + 2^-22)] and a Q4_0 block's to [-7 (1 + 2^-22), 7 (1 +
    // 2^-22)], so there only NaN (from non-finite inputs) needs the lower
    // clamp, which maps it to the level the exact rule gives it.  Rounding the
    // clamped value equals clamping the rounded one: the bounds are integers.
    constexpr float OFF = Q40 ? 8.0f : (BITS == 8 ? -128.0f : 0.0f);
    constexpr float MAGIC = 0x1.8p23f + OFF;
    auto clamp = [&](float t) { return CHAN ? fminf(fmaxf(t, LO), HI) : fmaxf(t, LO); };
    uint8_t* o = out + part * (kPart * BITS / 8);
    constexpr int UB = S::UE * BITS / 8;   // bytes per unit: 2, 4 or 8
#pragma unroll
    for (int jj = 0; jj < S::NU; ++jj) {
      const int uu = (jj + rot) % S::NU;
      [[maybe_unused]] const bool second = G16 && uu * S::UE >= 16;
      float y[S::UE], dd[S::UE];
      float far = 0.0f;   // the unit's largest distance of a rounded quotient from its integer
#pragma unroll
      for (int e = 0; e < S::UE; ++e) {
        float inv;
        if constexpr (Q40) {
          dd[e] = x[jj * S::UE + e];
          inv = i0;
        } else if constexpr (CHAN) {
          dd[e] = __fsub_rn(x[jj * S::UE + e], pzr[uu * S::UE + e]);
          inv = pinv[uu * S::UE + e];
        } else {
          dd[e] = __fsub_rn(x[jj * S::UE + e], second ? z1 : z0);
          inv = second ? i1 : i0;
        }
        const float tc = clamp(__fmul_rn(dd[e], inv));
        y[e] = __fadd_rn(tc, MAGIC);
        far = fmaxf(far, fabsf(__fsub_rn(tc, __fsub_rn(y[e], MAGIC))));
      }
      if (far > 0.5f - 0x1p-13f) {
        // a quotient within 2^-13 of a tie: there the exact quotient decides
        // (the reciprocal's is within 2^-15 of it for |quotient| <= 256)
#pragma unroll
        for (int e = 0; e < S::UE; ++e) {
          float sc, inv;
          if constexpr (Q40) {
            sc = s0;
            inv = i0;
          } else if constexpr (CHAN) {
            sc = psc[uu * S::UE + e];
            inv = pinv[uu * S::UE + e];
          } else {
            sc = second ? s1 : s0;
            inv = second ? i1 : i0;
          }
          const float tc = clamp(__fmul_rn(dd[e], inv));
          if (fabsf(__fsub_rn(tc, __fsub_rn(y[e], MAGIC))) > 0.5f - 0x1p-13f)
            y[e] = __fadd_rn(clamp(__fdiv_rn(dd[e], sc)), MAGIC);
        }
      }
      if constexpr (Q40) {
        if (s0 == 0.0f) {   // an all-zero block stores level 0 (nibble 8) throughout
#pragma unroll
          for (int e = 0; e < S::UE; ++e) y[e] = MAGIC;
        }
      }
      // the low byte of each sum is the stored byte (8-bit) or nibble (4-bit)
      uint32_t b[S::UE / 4];
#pragma unroll
      for (int q = 0; q < S::UE / 4; ++q) {
        const uint32_t lo = __byte_perm(__float_as_uint(y[4 * q]), __float_as_uint(y[4 * q + 1]), 0x0040);
        const uint32_t hi = __byte_perm(__float_as_uint(y[4 * q + 2]), __float_as_uint(y[4 * q + 3]), 0x0040);
        b[q] = __byte_perm(lo, hi, 0x5410);
      }
      uint8_t* dst = o + uu * UB;
      if constexpr (BITS == 8) {
        if constexpr (UB == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(b[0], b[1]);
        else *reinterpret_cast<uint32_t*>(dst) = b[0];
      } else {
        // bytes c0..c3 (each < 16) -> nibble pairs c0 | c1 << 4 and c2 | c3 << 4 in bytes 0 and 2
#pragma unroll
        for (int q = 0; q < S::UE / 4; ++q) b[q] |= b[q] >> 4;
        if constexpr (UB == 4) *reinterpret_cast<uint32_t*>(dst) = __byte_perm(b[0], b[1], 0x6420);
        else *reinterpret_cast<uint16_t*>(dst) = (uint16_t)__byte_perm(b[0], 0u, 0x0020);
      }
    }
  }
}

template <typename T>
__device__ __forceinline__ void code_side_any(int kind, const SideView& sv, float (&x)[kPart], int rot, int part,
                                              int lane, size_t orow, const float* bias, const KiviParams& kp) {
  switch (kind) {
    case BK_FP16: code_side<T, BK_FP16>(sv, x, rot, part, lane, orow, bias, kp); break;
    case BK_Q40: code_side<T, BK_Q40>(sv, x, rot, part, lane, orow, bias, kp); break;
    case BK_KIVI8: code_side<T, BK_KIVI8>(sv, x, rot, part, lane, orow, bias, kp); break;
    case BK_KIVI4: code_side<T, BK_KIVI4>(sv, x, rot, part, lane, orow, bias, kp); break;
    case BK_AFF8: code_side<T, BK_AFF8>(sv, x, rot, part, lane, orow, bias, kp); break;
    case BK_AFF4: code_side<T, BK_AFF4>(sv, x, rot, part, lane, orow, bias, kp); break;
    case BK_AFF8_G16: code_side<T, BK_AFF8_G16>(sv, x, rot, part, lane, orow, bias, kp); break;
    default: code_side<T, BK_AFF4_G16>(sv, x, rot, part, lane, orow, bias, kp); break;
  }
}

template <typename T, int E>
__global__ void __launch_bounds__(kBulkThreads, 3) append_bulk_kernel(CacheView c, const T* __restrict__ k,
                                                                    const T* __restrict__ v, int n,
                                                                    long long hstride) {
  using S = BulkShape<T>;
  constexpr int D = 32 * E;
  constexpr int P = D / kPart;          // parts per row
  constexpr int CH = kBulkThreads / P;  // tokens per chunk
  constexpr int NS = S::stages;
  constexpr int half = S::stage_bytes / 2;
  extern __shared__ __align__(128) unsigned char bulk_smem[];
  __shared__ __align__(8) uint64_t full[NS];
  __shared__ AppendCounters s_cnt;
  __shared__ KiviParams s_kp;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int part = tid % P;
  const int row = tid / P;
  const int nch = (n + CH - 1) / CH;                 // chunks per (b, kv head)
  const int units = c.B * c.Hkv * nch;               // < rows < 2^31
  const int G = gridDim.x;
  const int kind_k = bulk_kind(c.k), kind_v = bulk_kind(c.v);
  auto stage_k = [&](int s) { return reinterpret_cast<T*>(bulk_smem + s * S::stage_bytes); };
  auto stage_v = [&](int s) { return reinterpret_cast<T*>(bulk_smem + s * S::stage_bytes + half); };
  // chunk j of this CTA (global chunk blockIdx.x + j G) into stage j % NS
  auto issue = [&](int j) {
    const int u = blockIdx.x + j * G;
    const int bh = u / nch, i0 = (u - bh * nch) * CH;
    const uint32_t bytes = (uint32_t)min(CH, n - i0) * (uint32_t)(D * sizeof(T));
    const int s = j % NS;
    const size_t src = ((size_t)bh * hstride + i0) * D;
    mbar_expect_tx(&full[s], 2 * bytes);
    bulk_copy(stage_k(s), k + src, bytes, &full[s]);
    bulk_copy(stage_v(s), v + src, bytes, &full[s]);
  };
  int issued = 0;   // chunks requested so far (thread 0)
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  // launched as a programmatic dependent: the inputs and counters may come
  // from the previous kernel; the next launch may start its prologue now
  grid_dependency_wait();
  grid_launch_dependents();
  if (tid == 0) {
    for (; issued < NS && (int)blockIdx.x + issued * G < units; ++issued) issue(issued);
    read_append_counters(c, n, s_cnt);
  }
  __syncthreads();
  const AppendCounters a = s_cnt;
  // bank spread: the 8 threads of a shared-memory wavefront start at distinct 16-byte columns
  const int rot = S::NU >= 8 ? lane % S::NU : (lane * S::NU / 8) % S::NU;
  bool timed_out = false;
  int j = 0;
  for (; a.ok && (int)blockIdx.x + j * G < units; ++j) {
    const int s = j % NS;
    const int u = blockIdx.x + j * G;
    const int bh = u / nch, i0 = (u - bh * nch) * CH;
    const bool ready = mbar_wait_bounded(&full[s], (uint32_t)(j / NS) & 1u);
    // every thread has coded chunk j - 1: its stage takes the next chunk
    if (__syncthreads_or(!ready)) {
      timed_out = true;
      break;
    }
    if (tid == 0 && j > 0 && (int)blockIdx.x + issued * G < units) {
      fence_async_smem();   // the stage's shared-memory reads come before the copy engine's writes
      issue(issued++);
    }
    if (kind_k == BK_KIVI8 || kind_k == BK_KIVI4) {   // the chunk's per-channel K parameters
      if (tid < D) {
        const float sc = c.k.ch_scale32[(size_t)bh * D + tid];
        s_kp.sc[tid] = sc;
        s_kp.inv[tid] = __frcp_rn(sc);
        s_kp.zr[tid] = c.k.ch_zero32[(size_t)bh * D + tid];
      }
      __syncthreads();
    }
    const int slot = row < min(CH, n - i0) ? append_slot(c, a, n, i0 + row) : -1;
    if (slot < 0) continue;   // all parts of the row skip together
    const size_t orow = (size_t)bh * c.cap_alloc + slot;
    const float* bias = c.k_bias ? c.k_bias + (size_t)(bh % c.Hkv) * D : kZeroBias;
#pragma unroll 1
    for (int side = 0; side < 2; ++side) {
      const T* src = (side == 0 ? stage_k(s) : stage_v(s)) + row * D + part * kPart;
      float x[kPart];
#pragma unroll
      for (int jj = 0; jj < S::NU; ++jj) {
        alignas(16) T t[S::UE];
        *reinterpret_cast<uint4*>(t) = *reinterpret_cast<const uint4*>(src + ((jj + rot) % S::NU) * S::UE);
#pragma unroll
        for (int e = 0; e < S::UE; ++e) x[jj * S::UE + e] = In<T>::ld(&t[e]);
      }
      code_side_any<T>(side == 0 ? kind_k : kind_v, side == 0 ? c.k : c.v, x, rot, part, lane, orow, bias, s_kp);
    }
  }
  __syncthreads();
  if (tid != 0) return;
  // copies still in flight after an overflow or a timeout land before the CTA exits
  for (; j < issued; ++j) mbar_wait_bounded(&full[j % NS], (uint32_t)(j / NS) & 1u);
  if (timed_out) set_status(c.state, KVQ_DEV_TIMEOUT);
  finish_append(c, a, n);
}

// ---------------------------------------------------------------------------
// KIVI residual buffer (KIVI_BLOCK keys; the format's description in kvq.h).
// The tail (t rows) followed by the n new tokens is one sequence; each run of
// R that completes is a closed block.  Grid (nbm + 1, B * Hkv), nbm the most
// blocks an append of n can close: CTA x < nbm codes block x of its (b, kv
// head) if that block closes; the new tail is written by CTA 0 after its block
// has read the old tail, or by CTA nbm when no block closes.  The last CTA to
// arrive advances the counters, once every CTA has read them.
template <typename T, int E>
__global__ void __launch_bounds__(256) residual_append_kernel(CacheView c, const T* __restrict__ k,
                                                              const T* __restrict__ v, int n, long long hstride) {
  constexpr int D = 32 * E;
  constexpr int NW = 8;
  __shared__ long long s_pos;
  __shared__ int s_stored, s_tail, s_ok;
  __shared__ float s_part[2][NW][D];   // per-warp channel min / max
  __shared__ float s_sc[D], s_zr[D];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int R = c.k.group;
  const size_t bh = blockIdx.y;
  const int nbm = gridDim.x - 1;
  if (threadIdx.x == 0) {
    s_pos = c.state->pos;
    s_stored = c.state->stored;
    s_tail = c.state->tail;
    const long long nb = ((long long)s_tail + n) / R;
    const bool ok = (long long)s_stored + nb * R <= (c.cap / R) * R;
    s_ok = ok ? 1 : 0;
    if (!ok && blockIdx.x == 0 && blockIdx.y == 0) set_status(c.state, KVQ_DEV_OVERFLOW);
  }
  __syncthreads();
  const int t_old = s_tail;
  const int nb = (t_old + n) / R;
  const int j = blockIdx.x;
  // token i of the sequence (tail, then input), this lane's E channels, as fp32
  auto load_tok = [&](const float* tail, const T* in, int i, float (&x)[E]) {
    if (i < t_old) {
      const float* p = tail + (bh * R + i) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) x[e] = p[e];
    } else {
      load_row_slice<T, E>(in + ((long long)bh * hstride + (i - t_old)) * D + lane * E, x);
    }
  };
  if (s_ok && j < nb) {
    const float levels = (c.k.bits == 8) ? 255.0f : 15.0f;
    // keys: each channel's range over the block's R tokens
    float mn[E], mx[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      mn[e] = __int_as_float(0x7f800000);    // +inf
      mx[e] = __int_as_float(0xff800000);    // -inf
    }
    for (int r = warp; r < R; r += NW) {
      float x[E];
      load_tok(c.tail_k, k, j * R + r, x);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        mn[e] = fminf(mn[e], x[e]);
        mx[e] = fmaxf(mx[e], x[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      s_part[0][warp][lane * E + e] = mn[e];
      s_part[1][warp][lane * E + e] = mx[e];
    }
    __syncthreads();
    const int blk = s_stored / R + j;
    for (int ch = threadIdx.x; ch < D; ch += blockDim.x) {
      float a = s_part[0][0][ch], z = s_part[1][0][ch];
#pragma unroll
      for (int w = 1; w < NW; ++w) {
        a = fminf(a, s_part[0][w][ch]);
        z = fmaxf(z, s_part[1][w][ch]);
      }
      const float sc = affine_scale(a, z, levels);
      s_sc[ch] = sc;
      s_zr[ch] = a;
      const size_t mrow = (bh * (c.cap_alloc / R) + blk) * D + ch;
      c.k.blk_scale[mrow] = __float2half_rn(sc);
      c.k.blk_zero[mrow] = __float2half_rn(a);
    }
    __syncthreads();
    for (int r = warp; r < R; r += NW) {
      const int slot = s_stored + j * R + r;
      float x[E];
      load_tok(c.tail_k, k, j * R + r, x);
      int u[E];
#pragma unroll
      for (int e = 0; e < E; ++e) u[e] = affine_code(x[e], s_sc[lane * E + e], s_zr[lane * E + e], levels);
      store_codes<E>(c.k.codes + (bh * c.cap_alloc + slot) * c.k.row_bytes, lane, c.k.bits, u);
      float y[E];
      load_tok(c.tail_v, v, j * R + r, y);
      quantize_row<E>(c.v, nullptr, y, bh, c.cap_alloc, slot, lane);
    }
  }
  // the new tail: sequence tokens [nb R, t_old + n) become tail rows 0 ..
  if (s_ok && (nb == 0 ? j == nbm : j == 0)) {
    __syncthreads();   // CTA 0's reads of the old tail are done
    const int first = nb == 0 ? t_old : 0;               // first tail row written
    const int count = nb == 0 ? n : t_old + n - nb * R;  // rows written (all from the input)
    const int in0 = nb == 0 ? 0 : nb * R - t_old;        // their first input token
    for (int r = warp; r < count; r += NW) {
      float x[E], y[E];
      load_row_slice<T, E>(k + ((long long)bh * hstride + in0 + r) * D + lane * E, x);
      load_row_slice<T, E>(v + ((long long)bh * hstride + in0 + r) * D + lane * E, y);
      float* pk = c.tail_k + (bh * R + first + r) * D + lane * E;
      float* pv = c.tail_v + (bh * R + first + r) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        pk[e] = x[e];
        pv[e] = y[e];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  __threadfence();
  if (atomicAdd(&c.state->append_arrive, 1u) == gridDim.x * gridDim.y - 1) {
    if (s_ok) {
      c.state->pos = s_pos + n;
      c.state->stored = s_stored + nb * R;
      c.state->tail = t_old + n - nb * R;
    }
    c.state->append_arrive = 0u;
    __threadfence();
  }
}

// ---------------------------------------------------------------- launch --

// The staged bulk kernel: shared memory opted in and the resident CTA count
// looked up once per device, the grid that count (or the chunk count).
template <typename T, int E>
static cudaError_t launch_bulk(const CacheView& c, const T* k, const T* v, int n, long long hstride, int sms,
                               cudaLaunchConfig_t cfg) {
  static std::atomic<unsigned long long> done{0};
  static std::atomic<int> per_sm[64];   // resident CTAs per SM, per device (0 until looked up)
  constexpr int smem = BulkShape<T>::smem;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = once_per_device(done, [&]() {
    cudaError_t r = cudaFuncSetAttribute(append_bulk_kernel<T, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (r != cudaSuccess) return r;
    int b = 0;
    r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, append_bulk_kernel<T, E>, kBulkThreads, smem);
    if (r == cudaSuccess && dev >= 0 && dev < 64) per_sm[dev].store(b > 0 ? b : 1, std::memory_order_relaxed);
    return r;
  });
  if (e != cudaSuccess) return e;
  constexpr int rows = kBulkThreads / (E * 32 / kPart);   // tokens per chunk
  const int b = dev >= 0 && dev < 64 ? per_sm[dev].load(std::memory_order_relaxed) : 0;
  const long long resident = (long long)(b > 0 ? b : 1) * sms;
  const long long units = (long long)c.B * c.Hkv * ((n + rows - 1) / rows);
  cfg.gridDim = dim3((unsigned)(units < resident ? units : resident));
  cfg.blockDim = dim3(kBulkThreads);
  cfg.dynamicSmemBytes = smem;
  return cudaLaunchKernelEx(&cfg, append_bulk_kernel<T, E>, c, k, v, n, hstride);
}

template <typename T>
static cudaError_t launch_append_t(const CacheView& c, const void* k, const void* v, int n, long long hstride,
                                   bool calibrate, bool recompute, cudaStream_t st) {
  if (calibrate) {
    constexpr int VE = 16 / (int)sizeof(T);
    if ((reinterpret_cast<uintptr_t>(k) & 15) == 0 && c.D % VE == 0)
      calibrate_kivi_kernel<T, VE><<<c.B * c.Hkv, kCalibThreads, 0, st>>>(c, static_cast<const T*>(k), n, hstride);
    else
      calibrate_kivi_kernel<T, 1><<<c.B * c.Hkv, kCalibThreads, 0, st>>>(c, static_cast<const T*>(k), n, hstride);
    note_launch();
  }
  if (recompute) {
    recompute_kivi_kernel<T><<<c.B * c.Hkv, 256, 0, st>>>(c, static_cast<const T*>(k), n, hstride);
    note_launch();
  }
  const T* kk = static_cast<const T*>(k);
  const T* vv = static_cast<const T*>(v);
  if (c.k.fmt == KVQ_FMT_KIVI_BLOCK) {
    const int R = c.k.group;
    const dim3 grid((unsigned)((R - 1 + n) / R + 1), (unsigned)(c.B * c.Hkv));
    switch (c.D) {
      case 32: residual_append_kernel<T, 1><<<grid, 256, 0, st>>>(c, kk, vv, n, hstride); break;
      case 64: residual_append_kernel<T, 2><<<grid, 256, 0, st>>>(c, kk, vv, n, hstride); break;
      case 128: residual_append_kernel<T, 4><<<grid, 256, 0, st>>>(c, kk, vv, n, hstride); break;
      default: return cudaErrorInvalidValue;
    }
    note_launch();
    return cudaGetLastError();
  }
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const int sms = c.sms > 0 ? c.sms : 132;
  // prefill-sized appends with 16-byte aligned inputs: the staged kernel
  const bool aligned = ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) == 0;
  if (n >= kBulkMinTokens && aligned) {
    cudaError_t e;
    switch (c.D) {
      case 32: e = launch_bulk<T, 1>(c, kk, vv, n, hstride, sms, cfg); break;
      case 64: e = launch_bulk<T, 2>(c, kk, vv, n, hstride, sms, cfg); break;
      case 128: e = launch_bulk<T, 4>(c, kk, vv, n, hstride, sms, cfg); break;
      default: return cudaErrorInvalidValue;
    }
    note_launch();
    return e;
  }
  const long long rows = (long long)c.B * c.Hkv * n;
  // at most kAppendCtasPerSm CTAs per SM; their warps sweep the rows
  const long long need = (rows + kAppendWarps - 1) / kAppendWarps;
  const long long cap = (long long)kAppendCtasPerSm * sms;
  cfg.gridDim = dim3((unsigned)(need < cap ? need : cap));
  cfg.blockDim = dim3(32 * kAppendWarps);
  cudaError_t e;
  switch (c.D) {
    case 32: e = cudaLaunchKernelEx(&cfg, append_kernel<T, 1>, c, kk, vv, n, rows, hstride); break;
    case 64: e = cudaLaunchKernelEx(&cfg, append_kernel<T, 2>, c, kk, vv, n, rows, hstride); break;
    case 128: e = cudaLaunchKernelEx(&cfg, append_kernel<T, 4>, c, kk, vv, n, rows, hstride); break;
    default: return cudaErrorInvalidValue;
  }
  note_launch();
  return e;
}

cudaError_t launch_append(const CacheView& c, const void* k, const void* v, int n, long long hstride, int in_dtype,
                          bool calibrate, bool recompute, cudaStream_t st) {
  switch (in_dtype) {
    case KVQ_DTYPE_F32: return launch_append_t<float>(c, k, v, n, hstride, calibrate, recompute, st);
    case KVQ_DTYPE_BF16: return launch_append_t<__nv_bfloat16>(c, k, v, n, hstride, calibrate, recompute, st);
    case KVQ_DTYPE_F16: return launch_append_t<__half>(c, k, v, n, hstride, calibrate, recompute, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
