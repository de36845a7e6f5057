// Fused single-query GQA decode attention over the packed cache.
//
// "Low-bit KV caches on MLX", section 5: decode attention spends its time
// reading the cache; fused kernels read packed bytes and dequantise in
// registers.  "StreamingLLM + KIVI", "Affine quantisation formula": the
// attention runs on x_dq = (q - qMin) * scale + zero with the stored fp16
// scales upcast to fp32.  mlx-qsdpa (same memo, section 5) splits long
// contexts; here every (b, kv head) is split over `nsplit` CTAs whose
// partial (max, sum, accumulator) triples are merged with the online-softmax
// rule by the last CTA of the (b, kv head) to finish.
//
// Data movement: a CTA streams its token range through shared memory in
// 64-token tiles.  A tile is a handful of contiguous byte ranges (K codes,
// V codes and each metadata plane for those 64 rows), copied with 16-byte
// cp.async by all threads, NSTAGE tiles ahead of the one being computed.
//
// Work mapping: a token row of D channels is read by D/16 lanes, each lane
// owning 16 consecutive channels (8, 16 or 32 bytes of codes: one shared-
// memory vector load).  A warp covers 32/(D/16) tokens at a time.  The G
// query heads that share a kv head are computed together so each code is
// read once.
//
// Arithmetic kept out of the per-element loop:
//  * per-token affine keys: q . k_hat = s * sum(q_i u_i) + z * sum(q_i) over
//    the lane's channels (one group), so the inner loop is one FMA per head;
//  * Q4_0 keys: d * (sum(q_i u_i) - 8 sum(q_i));
//  * per-channel KIVI keys: q_i * s_i is folded into the query once; the
//    sum(q_i z_i) term is the same for every token of a row and is dropped,
//    which the softmax does not see (the shift-invariance argument of the
//    mean-centering page, "Why this is safe");
//  * per-token affine values: acc += (p * s) u_i, plus p * z once per token.
// Codes become floats exactly through the IEEE bit pattern 2^23 + u
// (byte-permute into the mantissa, subtract 2^23).
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

constexpr int kDecodeWarps = 4;
constexpr int kDecodeThreads = 32 * kDecodeWarps;
constexpr int kTileTokens = 64;       // divides kRowAlign: whole tiles stay inside cap_alloc

template <int F> struct FmtBits {
  static constexpr int v = (F == F_FP16) ? 16 : ((F == F_KIVI8 || F == F_AFF8 || F == F_KIVIB8) ? 8 : 4);
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Codes of one lane's 16 channels.
template <int BITS> struct Codes { uint32_t w[BITS / 2]; };

template <int BITS>
__device__ __forceinline__ void load_codes_smem(Codes<BITS>& c, const uint8_t* p) {
  if constexpr (BITS == 16) {
    const uint4 a = reinterpret_cast<const uint4*>(p)[0];
    const uint4 b = reinterpret_cast<const uint4*>(p)[1];
    c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
    c.w[4] = b.x; c.w[5] = b.y; c.w[6] = b.z; c.w[7] = b.w;
  } else if constexpr (BITS == 8) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
  } else {
    const uint2 a = *reinterpret_cast<const uint2*>(p);
    c.w[0] = a.x; c.w[1] = a.y;
  }
}

// float(byte k of w), exact: the pattern 0x4B0000bb is 2^23 + bb.
__device__ __forceinline__ float byte_to_float(uint32_t w, int k) {
  return __int_as_float(__byte_perm(w, 0x4B000000u, 0x7440u + k)) - 8388608.0f;
}

// Unsigned codes u (or the fp16 values) of the lane's 16 channels, in order.
template <int BITS>
__device__ __forceinline__ void unpack(const Codes<BITS>& c, float (&x)[16]) {
  if constexpr (BITS == 16) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      __half2 h;
      *reinterpret_cast<uint32_t*>(&h) = c.w[i];
      const float2 f = __half22float2(h);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  } else if constexpr (BITS == 8) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w = c.w[i] ^ 0x80808080u;   // signed level q -> u = q + 128
#pragma unroll
      for (int k = 0; k < 4; ++k) x[4 * i + k] = byte_to_float(w, k);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t lo = c.w[i] & 0x0F0F0F0Fu;          // channels 8i + 2k
      const uint32_t hi = (c.w[i] >> 4) & 0x0F0F0F0Fu;   // channels 8i + 2k + 1
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[8 * i + 2 * k] = byte_to_float(lo, k);
        x[8 * i + 2 * k + 1] = byte_to_float(hi, k);
      }
    }
  }
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Byte offsets of one pipeline stage (one 64-token tile) in shared memory.
struct TileLayout {
  int kc, vc, ks, kz, vs, vz, kbs, kbz, bytes;
  int tx;   // bytes actually transferred into a stage
};

template <int D, int KF, int VF>
__host__ __device__ __forceinline__ TileLayout tile_layout(int kng, int vng) {
  constexpr int KROW = D * FmtBits<KF>::v / 8;
  constexpr int VROW = D * FmtBits<VF>::v / 8;
  constexpr bool K_AFF = (KF == F_AFF8 || KF == F_AFF4);
  constexpr bool K_Q40 = (KF == F_Q40);
  constexpr bool V_AFF = (VF == F_AFF8 || VF == F_AFF4);
  TileLayout L;
  int off = 0;
  L.kc = off; off += kTileTokens * KROW;
  L.vc = off; off += kTileTokens * VROW;
  L.ks = off; off += (K_AFF || K_Q40) ? kTileTokens * kng * 2 : 0;
  L.kz = off; off += K_AFF ? kTileTokens * kng * 2 : 0;
  L.vs = off; off += V_AFF ? kTileTokens * vng * 2 : 0;
  L.vz = off; off += V_AFF ? kTileTokens * vng * 2 : 0;
  // KIVI_BLOCK keys: the per-channel scale and zero of the tile's block (a tile
  // never spans two blocks: the block length is a multiple of 64)
  constexpr bool K_KIVIB = (KF == F_KIVIB8 || KF == F_KIVIB4);
  L.kbs = off; off += K_KIVIB ? D * 2 : 0;
  L.kbz = off; off += K_KIVIB ? D * 2 : 0;
  L.bytes = off;   // every term is a multiple of 64 bytes
  L.tx = off;
  return L;
}

// Rows [t0, t1) of split `split` and the number of live splits `nse` for a
// cache holding T rows, with at most `nsplit` splits (the grid): whole 64-row
// tiles spread evenly, at least 4 tiles per split from 4096 rows on and 1
// below.  Every CTA reads the same T, so all agree on nse; splits past nse
// have no rows and take no part in the merge.
__device__ __forceinline__ void split_rows(int T, int nsplit, int split, int& t0, int& t1, int& nse) {
  const int nt = (T + kTileTokens - 1) / kTileTokens;
  int tps = (nt + nsplit - 1) / nsplit;
  const int min_tiles = T >= 4096 ? 4 : 1;
  if (tps < min_tiles) tps = min_tiles;
  nse = nt > 0 ? (nt + tps - 1) / tps : 1;
  t0 = min(T, split * tps * kTileTokens);
  t1 = min(T, t0 + tps * kTileTokens);
}

// Global add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// The counter update of a fused append + decode step: every CTA of the grid
// reads the counters first, then the last merge of the grid writes these.
struct StepUpdate {
  bool on = false;    // a fused step
  bool ok = false;    // the token was stored (a LINEAR cache was not full)
  long long pos = 0;  // counters after the step
  int stored = 0;
};

// Threads per output float4 in the cross-split merge: the largest of 8, 4, 2
// that fits the CTA with a whole number of warps, else 1.
__host__ __device__ constexpr int merge_lanes(int items, int threads) {
  return (items * 8 <= threads && (items * 8) % 32 == 0)   ? 8
         : (items * 4 <= threads && (items * 4) % 32 == 0) ? 4
         : (items * 2 <= threads && (items * 2) % 32 == 0) ? 2
                                                            : 1;
}

// Merges the per-warp (max, sum, accumulator) triples in shared memory and writes
// the output (one split) or this split's partial; the last split of a (b, kv head)
// to finish merges every partial with the online-softmax rule.
// Accumulator layout: ACCPAD == 0: acc[warp][h][d]; ACCPAD > 0 (tensor-core
// kernel): rows of D + ACCPAD floats, channel d at (d % (D/8)) * 8 + d / (D/8).
// HG > 1: warp w holds only heads 4 j .. 4 j + 3, j = (w / 4) % HG, and the
// other heads' entries of that warp are not read.  EXTRA = 1: one more state
// per head after the warps' (row NWARP of sm_m / sm_l), whose accumulator row
// ex_acc (laid out like a warp's, the same for every head) enters only when
// its weight is not zero.
// One (b, kv head) of a fused step is done: the last of the grid's B * Hkv
// to get here (after every CTA of the grid has read the counters) writes the
// new counters.
__device__ __forceinline__ void step_arrive(const CacheView& c, const StepUpdate& step) {
  const unsigned units = (unsigned)c.B * (unsigned)c.Hkv;
  if (atom_add_acq_rel_gpu(&c.state->step_arrive, 1u) == units - 1) {
    if (step.ok) {
      c.state->pos = step.pos;
      c.state->stored = step.stored;
    } else {
      set_status(c.state, KVQ_DEV_OVERFLOW);
    }
    c.state->step_arrive = 0u;
  }
}

// STEP (a fused step): every CTA of the (b, kv head) arrives, with rows or
// without (splits >= nse write nothing), the last arrival merges when there
// are several live splits, and the last such arrival of the grid advances
// the cache counters (or reports an overflow).
template <int D, int G, int ACCPAD, int NWARP = kDecodeWarps, int HG = 1, int EXTRA = 0, bool STEP = false>
__device__ __forceinline__ void merge_store(const CacheView& c, const DecodeArgs& a, int b, int kvh, int split, int nse,
                                            float (*sm_m)[G], float (*sm_l)[G], const float* sm_acc,
                                            const float* ex_acc = nullptr, StepUpdate step = StepUpdate{}) {
  constexpr int PROW = D + kPartialPad;
  constexpr int AROW = D + ACCPAD;
  constexpr int NTHR = 32 * NWARP;
  constexpr int NW = NWARP + EXTRA;
  static_assert(NW <= 32 && EXTRA <= 1, "one lane per state in the per-head reduction");
  __shared__ float sm_w[kMaxSplits][G];
  __shared__ float sm_lsum[kMaxSplits][G];
  __shared__ float sm_inv[G];
  __shared__ float sm_we[NW][G];      // weight of state w in head h's CTA merge
  __shared__ float sm_hm[G];          // CTA max and sum of each head
  __shared__ float sm_hl[G];
  __shared__ int s_last;
  const size_t bh = (size_t)b * c.Hkv + kvh;
  // Merge the warps.  One warp per head first finds the CTA's max over the
  // warps holding that head, each warp's weight 2^(m_w - M) and the weighted
  // sum, so that every (head, channel) output then takes one multiply-add per
  // warp; then write the output (one split) or this split's partial.
  {
    const int lane = threadIdx.x & 31;
    for (int h = threadIdx.x >> 5; h < G; h += NWARP) {
      const bool mine = lane < NW && (lane >= NWARP || HG == 1 || ((lane >> 2) % HG) == (h >> 2));
      const float mw = mine ? sm_m[lane][h] : neg_inf();
      float M = mw;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float e = (mw == neg_inf()) ? 0.0f : exp2f(mw - M);
      float L = mine ? sm_l[lane][h] * e : 0.0f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
      if (lane < NW) sm_we[lane][h] = e;
      if (lane == 0) {
        sm_hm[h] = M;
        sm_hl[h] = L;
      }
    }
  }
  __syncthreads();
  // Consecutive threads read consecutive accumulator words (no bank
  // conflicts): with ACCPAD > 0 word p of a row holds channel
  // (p % 8) * (D / 8) + p / 8.
  for (int idx = threadIdx.x; idx < G * D; idx += NTHR) {
    const int h = idx / D, p = idx % D;
    const int d = ACCPAD ? (p % 8) * (D / 8) + p / 8 : p;
    const int pos = h * AROW + p;
    const float M = sm_hm[h], L = sm_hl[h];
    float A = 0.0f;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) {
      if (HG > 1 && ((w >> 2) % HG) != (h >> 2)) continue;
      A = fmaf(sm_acc[w * G * AROW + pos], sm_we[w][h], A);
    }
    if constexpr (EXTRA) {
      const float e = sm_we[NWARP][h];
      A = e != 0.0f ? fmaf(ex_acc[p], e, A) : A;
    }
    if (STEP && split >= nse) {
      // a fused step's CTA without rows: nothing to write
    } else if (nse == 1) {
      const size_t oo = ((size_t)b * a.Hq + (size_t)kvh * G + h) * D + d;
      store_io(a.out, oo, a.io_dtype, L > 0.0f ? A / L : 0.0f);
    } else {
      float* P = a.partials + ((bh * a.nsplit + split) * G + h) * PROW;
      P[d] = A;
      if (d == 0) {
        P[D] = M;
        P[D + 1] = L;
      }
    }
  }
  if (!STEP && nse == 1) return;

  // The last split of this (b, kv head) to finish merges all partials.  The
  // barrier orders every thread's partial stores before thread 0's arrival,
  // whose release side publishes them at GPU scope and whose acquire side
  // (for the last arrival) makes the other splits' partials visible to the
  // whole CTA after the second barrier.
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned arrivals = STEP ? gridDim.x : (unsigned)nse;
    const bool last = atom_add_acq_rel_gpu(&c.split_sem[bh], 1u) == arrivals - 1;
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  if (STEP && nse == 1) {   // a fused step with one live split: its output is written
    if (threadIdx.x == 0) {
      c.split_sem[bh] = 0u;
      step_arrive(c, step);
    }
    return;
  }
  if (threadIdx.x == NTHR - 1) {
    // every CTA of this (b, kv head) has arrived, so the counter can be reset
    // and (fused step) every one of them has read the cache counters: the
    // grid-wide arrival goes out now, its round trip overlapping the merge's
    // loads, from the last thread (whose warp the float4 merge leaves idle
    // whenever it needs fewer threads than the CTA has)
    c.split_sem[bh] = 0u;
    if constexpr (STEP) step_arrive(c, step);
  }
  const float* P0 = a.partials + bh * a.nsplit * G * PROW;
  // Thread layout of the merge: SPL threads (adjacent lanes) per float4 of the
  // G x D output, each summing every SPL-th split.  The first PF partial
  // vectors of a thread's first float4 are requested before the weights are
  // known, so the partial data costs about one round trip to L2.
  constexpr int ITEMS = G * D / 4;
  constexpr int SPL = merge_lanes(ITEMS, NTHR);
  constexpr int PF = SPL <= 2 ? 16 : 8;
  constexpr int kStrideF4 = G * PROW / 4;   // float4 stride between splits
  float4 pre[PF];
  if (threadIdx.x < ITEMS * SPL) {
    const int item = threadIdx.x / SPL, sub = threadIdx.x % SPL;
    const float4* src = reinterpret_cast<const float4*>(P0 + (item / (D / 4)) * PROW) + item % (D / 4);
#pragma unroll
    for (int j = 0; j < PF; ++j) {
      const int sp = sub + j * SPL;
      pre[j] = sp < nse ? __ldcg(src + (size_t)sp * kStrideF4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // Every split's (max, sum) at once; then one warp per head reduces them with
  // shuffles and leaves one weight per (split, head).
  for (int i = threadIdx.x; i < nse * G; i += NTHR) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(P0 + i * PROW + D));
    sm_w[i / G][i % G] = ml.x;
    sm_lsum[i / G][i % G] = ml.y;
  }
  __syncthreads();
  {
    const int lane = threadIdx.x & 31;
    for (int h = threadIdx.x >> 5; h < G; h += NWARP) {
      float M = neg_inf();
      for (int sp = lane; sp < nse; sp += 32) M = fmaxf(M, sm_w[sp][h]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float L = 0.0f;
      for (int sp = lane; sp < nse; sp += 32) {
        const float ms = sm_w[sp][h];
        const float e = (ms == neg_inf()) ? 0.0f : exp2f(ms - M);
        L = fmaf(sm_lsum[sp][h], e, L);
        sm_w[sp][h] = e;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
      if (lane == 0) sm_inv[h] = L > 0.0f ? 1.0f / L : 0.0f;
    }
  }
  __syncthreads();
  // ITEMS * SPL is a multiple of 32 whenever SPL > 1, so every lane of a warp
  // runs the same iterations and the shuffles below see the whole warp.
  for (int base = threadIdx.x; base < ITEMS * SPL; base += NTHR) {
    const int item = base / SPL, sub = base % SPL;
    const int h = item / (D / 4), d4 = item % (D / 4);
    const float4* src = reinterpret_cast<const float4*>(P0 + h * PROW) + d4;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    int j0 = 0;
    if (base == threadIdx.x) {
#pragma unroll
      for (int j = 0; j < PF; ++j) {
        const int sp = sub + j * SPL;
        const float e = sp < nse ? sm_w[sp][h] : 0.0f;
        A.x = fmaf(pre[j].x, e, A.x);
        A.y = fmaf(pre[j].y, e, A.y);
        A.z = fmaf(pre[j].z, e, A.z);
        A.w = fmaf(pre[j].w, e, A.w);
      }
      j0 = PF;
    }
    for (int j1 = j0; sub + j1 * SPL < nse; j1 += 8) {
      float4 p[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int sp = sub + (j1 + j) * SPL;
        p[j] = sp < nse ? __ldcg(src + (size_t)sp * kStrideF4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int sp = sub + (j1 + j) * SPL;
        const float e = sp < nse ? sm_w[sp][h] : 0.0f;
        A.x = fmaf(p[j].x, e, A.x);
        A.y = fmaf(p[j].y, e, A.y);
        A.z = fmaf(p[j].z, e, A.z);
        A.w = fmaf(p[j].w, e, A.w);
      }
    }
#pragma unroll
    for (int o = SPL / 2; o > 0; o >>= 1) {
      A.x += __shfl_xor_sync(0xffffffffu, A.x, o);
      A.y += __shfl_xor_sync(0xffffffffu, A.y, o);
      A.z += __shfl_xor_sync(0xffffffffu, A.z, o);
      A.w += __shfl_xor_sync(0xffffffffu, A.w, o);
    }
    if (sub != 0) continue;
    const float inv = sm_inv[h];
    const size_t oo = ((size_t)b * a.Hq + (size_t)kvh * G + h) * D + 4 * d4;
    store_io(a.out, oo + 0, a.io_dtype, A.x * inv);
    store_io(a.out, oo + 1, a.io_dtype, A.y * inv);
    store_io(a.out, oo + 2, a.io_dtype, A.z * inv);
    store_io(a.out, oo + 3, a.io_dtype, A.w * inv);
  }
}

template <int KF> struct Stages { static constexpr int v = (KF == F_FP16) ? 3 : 4; };

// Copies rows [row0, row0 + 64) of every plane of one (b, kv head) into a stage.
template <int D, int KF, int VF>
__device__ __forceinline__ void issue_tile(uint8_t* st, const TileLayout& L, const CacheView& c, size_t bh,
                                           int row0) {
  constexpr int KROW = D * FmtBits<KF>::v / 8;
  constexpr int VROW = D * FmtBits<VF>::v / 8;
  constexpr bool K_AFF = (KF == F_AFF8 || KF == F_AFF4);
  constexpr bool K_Q40 = (KF == F_Q40);
  constexpr bool V_AFF = (VF == F_AFF8 || VF == F_AFF4);
  const size_t row = bh * c.cap_alloc + row0;
  const int tid = threadIdx.x;
  {
    const uint8_t* src = c.k.codes + row * KROW;
    for (int i = tid; i < kTileTokens * KROW / 16; i += kDecodeThreads) cp_async16(st + L.kc + 16 * i, src + 16 * i);
  }
  {
    const uint8_t* src = c.v.codes + row * VROW;
    for (int i = tid; i < kTileTokens * VROW / 16; i += kDecodeThreads) cp_async16(st + L.vc + 16 * i, src + 16 * i);
  }
  if constexpr (K_AFF || K_Q40) {
    const int n16 = kTileTokens * c.k.n_groups * 2 / 16;
    const uint8_t* s1 = reinterpret_cast<const uint8_t*>(c.k.tok_scale + row * c.k.n_groups);
    for (int i = tid; i < n16; i += kDecodeThreads) cp_async16(st + L.ks + 16 * i, s1 + 16 * i);
    if constexpr (K_AFF) {
      const uint8_t* s2 = reinterpret_cast<const uint8_t*>(c.k.tok_zero + row * c.k.n_groups);
      for (int i = tid; i < n16; i += kDecodeThreads) cp_async16(st + L.kz + 16 * i, s2 + 16 * i);
    }
  }
  if constexpr (V_AFF) {
    const int n16 = kTileTokens * c.v.n_groups * 2 / 16;
    const uint8_t* s1 = reinterpret_cast<const uint8_t*>(c.v.tok_scale + row * c.v.n_groups);
    const uint8_t* s2 = reinterpret_cast<const uint8_t*>(c.v.tok_zero + row * c.v.n_groups);
    for (int i = tid; i < n16; i += kDecodeThreads) {
      cp_async16(st + L.vs + 16 * i, s1 + 16 * i);
      cp_async16(st + L.vz + 16 * i, s2 + 16 * i);
    }
  }
  if constexpr (KF == F_KIVIB8 || KF == F_KIVIB4) {
    const size_t m = (bh * (c.cap_alloc / c.k.group) + row0 / c.k.group) * D;
    const uint8_t* s1 = reinterpret_cast<const uint8_t*>(c.k.blk_scale + m);
    const uint8_t* s2 = reinterpret_cast<const uint8_t*>(c.k.blk_zero + m);
    for (int i = tid; i < D * 2 / 16; i += kDecodeThreads) {
      cp_async16(st + L.kbs + 16 * i, s1 + 16 * i);
      cp_async16(st + L.kbz + 16 * i, s2 + 16 * i);
    }
  }
}

template <int D, int G, int KF, int VF>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(CacheView c, DecodeArgs a) {
  constexpr int NL = D / 16;                  // lanes per token
  constexpr int TPW = 32 / NL;                // tokens per warp per step
  constexpr int TPC = TPW * kDecodeWarps;     // tokens per CTA per step
  constexpr int C = kTileTokens / TPC;        // steps per tile
  constexpr int NSTAGE = Stages<KF>::v;
  constexpr int KB = FmtBits<KF>::v;
  constexpr int VB = FmtBits<VF>::v;
  constexpr int KROW = D * KB / 8;
  constexpr int VROW = D * VB / 8;
  constexpr bool K_AFF = (KF == F_AFF8 || KF == F_AFF4);
  constexpr bool K_KIVI = (KF == F_KIVI8 || KF == F_KIVI4);
  constexpr bool K_Q40 = (KF == F_Q40);
  constexpr bool V_AFF = (VF == F_AFF8 || VF == F_AFF4);
  constexpr bool K_KIVIB = (KF == F_KIVIB8 || KF == F_KIVIB4);

  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_tail;
  __shared__ float sm_m[kDecodeWarps][G];
  __shared__ float sm_l[kDecodeWarps][G];
  __shared__ __align__(16) float sm_acc[kDecodeWarps][G][D];
  __shared__ int s_T;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int j = lane % NL;                    // channel slice [16j, 16j + 16)
  const int grp = lane / NL;
  const int slot = warp * TPW + grp;
  const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
  const size_t bh = (size_t)b * c.Hkv + kvh;
  const int kng = c.k.n_groups;
  const int vng = c.v.n_groups;
  const TileLayout TL = tile_layout<D, KF, VF>(kng, vng);

  if (threadIdx.x == 0) {
    s_T = c.state->stored;
    s_tail = K_KIVIB ? c.state->tail : 0;
  }
  __syncthreads();
  const int T = s_T;
  int t0, t1, nse;
  split_rows(T, a.nsplit, split, t0, t1, nse);
  // KIVI_BLOCK: CTA a.nsplit attends over the full-precision tail and merges as
  // one more split (partial slot nse, after the bulk's); a cache with no
  // closed block has no bulk splits.
  const int TT = s_tail;
  const bool is_tail = K_KIVIB && split == a.nsplit;
  if (K_KIVIB && T == 0) nse = TT > 0 ? 0 : 1;
  const int nse_all = nse + (TT > 0 ? 1 : 0);
  if (is_tail ? TT == 0 : split >= nse) return;   // no rows for this CTA
  const int ntiles = is_tail ? 0 : (t1 - t0 + kTileTokens - 1) / kTileTokens;

  // Start streaming before anything else.
#pragma unroll
  for (int s = 0; s < NSTAGE - 1; ++s) {
    if (s < ntiles) issue_tile<D, KF, VF>(smem + s * TL.bytes, TL, c, bh, t0 + s * kTileTokens);
    cp_async_commit();
  }

  // Query slice, pre-scaled by softmax_scale * log2(e) so exp2 can be used.
  float qf[G][16];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const size_t qo = ((size_t)b * a.Hq + (size_t)kvh * G + h) * D + 16 * j;
#pragma unroll
    for (int i = 0; i < 16; ++i) qf[h][i] = load_io(a.q, qo + i, a.io_dtype) * a.qscale;
  }
  if constexpr (K_KIVI) {
    const __half* cs = c.k.ch_scale + bh * D + 16 * j;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float s = __half2float(cs[i]);
#pragma unroll
      for (int h = 0; h < G; ++h) qf[h][i] *= s;
    }
  }
  float qsum[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += qf[h][i];
    qsum[h] = s;
  }
  const int kg = K_AFF ? (16 * j) / c.k.group : (K_Q40 ? (j >> 1) : 0);
  const int vg = V_AFF ? (16 * j) / c.v.group : 0;

  float m[G], l[G], zacc[G], acc[G][16];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = neg_inf();
    l[h] = 0.0f;
    zacc[h] = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[h][i] = 0.0f;
  }

  for (int it = 0; it < ntiles; ++it) {
    cp_async_wait<NSTAGE - 2>();
    __syncthreads();
    {
      const int nx = it + NSTAGE - 1;
      if (nx < ntiles) issue_tile<D, KF, VF>(smem + (nx % NSTAGE) * TL.bytes, TL, c, bh, t0 + nx * kTileTokens);
      cp_async_commit();
    }
    const uint8_t* st = smem + (it % NSTAGE) * TL.bytes;
    const int tbase = t0 + it * kTileTokens;

    // Scores (log2 domain) of this lane-group's C tokens of the tile.
    float s[C][G];
#pragma unroll
    for (int cc = 0; cc < C; ++cc) {
      const int r = cc * TPC + slot;
      Codes<KB> kc;
      load_codes_smem<KB>(kc, st + TL.kc + r * KROW + j * (KROW / NL));
      float x[16];
      unpack<KB>(kc, x);
      if constexpr (K_KIVIB) {
        // the block's per-channel scale and zero, in fp32: k = s u + z
        const __half* bs = reinterpret_cast<const __half*>(st + TL.kbs) + 16 * j;
        const __half* bz = reinterpret_cast<const __half*>(st + TL.kbz) + 16 * j;
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = fmaf(__half2float(bs[i]), x[i], __half2float(bz[i]));
      }
      float ksc = 0.0f, kzr = 0.0f;
      if constexpr (K_AFF || K_Q40) ksc = __half2float(reinterpret_cast<const __half*>(st + TL.ks)[r * kng + kg]);
      if constexpr (K_AFF) kzr = __half2float(reinterpret_cast<const __half*>(st + TL.kz)[r * kng + kg]);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float p = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) p = fmaf(qf[h][i], x[i], p);
        if constexpr (K_AFF) p = fmaf(ksc, p, kzr * qsum[h]);
        if constexpr (K_Q40) p = ksc * fmaf(-8.0f, qsum[h], p);
        s[cc][h] = p;
      }
    }
#pragma unroll
    for (int cc = 0; cc < C; ++cc) {
      const bool valid = tbase + cc * TPC + slot < t1;
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int o = NL / 2; o >= 1; o >>= 1) s[cc][h] += __shfl_xor_sync(0xffffffffu, s[cc][h], o);
        if (!valid) s[cc][h] = neg_inf();
      }
    }

    // Online softmax: one rescale per tile.
    float pw[C][G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float mc = s[0][h];
#pragma unroll
      for (int cc = 1; cc < C; ++cc) mc = fmaxf(mc, s[cc][h]);
      const float mn = fmaxf(m[h], mc);
      if (mn == neg_inf()) {
#pragma unroll
        for (int cc = 0; cc < C; ++cc) pw[cc][h] = 0.0f;
        continue;
      }
      const float alpha = exp2f(m[h] - mn);
      l[h] *= alpha;
      zacc[h] *= alpha;
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[h][i] *= alpha;
      m[h] = mn;
#pragma unroll
      for (int cc = 0; cc < C; ++cc) {
        pw[cc][h] = exp2f(s[cc][h] - mn);
        l[h] += pw[cc][h];
      }
    }
#pragma unroll
    for (int cc = 0; cc < C; ++cc) {
      // rows past the split's end hold whatever the buffer held (possibly NaN
      // metadata or fp16 values): skip them rather than weight them by zero
      if (tbase + cc * TPC + slot >= t1) continue;
      const int r = cc * TPC + slot;
      Codes<VB> vcod;
      load_codes_smem<VB>(vcod, st + TL.vc + r * VROW + j * (VROW / NL));
      float x[16];
      unpack<VB>(vcod, x);
      float vsc = 0.0f, vzr = 0.0f;
      if constexpr (V_AFF) {
        vsc = __half2float(reinterpret_cast<const __half*>(st + TL.vs)[r * vng + vg]);
        vzr = __half2float(reinterpret_cast<const __half*>(st + TL.vz)[r * vng + vg]);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if constexpr (V_AFF) {
          const float w = pw[cc][h] * vsc;
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[h][i] = fmaf(w, x[i], acc[h][i]);
          zacc[h] = fmaf(pw[cc][h], vzr, zacc[h]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[h][i] = fmaf(pw[cc][h], x[i], acc[h][i]);
        }
      }
    }
  }
  cp_async_wait<0>();

  if constexpr (K_KIVIB) {
    if (is_tail) {
      // The fp32 tail rows [0, TT), one token per lane group per step.
      const float* tk = c.tail_k + bh * c.k.group * D + 16 * j;
      const float* tv = c.tail_v + bh * c.k.group * D + 16 * j;
      for (int base = 0; base < TT; base += TPC) {
        const int r = base + slot;
        const bool valid = r < TT;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = valid ? tk[(size_t)r * D + i] : 0.0f;
        float sc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float p = 0.0f;
#pragma unroll
          for (int i = 0; i < 16; ++i) p = fmaf(qf[h][i], x[i], p);
#pragma unroll
          for (int o = NL / 2; o >= 1; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
          sc[h] = valid ? p : neg_inf();
        }
        if (!valid) continue;   // uniform over the lane group
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = tv[(size_t)r * D + i];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float mn = fmaxf(m[h], sc[h]);
          const float alpha = exp2f(m[h] - mn);
          const float pw = exp2f(sc[h] - mn);
          l[h] = fmaf(l[h], alpha, pw);
          zacc[h] *= alpha;
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[h][i] = fmaf(acc[h][i], alpha, pw * x[i]);
          m[h] = mn;
        }
      }
    }
  }

  if constexpr (V_AFF) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[h][i] += zacc[h];
  }
  // Merge the lane-groups of the warp (lanes that share a channel slice).
#pragma unroll
  for (int o = NL; o < 32; o <<= 1) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[h], o);
      const float lo = __shfl_xor_sync(0xffffffffu, l[h], o);
      const float mn = fmaxf(m[h], mo);
      const float ea = (m[h] == neg_inf()) ? 0.0f : exp2f(m[h] - mn);
      const float eb = (mo == neg_inf()) ? 0.0f : exp2f(mo - mn);
      l[h] = l[h] * ea + lo * eb;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float ao = __shfl_xor_sync(0xffffffffu, acc[h][i], o);
        acc[h][i] = acc[h][i] * ea + ao * eb;
      }
      m[h] = mn;
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4*>(&sm_acc[warp][h][16 * j + i]) =
            make_float4(acc[h][i], acc[h][i + 1], acc[h][i + 2], acc[h][i + 3]);
      if (j == 0) {
        sm_m[warp][h] = m[h];
        sm_l[warp][h] = l[h];
      }
    }
  }
  __syncthreads();

  if constexpr (K_KIVIB) {
    DecodeArgs am = a;
    am.nsplit = a.nsplit + 1;   // partial slots per (b, kv head): the splits and the tail
    merge_store<D, G, 0>(c, am, b, kvh, is_tail ? nse : split, nse_all, sm_m, sm_l, &sm_acc[0][0][0]);
  } else {
    merge_store<D, G, 0>(c, a, b, kvh, split, nse, sm_m, sm_l, &sm_acc[0][0][0]);
  }
}

template <int D, int G, int KF, int VF>
cudaError_t launch_decode_dg(const CacheView& c, const DecodeArgs& a, cudaStream_t st) {
  constexpr int NSTAGE = Stages<KF>::v;
  const TileLayout L = tile_layout<D, KF, VF>(c.k.n_groups, c.v.n_groups);
  const int smem = NSTAGE * L.bytes;
  if (a.nsplit > kMaxSplits) return cudaErrorInvalidValue;
  // dynamic shared memory above 48 KB needs an opt-in, per device (the
  // attribute is set for the largest stage this kernel accepts)
  static std::atomic<unsigned long long> configured{0};
  {
    const cudaError_t e = once_per_device(configured, []() {
      return cudaFuncSetAttribute(decode_kernel<D, G, KF, VF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  NSTAGE * tile_layout<D, KF, VF>(D / 16, D / 16).bytes);
    });
    if (e != cudaSuccess) return e;
  }
  // KIVI_BLOCK keys: one more CTA per (b, kv head) for the full-precision tail
  const dim3 grid(a.nsplit + ((KF == F_KIVIB8 || KF == F_KIVIB4) ? 1 : 0), c.Hkv, c.B);
  decode_kernel<D, G, KF, VF><<<grid, kDecodeThreads, smem, st>>>(c, a);
  note_launch();
  return cudaGetLastError();
}

template <int D, int KF, int VF>
cudaError_t launch_decode_d(const CacheView& c, int G, const DecodeArgs& a, cudaStream_t st) {
  switch (G) {
    case 1: return launch_decode_dg<D, 1, KF, VF>(c, a, st);
    case 2: return launch_decode_dg<D, 2, KF, VF>(c, a, st);
    case 3: return launch_decode_dg<D, 3, KF, VF>(c, a, st);
    case 4: return launch_decode_dg<D, 4, KF, VF>(c, a, st);
    default: return cudaErrorNotSupported;
  }
}

// CUDA-core path: exact fp32 arithmetic on the codes, up to 4 query heads per kv head.
template <int KF, int VF>
cudaError_t launch_decode_cc(const CacheView& c, int G, const DecodeArgs& a, cudaStream_t st) {
  switch (c.D) {
    case 32: return launch_decode_d<32, KF, VF>(c, G, a, st);
    case 64: return launch_decode_d<64, KF, VF>(c, G, a, st);
    case 128: return launch_decode_d<128, KF, VF>(c, G, a, st);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace kvq
