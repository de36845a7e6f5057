// SnapKV observation-window scoring and sink-forced top-k selection.
//
// "SnapKV -- Prefill Observation-Window Token Eviction", "How it works": per
// head, the last w key rows act as proxy queries; attn = softmax(K[-w:] K^T /
// sqrt(D)) over all S keys; the mean over the w rows scores each key; the
// first n_sink positions are always kept, the top (budget - n_sink) of the
// rest are chosen and the union is returned in ascending order.
//
// Scoring is a [w x D] x [D x S] contraction per head, run on the tensor
// cores (fp16 inputs, fp32 accumulation, mma.sync m16n8k16).  Each CTA takes
// kSnapChunk keys: it computes their logits once, keeps them in shared
// memory and publishes its per-row (max, sum of exp); once every chunk of
// its head has published (a per-head arrival count, bounded wait, in a
// cooperative launch whose CTAs are all resident), it merges the row
// statistics and turns its logits into probabilities summed over the w rows.
// K is read once.  Where the grid cannot be resident at once, two launches do
// the same: pass 1 the statistics, pass 2 the logits again (K from L2 for the
// prompt sizes the page discusses) and the scores; both give the same bits.
// Each warp keeps the next 8 keys' fragments in flight while it multiplies
// the current ones.
//
// Selection is a radix select on the fp32 score bit patterns (4 passes of 8
// bits, the scores held in shared memory) that finds the (budget - n_sink)-th
// largest score exactly, followed by one ordered pass that keeps every larger
// score and the lowest-indexed equal ones, emitting positions in ascending
// order with a block scan.
#include <cooperative_groups.h>

#include "kvq_internal.cuh"

namespace kvq {

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ uint2 ld_quad(const __half* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }

// A hint: request this CTA's keys [key0, key0 + kSnapChunk) (clipped to S)
// into L2 with one bulk copy per 32 KB, so that the warps' loads, a tile of 8
// keys ahead each, are served from L2 while HBM streams at full rate.  The
// rows are contiguous (head_stride >= S) and 16-byte aligned when D * 2 is.
template <int D>
__device__ __forceinline__ void prefetch_chunk_l2(const __half* kh, int key0, int S) {
  if (threadIdx.x != 0 || key0 >= S) return;
  const uint8_t* p = reinterpret_cast<const uint8_t*>(kh + (size_t)key0 * D);
  if (reinterpret_cast<uintptr_t>(p) & 15) return;
  const uint32_t bytes = (uint32_t)(min(kSnapChunk, S - key0) * D * 2);
  for (uint32_t off = 0; off < bytes; off += 32768)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p + off), "r"(min(32768u, bytes - off))
                 : "memory");
}

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ unsigned long long clock_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Channel order shared by the observation rows (A) and the keys (B): k-step
// ks, mma k index 2t + j (j < 2) is channel 16 ks + 4t + j and 2t + 8 + j is
// 16 ks + 4t + 2 + j, so each thread reads 8 contiguous bytes of a row per
// k-step.  Both operands use it, so the dot products are unchanged.

// Observation rows as A fragments: row r (0..16*MT) is key S - w + r, zero when r >= w.
template <int D, int MT>
__device__ __forceinline__ void load_obs_perm(uint32_t (&A)[MT][D / 16][4], const __half* kh, int S, int w, int g,
                                              int t) {
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int r0 = mt * 16 + g, r1 = r0 + 8;
    const __half* p0 = kh + (size_t)(S - w + r0) * D;
    const __half* p1 = kh + (size_t)(S - w + r1) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int c0 = ks * 16 + 4 * t;
      const uint2 v0 = r0 < w ? ld_quad(p0 + c0) : make_uint2(0u, 0u);
      const uint2 v1 = r1 < w ? ld_quad(p1 + c0) : make_uint2(0u, 0u);
      A[mt][ks][0] = v0.x;
      A[mt][ks][1] = v1.x;
      A[mt][ks][2] = v0.y;
      A[mt][ks][3] = v1.y;
    }
  }
}

// B fragments of 8 keys [key0, key0 + 8): thread (g, t) holds key key0 + g,
// channels 16 ks + 4t .. 4t + 3.  Keys past the end repeat the last key (their
// logits are never used).
template <int D>
__device__ __forceinline__ void load_keys(uint32_t (&Bf)[D / 16][2], const __half* kh, int key0, int S, int g, int t) {
  const __half* p = kh + (size_t)min(key0 + g, S - 1) * D;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint2 v = ld_quad(p + ks * 16 + 4 * t);
    Bf[ks][0] = v.x;
    Bf[ks][1] = v.y;
  }
}

// Logits of those 8 keys against the 16*MT observation rows.
// cacc[mt][0..1] = rows mt*16+g, keys key0+2t, +1; cacc[mt][2..3] = rows +8.
// Even and odd k-steps accumulate apart (two short dependency chains).
template <int D, int MT>
__device__ __forceinline__ void tile_logits(float (&cacc)[MT][4], const uint32_t (&A)[MT][D / 16][4],
                                            const uint32_t (&Bf)[D / 16][2]) {
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    float odd[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    cacc[mt][0] = cacc[mt][1] = cacc[mt][2] = cacc[mt][3] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint32_t b[2] = {Bf[ks][0], Bf[ks][1]};
      mma16816((ks & 1) ? odd : cacc[mt], A[mt][ks], b);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) cacc[mt][i] += odd[i];
  }
}

// Per-row (max, sum) of this CTA: the 4 lanes sharing a row merge by
// shuffles, the 4 warps through shared memory; written as stats[r], r < 64.
template <int MT>
__device__ __forceinline__ void snap_row_stats(float (&rm)[MT][2], float (&rz)[MT][2], float (*sm_m)[MT * 16],
                                               float (*sm_z)[MT * 16], float2* stats, int g, int t, int warp) {
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const float mo = __shfl_xor_sync(0xffffffffu, rm[mt][hf], o);
        const float zo = __shfl_xor_sync(0xffffffffu, rz[mt][hf], o);
        const float mn = fmaxf(rm[mt][hf], mo);
        const float ea = (rm[mt][hf] == ninf()) ? 0.0f : exp2f(rm[mt][hf] - mn);
        const float eb = (mo == ninf()) ? 0.0f : exp2f(mo - mn);
        rz[mt][hf] = rz[mt][hf] * ea + zo * eb;
        rm[mt][hf] = mn;
      }
    }
  }
  if (t == 0) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        sm_m[warp][mt * 16 + g + 8 * hf] = rm[mt][hf];
        sm_z[warp][mt * 16 + g + 8 * hf] = rz[mt][hf];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < MT * 16) {
    const int r = threadIdx.x;
    float M = sm_m[0][r];
    for (int wi = 1; wi < 4; ++wi) M = fmaxf(M, sm_m[wi][r]);
    float Z = 0.0f;
    if (M != ninf()) {
      for (int wi = 0; wi < 4; ++wi) {
        if (sm_m[wi][r] != ninf()) Z += sm_z[wi][r] * exp2f(sm_m[wi][r] - M);
      }
    }
    stats[r] = make_float2(M, Z);
  }
}

// Every chunk's (max, sum) of each observation row merged into the row's max
// and 1 / sum (rows >= w: 0, 0): TPR adjacent threads per row, each over every
// TPR-th chunk, then a shuffle merge.  Ends with a barrier.
template <int MT>
__device__ __forceinline__ void merge_row_stats(const float2* __restrict__ stats, int nchunk, int w, float* row_m,
                                                float* row_iz) {
  constexpr int R = MT * 16;
  constexpr int TPR = (128 / R) >= 4 ? 4 : ((128 / R) >= 2 ? 2 : 1);
  const int r = threadIdx.x / TPR, part = threadIdx.x % TPR;
  float M = ninf(), Z = 0.0f;
  if (r < R && r < w) {
#pragma unroll 8
    for (int cch = part; cch < nchunk; cch += TPR) {
      const float2 st = __ldcg(&stats[cch * 64 + r]);
      if (st.x != ninf()) {
        const float mn = fmaxf(M, st.x);
        Z = Z * exp2f(M - mn) + st.y * exp2f(st.x - mn);
        M = mn;
      }
    }
  }
#pragma unroll
  for (int o = 1; o < TPR; o <<= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, M, o);
    const float zo = __shfl_xor_sync(0xffffffffu, Z, o);
    const float mn = fmaxf(M, mo);
    const float ea = (M == ninf()) ? 0.0f : exp2f(M - mn);
    const float eb = (mo == ninf()) ? 0.0f : exp2f(mo - mn);
    Z = Z * ea + zo * eb;
    M = mn;
  }
  if (r < R && part == 0) {
    const bool live = r < w;
    row_m[r] = live ? M : 0.0f;
    row_iz[r] = live ? 1.0f / Z : 0.0f;
  }
  __syncthreads();
}

// score[key] = (1/w) sum_r 2^(logit_r,key - M_r) / Z_r for the tile's 8 keys.
template <int MT>
__device__ __forceinline__ void snap_score_tile(const float (&cacc)[MT][4], const float (&Mr)[MT][2],
                                                const float (&Ir)[MT][2], float cscale, float inv_w,
                                                float* __restrict__ score_row, int key0, int S, int g, int t) {
  float col[2] = {0.0f, 0.0f};
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        // padded rows carry Ir = 0 and logit 0, contributing exactly 0
        col[e] += exp2f(cacc[mt][2 * hf + e] * cscale - Mr[mt][hf]) * Ir[mt][hf];
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 2; ++e) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) col[e] += __shfl_xor_sync(0xffffffffu, col[e], o);
  }
  if (g == 0) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = key0 + 2 * t + e;
      if (key < S) score_row[key] = col[e] * inv_w;
    }
  }
}

// Pass 1: per-row (max, sum 2^(logit - max)) over this CTA's keys, log2 domain.
template <int D, int MT>
__global__ void __launch_bounds__(128) snapkv_stats_kernel(const __half* __restrict__ k, long long head_stride,
                                                           int Hkv, int S, int w, float cscale, float2* stats,
                                                           int nchunk) {
  __shared__ float sm_m[4][MT * 16];
  __shared__ float sm_z[4][MT * 16];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const size_t bh = (size_t)blockIdx.z * Hkv + blockIdx.y;
  const int chunk = blockIdx.x;
  const __half* kh = k + bh * head_stride * D;
  prefetch_chunk_l2<D>(kh, chunk * kSnapChunk, S);

  uint32_t A[MT][D / 16][4];
  load_obs_perm<D, MT>(A, kh, S, w, g, t);

  float rm[MT][2], rz[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) rm[mt][0] = rm[mt][1] = ninf(), rz[mt][0] = rz[mt][1] = 0.0f;

  constexpr int kPerWarp = kSnapChunk / 4;
  const int wbase = chunk * kSnapChunk + warp * kPerWarp;
  const int ntile = max(0, min(kPerWarp / 8, (S - wbase + 7) / 8));
  uint32_t Bn[D / 16][2];
  if (ntile > 0) load_keys<D>(Bn, kh, wbase, S, g, t);
  for (int tile = 0; tile < ntile; ++tile) {
    const int key0 = wbase + tile * 8;
    uint32_t Bc[D / 16][2];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) Bc[ks][0] = Bn[ks][0], Bc[ks][1] = Bn[ks][1];
    if (tile + 1 < ntile) load_keys<D>(Bn, kh, key0 + 8, S, g, t);   // next tile's keys in flight
    float cacc[MT][4];
    tile_logits<D, MT>(cacc, A, Bc);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (key0 + 2 * t + e < S) {
            const float v = cacc[mt][2 * hf + e] * cscale;
            const float mn = fmaxf(rm[mt][hf], v);
            rz[mt][hf] = rz[mt][hf] * exp2f(rm[mt][hf] - mn) + exp2f(v - mn);
            rm[mt][hf] = mn;
          }
        }
      }
    }
  }
  snap_row_stats<MT>(rm, rz, sm_m, sm_z, stats + (bh * nchunk + chunk) * 64, g, t, warp);
}

// Pass 2: score[j] = (1/w) sum_r 2^(logit_rj - M_r) / Z_r.
template <int D, int MT>
__global__ void __launch_bounds__(128) snapkv_scores_kernel(const __half* __restrict__ k, long long head_stride,
                                                            int Hkv, int S, int w, float cscale,
                                                            const float2* __restrict__ stats, int nchunk,
                                                            float* __restrict__ scores) {
  __shared__ float row_m[64];
  __shared__ float row_iz[64];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const size_t bh = (size_t)blockIdx.z * Hkv + blockIdx.y;
  const int chunk = blockIdx.x;
  const __half* kh = k + bh * head_stride * D;

  merge_row_stats<MT>(stats + bh * nchunk * 64, nchunk, w, row_m, row_iz);   // ends with __syncthreads

  uint32_t A[MT][D / 16][4];
  load_obs_perm<D, MT>(A, kh, S, w, g, t);
  float Mr[MT][2], Ir[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      Mr[mt][hf] = row_m[mt * 16 + g + 8 * hf];
      Ir[mt][hf] = row_iz[mt * 16 + g + 8 * hf];
    }
  }
  const float inv_w = 1.0f / (float)w;
  constexpr int kPerWarp = kSnapChunk / 4;
  const int wbase = chunk * kSnapChunk + warp * kPerWarp;
  const int ntile = max(0, min(kPerWarp / 8, (S - wbase + 7) / 8));
  uint32_t Bn[D / 16][2];
  if (ntile > 0) load_keys<D>(Bn, kh, wbase, S, g, t);
  for (int tile = 0; tile < ntile; ++tile) {
    const int key0 = wbase + tile * 8;
    uint32_t Bc[D / 16][2];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) Bc[ks][0] = Bn[ks][0], Bc[ks][1] = Bn[ks][1];
    if (tile + 1 < ntile) load_keys<D>(Bn, kh, key0 + 8, S, g, t);   // next tile's keys in flight
    float cacc[MT][4];
    tile_logits<D, MT>(cacc, A, Bc);
    snap_score_tile<MT>(cacc, Mr, Ir, cscale, inv_w, scores + bh * S, key0, S, g, t);
  }
}

// One pass (cooperative launch): the logits of this CTA's keys once, kept in
// shared memory (each thread its own fragments: [warp][tile][mt][4][lane]),
// the chunk's row statistics published, a per-head arrival count waited for
// (bounded: after ~200 ms *fail is set and the scores are not valid), then
// the scores exactly as pass 2 computes them from the same logits.
template <int D, int MT>
__global__ void __launch_bounds__(128) snapkv_fused_kernel(const __half* __restrict__ k, long long head_stride,
                                                           int Hkv, int S, int w, float cscale, float2* stats,
                                                           int nchunk, float* __restrict__ scores,
                                                           unsigned* arrive, int* fail) {
  constexpr int kPerWarp = kSnapChunk / 4;
  constexpr int NT = kPerWarp / 8;   // tiles of 8 keys per warp
  extern __shared__ float sm_logit[];
  __shared__ float sm_m[4][MT * 16];
  __shared__ float sm_z[4][MT * 16];
  __shared__ float row_m[64];
  __shared__ float row_iz[64];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const size_t bh = (size_t)blockIdx.z * Hkv + blockIdx.y;
  const int chunk = blockIdx.x;
  const __half* kh = k + bh * head_stride * D;
  // the top-k that follows is a programmatic dependent: it may be scheduled
  // now (it waits for this grid to complete before reading anything)
  grid_launch_dependents();
  prefetch_chunk_l2<D>(kh, chunk * kSnapChunk, S);
  float* mylog = sm_logit + (size_t)warp * NT * MT * 4 * 32 + lane;

  uint32_t A[MT][D / 16][4];
  load_obs_perm<D, MT>(A, kh, S, w, g, t);
  float rm[MT][2], rz[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) rm[mt][0] = rm[mt][1] = ninf(), rz[mt][0] = rz[mt][1] = 0.0f;
  const int wbase = chunk * kSnapChunk + warp * kPerWarp;
  const int ntile = max(0, min(NT, (S - wbase + 7) / 8));
  uint32_t Bn[D / 16][2];
  if (ntile > 0) load_keys<D>(Bn, kh, wbase, S, g, t);
  for (int tile = 0; tile < ntile; ++tile) {
    const int key0 = wbase + tile * 8;
    uint32_t Bc[D / 16][2];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) Bc[ks][0] = Bn[ks][0], Bc[ks][1] = Bn[ks][1];
    if (tile + 1 < ntile) load_keys<D>(Bn, kh, key0 + 8, S, g, t);
    float cacc[MT][4];
    tile_logits<D, MT>(cacc, A, Bc);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) mylog[((tile * MT + mt) * 4 + i) * 32] = cacc[mt][i];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (key0 + 2 * t + e < S) {
            const float v = cacc[mt][2 * hf + e] * cscale;
            const float mn = fmaxf(rm[mt][hf], v);
            rz[mt][hf] = rz[mt][hf] * exp2f(rm[mt][hf] - mn) + exp2f(v - mn);
            rm[mt][hf] = mn;
          }
        }
      }
    }
  }
  snap_row_stats<MT>(rm, rz, sm_m, sm_z, stats + (bh * nchunk + chunk) * 64, g, t, warp);
  __syncthreads();   // this CTA's statistics are written
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&arrive[bh], 1u);
    const unsigned long long t0 = clock_ns();
    unsigned n;
    do {
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(n) : "l"(&arrive[bh]) : "memory");
      if (n >= (unsigned)nchunk) break;
      if (clock_ns() - t0 > kWaitNs) {
        atomicExch(fail, 1);
        break;
      }
    } while (true);
  }
  __syncthreads();
  merge_row_stats<MT>(stats + bh * nchunk * 64, nchunk, w, row_m, row_iz);   // ends with __syncthreads
  float Mr[MT][2], Ir[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      Mr[mt][hf] = row_m[mt * 16 + g + 8 * hf];
      Ir[mt][hf] = row_iz[mt * 16 + g + 8 * hf];
    }
  }
  const float inv_w = 1.0f / (float)w;
  for (int tile = 0; tile < ntile; ++tile) {
    float cacc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) cacc[mt][i] = mylog[((tile * MT + mt) * 4 + i) * 32];
    }
    snap_score_tile<MT>(cacc, Mr, Ir, cscale, inv_w, scores + bh * S, wbase + tile * 8, S, g, t);
  }
}

// ----------------------------------------------------------------- top-k --

// Monotone map from fp32 to uint32 order; -0.0 ranks with +0.0.
__device__ __forceinline__ unsigned order_key(float f) {
  unsigned u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}


// The (budget - n_sink)-th largest key among `need` remaining: given the
// 256-bin histogram of the current digit, warp 0 finds the bin where the
// count of larger-or-equal digits reaches `need` (a suffix scan, 8 bins per
// lane) and how many of that bin are still needed.
__device__ __forceinline__ void pick_bin(const unsigned* hist, unsigned need, unsigned* s_bin, unsigned* s_need) {
  const int lane = threadIdx.x & 31;
  // lane l owns bins 255 - 8l ... 248 - 8l (descending digit order)
  unsigned cnt[8], own = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    cnt[i] = hist[255 - 8 * lane - i];
    own += cnt[i];
  }
  unsigned incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  const unsigned before = incl - own;   // keys in larger digits than this lane's bins
  const bool here = before < need && incl >= need;
  if (here) {
    unsigned cum = before;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (cum + cnt[i] >= need) {
        *s_bin = 255u - 8u * lane - i;
        *s_need = need - cum;
        break;
      }
      cum += cnt[i];
    }
  }
}

// Scores live in shared memory when they fit (dynamic size S floats); larger
// prompts read them from global memory on every pass.
constexpr int kTopkSmemKeys = 48 * 1024;

// Exclusive prefix sum of `v` over the block (blockDim.x a multiple of 32,
// at most 1024); *total gets the block's sum.
__device__ __forceinline__ int block_excl_count_n(int v, int* total, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    const int ws = lane < nw ? warp_sums[lane] : 0;
    int wincl = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wincl, o);
      if (lane >= o) wincl += n;
    }
    warp_sums[lane] = wincl - ws;
    if (lane == 31) warp_sums[32] = wincl;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  *total = warp_sums[32];
  __syncthreads();
  return r;
}

// fail (nullable): set by a scoring launch whose wait ran out; the indices
// are then all -1.
__global__ void __launch_bounds__(1024) topk_kernel(const float* __restrict__ scores, int S, int budget, int n_sink,
                                                    int* __restrict__ idx_out, const int* fail) {
  grid_dependency_wait();   // launched as a programmatic dependent of the scoring
  extern __shared__ float sm_sc[];
  __shared__ unsigned hist[256];
  __shared__ unsigned s_bin, s_need;
  __shared__ int warp_sums[33];
  const size_t bh = blockIdx.x;
  const float* sc = scores + bh * S;
  const int n_keep = min(budget, S);
  int* out = idx_out + bh * n_keep;
  if (fail && *fail) {
    for (int j = threadIdx.x; j < n_keep; j += blockDim.x) out[j] = -1;
    return;
  }
  if (budget >= S) {
    for (int j = threadIdx.x; j < S; j += blockDim.x) out[j] = j;
    return;
  }
  const bool in_smem = S <= kTopkSmemKeys;
  if (in_smem) {
    // coalesced copy; the row start is 16-byte aligned when S % 4 == 0
    if ((S & 3) == 0 && (reinterpret_cast<uintptr_t>(sc) & 15) == 0) {
      const float4* src = reinterpret_cast<const float4*>(sc);
      for (int i = threadIdx.x; i < S / 4; i += blockDim.x) reinterpret_cast<float4*>(sm_sc)[i] = __ldg(src + i);
    } else {
      for (int i = threadIdx.x; i < S; i += blockDim.x) sm_sc[i] = __ldg(sc + i);
    }
    __syncthreads();
  }
  const float* src = in_smem ? sm_sc : sc;
  const int ns = min(n_sink, S);
  const int k = budget - ns;   // 0 <= k < S - ns
  unsigned prefix = 0u, mask = 0u, need = (unsigned)k;
  if (k > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
      __syncthreads();
      for (int j = ns + threadIdx.x; j < S; j += blockDim.x) {
        const unsigned key = order_key(src[j]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFFu], 1u);
      }
      __syncthreads();
      if (threadIdx.x < 32) pick_bin(hist, need, &s_bin, &s_need);
      __syncthreads();
      prefix |= s_bin << shift;
      mask |= 0xFFu << shift;
      need = s_need;
      __syncthreads();
    }
  }
  // prefix is the exact key of the k-th largest score; `need` equal keys are
  // kept, the lowest positions first.  Thread i owns positions
  // [i * seg, (i + 1) * seg): it counts its sinks, larger keys and ties, two
  // block scans place its ties and its selected positions, and it writes
  // them in ascending order.
  const int seg = (S + blockDim.x - 1) / blockDim.x;
  const int j0 = min(S, (int)threadIdx.x * seg), j1 = min(S, j0 + seg);
  int n_big = 0, n_tie = 0;
  for (int j = j0; j < j1; ++j) {
    if (j < ns) {
      ++n_big;
    } else if (k > 0) {
      const unsigned key = order_key(src[j]);
      n_big += key > prefix;
      n_tie += key == prefix;
    }
  }
  int tie_total;
  const int tie_before = block_excl_count_n(n_tie, &tie_total, warp_sums);
  const int ties_kept = max(0, min(n_tie, (int)need - tie_before));
  int sel_total;
  int pos = block_excl_count_n(n_big + ties_kept, &sel_total, warp_sums);
  int ties_left = ties_kept;
  for (int j = j0; j < j1; ++j) {
    bool sel;
    if (j < ns) {
      sel = true;
    } else if (k > 0) {
      const unsigned key = order_key(src[j]);
      sel = key > prefix;
      if (key == prefix && ties_left > 0) {
        sel = true;
        --ties_left;
      }
    } else {
      sel = false;
    }
    if (sel) out[pos++] = j;
  }
}

// The same selection with a cluster of kTopkCluster CTAs per (b, kv head), so
// that a long prompt's scores are worked by that many SMs instead of one.
// CTA rank r holds positions [r * chunk, (r + 1) * chunk) in shared memory.
// Each radix pass builds the CTA's histogram (double-buffered by pass), and
// after one cluster barrier every CTA sums the cluster's histograms through
// distributed shared memory and picks the same bin.  The positions kept come
// out in ascending order: rank r writes after the kept positions of the lower
// ranks (sinks, larger keys and the ties they keep, lowest positions first),
// which each CTA counts from the lower ranks' (larger, tie) counts.
constexpr int kTopkCluster = 8;
constexpr int kTopkClusterThreads = 512;
constexpr int kTopkClusterMaxChunk = 8192;   // positions per CTA (32 KB of shared memory)

__global__ void __launch_bounds__(kTopkClusterThreads) topk_cluster_kernel(const float* __restrict__ scores, int S,
                                                                           int budget, int n_sink,
                                                                           int* __restrict__ idx_out,
                                                                           const int* fail) {
  grid_dependency_wait();   // launched as a programmatic dependent of the scoring
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ float sm_sc[];
  __shared__ unsigned hist[2][256];
  __shared__ unsigned tot[256];
  __shared__ unsigned s_bin, s_need;
  __shared__ int warp_sums[33];
  __shared__ int s_cnt[2];   // this CTA's positions kept outright (sinks, larger keys) and ties
  const int rank = (int)cluster.block_rank();
  const size_t bh = blockIdx.y;
  const float* sc = scores + bh * S;
  int* out = idx_out + bh * budget;   // budget < S (the host takes the other case)
  if (fail && *fail) {   // every CTA of the cluster reads the same flag: none reaches a cluster barrier
    if (rank == 0)
      for (int j = threadIdx.x; j < budget; j += blockDim.x) out[j] = -1;
    return;
  }
  const int chunk = (S + kTopkCluster - 1) / kTopkCluster;
  const int c0 = min(S, rank * chunk), c1 = min(S, c0 + chunk);
  for (int i = threadIdx.x; i < c1 - c0; i += blockDim.x) sm_sc[i] = __ldg(sc + c0 + i);
  __syncthreads();
  const int ns = min(n_sink, S);
  const int k = budget - ns;
  unsigned prefix = 0u, mask = 0u, need = (unsigned)k;
  if (k > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      unsigned* h = hist[pass & 1];
      for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0u;
      __syncthreads();
      for (int j = max(c0, ns) + threadIdx.x; j < c1; j += blockDim.x) {
        const unsigned key = order_key(sm_sc[j - c0]);
        if ((key & mask) == prefix) atomicAdd(&h[(key >> shift) & 0xFFu], 1u);
      }
      // every CTA's histogram of this pass is complete; the buffer of the
      // previous pass is free (each CTA finished reading it before arriving)
      cluster.sync();
      for (int i = threadIdx.x; i < 256; i += blockDim.x) {
        unsigned t = 0u;
#pragma unroll
        for (int r = 0; r < kTopkCluster; ++r) t += cluster.map_shared_rank(h, r)[i];
        tot[i] = t;
      }
      __syncthreads();
      if (threadIdx.x < 32) pick_bin(tot, need, &s_bin, &s_need);
      __syncthreads();
      prefix |= s_bin << shift;
      mask |= 0xFFu << shift;
      need = s_need;
      __syncthreads();
    }
  }
  // This thread's positions, their counts, and the CTA's totals.
  const int seg = (c1 - c0 + (int)blockDim.x - 1) / (int)blockDim.x;
  const int j0 = min(c1, c0 + (int)threadIdx.x * seg), j1 = min(c1, j0 + seg);
  int n_big = 0, n_tie = 0;
  for (int j = j0; j < j1; ++j) {
    if (j < ns) {
      ++n_big;
    } else if (k > 0) {
      const unsigned key = order_key(sm_sc[j - c0]);
      n_big += key > prefix;
      n_tie += key == prefix;
    }
  }
  int big_total, tie_total;
  const int big_before = block_excl_count_n(n_big, &big_total, warp_sums);
  const int tie_before = block_excl_count_n(n_tie, &tie_total, warp_sums);
  if (threadIdx.x == 0) {
    s_cnt[0] = big_total;
    s_cnt[1] = tie_total;
  }
  cluster.sync();
  // positions the lower ranks keep, and the ties they take
  int out_before = 0, ties_before_cta = 0;
  for (int r = 0; r < rank; ++r) {
    const int* rc = cluster.map_shared_rank(s_cnt, r);
    const int kept = max(0, min(rc[1], (int)need - ties_before_cta));
    out_before += rc[0] + kept;
    ties_before_cta += rc[1];
  }
  cluster.sync();   // no CTA leaves while another may still read its counts
  const int ties_cta = max(0, min(tie_total, (int)need - ties_before_cta));
  const int ties_kept = max(0, min(n_tie, ties_cta - tie_before));
  // the CTA's kept ties come from its lowest positions: threads before this
  // one keep min(tie_before, ties_cta) of them
  int pos = out_before + big_before + min(tie_before, ties_cta);
  int ties_left = ties_kept;
  for (int j = j0; j < j1; ++j) {
    bool sel;
    if (j < ns) {
      sel = true;
    } else if (k > 0) {
      const unsigned key = order_key(sm_sc[j - c0]);
      sel = key > prefix;
      if (key == prefix && ties_left > 0) {
        sel = true;
        --ties_left;
      }
    } else {
      sel = false;
    }
    if (sel) out[pos++] = j;
  }
}

// ------------------------------------------------------------ smoothing --
// The SnapKV paper's max-pool smoothing of the scores (the page leaves it out,
// "Proxy limitation"): out[j] = max of in[j - r .. j + r] clipped to [0, S),
// r = kernel_size / 2.  One CTA of 256 threads per 256 positions of one
// (b, kv head), with the positions and an r-wide halo on each side staged in
// shared memory.

constexpr int kPoolTile = 256;
constexpr int kPoolMaxR = 31;

__global__ void __launch_bounds__(kPoolTile) snapkv_pool_kernel(const float* __restrict__ in,
                                                                float* __restrict__ out, int S, int r) {
  __shared__ float tile[kPoolTile + 2 * kPoolMaxR];
  const size_t bh = blockIdx.y;
  const int j0 = blockIdx.x * kPoolTile;
  const float* row = in + bh * S;
  for (int i = threadIdx.x; i < kPoolTile + 2 * r; i += kPoolTile) {
    const int j = j0 - r + i;
    tile[i] = (j >= 0 && j < S) ? row[j] : ninf();
  }
  __syncthreads();
  const int j = j0 + threadIdx.x;
  if (j < S) {
    float m = tile[threadIdx.x];
    for (int i = 1; i <= 2 * r; ++i) m = fmaxf(m, tile[threadIdx.x + i]);
    out[bh * S + j] = m;
  }
}

cudaError_t launch_snapkv_pool(const float* in, float* out, int BH, int S, int kernel_size, cudaStream_t st) {
  const int r = kernel_size / 2;
  if (r > kPoolMaxR) return cudaErrorInvalidValue;
  const dim3 grid((S + kPoolTile - 1) / kPoolTile, BH);
  snapkv_pool_kernel<<<grid, kPoolTile, 0, st>>>(in, out, S, r);
  note_launch();
  return cudaGetLastError();
}

// ---------------------------------------------------------------- launch --

// Whether a cooperative grid of `ctas` fused scoring CTAs is resident at once
// on the current device (remembered per device and shape).
template <int D, int MT>
static bool fused_grid_fits(long long ctas, int smem) {
  static std::atomic<int> per_dev[64];   // CTAs resident at once + 1, 0 unknown
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  int known = per_dev[dev].load(std::memory_order_relaxed);
  if (!known) {
    int sms = 0, per_sm = 0, coop = 0;
    bool ok = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
              cudaFuncSetAttribute(snapkv_fused_kernel<D, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
                  cudaSuccess &&
              cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, snapkv_fused_kernel<D, MT>, 128, smem) ==
                  cudaSuccess;
    (void)cudaGetLastError();
    known = (ok ? per_sm * sms : 0) + 1;
    per_dev[dev].store(known, std::memory_order_relaxed);
  }
  return ctas <= known - 1;
}

template <int D, int MT>
static cudaError_t launch_snapkv_dm(const void* k, long long hs, int B, int Hkv, int S, int w,
                                    float* scores, float2* stats, int nchunk, unsigned* arrive, int* fail,
                                    cudaStream_t st) {
  const float cscale = 1.4426950408889634f / sqrtf((float)D);
  const dim3 grid(nchunk, Hkv, B);
  const __half* kk = static_cast<const __half*>(k);
  const int smem = 4 * (kSnapChunk / 4 / 8) * MT * 4 * 32 * (int)sizeof(float);
  // the arrival counts and the failure flag (read by the top-k) start at zero
  cudaError_t e = cudaMemsetAsync(arrive, 0, ((size_t)B * Hkv + 1) * sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  if (fused_grid_fits<D, MT>((long long)nchunk * Hkv * B, smem)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, snapkv_fused_kernel<D, MT>, kk, hs, Hkv, S, w, cscale, stats, nchunk, scores, arrive,
                           fail);
    note_launch();
    return e;
  }
  snapkv_stats_kernel<D, MT><<<grid, 128, 0, st>>>(kk, hs, Hkv, S, w, cscale, stats, nchunk);
  note_launch();
  snapkv_scores_kernel<D, MT><<<grid, 128, 0, st>>>(kk, hs, Hkv, S, w, cscale, stats, nchunk, scores);
  note_launch();
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_snapkv_d(const void* k, long long hs, int B, int Hkv, int S, int w,
                                   float* scores, float2* stats, int nchunk, unsigned* arrive, int* fail,
                                   cudaStream_t st) {
  switch ((w + 15) / 16) {
    case 1: return launch_snapkv_dm<D, 1>(k, hs, B, Hkv, S, w, scores, stats, nchunk, arrive, fail, st);
    case 2: return launch_snapkv_dm<D, 2>(k, hs, B, Hkv, S, w, scores, stats, nchunk, arrive, fail, st);
    case 3: return launch_snapkv_dm<D, 3>(k, hs, B, Hkv, S, w, scores, stats, nchunk, arrive, fail, st);
    case 4: return launch_snapkv_dm<D, 4>(k, hs, B, Hkv, S, w, scores, stats, nchunk, arrive, fail, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_topk(const float* scores, int B, int Hkv, int S, int budget, int n_sink, int* idx,
                        const int* fail, cudaStream_t st) {
  if (budget < S && S >= 4096 && (S + kTopkCluster - 1) / kTopkCluster <= kTopkClusterMaxChunk) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kTopkCluster, B * Hkv);
    cfg.blockDim = dim3(kTopkClusterThreads);
    cfg.dynamicSmemBytes = ((S + kTopkCluster - 1) / kTopkCluster) * sizeof(float);
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kTopkCluster;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, topk_cluster_kernel, scores, S, budget, n_sink, idx, fail);
    note_launch();
    return e;
  }
  const int smem = S <= kTopkSmemKeys ? S * (int)sizeof(float) : 0;
  static std::atomic<unsigned long long> configured{0};   // the opt-in is per device
  const cudaError_t e = once_per_device(configured, []() {
    return cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kTopkSmemKeys * (int)sizeof(float));
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B * Hkv);
  cfg.blockDim = dim3(1024);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e2 = cudaLaunchKernelEx(&cfg, topk_kernel, scores, S, budget, n_sink, idx, fail);
  note_launch();
  return e2;
}

cudaError_t launch_snapkv(const void* k, long long head_stride, int B, int Hkv, int S, int D, int w, int budget,
                          int n_sink, float* scores, int* idx, float2* stats, int nchunk, unsigned* arrive,
                          cudaStream_t st) {
  // the failure flag sits after the B * Hkv arrival counts
  int* fail = reinterpret_cast<int*>(arrive + (size_t)B * Hkv);
  cudaError_t e;
  switch (D) {
    case 32: e = launch_snapkv_d<32>(k, head_stride, B, Hkv, S, w, scores, stats, nchunk, arrive, fail, st); break;
    case 64: e = launch_snapkv_d<64>(k, head_stride, B, Hkv, S, w, scores, stats, nchunk, arrive, fail, st); break;
    case 128: e = launch_snapkv_d<128>(k, head_stride, B, Hkv, S, w, scores, stats, nchunk, arrive, fail, st); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch_topk(scores, B, Hkv, S, budget, n_sink, idx, fail, st);
}

}  // namespace kvq
