// SnapKV observation-window scoring and sink-forced top-k selection.
//
// "SnapKV -- Prefill Observation-Window Token Eviction", "How it works": per
// head, the last w key rows act as proxy queries; attn = softmax(K[-w:] K^T /
// sqrt(D)) over all S keys; the mean over the w rows scores each key; the
// first n_sink positions are always kept, the top (budget - n_sink) of the
// rest are chosen and the union is returned in ascending order.
//
// Scoring is a [w x D] x [D x S] contraction per head, run on the tensor
// cores (fp16 inputs, fp32 accumulation, mma.sync m16n8k16) in two passes
// over the keys: pass 1 gives each CTA's per-row (max, sum of exp) over its
// 512 keys, pass 2 merges those row statistics and turns every logit into
// its probability, summing over the w rows.  The second read of K is served
// by L2 for the prompt sizes the page discusses (16K keys x 8 heads x 256 B).
//
// Selection is a radix select on the fp32 score bit patterns (4 passes of 8
// bits) that finds the (budget - n_sink)-th largest score exactly, followed
// by one ordered pass that keeps every larger score and the lowest-indexed
// equal ones, emitting positions in ascending order with a block scan.
#include "kvq_internal.cuh"

namespace kvq {

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ uint32_t ld_pair(const __half* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }

// Observation rows as A fragments: row r (0..16*MT) is key S - w + r, zero when r >= w.
template <int D, int MT>
__device__ __forceinline__ void load_obs(uint32_t (&A)[MT][D / 16][4], const __half* kh, int S, int w, int g,
                                         int t) {
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int r0 = mt * 16 + g, r1 = r0 + 8;
    const __half* p0 = kh + (size_t)(S - w + r0) * D;
    const __half* p1 = kh + (size_t)(S - w + r1) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int c0 = ks * 16 + 2 * t;
      A[mt][ks][0] = r0 < w ? ld_pair(p0 + c0) : 0u;
      A[mt][ks][1] = r1 < w ? ld_pair(p1 + c0) : 0u;
      A[mt][ks][2] = r0 < w ? ld_pair(p0 + c0 + 8) : 0u;
      A[mt][ks][3] = r1 < w ? ld_pair(p1 + c0 + 8) : 0u;
    }
  }
}

// Logits of 8 keys [key0, key0 + 8) against the 16*MT observation rows.
// cacc[mt][0..1] = rows mt*16+g, keys key0+2t, +1; cacc[mt][2..3] = rows +8.
template <int D, int MT>
__device__ __forceinline__ void tile_logits(float (&cacc)[MT][4], const uint32_t (&A)[MT][D / 16][4],
                                            const __half* kh, int key0, int S, int g, int t) {
  const int kr = min(key0 + g, S - 1);
  const __half* p = kh + (size_t)kr * D;
  uint32_t Bf[D / 16][2];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    Bf[ks][0] = ld_pair(p + ks * 16 + 2 * t);
    Bf[ks][1] = ld_pair(p + ks * 16 + 2 * t + 8);
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    cacc[mt][0] = cacc[mt][1] = cacc[mt][2] = cacc[mt][3] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint32_t b[2] = {Bf[ks][0], Bf[ks][1]};
      mma16816(cacc[mt], A[mt][ks], b);
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

  uint32_t A[MT][D / 16][4];
  load_obs<D, MT>(A, kh, S, w, g, t);

  float rm[MT][2], rz[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) rm[mt][0] = rm[mt][1] = ninf(), rz[mt][0] = rz[mt][1] = 0.0f;

  constexpr int kPerWarp = kSnapChunk / 4;
  const int wbase = chunk * kSnapChunk + warp * kPerWarp;
  for (int tile = 0; tile < kPerWarp / 8; ++tile) {
    const int key0 = wbase + tile * 8;
    if (key0 >= S) break;
    float cacc[MT][4];
    tile_logits<D, MT>(cacc, A, kh, key0, S, g, t);
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
  // merge the 4 lanes that share a row
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
    stats[(bh * nchunk + chunk) * 64 + r] = make_float2(M, Z);
  }
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

  if (threadIdx.x < MT * 16) {
    const int r = threadIdx.x;
    float M = 0.0f, iz = 0.0f;
    if (r < w) {
      M = ninf();
      for (int cch = 0; cch < nchunk; ++cch) M = fmaxf(M, stats[(bh * nchunk + cch) * 64 + r].x);
      float Z = 0.0f;
      for (int cch = 0; cch < nchunk; ++cch) {
        const float2 st = stats[(bh * nchunk + cch) * 64 + r];
        if (st.x != ninf()) Z += st.y * exp2f(st.x - M);
      }
      iz = 1.0f / Z;
    }
    row_m[r] = M;
    row_iz[r] = iz;
  }
  __syncthreads();

  uint32_t A[MT][D / 16][4];
  load_obs<D, MT>(A, kh, S, w, g, t);
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
  for (int tile = 0; tile < kPerWarp / 8; ++tile) {
    const int key0 = wbase + tile * 8;
    if (key0 >= S) break;
    float cacc[MT][4];
    tile_logits<D, MT>(cacc, A, kh, key0, S, g, t);
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
        if (key < S) scores[bh * S + key] = col[e] * inv_w;
      }
    }
  }
}

// ----------------------------------------------------------------- top-k --

// Monotone map from fp32 to uint32 order; -0.0 ranks with +0.0.
__device__ __forceinline__ unsigned order_key(float f) {
  unsigned u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix count of `flag` over the block (blockDim.x == 1024);
// *total gets the block's count.
__device__ __forceinline__ int block_excl_count(bool flag, int* total, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_sums[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    const int v = warp_sums[lane];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    warp_sums[lane] = incl - v;
    if (lane == 31) warp_sums[32] = incl;
  }
  __syncthreads();
  const int r = warp_sums[warp] + in_warp;
  *total = warp_sums[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024) topk_kernel(const float* __restrict__ scores, int S, int budget, int n_sink,
                                                    int* __restrict__ idx_out) {
  __shared__ unsigned hist[256];
  __shared__ unsigned s_bin, s_need;
  __shared__ int warp_sums[33];
  const size_t bh = blockIdx.x;
  const float* sc = scores + bh * S;
  const int n_keep = min(budget, S);
  int* out = idx_out + bh * n_keep;
  if (budget >= S) {
    for (int j = threadIdx.x; j < S; j += blockDim.x) out[j] = j;
    return;
  }
  const int ns = min(n_sink, S);
  const int k = budget - ns;   // 0 <= k < S - ns
  unsigned prefix = 0u, mask = 0u, need = (unsigned)k;
  if (k > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
      __syncthreads();
      for (int j = ns + threadIdx.x; j < S; j += blockDim.x) {
        const unsigned key = order_key(sc[j]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFFu], 1u);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        unsigned cum = 0u;
        for (int bin = 255; bin >= 0; --bin) {
          const unsigned hcount = hist[bin];
          if (cum + hcount >= need) {
            s_bin = (unsigned)bin;
            s_need = need - cum;
            break;
          }
          cum += hcount;
        }
      }
      __syncthreads();
      prefix |= s_bin << shift;
      mask |= 0xFFu << shift;
      need = s_need;
      __syncthreads();
    }
  }
  // prefix is the exact key of the k-th largest score; `need` equal keys are kept.
  int running = 0, tie_running = 0;
  for (int base = 0; base < S; base += blockDim.x) {
    const int j = base + threadIdx.x;
    const bool in_rest = (j >= ns) && (j < S);
    const unsigned key = (j < S) ? order_key(sc[j]) : 0u;
    const bool tie = (k > 0) && in_rest && key == prefix;
    int tie_total;
    const int tie_rank = block_excl_count(tie, &tie_total, warp_sums) + tie_running;
    const bool sel = (j < ns) || ((k > 0) && in_rest && (key > prefix || (tie && tie_rank < (int)need)));
    int sel_total;
    const int rank = block_excl_count(sel, &sel_total, warp_sums) + running;
    if (sel) out[rank] = j;
    running += sel_total;
    tie_running += tie_total;
  }
}

// ---------------------------------------------------------------- launch --

template <int D, int MT>
static cudaError_t launch_snapkv_dm(const void* k, long long hs, int B, int Hkv, int S, int w, float* scores,
                                    float2* stats, int nchunk, cudaStream_t st) {
  const float cscale = 1.4426950408889634f / sqrtf((float)D);
  const dim3 grid(nchunk, Hkv, B);
  const __half* kk = static_cast<const __half*>(k);
  snapkv_stats_kernel<D, MT><<<grid, 128, 0, st>>>(kk, hs, Hkv, S, w, cscale, stats, nchunk);
  note_launch();
  snapkv_scores_kernel<D, MT><<<grid, 128, 0, st>>>(kk, hs, Hkv, S, w, cscale, stats, nchunk, scores);
  note_launch();
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_snapkv_d(const void* k, long long hs, int B, int Hkv, int S, int w, float* scores,
                                   float2* stats, int nchunk, cudaStream_t st) {
  switch ((w + 15) / 16) {
    case 1: return launch_snapkv_dm<D, 1>(k, hs, B, Hkv, S, w, scores, stats, nchunk, st);
    case 2: return launch_snapkv_dm<D, 2>(k, hs, B, Hkv, S, w, scores, stats, nchunk, st);
    case 3: return launch_snapkv_dm<D, 3>(k, hs, B, Hkv, S, w, scores, stats, nchunk, st);
    case 4: return launch_snapkv_dm<D, 4>(k, hs, B, Hkv, S, w, scores, stats, nchunk, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_topk(const float* scores, int B, int Hkv, int S, int budget, int n_sink, int* idx,
                        cudaStream_t st) {
  topk_kernel<<<B * Hkv, 1024, 0, st>>>(scores, S, budget, n_sink, idx);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_snapkv(const void* k, long long head_stride, int B, int Hkv, int S, int D, int w, int budget,
                          int n_sink, float* scores, int* idx, float2* stats, int nchunk, cudaStream_t st) {
  cudaError_t e;
  switch (D) {
    case 32: e = launch_snapkv_d<32>(k, head_stride, B, Hkv, S, w, scores, stats, nchunk, st); break;
    case 64: e = launch_snapkv_d<64>(k, head_stride, B, Hkv, S, w, scores, stats, nchunk, st); break;
    case 128: e = launch_snapkv_d<128>(k, head_stride, B, Hkv, S, w, scores, stats, nchunk, st); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch_topk(scores, B, Hkv, S, budget, n_sink, idx, st);
}

}  // namespace kvq
