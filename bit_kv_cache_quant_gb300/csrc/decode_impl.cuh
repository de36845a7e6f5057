// Fused single-query GQA decode attention over the packed cache.
//
// "Low-bit KV caches on MLX", section 5: decode attention spends its time
// reading the cache; fused kernels read packed bytes and dequantise in
// registers.  "StreamingLLM + KIVI", "Affine quantisation formula": the
// attention runs on x_dq = (q - qMin) * scale + zero with the stored fp16
// scales upcast to fp32.  mlx-qsdpa (same memo, section 5) splits long
// contexts; here every (b, kv head) is split over `nsplit` CTAs whose
// partial (max, sum, accumulator) triples are merged with the online-softmax
// rule by the last CTA to finish.
//
// Work mapping: a token row of D channels is read by D/16 lanes, each lane
// owning 16 consecutive channels (8, 16 or 32 bytes of codes: one 64- or
// 128-bit load).  A warp covers 32/(D/16) tokens at a time, the CTA (4 warps)
// processes C such token groups per step, loading all their codes before
// using any.  The G query heads that share a kv head are computed together so
// each code is read once.
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
constexpr float kLog2e = 1.4426950408889634f;

template <int F> struct FmtBits {
  static constexpr int v = (F == F_FP16) ? 16 : ((F == F_KIVI8 || F == F_AFF8) ? 8 : 4);
};

// Codes of one lane's 16 channels.
template <int BITS> struct Codes { uint32_t w[BITS / 2]; };

template <int BITS>
__device__ __forceinline__ void load_codes(Codes<BITS>& c, const uint8_t* p) {
  if constexpr (BITS == 16) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
    c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
    c.w[4] = b.x; c.w[5] = b.y; c.w[6] = b.z; c.w[7] = b.w;
  } else if constexpr (BITS == 8) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
  } else {
    const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
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

template <int D, int G, int KF, int VF, int C>
__global__ void __launch_bounds__(128) decode_kernel(CacheView c, DecodeArgs a) {
  constexpr int NL = D / 16;                  // lanes per token
  constexpr int TPW = 32 / NL;                // tokens per warp per step
  constexpr int TPC = TPW * kDecodeWarps;     // tokens per CTA per step
  constexpr int KB = FmtBits<KF>::v;
  constexpr int VB = FmtBits<VF>::v;
  constexpr int KROW = D * KB / 8;
  constexpr int VROW = D * VB / 8;
  constexpr bool K_AFF = (KF == F_AFF8 || KF == F_AFF4);
  constexpr bool K_KIVI = (KF == F_KIVI8 || KF == F_KIVI4);
  constexpr bool K_Q40 = (KF == F_Q40);
  constexpr bool V_AFF = (VF == F_AFF8 || VF == F_AFF4);

  __shared__ float sm_m[kDecodeWarps][G];
  __shared__ float sm_l[kDecodeWarps][G];
  __shared__ float sm_acc[kDecodeWarps][G][D];
  __shared__ int s_T;
  __shared__ int s_last;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int j = lane % NL;                    // channel slice [16j, 16j + 16)
  const int grp = lane / NL;
  const int slot = warp * TPW + grp;
  const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
  const size_t bh = (size_t)b * c.Hkv + kvh;

  if (threadIdx.x == 0) s_T = c.state->stored;
  __syncthreads();
  const int T = s_T;
  const int per = (T + a.nsplit - 1) / a.nsplit;
  const int t0 = min(T, split * per);
  const int t1 = min(T, t0 + per);

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

  const int kng = c.k.n_groups;
  const int vng = c.v.n_groups;
  const int kg = K_AFF ? (16 * j) / c.k.group : (K_Q40 ? (j >> 1) : 0);
  const int vg = V_AFF ? (16 * j) / c.v.group : 0;
  const uint8_t* kbase = c.k.codes + bh * c.cap_alloc * KROW + j * (KROW / NL);
  const uint8_t* vbase = c.v.codes + bh * c.cap_alloc * VROW + j * (VROW / NL);
  const __half* ksb = (K_AFF || K_Q40) ? c.k.tok_scale + bh * c.cap_alloc * kng + kg : nullptr;
  const __half* kzb = K_AFF ? c.k.tok_zero + bh * c.cap_alloc * kng + kg : nullptr;
  const __half* vsb = V_AFF ? c.v.tok_scale + bh * c.cap_alloc * vng + vg : nullptr;
  const __half* vzb = V_AFF ? c.v.tok_zero + bh * c.cap_alloc * vng + vg : nullptr;

  float m[G], l[G], zacc[G], acc[G][16];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = neg_inf();
    l[h] = 0.0f;
    zacc[h] = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[h][i] = 0.0f;
  }

  for (int base = t0; base < t1; base += TPC * C) {
    Codes<KB> kc[C];
    Codes<VB> vc[C];
    float ksc[C], kzr[C], vsc[C], vzr[C];
    bool valid[C];
#pragma unroll
    for (int cc = 0; cc < C; ++cc) {
      const int t = base + cc * TPC + slot;
      valid[cc] = t < t1;
      const size_t tt = valid[cc] ? (size_t)t : (size_t)t0;
      load_codes<KB>(kc[cc], kbase + tt * KROW);
      load_codes<VB>(vc[cc], vbase + tt * VROW);
      if constexpr (K_AFF || K_Q40) ksc[cc] = __half2float(ksb[tt * kng]);
      if constexpr (K_AFF) kzr[cc] = __half2float(kzb[tt * kng]);
      if constexpr (V_AFF) {
        vsc[cc] = __half2float(vsb[tt * vng]);
        vzr[cc] = __half2float(vzb[tt * vng]);
      }
    }

    // Scores (log2 domain) of this lane-group's C tokens.
    float s[C][G];
#pragma unroll
    for (int cc = 0; cc < C; ++cc) {
      float x[16];
      unpack<KB>(kc[cc], x);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float p = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) p = fmaf(qf[h][i], x[i], p);
        if constexpr (K_AFF) p = fmaf(ksc[cc], p, kzr[cc] * qsum[h]);
        if constexpr (K_Q40) p = ksc[cc] * fmaf(-8.0f, qsum[h], p);
        s[cc][h] = p;
      }
    }
#pragma unroll
    for (int cc = 0; cc < C; ++cc) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int o = NL / 2; o >= 1; o >>= 1) s[cc][h] += __shfl_xor_sync(0xffffffffu, s[cc][h], o);
        if (!valid[cc]) s[cc][h] = neg_inf();
      }
    }

    // Online softmax: one rescale per step.
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
      float x[16];
      unpack<VB>(vc[cc], x);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if constexpr (V_AFF) {
          const float w = pw[cc][h] * vsc[cc];
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[h][i] = fmaf(w, x[i], acc[h][i]);
          zacc[h] = fmaf(pw[cc][h], vzr[cc], zacc[h]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[h][i] = fmaf(pw[cc][h], x[i], acc[h][i]);
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
      for (int i = 0; i < 16; ++i) sm_acc[warp][h][16 * j + i] = acc[h][i];
      if (j == 0) {
        sm_m[warp][h] = m[h];
        sm_l[warp][h] = l[h];
      }
    }
  }
  __syncthreads();

  // Merge the warps; write the output (one split) or this split's partial.
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int h = idx / D, d = idx % D;
    float M = sm_m[0][h];
#pragma unroll
    for (int w = 1; w < kDecodeWarps; ++w) M = fmaxf(M, sm_m[w][h]);
    float A = 0.0f, L = 0.0f;
    if (M != neg_inf()) {
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) {
        const float e = (sm_m[w][h] == neg_inf()) ? 0.0f : exp2f(sm_m[w][h] - M);
        A = fmaf(sm_acc[w][h][d], e, A);
        L = fmaf(sm_l[w][h], e, L);
      }
    }
    if (a.nsplit == 1) {
      const size_t oo = ((size_t)b * a.Hq + (size_t)kvh * G + h) * D + d;
      store_io(a.out, oo, a.io_dtype, L > 0.0f ? A / L : 0.0f);
    } else {
      float* P = a.partials + ((bh * a.nsplit + split) * G + h) * (D + 2);
      P[d] = A;
      if (d == 0) {
        P[D] = M;
        P[D + 1] = L;
      }
    }
  }
  if (a.nsplit == 1) return;

  // The last split of this (b, kv head) to finish merges all partials.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&c.split_sem[bh], 1u) == (unsigned)(a.nsplit - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int h = idx / D, d = idx % D;
    const float* P0 = a.partials + (bh * a.nsplit * G + h) * (D + 2);
    const size_t stride = (size_t)G * (D + 2);
    float M = neg_inf();
    for (int sp = 0; sp < a.nsplit; ++sp) M = fmaxf(M, __ldcg(P0 + sp * stride + D));
    float A = 0.0f, L = 0.0f;
    if (M != neg_inf()) {
      for (int sp = 0; sp < a.nsplit; ++sp) {
        const float ms = __ldcg(P0 + sp * stride + D);
        const float e = (ms == neg_inf()) ? 0.0f : exp2f(ms - M);
        A = fmaf(__ldcg(P0 + sp * stride + d), e, A);
        L = fmaf(__ldcg(P0 + sp * stride + D + 1), e, L);
      }
    }
    const size_t oo = ((size_t)b * a.Hq + (size_t)kvh * G + h) * D + d;
    store_io(a.out, oo, a.io_dtype, L > 0.0f ? A / L : 0.0f);
  }
  if (threadIdx.x == 0) c.split_sem[bh] = 0u;
}

template <int D, int G, int KF, int VF>
cudaError_t launch_decode_dg(const CacheView& c, const DecodeArgs& a, cudaStream_t st) {
  constexpr int C = (G >= 3) ? 2 : 4;
  const dim3 grid(a.nsplit, c.Hkv, c.B);
  decode_kernel<D, G, KF, VF, C><<<grid, 128, 0, st>>>(c, a);
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

template <int KF, int VF>
cudaError_t launch_decode(const CacheView& c, int G, const DecodeArgs& a, cudaStream_t st) {
  switch (c.D) {
    case 32: return launch_decode_d<32, KF, VF>(c, G, a, st);
    case 64: return launch_decode_d<64, KF, VF>(c, G, a, st);
    case 128: return launch_decode_d<128, KF, VF>(c, G, a, st);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace kvq
