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
#include "quantize_row.cuh"

namespace kvq {

// ---------------------------------------------------------------------------
// Per-channel K calibration: min / max over the n tokens of one (b, kv head),
// then the fp32 scale / zero that codes are computed from and their fp16
// stored copies.  One CTA of 256 threads per (b, kv head); 256 % D == 0.
// Token t of (b, kv head) bh is row bh * hstride + t of k.
template <typename T>
__global__ void __launch_bounds__(256) calibrate_kivi_kernel(CacheView c, const T* __restrict__ k, int n,
                                                             long long hstride) {
  __shared__ float smn[256];
  __shared__ float smx[256];
  const int D = c.D;
  const int bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int d = tid % D;
  const int tg = tid / D;
  const int ntg = blockDim.x / D;
  float mn = __int_as_float(0x7f800000);   // +inf
  float mx = __int_as_float(0xff800000);   // -inf
  const T* base = k + (size_t)bh * hstride * D;
  for (int t = tg; t < n; t += ntg) {
    float x = In<T>::ld(base + (size_t)t * D + d);
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
    const float levels = (c.k.bits == 8) ? 255.0f : 15.0f;
    const float s = affine_scale(mn, mx, levels);
    const size_t o = (size_t)bh * D + d;
    c.k.ch_scale32[o] = s;
    c.k.ch_zero32[o] = mn;
    c.k.ch_scale[o] = __float2half_rn(s);
    c.k.ch_zero[o] = __float2half_rn(mn);
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

// One warp per (b, kv head, token) row of the append; 8 warps per CTA.  The
// input rows are requested before the counters are read (they do not depend
// on them).  With more than one CTA the last to arrive advances the counters,
// once every CTA has read them; a one-CTA append advances them directly.
constexpr int kAppendWarps = 8;
constexpr int kAppendCtasPerSm = 8;

template <typename T, int E>
__global__ void __launch_bounds__(32 * kAppendWarps) append_kernel(CacheView c, const T* __restrict__ k,
                                                                    const T* __restrict__ v, int n, long long rows,
                                                                    long long hstride) {
  __shared__ long long s_pos;
  __shared__ int s_stored;
  __shared__ int s_ok;
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
  if (threadIdx.x == 0) {
    s_pos = c.state->pos;
    s_stored = c.state->stored;
    const bool ok = (c.layout == KVQ_LAYOUT_RING) || ((long long)s_stored + n <= c.cap);
    s_ok = ok ? 1 : 0;
    if (!ok && blockIdx.x == 0) set_status(c.state, KVQ_DEV_OVERFLOW);
  }
  __syncthreads();
  // a warp codes rows row, row + stride, ...: the grid is capped at a few
  // CTAs per SM (one arrival each on the append counter), and each warp
  // requests its next row before coding the current one
  for (; s_ok && row < rows; row += stride) {
    float nk[E], nv[E];
    const bool more = row + stride < rows;
    if (more) load(row + stride, nk, nv);
    const int i = (int)((unsigned)row % (unsigned)n);
    const long long bh = (unsigned)row / (unsigned)n;
    const int kvh = (int)((unsigned)bh % (unsigned)c.Hkv);
    const long long p = s_pos + i;
    bool write = true;
    int slot;
    if (c.layout == KVQ_LAYOUT_RING) {
      if (p < c.sink) {
        slot = (int)p;
      } else {
        // a later token of this same append lands in the slot: skip this one
        write = p >= s_pos + n - c.window;
        slot = c.sink + (int)((p - c.sink) % c.window);
      }
    } else {
      slot = s_stored + i;
    }
    if (write) {
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
  if (threadIdx.x != 0) return;
  bool last = true;
  if (gridDim.x > 1) {
    __threadfence();
    last = atomicAdd(&c.state->append_arrive, 1u) == gridDim.x - 1;
  }
  if (last) {
    if (s_ok) {
      const long long np = s_pos + n;
      c.state->pos = np;
      if (c.layout == KVQ_LAYOUT_RING) {
        const long long w = (long long)c.sink + c.window;
        c.state->stored = (int)(np < w ? np : w);
      } else {
        c.state->stored = s_stored + n;
      }
    }
    if (gridDim.x > 1) {
      c.state->append_arrive = 0u;
      __threadfence();
    }
  }
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

template <typename T>
static cudaError_t launch_append_t(const CacheView& c, const void* k, const void* v, int n, long long hstride,
                                   bool calibrate, bool recompute, cudaStream_t st) {
  if (calibrate) {
    calibrate_kivi_kernel<T><<<c.B * c.Hkv, 256, 0, st>>>(c, static_cast<const T*>(k), n, hstride);
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
  const long long rows = (long long)c.B * c.Hkv * n;
  // at most kAppendCtasPerSm CTAs per SM; their warps sweep the rows
  const long long need = (rows + kAppendWarps - 1) / kAppendWarps;
  const long long cap = (long long)kAppendCtasPerSm * (c.sms > 0 ? c.sms : 132);
  const unsigned grid = (unsigned)(need < cap ? need : cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(32 * kAppendWarps);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
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
