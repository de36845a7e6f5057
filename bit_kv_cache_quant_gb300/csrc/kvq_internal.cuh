// Internal definitions shared by the kvq kernels and the C-ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kRowAlign = 64;      // cap_alloc granularity: whole tiles are always in bounds
constexpr int kPlaneAlign = 256;   // byte alignment of every plane

// Device-resident counters of one cache (first 256 bytes of the cache buffer).
struct DevState {
  long long pos;            // absolute position of the next token
  int stored;               // rows holding live tokens
  int status;               // first KVQ_DEV_* error, 0 if none
  unsigned append_arrive;   // CTA arrival counter of the append in flight
  unsigned evict_arrive;    // CTA arrival counter of the eviction in flight
  int k_calibrated;         // per-channel K scales frozen
  int tail;                 // KIVI_BLOCK: rows in the full-precision tail
  unsigned step_arrive;     // CTA arrival counter of the fused append + decode in flight
  int pad[55];
};
static_assert(sizeof(DevState) == 256, "DevState must be 256 bytes");

// Format codes used as template parameters of the decode kernels.
enum Fmt : int {
  F_FP16 = 0,
  F_KIVI8 = 1,
  F_KIVI4 = 2,
  F_AFF8 = 3,
  F_AFF4 = 4,
  F_Q40 = 5,
  F_KIVIB8 = 6,   // KIVI_BLOCK keys, 8 / 4 bits
  F_KIVIB4 = 7,
};

struct SideView {
  uint8_t* codes;        // [B][Hkv][cap_alloc][row_bytes]
  __half* tok_scale;     // [B][Hkv][cap_alloc][n_groups]
  __half* tok_zero;      // [B][Hkv][cap_alloc][n_groups]
  __half* ch_scale;      // [B][Hkv][D]
  __half* ch_zero;       // [B][Hkv][D]
  float* ch_scale32;     // [B][Hkv][D]
  float* ch_zero32;      // [B][Hkv][D]
  __half* blk_scale;     // [B][Hkv][cap_alloc / R][D] (KIVI_BLOCK)
  __half* blk_zero;      // [B][Hkv][cap_alloc / R][D] (KIVI_BLOCK)
  int fmt;               // kvq_format
  int bits;
  int group;             // channels per (scale, zero) group
  int row_bytes;
  int n_groups;          // per-token metadata entries per row
};

struct CacheView {
  // TMA descriptors of the K and V code planes, viewed as [B*Hkv*cap_alloc rows,
  // row_bytes] and copied 64 rows at a time with a 32/64/128-byte swizzle (rows
  // of 256 bytes as [rows][2][128]).  Encoded once per cache; has_maps = 0 when
  // the driver cannot encode them (the CUDA-core decode kernel is used then).
  CUtensorMap kmap;
  CUtensorMap vmap;
  DevState* state;
  unsigned* split_sem;   // [B*Hkv]
  const float* k_bias;   // [Hkv][D] or null
  SideView k, v;
  float* tail_k;         // [B][Hkv][R][D] full-precision tail (KIVI_BLOCK), else null
  float* tail_v;
  int B, Hkv, D, cap, cap_alloc, layout, sink, window;
  int has_maps;
  int sms;               // SMs of the device the cache was bound on
};

// Programmatic dependent launch: wait until the grids this launch depends on
// have completed (a no-op for a launch without the attribute), and allow the
// next dependent launch to start its prologue.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ void set_status(DevState* st, int code) {
  atomicCAS(&st->status, 0, code);
}

// ------------------------------------------------------------ input loads --

template <typename T> struct In;
template <> struct In<float> {
  static __device__ __forceinline__ float ld(const float* p) { return *p; }
};
template <> struct In<__nv_bfloat16> {
  static __device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
};
template <> struct In<__half> {
  static __device__ __forceinline__ float ld(const __half* p) { return __half2float(*p); }
};

// Reads E consecutive input elements as fp32 (exact for bf16 / fp16 inputs).
template <typename T, int E>
__device__ __forceinline__ void load_row_slice(const T* p, float (&x)[E]) {
#pragma unroll
  for (int i = 0; i < E; ++i) x[i] = In<T>::ld(p + i);
}

// Loads element i of an io-dtype tensor as fp32; stores fp32 as io dtype (RNE).
__device__ __forceinline__ float load_io(const void* p, size_t i, int dtype) {
  if (dtype == KVQ_DTYPE_F32) return static_cast<const float*>(p)[i];
  if (dtype == KVQ_DTYPE_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  return __half2float(static_cast<const __half*>(p)[i]);
}
__device__ __forceinline__ void store_io(void* p, size_t i, int dtype, float x) {
  if (dtype == KVQ_DTYPE_F32) static_cast<float*>(p)[i] = x;
  else if (dtype == KVQ_DTYPE_BF16) static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  else static_cast<__half*>(p)[i] = __float2half_rn(x);
}

// -------------------------------------------------------- exact arithmetic --
// The quantiser's decisions: IEEE fp32, round to nearest even, no contraction.

__device__ __forceinline__ float affine_scale(float mn, float mx, float levels) {
  return fmaxf(1e-5f, __fdiv_rn(__fsub_rn(mx, mn), levels));
}

__device__ __forceinline__ int affine_code(float x, float scale, float zero, float levels) {
  float t = __fdiv_rn(__fsub_rn(x, zero), scale);
  float u = fminf(fmaxf(rintf(t), 0.0f), levels);
  return (int)u;
}

// affine_code from inv = 1 / scale (rounded once per group): q = (x - zero) * inv
// is within 2^-23 of (x - zero) / scale relative to it, so wherever the
// clamped code depends on the quotient (|quotient| <= 256) q is within 2^-14 of
// it and rint(q) == rint(quotient) unless q lies within 2^-12 of a
// half-integer; only there (rarely) does the exact division decide.  Larger
// quotients clamp to the same code either way; NaN and infinities take the
// same path as in affine_code.  Bit-identical to affine_code.
__device__ __forceinline__ int affine_code_inv(float x, float scale, float inv, float zero, float levels) {
  const float d = __fsub_rn(x, zero);
  float t = __fmul_rn(d, inv);
  if (fabsf(__fsub_rn(__fsub_rn(t, floorf(t)), 0.5f)) < 0x1p-12f) t = __fdiv_rn(d, scale);
  const float u = fminf(fmaxf(rintf(t), 0.0f), levels);
  return (int)u;
}

// Symmetric Q4_0 nibble: d == 0 stores level 0 (nibble 8).
__device__ __forceinline__ int q40_code(float x, float d) {
  if (d == 0.0f) return 8;
  float t = __fdiv_rn(x, d);
  float q = fminf(fmaxf(rintf(t), -8.0f), 7.0f);
  return (int)q + 8;
}

// q40_code from inv = 1 / d, by the argument of affine_code_inv (quotients
// that matter are within [-9, 8]).  Bit-identical to q40_code.
__device__ __forceinline__ int q40_code_inv(float x, float d, float inv) {
  if (d == 0.0f) return 8;
  float t = __fmul_rn(x, inv);
  if (fabsf(__fsub_rn(__fsub_rn(t, floorf(t)), 0.5f)) < 0x1p-12f) t = __fdiv_rn(x, d);
  const float q = fminf(fmaxf(rintf(t), -8.0f), 7.0f);
  return (int)q + 8;
}

// Runs fn (a cudaError_t() callable that must be idempotent) unless it has
// already succeeded for the current device at this call site; `done` holds one
// bit per device ordinal below 64 (higher ordinals run fn every time).  A
// function attribute set with cudaFuncSetAttribute applies to the current
// device only, hence per device.  Concurrent first calls may both run fn.
template <typename F>
cudaError_t once_per_device(std::atomic<unsigned long long>& done, F fn) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = fn();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Counts kernels enqueued by the current API call (host side, per thread).
void note_launch(int n = 1);

// Records `msg` as the calling thread's last error and returns `s`.
kvq_status report_error(kvq_status s, const char* msg);

// Launchers (defined in the kernel files).
// Token t of (b, kv head) bh is row bh * hstride + t of k and v (hstride >= n).
// recompute: KIVI keys, recompute the per-channel range over the stored and new keys first.
cudaError_t launch_append(const CacheView& c, const void* k, const void* v, int n, long long hstride, int in_dtype,
                          bool calibrate, bool recompute, cudaStream_t st);
cudaError_t launch_evict_middle(const CacheView& c, cudaStream_t st);
cudaError_t launch_evict_keepset(const CacheView& c, const int* idx, int n_keep, cudaStream_t st);

struct DecodeArgs {
  const void* q;
  void* out;
  int io_dtype;
  int Hq;
  float qscale;      // softmax scale * log2(e)
  float* partials;   // [B*Hkv][nsplit][G][D + kPartialPad] or null when nsplit == 1
  int nsplit;        // splits per (b, kv head): the CUDA-core kernel's grid x extent
  int nsplit_tc;     // the same for the tensor-core kernel
  int wide;          // tensor-core kernel: 1 = two tile groups of warps per CTA (the grid fits
                     // in one wave at the CTAs per SM of that shape) instead of one; 2 = four
                     // tile groups, one CTA per SM
  // Fused append (tensor-core kernel): the new token's key and value rows
  // [B][Hkv][D] of in_dtype, coded into the cache by this launch before it
  // attends over the cache including that token; null for a plain decode.
  const void* k_new;
  const void* v_new;
  int in_dtype;
  // Test hook (0 in use): bytes the first tile's barrier of every CTA expects
  // beyond what its copies bring, so that the wait for that tile runs out
  // and the launch reports KVQ_DEV_TIMEOUT.
  unsigned stall_tx;
  // The kernel just before this launch on the stream writes neither this
  // cache nor its counters (kvq_append_decode's KVQ_STEP_EARLY_READ): the
  // launch reads them before its dependency wait.
  int early;
};
// Defined once per (K format, V format) pair; returns cudaErrorNotSupported for
// an (D, G) outside the instantiated set.
template <int KF, int VF>
cudaError_t launch_decode(const CacheView& c, int G, const DecodeArgs& a, cudaStream_t st);

// arrive: B * Hkv arrival counts then one failure flag (device, zeroed by the launcher).
cudaError_t launch_snapkv(const void* k, long long head_stride, int B, int Hkv, int S, int D, int w, int budget,
                          int n_sink, float* scores, int* idx, float2* stats, int nchunk, unsigned* arrive,
                          cudaStream_t st);
// Max-pool smoothing of [BH][S] scores, odd kernel_size <= 63, in != out.
cudaError_t launch_snapkv_pool(const float* in, float* out, int BH, int S, int kernel_size, cudaStream_t st);
// fail (device, nullable): a scoring launch's failure flag; when set the indices are all -1.
cudaError_t launch_topk(const float* scores, int B, int Hkv, int S, int budget, int n_sink, int* idx,
                        const int* fail, cudaStream_t st);

constexpr unsigned long long kWaitNs = 200000000ull;   // default limit of a bounded device wait (200 ms)
constexpr int kSnapChunk = 256;   // keys per CTA of the SnapKV scoring kernels
constexpr int kTmaRows = 64;      // rows per TMA box of a code plane (one decode tile)
constexpr int kMaxSplits = 128;   // decode splits per (b, kv head)
constexpr int kTcStagesNarrow = 2;   // tensor-core decode, four-warp CTAs: pipeline stages at most
constexpr int kTcWaves = 2;       // tensor-core decode, four-warp CTAs: waves of CTAs the splits fill
constexpr int kTcCtasPerSm = 4;   // tensor-core decode, four-warp CTAs resident per SM (five measured slower: 96 registers)
constexpr int kPartialPad = 4;    // decode partial row: D accumulators, max, sum, 2 pad (16-byte rows)

}  // namespace kvq
