// Eviction kernels.
//
// "StreamingLLM + KIVI" page, "Implementation": when the stored length passes
// sink + window, logical rows [sink, len - window) are dropped and the window
// is concatenated after the sinks; per-token V metadata moves with its token,
// K's per-channel scales do not.  "SnapKV" page, "How it works", step 4: only
// the selected rows are kept, in ascending order.
//
// Both moves run in place.  Destination rows never lie above their sources
// (dst = sink + i <= sink + shift + i; a keep-set has idx[j] >= j), so a CTA
// that owns one (b, kv head) and copies its rows in increasing order, reading
// each chunk completely before writing it, never overwrites a row it has not
// read yet.
#include "kvq_internal.cuh"

namespace kvq {

template <typename U>
__device__ __forceinline__ void block_move_forward(uint8_t* dst, const uint8_t* src, size_t nbytes) {
  const size_t units = nbytes / sizeof(U);
  U* d = reinterpret_cast<U*>(dst);
  const U* s = reinterpret_cast<const U*>(src);
  for (size_t base = 0; base < units; base += blockDim.x) {
    const size_t i = base + threadIdx.x;
    U val;
    const bool has = i < units;
    if (has) val = s[i];
    __syncthreads();
    if (has) d[i] = val;
    __syncthreads();
  }
}

// Forward (dst < src) block-wide move with the widest unit that divides the
// two addresses and the length.
__device__ void block_move(uint8_t* dst, const uint8_t* src, size_t nbytes) {
  const uintptr_t a = (uintptr_t)dst | (uintptr_t)src | (uintptr_t)nbytes;
  if ((a & 15) == 0) block_move_forward<uint4>(dst, src, nbytes);
  else if ((a & 7) == 0) block_move_forward<uint2>(dst, src, nbytes);
  else if ((a & 3) == 0) block_move_forward<uint32_t>(dst, src, nbytes);
  else if ((a & 1) == 0) block_move_forward<uint16_t>(dst, src, nbytes);
  else block_move_forward<uint8_t>(dst, src, nbytes);
}

__device__ void move_side_rows(const SideView& s, size_t bh, int cap_alloc, int dst_row, int src_row, int nrows) {
  {
    const size_t rb = s.row_bytes;
    uint8_t* base = s.codes + bh * cap_alloc * rb;
    block_move(base + dst_row * rb, base + src_row * rb, nrows * rb);
  }
  const size_t mb = (size_t)s.n_groups * sizeof(__half);
  if (s.tok_scale) {
    uint8_t* base = reinterpret_cast<uint8_t*>(s.tok_scale) + bh * cap_alloc * mb;
    block_move(base + dst_row * mb, base + src_row * mb, nrows * mb);
  }
  if (s.tok_zero) {
    uint8_t* base = reinterpret_cast<uint8_t*>(s.tok_zero) + bh * cap_alloc * mb;
    block_move(base + dst_row * mb, base + src_row * mb, nrows * mb);
  }
}

__device__ __forceinline__ void arrive_and_update(const CacheView& c, int new_stored, bool apply) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(&c.state->evict_arrive, 1u);
    if (prev == gridDim.x - 1) {
      if (apply) c.state->stored = new_stored;
      c.state->evict_arrive = 0u;
      __threadfence();
    }
  }
}

// One CTA per (b, kv head).
__global__ void __launch_bounds__(256) evict_middle_kernel(CacheView c) {
  __shared__ int s_len;
  if (threadIdx.x == 0) s_len = c.state->stored;
  __syncthreads();
  const int len = s_len;
  const int keep = c.sink + c.window;
  const size_t bh = blockIdx.x;
  if (len > keep) {
    const int shift = len - keep;
    move_side_rows(c.k, bh, c.cap_alloc, c.sink, c.sink + shift, c.window);
    move_side_rows(c.v, bh, c.cap_alloc, c.sink, c.sink + shift, c.window);
  }
  arrive_and_update(c, keep, len > keep);
}

// Gathers rows idx[0..n_keep) of one plane into rows [0, n_keep), chunk by
// chunk through shared memory.
__device__ void gather_plane(uint8_t* base, size_t rb, const int* __restrict__ idx, int n_keep, uint8_t* stage,
                             int stage_bytes) {
  const int rows_per_chunk = (int)(stage_bytes / rb);
  const bool w4 = (rb % 4) == 0;
  for (int j0 = 0; j0 < n_keep; j0 += rows_per_chunk) {
    const int nr = min(rows_per_chunk, n_keep - j0);
    if (w4) {
      const int wpr = (int)(rb / 4);
      for (int u = threadIdx.x; u < nr * wpr; u += blockDim.x) {
        const int r = u / wpr, col = u % wpr;
        reinterpret_cast<uint32_t*>(stage)[u] =
            reinterpret_cast<const uint32_t*>(base + (size_t)idx[j0 + r] * rb)[col];
      }
      __syncthreads();
      for (int u = threadIdx.x; u < nr * wpr; u += blockDim.x) {
        const int r = u / wpr, col = u % wpr;
        reinterpret_cast<uint32_t*>(base + (size_t)(j0 + r) * rb)[col] = reinterpret_cast<uint32_t*>(stage)[u];
      }
    } else {
      const int hpr = (int)(rb / 2);
      for (int u = threadIdx.x; u < nr * hpr; u += blockDim.x) {
        const int r = u / hpr, col = u % hpr;
        reinterpret_cast<uint16_t*>(stage)[u] =
            reinterpret_cast<const uint16_t*>(base + (size_t)idx[j0 + r] * rb)[col];
      }
      __syncthreads();
      for (int u = threadIdx.x; u < nr * hpr; u += blockDim.x) {
        const int r = u / hpr, col = u % hpr;
        reinterpret_cast<uint16_t*>(base + (size_t)(j0 + r) * rb)[col] = reinterpret_cast<uint16_t*>(stage)[u];
      }
    }
    __syncthreads();
  }
}

__device__ void gather_side(const SideView& s, size_t bh, int cap_alloc, const int* idx, int n_keep, uint8_t* stage,
                            int stage_bytes) {
  gather_plane(s.codes + bh * cap_alloc * s.row_bytes, s.row_bytes, idx, n_keep, stage, stage_bytes);
  const size_t mb = (size_t)s.n_groups * sizeof(__half);
  if (s.tok_scale)
    gather_plane(reinterpret_cast<uint8_t*>(s.tok_scale) + bh * cap_alloc * mb, mb, idx, n_keep, stage, stage_bytes);
  if (s.tok_zero)
    gather_plane(reinterpret_cast<uint8_t*>(s.tok_zero) + bh * cap_alloc * mb, mb, idx, n_keep, stage, stage_bytes);
}

constexpr int kStageBytes = 32768;

// One CTA per (b, kv head): validate the keep-set, then gather in place.
__global__ void __launch_bounds__(256) evict_keepset_kernel(CacheView c, const int* __restrict__ keep_idx,
                                                            int n_keep) {
  __shared__ __align__(16) uint8_t stage[kStageBytes];
  __shared__ int s_len;
  if (threadIdx.x == 0) s_len = c.state->stored;
  __syncthreads();
  const int len = s_len;
  const size_t bh = blockIdx.x;
  const int* idx = keep_idx + bh * n_keep;
  int bad = (n_keep > len) ? 1 : 0;
  for (int j = threadIdx.x; j < n_keep && !bad; j += blockDim.x) {
    const int x = idx[j];
    if (x < 0 || x >= len) bad = 1;
    if (j > 0 && idx[j - 1] >= x) bad = 1;
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (threadIdx.x == 0) set_status(c.state, KVQ_DEV_BAD_KEEPSET);
  } else {
    gather_side(c.k, bh, c.cap_alloc, idx, n_keep, stage, kStageBytes);
    gather_side(c.v, bh, c.cap_alloc, idx, n_keep, stage, kStageBytes);
  }
  // The stored count becomes n_keep; an invalid set anywhere leaves the status
  // word set and the cache contents unspecified.
  arrive_and_update(c, n_keep, true);
}

cudaError_t launch_evict_middle(const CacheView& c, cudaStream_t st) {
  evict_middle_kernel<<<c.B * c.Hkv, 256, 0, st>>>(c);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_evict_keepset(const CacheView& c, const int* idx, int n_keep, cudaStream_t st) {
  evict_keepset_kernel<<<c.B * c.Hkv, 256, 0, st>>>(c, idx, n_keep);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvq
