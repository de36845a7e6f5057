// kvq_decode_attn_noalloc: decode attention whose split-KV scratch lives in a
// fixed device array owned by this library, for callers that cannot allocate
// device memory themselves.
//
// Some callers run where a cudaMalloc is not allowed or not possible: code
// inside an allocator or a memory-pool callback, a plugin host that forbids
// device allocations after start-up, or a latency-critical loop that must
// never reach the driver's allocator.  They still own the cache, the query and
// the output; only the per-split partial results need somewhere to go.  This
// file keeps them in `g_decode_scratch`, a file-scope device array of
// kvq_noalloc_scratch_bytes() bytes that every GPU which loads the library
// holds until the process exits.
//
// The array's name is only a host-side stand-in in host code, not a device
// address, so the real address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached here, together
// with the unique id of the CUDA context it belongs to.  That look-up happens
// inside the first call on each device, and again in the first call after
// the device's context was replaced (cudaDeviceReset ends the context, and
// the array then lives at an address of the new one); make those calls
// before any stream capture.
//
// Every call on a device shares the one array and leaves its last contents
// there.  Nothing in it has to start at zero: each split writes its partial
// before the merging CTA reads it, and the arrival counters that decide which
// CTA merges live in the cache buffer (zeroed at init, reset by every call).
// Calls that overlap on the GPU, on any cache or stream of the same device,
// race on the array and give wrong results; serialise them.
#include <stdio.h>

#include <mutex>

#include <cudaTypedefs.h>

#include "kvq_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;   // 4 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};   // id of the context the address belongs to

// Unique id of the calling thread's current CUDA context (never reused within
// the process), or 0 when there is none yet or the driver cannot tell.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_decode_scratch on the current device: looked up once
// per device and context (again when the context id changed or is unknown).
kvq_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvq::report_error(KVQ_ERR_CUDA, "kvq_decode_attn_noalloc: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return kvq::report_error(KVQ_ERR_UNSUPPORTED, "kvq_decode_attn_noalloc: device index beyond 63");
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long ctx = current_context_id();
  if (g_scratch_addr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);   // makes the device's context current if needed
    if (e != cudaSuccess || p == nullptr)
      return kvq::report_error(KVQ_ERR_CUDA, "kvq_decode_attn_noalloc: cudaGetSymbolAddress of the scratch failed");
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = current_context_id();
  }
  *out = g_scratch_addr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" {

size_t kvq_noalloc_scratch_bytes(void) { return kScratchBytes; }

kvq_status kvq_decode_attn_noalloc(kvq_cache cache, const void* q, void* out, int32_t n_q_heads, int32_t io_dtype,
                                   float softmax_scale, cudaStream_t stream) {
  if (!cache) return kvq::report_error(KVQ_ERR_INVALID_ARG, "kvq_decode_attn_noalloc: null cache");
  const size_t need = kvq_decode_workspace_bytes(cache, n_q_heads);
  if (need > kScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "kvq_decode_attn_noalloc: this cache needs %zu bytes of split scratch, the built-in array holds %zu; "
             "use kvq_decode_attn with a workspace",
             need, kScratchBytes);
    return kvq::report_error(KVQ_ERR_CAPACITY, msg);
  }
  void* scratch = nullptr;
  if (need > 0) {
    const kvq_status s = scratch_address(&scratch);
    if (s != KVQ_OK) return s;
  }
  return kvq_decode_attn(cache, q, out, n_q_heads, io_dtype, softmax_scale, scratch, need, stream);
}

}  // extern "C"
