// The per-layer floor of a chain of dependent launches on this GPU: what a
// decode step of L layers costs when each layer's launch does nothing but
// read its share of the cache.  Each mode captures L launches (one per
// layer, programmatic dependent launches) in one CUDA graph; every launch
// reads its own `bytes`-sized buffer (distinct buffers, L2 flushed before
// each replay), split over `ctas` CTAs that copy their contiguous chunk into
// shared memory with bulk copies and an mbarrier (bounded wait).
//   0 empty: dependency wait and trigger only
//   1 the chunk copied after the dependency wait, trigger after the copy
//   2 trigger at entry, the chunk requested into L2 before the wait, copied after it
//   3 trigger at entry, the chunk copied before the wait (an upper bound:
//     legal here only because no launch writes these buffers)
//   4 mode 2 plus a last-arriver merge of per-CTA partials per head (8 heads)
//   5 mode 1 without the programmatic-dependent launch attribute
// Prints one JSON line per (mode, ctas): microseconds per launch (median of
// 20 replays) and the read rate per layer.  Used by `bench.py --floor`.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#define CK(x)                                                                          \
  do {                                                                                 \
    cudaError_t e_ = (x);                                                              \
    if (e_ != cudaSuccess) {                                                           \
      fprintf(stderr, "%s at line %d: %s\n", #x, __LINE__, cudaGetErrorString(e_));   \
      exit(1);                                                                         \
    }                                                                                  \
  } while (0)

namespace {

__device__ __forceinline__ uint32_t s32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool mbar_ready(uint64_t* m, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(s32(m)), "r"(parity)
      : "memory");
  return ok != 0;
}

struct Args {
  const uint8_t* buf;   // this launch's buffer
  uint32_t chunk;       // bytes per CTA, a multiple of 16 (<= dynamic shared memory)
  float* out;           // one float per CTA
  float* part;          // [ctas][400] partials (mode 4)
  unsigned* sem;        // [8] arrival counters (mode 4)
  int mode;
  int per_head;         // CTAs per head (mode 4)
};

extern __shared__ __align__(128) uint8_t sm[];

__global__ void __launch_bounds__(256) floor_kernel(Args a) {
  __shared__ __align__(8) uint64_t mb;
  __shared__ int s_last;
  __shared__ int s_fail;
  const uint8_t* src = a.buf + (size_t)blockIdx.x * a.chunk;
  if (a.mode >= 2 && a.mode <= 4) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    s_fail = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(s32(&mb)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (a.mode == 2 || a.mode == 4)
      for (uint32_t o = 0; o < a.chunk; o += 16384)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src + o), "r"(min(16384u, a.chunk - o))
                     : "memory");
  }
  __syncthreads();
  auto issue = [&]() {
    if (threadIdx.x == 0 && a.mode != 0) {
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s32(&mb)), "r"(a.chunk) : "memory");
      for (uint32_t o = 0; o < a.chunk; o += 16384)
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                s32(sm + o)),
            "l"(src + o), "r"(min(16384u, a.chunk - o)), "r"(s32(&mb))
            : "memory");
    }
  };
  if (a.mode == 3) issue();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (a.mode != 3) issue();
  float acc = 0.f;
  if (a.mode != 0) {
    const uint64_t t0 = now_ns();
    while (!mbar_ready(&mb, 0)) {
      if (now_ns() - t0 > 100000000ull) {   // 100 ms: give up, flag the result
        s_fail = 1;
        break;
      }
    }
    if (!s_fail)
      for (uint32_t i = threadIdx.x * 16; i < a.chunk; i += 256 * 16)
        acc += __int_as_float(*(const int*)(sm + i) & 0x3f800000);
  }
  if (a.mode == 1 || a.mode == 5) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (a.mode == 4) {
    for (int i = threadIdx.x; i < 390; i += 256) a.part[(size_t)blockIdx.x * 400 + i] = acc + i;
    __syncthreads();
    if (threadIdx.x == 0) {
      const int h = blockIdx.x / a.per_head;
      unsigned old;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.sem + h) : "memory");
      s_last = old == (unsigned)(a.per_head - 1);
    }
    __syncthreads();
    if (s_last) {
      const int h = blockIdx.x / a.per_head;
      for (int i = threadIdx.x; i < 390; i += 256) {
        float v[32];
        const int n = min(a.per_head, 32);
        for (int s = 0; s < n; ++s) v[s] = __ldcg(a.part + (size_t)(h * a.per_head + s) * 400 + i);
        float r = 0.f;
        for (int s = 0; s < n; ++s) r += v[s];
        if (i == 0) a.out[blockIdx.x] = r;
      }
      if (threadIdx.x == 0) a.sem[h] = 0;
    }
    return;
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  if (threadIdx.x == 0) a.out[blockIdx.x] = acc + (s_fail ? 1e9f : 0.f);
}

}  // namespace

int main(int argc, char** argv) {
  const int L = argc > 1 ? atoi(argv[1]) : 28;                       // launches (layers) per graph
  const size_t bytes = argc > 2 ? strtoull(argv[2], nullptr, 10) : 9468480;   // bytes read per launch
  const size_t alloc = (bytes + 1048575) / 1048576 * 1048576 + (1 << 20);
  int sms = 0, dev = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  std::vector<uint8_t*> bufs(L);
  for (int l = 0; l < L; ++l) {
    CK(cudaMalloc(&bufs[l], alloc));
    CK(cudaMemset(bufs[l], 1, alloc));
  }
  uint8_t* flush;
  const size_t flush_bytes = size_t(256) << 20;
  CK(cudaMalloc(&flush, flush_bytes));
  float* out;
  CK(cudaMalloc(&out, 4096 * sizeof(float)));
  float* part;
  CK(cudaMalloc(&part, (size_t)L * 1024 * 400 * sizeof(float)));
  unsigned* sem;
  CK(cudaMalloc(&sem, (size_t)L * 8 * sizeof(unsigned)));
  CK(cudaMemset(sem, 0, (size_t)L * 8 * sizeof(unsigned)));
  const int max_smem = 100 * 1024;
  CK(cudaFuncSetAttribute(floor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem));
  cudaStream_t st;
  CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  const int ctas_list[] = {sms, 256, 2 * sms, 4 * sms};
  const int modes[] = {0, 5, 1, 2, 3, 4};
  for (int mode : modes) {
    for (int nc : ctas_list) {
      const uint32_t chunk = (uint32_t)(((bytes + nc - 1) / nc + 15) / 16 * 16);
      if ((size_t)chunk * nc > alloc || chunk > (uint32_t)max_smem || nc > 1024) continue;
      if (mode == 4 && nc % 8) continue;
      cudaGraph_t g;
      cudaGraphExec_t ge;
      CK(cudaStreamBeginCapture(st, cudaStreamCaptureModeGlobal));
      for (int l = 0; l < L; ++l) {
        Args a{bufs[l], chunk, out, part + (size_t)l * 1024 * 400, sem + l * 8, mode, nc / 8};
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(nc);
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = chunk;
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = mode == 5 ? 0 : 1;
        CK(cudaLaunchKernelEx(&cfg, floor_kernel, a));
      }
      CK(cudaStreamEndCapture(st, &g));
      CK(cudaGraphInstantiate(&ge, g, 0));
      cudaEvent_t e0, e1;
      CK(cudaEventCreate(&e0));
      CK(cudaEventCreate(&e1));
      std::vector<float> ts;
      for (int r = 0; r < 25; ++r) {
        CK(cudaMemsetAsync(flush, r & 0xff, flush_bytes, st));
        CK(cudaEventRecord(e0, st));
        CK(cudaGraphLaunch(ge, st));
        CK(cudaEventRecord(e1, st));
        CK(cudaStreamSynchronize(st));
        float ms;
        CK(cudaEventElapsedTime(&ms, e0, e1));
        if (r >= 5) ts.push_back(ms);
      }
      std::sort(ts.begin(), ts.end());
      const double us = ts[ts.size() / 2] * 1000.0 / L;
      printf("{\"mode\": %d, \"ctas\": %d, \"layers\": %d, \"bytes_per_launch\": %zu, \"us_per_launch\": %.3f, "
             "\"gbs_per_layer\": %.1f}\n",
             mode, nc, L, bytes, us, mode ? (double)bytes / (us * 1e-6) / 1e9 : 0.0);
      fflush(stdout);
      CK(cudaEventDestroy(e0));
      CK(cudaEventDestroy(e1));
      CK(cudaGraphExecDestroy(ge));
      CK(cudaGraphDestroy(g));
    }
  }
  float h[4];
  CK(cudaMemcpy(h, out, sizeof(h), cudaMemcpyDeviceToHost));
  return 0;
}
