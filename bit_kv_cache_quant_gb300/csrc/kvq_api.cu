// The extern "C" entry points declared in include/kvq.h: argument checks,
// plane layout, the host handle and kernel dispatch.  No device memory is
// allocated here; every buffer comes from the caller.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <mutex>
#include <new>
#include <string>

#include <cudaTypedefs.h>

#include "kvq_internal.cuh"

struct kvq_cache_s {
  kvq_config cfg;
  kvq_cache_layout lay;
  uint8_t* base;
  size_t bytes;
  int sms;
  bool k_calibrated;
  kvq::CacheView view;
};

namespace {

thread_local std::string g_err;
thread_local int g_launches = 0;

kvq_status fail(kvq_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

kvq_status cuda_fail(cudaError_t e, const char* what) {
  if (e == cudaErrorNotSupported) return fail(KVQ_ERR_UNSUPPORTED, "%s: shape not instantiated", what);
  return fail(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

void begin_call() {
  g_err.clear();
  g_launches = 0;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool valid_dtype(int d) { return d == KVQ_DTYPE_F32 || d == KVQ_DTYPE_BF16 || d == KVQ_DTYPE_F16; }

int row_bytes(int fmt, int bits, int D) { return fmt == KVQ_FMT_FP16 ? 2 * D : D * bits / 8; }

int token_groups(int fmt, int group, int D) {
  if (fmt == KVQ_FMT_AFFINE_TOKEN) return D / group;
  if (fmt == KVQ_FMT_Q4_0) return D / 32;
  return 0;
}

bool group_ok(int group, int D) {
  return (group == 16 || group == 32 || group == 64 || group == 128) && group <= D && D % group == 0;
}

kvq_status check_side(int fmt, int bits, int group, int D, bool is_k) {
  switch (fmt) {
    case KVQ_FMT_FP16:
      if (bits != 16) return fail(KVQ_ERR_INVALID_ARG, "fp16 format needs bits = 16");
      return KVQ_OK;
    case KVQ_FMT_KIVI_CHAN:
      if (!is_k) return fail(KVQ_ERR_UNSUPPORTED, "per-channel (KIVI_CHAN) storage is a K-side format");
      if (bits != 8 && bits != 4) return fail(KVQ_ERR_INVALID_ARG, "KIVI_CHAN bits must be 8 or 4");
      return KVQ_OK;
    case KVQ_FMT_AFFINE_TOKEN:
      if (bits != 8 && bits != 4) return fail(KVQ_ERR_INVALID_ARG, "AFFINE_TOKEN bits must be 8 or 4");
      if (!group_ok(group, D)) return fail(KVQ_ERR_INVALID_ARG, "AFFINE_TOKEN group must be 16/32/64/128 and divide D");
      return KVQ_OK;
    case KVQ_FMT_Q4_0:
      if (!is_k) return fail(KVQ_ERR_UNSUPPORTED, "Q4_0 storage is a K-side format");
      if (bits != 4 || (group != 32 && group != 0)) return fail(KVQ_ERR_INVALID_ARG, "Q4_0 needs bits 4, group 32");
      return KVQ_OK;
    case KVQ_FMT_KIVI_BLOCK:
      if (!is_k) return fail(KVQ_ERR_UNSUPPORTED, "KIVI_BLOCK storage is a K-side format");
      if (bits != 8 && bits != 4) return fail(KVQ_ERR_INVALID_ARG, "KIVI_BLOCK bits must be 8 or 4");
      if (group != 64 && group != 128)
        return fail(KVQ_ERR_UNSUPPORTED, "KIVI_BLOCK block length (k_group) must be 64 or 128 tokens");
      return KVQ_OK;
    default:
      return fail(KVQ_ERR_INVALID_ARG, "unknown format %d", fmt);
  }
}

// Template code of a side's format for the decode kernels.
int fmt_code(int fmt, int bits) {
  switch (fmt) {
    case KVQ_FMT_FP16: return kvq::F_FP16;
    case KVQ_FMT_KIVI_CHAN: return bits == 8 ? kvq::F_KIVI8 : kvq::F_KIVI4;
    case KVQ_FMT_AFFINE_TOKEN: return bits == 8 ? kvq::F_AFF8 : kvq::F_AFF4;
    case KVQ_FMT_Q4_0: return kvq::F_Q40;
    case KVQ_FMT_KIVI_BLOCK: return bits == 8 ? kvq::F_KIVIB8 : kvq::F_KIVIB4;
  }
  return -1;
}

kvq_status compute_layout(const kvq_config* c, kvq_cache_layout* L) {
  if (!c || !L) return fail(KVQ_ERR_INVALID_ARG, "null config or layout");
  if (c->batch < 1 || c->n_kv_heads < 1) return fail(KVQ_ERR_INVALID_ARG, "batch and n_kv_heads must be >= 1");
  if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128)
    return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d not supported (32, 64, 128)", c->head_dim);
  if (c->capacity < 1) return fail(KVQ_ERR_INVALID_ARG, "capacity must be >= 1");
  const int D = c->head_dim;
  switch (c->layout) {
    case KVQ_LAYOUT_LINEAR: break;
    case KVQ_LAYOUT_COMPACT:
      if (c->sink < 0 || c->window < 1) return fail(KVQ_ERR_INVALID_ARG, "sink >= 0 and window >= 1 required");
      if ((long long)c->capacity < (long long)c->sink + c->window + 1)
        return fail(KVQ_ERR_INVALID_ARG, "COMPACT capacity must be >= sink + window + 1");
      break;
    case KVQ_LAYOUT_RING:
      if (c->sink < 0 || c->window < 1) return fail(KVQ_ERR_INVALID_ARG, "sink >= 0 and window >= 1 required");
      if ((long long)c->capacity < (long long)c->sink + c->window)
        return fail(KVQ_ERR_INVALID_ARG, "RING capacity must be >= sink + window");
      break;
    default: return fail(KVQ_ERR_INVALID_ARG, "unknown layout %d", c->layout);
  }
  kvq_status s = check_side(c->k_format, c->k_bits, c->k_group, D, true);
  if (s != KVQ_OK) return s;
  s = check_side(c->v_format, c->v_bits, c->v_group, D, false);
  if (s != KVQ_OK) return s;
  if (c->k_bias != nullptr && c->k_format != KVQ_FMT_Q4_0)
    return fail(KVQ_ERR_UNSUPPORTED, "a K mean-centering bias requires Q4_0 keys");
  if (c->k_format == KVQ_FMT_KIVI_BLOCK &&
      (c->layout != KVQ_LAYOUT_LINEAR || c->v_format != KVQ_FMT_AFFINE_TOKEN || c->capacity < c->k_group))
    return fail(KVQ_ERR_UNSUPPORTED, "KIVI_BLOCK keys need the LINEAR layout, AFFINE_TOKEN values and capacity >= "
                                     "the block length");

  const size_t B = c->batch, H = c->n_kv_heads, BH = B * H;
  const size_t cap_alloc = align_up((size_t)c->capacity, kvq::kRowAlign);
  // The decode kernels address a code plane as one tensor of B * Hkv * cap_alloc
  // rows whose row coordinate is a signed 32-bit integer; keep every row and the
  // 64-row tile after it below 2^31.
  if (BH > (size_t)INT32_MAX || BH * cap_alloc > (size_t)INT32_MAX - kvq::kRowAlign)
    return fail(KVQ_ERR_UNSUPPORTED,
                "batch * n_kv_heads * capacity (rounded up to a multiple of %d rows) must stay below 2^31 - %d rows",
                kvq::kRowAlign, kvq::kRowAlign);
  const size_t A = kvq::kPlaneAlign;
  *L = kvq_cache_layout{};
  L->cap_alloc = (int32_t)cap_alloc;
  L->k_row_bytes = row_bytes(c->k_format, c->k_bits, D);
  L->v_row_bytes = row_bytes(c->v_format, c->v_bits, D);
  const int kgroup = c->k_format == KVQ_FMT_Q4_0 ? 32 : c->k_group;
  L->k_n_groups = token_groups(c->k_format, kgroup, D);
  L->v_n_groups = token_groups(c->v_format, c->v_group, D);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, A);
    return o;
  };
  L->state = take(sizeof(kvq::DevState));
  L->split_sem = take(BH * sizeof(unsigned));
  L->k_codes = take(BH * cap_alloc * L->k_row_bytes);
  if (L->k_n_groups) L->k_tok_scale = take(BH * cap_alloc * L->k_n_groups * 2);
  if (c->k_format == KVQ_FMT_AFFINE_TOKEN) L->k_tok_zero = take(BH * cap_alloc * L->k_n_groups * 2);
  if (c->k_format == KVQ_FMT_KIVI_CHAN) {
    L->k_ch_scale = take(BH * D * 2);
    L->k_ch_zero = take(BH * D * 2);
    L->k_ch_scale32 = take(BH * D * 4);
    L->k_ch_zero32 = take(BH * D * 4);
  }
  if (c->k_bias) L->k_bias = take(H * D * 4);
  if (c->k_format == KVQ_FMT_KIVI_BLOCK) {
    const size_t R = c->k_group;
    L->k_blk_scale = take(BH * (cap_alloc / R) * D * 2);
    L->k_blk_zero = take(BH * (cap_alloc / R) * D * 2);
    L->k_tail = take(BH * R * D * 4);
    L->v_tail = take(BH * R * D * 4);
  }
  L->v_codes = take(BH * cap_alloc * L->v_row_bytes);
  if (L->v_n_groups) L->v_tok_scale = take(BH * cap_alloc * L->v_n_groups * 2);
  if (c->v_format == KVQ_FMT_AFFINE_TOKEN) L->v_tok_zero = take(BH * cap_alloc * L->v_n_groups * 2);
  L->total_bytes = off;
  return KVQ_OK;
}

kvq::SideView side_view(uint8_t* base, int fmt, int bits, int group, int row_b, int ng, size_t codes, size_t ts,
                        size_t tz, size_t cs, size_t cz, size_t cs32, size_t cz32) {
  kvq::SideView s{};
  s.codes = base + codes;
  s.tok_scale = ts ? reinterpret_cast<__half*>(base + ts) : nullptr;
  s.tok_zero = tz ? reinterpret_cast<__half*>(base + tz) : nullptr;
  s.ch_scale = cs ? reinterpret_cast<__half*>(base + cs) : nullptr;
  s.ch_zero = cz ? reinterpret_cast<__half*>(base + cz) : nullptr;
  s.ch_scale32 = cs32 ? reinterpret_cast<float*>(base + cs32) : nullptr;
  s.ch_zero32 = cz32 ? reinterpret_cast<float*>(base + cz32) : nullptr;
  s.fmt = fmt;
  s.bits = bits;
  s.group = fmt == KVQ_FMT_Q4_0 ? 32 : group;
  s.row_bytes = row_b;
  s.n_groups = ng;
  return s;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A code plane of `rows` rows of `row_bytes` bytes, copied 64 rows at a time
// into shared memory with the 16-byte-chunk swizzle matching the row length.
bool encode_rows_map(CUtensorMap* m, void* base, size_t rows, int row_bytes) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r;
  if (row_bytes <= 128) {
    const CUtensorMapSwizzle sw = row_bytes == 32    ? CU_TENSOR_MAP_SWIZZLE_32B
                                  : row_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                                  : row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                     : CU_TENSOR_MAP_SWIZZLE_NONE;
    if (sw == CU_TENSOR_MAP_SWIZZLE_NONE) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)row_bytes, (cuuint32_t)kvq::kTmaRows};
    r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
            sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else if (row_bytes == 256) {
    const cuuint64_t dims[3] = {128, 2, rows};
    const cuuint64_t strides[2] = {128, 256};
    const cuuint32_t box[3] = {128, 2, (cuuint32_t)kvq::kTmaRows};
    r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    return false;
  }
  return r == CUDA_SUCCESS;
}

int decode_nsplit(const kvq_cache_s* c) {
  // The grid's splits per (b, kv head), an upper bound: about eight CTAs per
  // SM in all (even waves), at least 256 rows per split of the capacity (one
  // 64-row tile under 4096 rows).  The kernel spreads the rows actually
  // stored over at most this many splits.
  const int units = c->cfg.batch * c->cfg.n_kv_heads;
  int rows = c->cfg.capacity;
  if (c->cfg.layout != KVQ_LAYOUT_LINEAR) rows = c->cfg.sink + c->cfg.window + (c->cfg.layout == KVQ_LAYOUT_COMPACT);
  const int target = 8 * c->sms;
  int ns = (target + units / 2) / units;
  const int min_rows = rows >= 4096 ? 256 : 64;
  const int max_by_len = rows / min_rows > 1 ? rows / min_rows : 1;
  if (ns > max_by_len) ns = max_by_len;
  if (ns > kvq::kMaxSplits) ns = kvq::kMaxSplits;
  if (ns < 1) ns = 1;
  return ns;
}

// Launch plan of kvq_decode_attn for G query heads per kv head.  nsplit
// (decode_nsplit) drives the CUDA-core kernel and decides the tensor-core
// kernel's shape: eight-warp CTAs when that grid fits in one wave (wide), with
// the same splits; otherwise four-warp CTAs (kTcCtasPerSm per SM; eight-warp,
// two per SM, over four heads per kv head) with as many splits as fill two
// whole waves without starting a third.  A one-wave grid of up to four heads
// per kv head whose (b, kv head) units can each take at least two splits of
// four tiles of the capacity at one CTA per SM runs sixteen-warp CTAs instead
// (wide == 2): SMs / units splits (one fewer with a KIVI_BLOCK tail CTA).
struct DecodePlan {
  int nsplit;
  int nsplit_tc;
  int wide;
};

DecodePlan decode_plan(const kvq_cache_s* c, int G) {
  DecodePlan p;
  p.nsplit = decode_nsplit(c);
  const long long units = (long long)c->cfg.batch * c->cfg.n_kv_heads;
  p.wide = units * p.nsplit <= (G > 4 ? 1LL : 2LL) * c->sms;
  p.nsplit_tc = p.nsplit;
  if (p.wide && G <= 4) {
    int rows = c->cfg.capacity;
    if (c->cfg.layout != KVQ_LAYOUT_LINEAR) rows = c->cfg.sink + c->cfg.window + (c->cfg.layout == KVQ_LAYOUT_COMPACT);
    long long ns = c->sms / units - (c->cfg.k_format == KVQ_FMT_KIVI_BLOCK ? 1 : 0);
    if (ns > rows / (4 * kvq::kTmaRows)) ns = rows / (4 * kvq::kTmaRows);
    if (ns > kvq::kMaxSplits) ns = kvq::kMaxSplits;
    if (ns >= 2) {
      p.wide = 2;
      p.nsplit_tc = (int)ns;
    }
  }
  if (!p.wide) {
    const long long slots = (long long)kvq::kTcWaves * (G > 4 ? 2 : kvq::kTcCtasPerSm) * c->sms;
    int rows = c->cfg.capacity;
    if (c->cfg.layout != KVQ_LAYOUT_LINEAR) rows = c->cfg.sink + c->cfg.window + (c->cfg.layout == KVQ_LAYOUT_COMPACT);
    const int min_rows = rows >= 4096 ? 256 : 64;
    long long ns = slots / units;
    if (ns > rows / min_rows) ns = rows / min_rows;
    if (ns > kvq::kMaxSplits) ns = kvq::kMaxSplits;
    p.nsplit_tc = ns < 1 ? 1 : (int)ns;
  }
  return p;
}

size_t live_bytes(const kvq_cache_s* c, int stored) {
  const kvq_config& f = c->cfg;
  const size_t BH = (size_t)f.batch * f.n_kv_heads;
  auto per_token = [&](int fmt, int rb, int ng) {
    return (size_t)rb + (size_t)ng * 2 * (fmt == KVQ_FMT_AFFINE_TOKEN ? 2 : 1);
  };
  size_t b = BH * (size_t)stored *
             (per_token(f.k_format, c->lay.k_row_bytes, c->lay.k_n_groups) +
              per_token(f.v_format, c->lay.v_row_bytes, c->lay.v_n_groups));
  if (f.k_format == KVQ_FMT_KIVI_CHAN) b += BH * f.head_dim * 4;
  if (f.k_format == KVQ_FMT_KIVI_BLOCK) b += BH * ((size_t)stored / f.k_group) * f.head_dim * 4;   // block scale, zero
  return b;
}

}  // namespace

void kvq::note_launch(int n) { g_launches += n; }

kvq_status kvq::report_error(kvq_status s, const char* msg) {
  begin_call();
  return fail(s, "%s", msg);
}

extern "C" {

int32_t kvq_abi_version(void) { return KVQ_ABI_VERSION; }

const char* kvq_last_error(void) { return g_err.c_str(); }

int32_t kvq_last_launch_count(void) { return g_launches; }

kvq_status kvq_cache_layout_query(const kvq_config* cfg, kvq_cache_layout* out) {
  begin_call();
  return compute_layout(cfg, out);
}

kvq_status kvq_cache_init(const kvq_config* cfg, void* dev_mem, size_t bytes, cudaStream_t stream,
                          kvq_cache* out) {
  begin_call();
  if (!out) return fail(KVQ_ERR_INVALID_ARG, "null output handle");
  *out = nullptr;
  kvq_cache_layout lay;
  kvq_status s = compute_layout(cfg, &lay);
  if (s != KVQ_OK) return s;
  if (!dev_mem) return fail(KVQ_ERR_INVALID_ARG, "null cache buffer");
  if (((uintptr_t)dev_mem & (kvq::kPlaneAlign - 1)) != 0) return fail(KVQ_ERR_INVALID_ARG, "cache buffer must be 256-byte aligned");
  if (bytes < lay.total_bytes)
    return fail(KVQ_ERR_CAPACITY, "cache buffer holds %zu bytes, layout needs %zu", bytes, lay.total_bytes);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  kvq_cache_s* c = new (std::nothrow) kvq_cache_s();
  if (!c) return fail(KVQ_ERR_CAPACITY, "host allocation of the cache handle failed");
  c->cfg = *cfg;
  c->lay = lay;
  c->base = static_cast<uint8_t*>(dev_mem);
  c->bytes = bytes;
  c->sms = sms;
  c->k_calibrated = false;
  uint8_t* b = c->base;
  kvq::CacheView& v = c->view;
  v.state = reinterpret_cast<kvq::DevState*>(b + lay.state);
  v.split_sem = reinterpret_cast<unsigned*>(b + lay.split_sem);
  v.k_bias = cfg->k_bias ? reinterpret_cast<const float*>(b + lay.k_bias) : nullptr;
  v.k = side_view(b, cfg->k_format, cfg->k_bits, cfg->k_group, lay.k_row_bytes, lay.k_n_groups, lay.k_codes,
                  lay.k_tok_scale, lay.k_tok_zero, lay.k_ch_scale, lay.k_ch_zero, lay.k_ch_scale32, lay.k_ch_zero32);
  v.v = side_view(b, cfg->v_format, cfg->v_bits, cfg->v_group, lay.v_row_bytes, lay.v_n_groups, lay.v_codes,
                  lay.v_tok_scale, lay.v_tok_zero, 0, 0, 0, 0);
  v.k.blk_scale = lay.k_blk_scale ? reinterpret_cast<__half*>(b + lay.k_blk_scale) : nullptr;
  v.k.blk_zero = lay.k_blk_zero ? reinterpret_cast<__half*>(b + lay.k_blk_zero) : nullptr;
  v.tail_k = lay.k_tail ? reinterpret_cast<float*>(b + lay.k_tail) : nullptr;
  v.tail_v = lay.v_tail ? reinterpret_cast<float*>(b + lay.v_tail) : nullptr;
  v.B = cfg->batch;
  v.Hkv = cfg->n_kv_heads;
  v.D = cfg->head_dim;
  v.cap = cfg->capacity;
  v.cap_alloc = lay.cap_alloc;
  v.layout = cfg->layout;
  v.sink = cfg->sink;
  v.window = cfg->window;
  v.sms = sms;
  {
    const size_t rows = (size_t)cfg->batch * cfg->n_kv_heads * lay.cap_alloc;
    v.has_maps = cfg->head_dim >= 64 && encode_rows_map(&v.kmap, b + lay.k_codes, rows, lay.k_row_bytes) &&
                 encode_rows_map(&v.vmap, b + lay.v_codes, rows, lay.v_row_bytes);
  }
  // zero the counters and the split semaphores (they are contiguous at the front)
  e = cudaMemsetAsync(b, 0, lay.k_codes, stream);
  if (e == cudaSuccess && cfg->k_bias)
    e = cudaMemcpyAsync(b + lay.k_bias, cfg->k_bias, (size_t)cfg->n_kv_heads * cfg->head_dim * sizeof(float),
                        cudaMemcpyDeviceToDevice, stream);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "cache init");
  }
  *out = c;
  return KVQ_OK;
}

void kvq_cache_release(kvq_cache cache) { delete cache; }

namespace {

kvq_status append_rows(kvq_cache c, const void* k, const void* v, int64_t head_stride, int32_t n_tokens,
                       int32_t in_dtype, int32_t flags, cudaStream_t stream, const char* what) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "null cache");
  if (!k || !v) return fail(KVQ_ERR_INVALID_ARG, "null k or v");
  if (n_tokens < 1) return fail(KVQ_ERR_INVALID_ARG, "n_tokens must be >= 1");
  if (head_stride < n_tokens) return fail(KVQ_ERR_INVALID_ARG, "head_stride must be >= n_tokens");
  if (!valid_dtype(in_dtype)) return fail(KVQ_ERR_INVALID_ARG, "unknown input dtype %d", in_dtype);
  if (flags & ~(KVQ_APPEND_CALIBRATE_K | KVQ_APPEND_RECOMPUTE_K))
    return fail(KVQ_ERR_INVALID_ARG, "unknown append flags 0x%x", flags);
  const bool calibrate = (flags & KVQ_APPEND_CALIBRATE_K) != 0;
  const bool recompute = (flags & KVQ_APPEND_RECOMPUTE_K) != 0;
  if (calibrate && recompute)
    return fail(KVQ_ERR_INVALID_ARG, "KVQ_APPEND_CALIBRATE_K and KVQ_APPEND_RECOMPUTE_K exclude each other");
  if ((calibrate || recompute) && c->cfg.k_format != KVQ_FMT_KIVI_CHAN)
    return fail(KVQ_ERR_UNSUPPORTED, "K calibration flags apply to KIVI_CHAN keys only");
  if (recompute && c->cfg.layout == KVQ_LAYOUT_RING)
    return fail(KVQ_ERR_UNSUPPORTED, "KVQ_APPEND_RECOMPUTE_K needs a LINEAR or COMPACT layout");
  if (c->cfg.k_format == KVQ_FMT_KIVI_CHAN && !calibrate && !recompute && !c->k_calibrated)
    return fail(KVQ_ERR_UNSUPPORTED, "per-channel K scales are not calibrated yet (pass KVQ_APPEND_CALIBRATE_K)");
  if (c->cfg.k_format == KVQ_FMT_KIVI_BLOCK && flags)
    return fail(KVQ_ERR_INVALID_ARG, "KIVI_BLOCK appends take no flags");
  if (c->cfg.layout != KVQ_LAYOUT_RING && n_tokens > c->cfg.capacity)
    return fail(KVQ_ERR_CAPACITY, "append of %d tokens exceeds capacity %d", n_tokens, c->cfg.capacity);
  cudaError_t e = kvq::launch_append(c->view, k, v, n_tokens, head_stride, in_dtype, calibrate, recompute, stream);
  if (e != cudaSuccess) return cuda_fail(e, what);
  if (calibrate || recompute) c->k_calibrated = true;
  return KVQ_OK;
}

}  // namespace

kvq_status kvq_append(kvq_cache c, const void* k, const void* v, int32_t n_tokens, int32_t in_dtype, int32_t flags,
                      cudaStream_t stream) {
  begin_call();
  return append_rows(c, k, v, n_tokens, n_tokens, in_dtype, flags, stream, "kvq_append");
}

kvq_status kvq_convert(kvq_cache c, const void* k, const void* v, int64_t head_stride, int32_t n_tokens,
                       int32_t in_dtype, int32_t flags, cudaStream_t stream) {
  begin_call();
  return append_rows(c, k, v, head_stride, n_tokens, in_dtype, flags, stream, "kvq_convert");
}

kvq_status kvq_evict(kvq_cache c, int32_t mode, const int32_t* keep_idx, int32_t n_keep, cudaStream_t stream) {
  begin_call();
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "null cache");
  if (mode == KVQ_EVICT_MIDDLE) {
    if (c->cfg.layout == KVQ_LAYOUT_RING) return KVQ_OK;   // the ring already holds the survivors
    if (c->cfg.layout != KVQ_LAYOUT_COMPACT)
      return fail(KVQ_ERR_INVALID_ARG, "middle eviction needs a COMPACT or RING layout");
    cudaError_t e = kvq::launch_evict_middle(c->view, stream);
    return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_evict");
  }
  if (mode == KVQ_EVICT_KEEPSET) {
    if (!keep_idx) return fail(KVQ_ERR_INVALID_ARG, "null keep_idx");
    if (n_keep < 1 || n_keep > c->cfg.capacity) return fail(KVQ_ERR_INVALID_ARG, "n_keep out of range");
    if (c->cfg.layout == KVQ_LAYOUT_RING) return fail(KVQ_ERR_UNSUPPORTED, "keep-sets apply to LINEAR or COMPACT caches");
    if (c->cfg.k_format == KVQ_FMT_KIVI_BLOCK)
      return fail(KVQ_ERR_UNSUPPORTED, "keep-sets do not apply to KIVI_BLOCK caches (closed blocks share K scales)");
    cudaError_t e = kvq::launch_evict_keepset(c->view, keep_idx, n_keep, stream);
    return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_evict");
  }
  return fail(KVQ_ERR_INVALID_ARG, "unknown evict mode %d", mode);
}

size_t kvq_decode_workspace_bytes(kvq_cache c, int32_t n_q_heads) {
  if (!c || n_q_heads < 1 || n_q_heads % c->cfg.n_kv_heads) return 0;
  const size_t G = n_q_heads / c->cfg.n_kv_heads;
  const DecodePlan p = decode_plan(c, (int)G);
  int ns = p.nsplit > p.nsplit_tc ? p.nsplit : p.nsplit_tc;
  if (c->cfg.k_format == KVQ_FMT_KIVI_BLOCK) ns += 1;   // the tail's partial
  if (ns == 1) return 0;
  return (size_t)c->cfg.batch * c->cfg.n_kv_heads * ns * G * (c->cfg.head_dim + kvq::kPartialPad) * sizeof(float);
}

kvq_status kvq_decode_plan_query(const kvq_config* cfg, int32_t n_q_heads, int32_t sms, int32_t* nsplit,
                                 int32_t* nsplit_tc, int32_t* wide) {
  begin_call();
  kvq_cache_layout lay;
  const kvq_status s = compute_layout(cfg, &lay);
  if (s != KVQ_OK) return s;
  if (n_q_heads < 1 || n_q_heads % cfg->n_kv_heads)
    return fail(KVQ_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
  if (sms < 1) return fail(KVQ_ERR_INVALID_ARG, "sms must be >= 1");
  if (!nsplit || !nsplit_tc || !wide) return fail(KVQ_ERR_INVALID_ARG, "null output");
  kvq_cache_s c{};   // only the configuration and the SM count enter the plan
  c.cfg = *cfg;
  c.sms = sms;
  const DecodePlan p = decode_plan(&c, n_q_heads / cfg->n_kv_heads);
  *nsplit = p.nsplit;
  *nsplit_tc = p.nsplit_tc;
  *wide = p.wide;
  return KVQ_OK;
}

}  // extern "C"

namespace {

// kvq_test_stall_decode_tiles: bytes every decode CTA's first tile barrier expects in excess.
std::atomic<unsigned> g_stall_tx{0};

// Argument checks shared by kvq_decode_attn and kvq_append_decode.
kvq_status check_decode_args(kvq_cache c, const void* q, void* out, int32_t n_q_heads, int32_t io_dtype,
                             void* workspace, size_t ws_bytes) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "null cache");
  if (!q || !out) return fail(KVQ_ERR_INVALID_ARG, "null q or out");
  if (!valid_dtype(io_dtype)) return fail(KVQ_ERR_INVALID_ARG, "unknown io dtype %d", io_dtype);
  if (n_q_heads < 1 || n_q_heads % c->cfg.n_kv_heads)
    return fail(KVQ_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
  const int G = n_q_heads / c->cfg.n_kv_heads;
  if (G > 8) return fail(KVQ_ERR_UNSUPPORTED, "query heads per kv head must be <= 8 (got %d)", G);
  if (c->cfg.k_format == KVQ_FMT_KIVI_CHAN && !c->k_calibrated)
    return fail(KVQ_ERR_UNSUPPORTED, "per-channel K scales are not calibrated yet");
  const size_t need = kvq_decode_workspace_bytes(c, n_q_heads);
  if (need && (!workspace || ws_bytes < need))
    return fail(KVQ_ERR_CAPACITY, "decode workspace needs %zu bytes, got %zu", need, ws_bytes);
  if (need && ((uintptr_t)workspace & 15)) return fail(KVQ_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  return KVQ_OK;
}

// One decode launch; k_new != null asks the tensor-core kernel to code the
// new token first (cudaErrorNotSupported, with nothing launched, where that
// kernel does not serve the cache and io dtype).
cudaError_t launch_decode_any(kvq_cache c, const void* q, void* out, int32_t n_q_heads, int32_t io_dtype,
                              float softmax_scale, void* workspace, const void* k_new, const void* v_new,
                              int32_t in_dtype, bool early, cudaStream_t stream) {
  const int G = n_q_heads / c->cfg.n_kv_heads;
  const size_t need = kvq_decode_workspace_bytes(c, n_q_heads);
  if (!(softmax_scale > 0.0f)) softmax_scale = 1.0f / sqrtf((float)c->cfg.head_dim);
  kvq::DecodeArgs a;
  a.q = q;
  a.out = out;
  a.io_dtype = io_dtype;
  a.Hq = n_q_heads;
  a.qscale = softmax_scale * 1.4426950408889634f;
  const DecodePlan plan = decode_plan(c, G);
  a.nsplit = plan.nsplit;
  a.nsplit_tc = plan.nsplit_tc;
  a.wide = plan.wide;
  a.partials = need ? static_cast<float*>(workspace) : nullptr;
  a.k_new = k_new;
  a.v_new = v_new;
  a.in_dtype = in_dtype;
  a.stall_tx = g_stall_tx.load(std::memory_order_relaxed);
  a.early = early ? 1 : 0;
  const int kf = fmt_code(c->cfg.k_format, c->cfg.k_bits);
  const int vf = fmt_code(c->cfg.v_format, c->cfg.v_bits);
  using namespace kvq;
  if (kf == F_KIVIB8 && vf == F_AFF8) return k_new ? cudaErrorNotSupported : launch_decode<F_KIVIB8, F_AFF8>(c->view, G, a, stream);
  if (kf == F_KIVIB4 && vf == F_AFF4) return k_new ? cudaErrorNotSupported : launch_decode<F_KIVIB4, F_AFF4>(c->view, G, a, stream);
  if (kf == F_FP16 && vf == F_FP16) return launch_decode<F_FP16, F_FP16>(c->view, G, a, stream);
  if (kf == F_KIVI8 && vf == F_AFF8) return launch_decode<F_KIVI8, F_AFF8>(c->view, G, a, stream);
  if (kf == F_KIVI4 && vf == F_AFF4) return launch_decode<F_KIVI4, F_AFF4>(c->view, G, a, stream);
  if (kf == F_AFF8 && vf == F_AFF8) return launch_decode<F_AFF8, F_AFF8>(c->view, G, a, stream);
  if (kf == F_AFF4 && vf == F_AFF4) return launch_decode<F_AFF4, F_AFF4>(c->view, G, a, stream);
  if (kf == F_Q40 && vf == F_AFF8) return launch_decode<F_Q40, F_AFF8>(c->view, G, a, stream);
  if (kf == F_Q40 && vf == F_AFF4) return launch_decode<F_Q40, F_AFF4>(c->view, G, a, stream);
  return cudaErrorInvalidValue;
}

// Whether the (K format, V format) pair and, for KIVI_BLOCK keys, the
// head count have a decode kernel.
kvq_status check_decode_pair(kvq_cache c, int G, int32_t io_dtype) {
  using namespace kvq;
  const int kf = fmt_code(c->cfg.k_format, c->cfg.k_bits);
  const int vf = fmt_code(c->cfg.v_format, c->cfg.v_bits);
  if (kf == F_KIVIB8 || kf == F_KIVIB4) {
    if (G > 4 && (io_dtype == KVQ_DTYPE_F32 || c->cfg.head_dim == 32 || !c->view.has_maps))
      return fail(KVQ_ERR_UNSUPPORTED, "KIVI_BLOCK decode on the fp32 CUDA-core path takes up to 4 query heads per kv head");
    if (!((kf == F_KIVIB8 && vf == F_AFF8) || (kf == F_KIVIB4 && vf == F_AFF4)))
      return fail(KVQ_ERR_UNSUPPORTED, "KIVI_BLOCK decode is built for 8-bit keys with 8-bit values and 4 with 4");
    return KVQ_OK;
  }
  const bool built = (kf == F_FP16 && vf == F_FP16) || (kf == F_KIVI8 && vf == F_AFF8) ||
                     (kf == F_KIVI4 && vf == F_AFF4) || (kf == F_AFF8 && vf == F_AFF8) ||
                     (kf == F_AFF4 && vf == F_AFF4) || (kf == F_Q40 && vf == F_AFF8) || (kf == F_Q40 && vf == F_AFF4);
  if (!built) return fail(KVQ_ERR_UNSUPPORTED, "decode for this (K format, V format) pair is not built");
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_decode_attn(kvq_cache c, const void* q, void* out, int32_t n_q_heads, int32_t io_dtype,
                           float softmax_scale, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  begin_call();
  kvq_status st = check_decode_args(c, q, out, n_q_heads, io_dtype, workspace, ws_bytes);
  if (st != KVQ_OK) return st;
  st = check_decode_pair(c, n_q_heads / c->cfg.n_kv_heads, io_dtype);
  if (st != KVQ_OK) return st;
  const cudaError_t e = launch_decode_any(c, q, out, n_q_heads, io_dtype, softmax_scale, workspace, nullptr, nullptr,
                                          0, false, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_decode_attn");
}

namespace {

// One layer's step of kvq_append_decode (the counters of the call are the caller's).
kvq_status append_decode_one(kvq_cache c, const void* k, const void* v, int32_t in_dtype, const void* q, void* out,
                             int32_t n_q_heads, int32_t io_dtype, float softmax_scale, void* workspace,
                             size_t ws_bytes, int32_t flags, cudaStream_t stream) {
  kvq_status st = check_decode_args(c, q, out, n_q_heads, io_dtype, workspace, ws_bytes);
  if (st != KVQ_OK) return st;
  st = check_decode_pair(c, n_q_heads / c->cfg.n_kv_heads, io_dtype);
  if (st != KVQ_OK) return st;
  if (!k || !v) return fail(KVQ_ERR_INVALID_ARG, "null k or v");
  if (!valid_dtype(in_dtype)) return fail(KVQ_ERR_INVALID_ARG, "unknown input dtype %d", in_dtype);
  if (flags & ~KVQ_STEP_EARLY_READ) return fail(KVQ_ERR_INVALID_ARG, "unknown step flags 0x%x", flags);
  const bool early = (flags & KVQ_STEP_EARLY_READ) != 0;
  // one launch: the tensor-core kernel codes the token and attends
  if (c->cfg.layout != KVQ_LAYOUT_COMPACT) {
    const cudaError_t e = launch_decode_any(c, q, out, n_q_heads, io_dtype, softmax_scale, workspace, k, v,
                                            in_dtype, early, stream);
    if (e == cudaSuccess) return KVQ_OK;
    if (e != cudaErrorNotSupported) return cuda_fail(e, "kvq_append_decode");
  }
  // otherwise the three steps in turn: append, StreamingLLM eviction of a
  // compact cache, decode
  st = append_rows(c, k, v, 1, 1, in_dtype, 0, stream, "kvq_append_decode");
  if (st != KVQ_OK) return st;
  if (c->cfg.layout == KVQ_LAYOUT_COMPACT) {
    const cudaError_t e = kvq::launch_evict_middle(c->view, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvq_append_decode");
  }
  const cudaError_t e = launch_decode_any(c, q, out, n_q_heads, io_dtype, softmax_scale, workspace, nullptr, nullptr,
                                          0, false, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_append_decode");
}

}  // namespace

kvq_status kvq_append_decode(kvq_cache c, const void* k, const void* v, int32_t in_dtype, const void* q, void* out,
                             int32_t n_q_heads, int32_t io_dtype, float softmax_scale, void* workspace,
                             size_t ws_bytes, int32_t flags, cudaStream_t stream) {
  begin_call();
  return append_decode_one(c, k, v, in_dtype, q, out, n_q_heads, io_dtype, softmax_scale, workspace, ws_bytes, flags,
                           stream);
}

kvq_status kvq_append_decode_layers(int32_t n_layers, const kvq_cache* caches, const void* const* k,
                                    const void* const* v, int32_t in_dtype, const void* const* q, void* const* out,
                                    int32_t n_q_heads, int32_t io_dtype, float softmax_scale,
                                    void* const* workspace, const size_t* ws_bytes, int32_t flags,
                                    cudaStream_t stream) {
  begin_call();
  if (n_layers < 1) return fail(KVQ_ERR_INVALID_ARG, "n_layers must be >= 1");
  if (!caches || !k || !v || !q || !out) return fail(KVQ_ERR_INVALID_ARG, "null per-layer array");
  if (flags & ~KVQ_STEP_EARLY_READ) return fail(KVQ_ERR_INVALID_ARG, "unknown step flags 0x%x", flags);
  // layers after the first read their caches early (their predecessor on the
  // stream is the previous layer's step, which writes only its own cache):
  // that needs distinct caches
  for (int32_t i = 0; i < n_layers; ++i)
    for (int32_t j = 0; j < i; ++j)
      if (caches[i] == caches[j]) return fail(KVQ_ERR_INVALID_ARG, "layers %d and %d share one cache", j, i);
  for (int32_t l = 0; l < n_layers; ++l) {
    const kvq_status st =
        append_decode_one(caches[l], k[l], v[l], in_dtype, q[l], out[l], n_q_heads, io_dtype, softmax_scale,
                          workspace ? workspace[l] : nullptr, ws_bytes ? ws_bytes[l] : 0,
                          l == 0 ? flags : (flags | KVQ_STEP_EARLY_READ), stream);
    if (st != KVQ_OK) {
      char msg[256];
      snprintf(msg, sizeof(msg), "layer %d: %s", l, kvq_last_error());
      return fail(st, "%s", msg);
    }
  }
  return KVQ_OK;
}

void kvq_test_stall_decode_tiles(int32_t on) { g_stall_tx.store(on ? 16u : 0u, std::memory_order_relaxed); }

size_t snapkv_workspace_bytes(int32_t batch, int32_t n_kv_heads, int32_t S, int32_t head_dim, int32_t obs_window) {
  (void)head_dim;
  (void)obs_window;
  if (batch < 1 || n_kv_heads < 1 || S < 1) return 0;
  const size_t BH = (size_t)batch * n_kv_heads;
  const size_t nchunk = (S + kvq::kSnapChunk - 1) / kvq::kSnapChunk;
  // row statistics, scores (when the caller passes none), arrival counts and a failure flag
  return align_up(BH * nchunk * 64 * sizeof(float2), 256) + align_up(BH * (size_t)S * sizeof(float), 256) +
         align_up((BH + 1) * sizeof(unsigned), 256);
}

kvq_status snapkv_select(const void* k, int64_t head_stride, int32_t batch, int32_t n_kv_heads, int32_t S,
                         int32_t head_dim, int32_t obs_window, int32_t budget, int32_t n_sink, float* scores_out,
                         int32_t* idx_out, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  begin_call();
  if (!k || !idx_out) return fail(KVQ_ERR_INVALID_ARG, "null k or idx_out");
  if (batch < 1 || n_kv_heads < 1 || S < 1) return fail(KVQ_ERR_INVALID_ARG, "batch, n_kv_heads, S must be >= 1");
  if (head_dim != 32 && head_dim != 64 && head_dim != 128)
    return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d not supported (32, 64, 128)", head_dim);
  if (head_stride < S) return fail(KVQ_ERR_INVALID_ARG, "head_stride must be >= S");
  if (obs_window < 1 || obs_window > 64) return fail(KVQ_ERR_UNSUPPORTED, "obs_window must be in 1..64");
  if (budget < 1 || n_sink < 0) return fail(KVQ_ERR_INVALID_ARG, "budget >= 1 and n_sink >= 0 required");
  if (n_sink > budget) return fail(KVQ_ERR_INVALID_ARG, "n_sink must not exceed budget");
  if (((uintptr_t)k & 7) != 0) return fail(KVQ_ERR_INVALID_ARG, "k must be 8-byte aligned");
  const size_t need = snapkv_workspace_bytes(batch, n_kv_heads, S, head_dim, obs_window);
  if (!workspace || ws_bytes < need)
    return fail(KVQ_ERR_CAPACITY, "snapkv workspace needs %zu bytes, got %zu", need, ws_bytes);
  if ((uintptr_t)workspace & 255) return fail(KVQ_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const size_t BH = (size_t)batch * n_kv_heads;
  const int nchunk = (S + kvq::kSnapChunk - 1) / kvq::kSnapChunk;
  float2* stats = static_cast<float2*>(workspace);
  const size_t off_scores = align_up(BH * nchunk * 64 * sizeof(float2), 256);
  const size_t off_arrive = off_scores + align_up(BH * (size_t)S * sizeof(float), 256);
  float* scores = scores_out;
  if (!scores) scores = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + off_scores);
  unsigned* arrive = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(workspace) + off_arrive);
  const int w = obs_window < S ? obs_window : S;
  cudaError_t e = kvq::launch_snapkv(k, head_stride, batch, n_kv_heads, S, head_dim, w, budget, n_sink, scores,
                                     idx_out, stats, nchunk, arrive, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "snapkv_select");
}

kvq_status snapkv_pool(const float* scores, float* pooled, int32_t batch, int32_t n_kv_heads, int32_t S,
                       int32_t kernel_size, cudaStream_t stream) {
  begin_call();
  if (!scores || !pooled) return fail(KVQ_ERR_INVALID_ARG, "null scores or pooled");
  if (batch < 1 || n_kv_heads < 1 || S < 1) return fail(KVQ_ERR_INVALID_ARG, "batch, n_kv_heads, S must be >= 1");
  if (kernel_size < 1 || kernel_size % 2 == 0 || kernel_size > 63)
    return fail(KVQ_ERR_INVALID_ARG, "kernel_size must be odd, 1..63 (got %d)", kernel_size);
  const size_t n = (size_t)batch * n_kv_heads * S;
  if (scores < pooled + n && pooled < scores + n) return fail(KVQ_ERR_INVALID_ARG, "scores and pooled overlap");
  const cudaError_t e = kvq::launch_snapkv_pool(scores, pooled, batch * n_kv_heads, S, kernel_size, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "snapkv_pool");
}

kvq_status snapkv_topk(const float* scores, int32_t batch, int32_t n_kv_heads, int32_t S, int32_t budget,
                       int32_t n_sink, int32_t* idx_out, cudaStream_t stream) {
  begin_call();
  if (!scores || !idx_out) return fail(KVQ_ERR_INVALID_ARG, "null scores or idx_out");
  if (batch < 1 || n_kv_heads < 1 || S < 1) return fail(KVQ_ERR_INVALID_ARG, "batch, n_kv_heads, S must be >= 1");
  if (budget < 1 || n_sink < 0) return fail(KVQ_ERR_INVALID_ARG, "budget >= 1 and n_sink >= 0 required");
  if (n_sink > budget) return fail(KVQ_ERR_INVALID_ARG, "n_sink must not exceed budget");
  cudaError_t e = kvq::launch_topk(scores, batch, n_kv_heads, S, budget, n_sink, idx_out, nullptr, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "snapkv_topk");
}

kvq_status kvq_stats_read(kvq_cache c, kvq_stats* out) {
  begin_call();
  if (!c || !out) return fail(KVQ_ERR_INVALID_ARG, "null cache or stats");
  kvq::DevState st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&st, c->view.state, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "kvq_stats_read");
  out->pos = st.pos;
  out->stored = st.stored;
  out->capacity = c->cfg.capacity;
  out->device_status = st.status;
  out->k_calibrated = st.k_calibrated;
  out->cache_bytes = c->lay.total_bytes;
  out->live_bytes = live_bytes(c, st.stored);
  out->tail = c->cfg.k_format == KVQ_FMT_KIVI_BLOCK ? st.tail : 0;
  if (out->tail) out->live_bytes += (size_t)c->cfg.batch * c->cfg.n_kv_heads * out->tail * c->cfg.head_dim * 8;
  return st.status ? fail(KVQ_ERR_DEVICE, "device status %d", st.status) : KVQ_OK;
}

kvq_status kvq_clear_status(kvq_cache c, cudaStream_t stream) {
  begin_call();
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "null cache");
  // the status word, and the decode merge's per-(b, kv head) arrival counters
  // (which a launch that stopped early could have left short of their reset)
  cudaError_t e = cudaMemsetAsync(&c->view.state->status, 0, sizeof(int), stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(c->view.split_sem, 0, (size_t)c->cfg.batch * c->cfg.n_kv_heads * sizeof(unsigned), stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_clear_status");
}

}  // extern "C"
