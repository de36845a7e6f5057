/*
 * kvq.h -- C ABI of the GB300 compressed KV cache for single-token LLM decode.
 *
 * The library quantises keys and values into a low-bit cache as they are
 * appended, evicts tokens (StreamingLLM sink + window, SnapKV keep-sets),
 * and runs grouped-query decode attention that reads the packed codes
 * directly.  It also scores and selects SnapKV keep-sets from a prompt's keys.
 *
 * Sources, cited by page title and section:
 *   [SLK]  "StreamingLLM + KIVI -- long-context decode without growing the KV
 *          cache" (tinygpt docs)
 *   [SKV]  "SnapKV -- Prefill Observation-Window Token Eviction"
 *          (veloxquant-mlx docs)
 *   [KMC]  "kv-cache: optional per-channel K-cache mean-centering for Q4_0"
 *          (llama.cpp PR #51)
 *   [MLX]  "Low-bit KV caches on MLX: what exists and what is missing"
 *
 * Conventions shared by every call
 *   - Pointers marked "device" must point to memory of the current CUDA
 *     device; pointers marked "host" to host memory.  The caller owns and
 *     allocates all device memory (cache buffer, workspaces); the library
 *     allocates none.  A kvq_cache handle is a small host-side object created
 *     by kvq_cache_init and freed by kvq_cache_release.
 *   - Calls that take a cudaStream_t are asynchronous and stream-ordered:
 *     they validate their host-side arguments, enqueue kernels and return.
 *     A host-side validation failure returns an error before anything is
 *     enqueued.  NULL means the legacy default stream.
 *   - The cache's counters (absolute position, stored rows) live in device
 *     memory and are advanced by the kernels, so a captured CUDA graph of
 *     append / evict / decode replays correctly.  Conditions only the device
 *     can see (capacity overflow, a malformed keep-set) set a device status
 *     word instead of trapping; kvq_stats_read reports it.
 *   - Tensors are dense and row-major with the last dimension contiguous.
 *     B = batch, Hkv = kv heads, Hq = query heads (a multiple of Hkv),
 *     D = head_dim, n = tokens in a call, S = prompt length.  Query head h
 *     attends with kv head h / (Hq / Hkv).
 *   - No call throws; errors are returned as kvq_status with a message
 *     available from kvq_last_error() on the calling thread.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_ABI_VERSION 2

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,   /* bad shape, pointer, size or mode                       */
  KVQ_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement, or a
                                K bias with non-Q4_0 keys ([KMC] "What's included":
                                the bias is gated to Q4_0 K caches, a mismatch fails) */
  KVQ_ERR_CAPACITY = 3,      /* buffer or workspace too small                          */
  KVQ_ERR_DEVICE = 4,        /* the device status word reports an error                */
  KVQ_ERR_CUDA = 5           /* a CUDA runtime call failed                             */
} kvq_status;

/* Storage format of one side (K or V) of the cache. */
typedef enum kvq_format {
  /* raw fp16 rows, 2 bytes per element ([SKV] "How it works": kept rows stay fp16) */
  KVQ_FMT_FP16 = 0,
  /* KIVI keys: asymmetric, one (scale, zero) per (b, kv head, channel) shared by all
     tokens, computed once from the tokens of a calibrating append and then frozen
     ([SLK] "KIVI", "Affine quantisation formula").  bits 8 or 4.  K side only.   */
  KVQ_FMT_KIVI_CHAN = 1,
  /* asymmetric, one (scale, zero) per (b, kv head, token, group of `group`
     consecutive channels): KIVI values with group = D ([SLK] "KIVI"), mlx-lm's
     QuantizedKVCache with group = 64 ([MLX] section 1).  bits 8 or 4; group a
     multiple of 16 dividing D.                                                      */
  KVQ_FMT_AFFINE_TOKEN = 2,
  /* symmetric blocks of 32 channels, one fp16 scale each, no zero point.  [KMC]
     "The idea" calls Q4_0 a symmetric block quantiser without a zero point; the
     32-channel block and its fp16 scale are the Q4_0 layout, which the page does
     not spell out.  bits 4, group 32.  K side only; the only format that accepts
     a K bias.                                                                       */
  KVQ_FMT_Q4_0 = 3,
  /* KIVI residual buffer ([MLX] section 3, "What KIVI and KVQuant found"): the most
     recent tokens stay at full precision (fp32) in a tail of fewer than `group` = R
     rows; each time R tokens have gathered, that closed block's keys are coded per
     (b, kv head, channel) with the block's own asymmetric scale and zero (the KIVI
     formula over exactly those R tokens) and its values per token with the V
     format, the codes go to the next R rows of the quantised bulk and the tail
     empties.  Decode attends over the bulk and then the exact tail.  K side only;
     bits 8 or 4; R a multiple of 64 (64 or 128); needs an AFFINE_TOKEN V side and
     the LINEAR layout.                                                              */
  KVQ_FMT_KIVI_BLOCK = 4
} kvq_format;

typedef enum kvq_layout {
  KVQ_LAYOUT_LINEAR = 0,   /* rows appended in order; no middle eviction (SnapKV, plain) */
  KVQ_LAYOUT_COMPACT = 1,  /* sink + window, evicted rows removed by moving the window down
                              ([SLK] "Implementation": concatenate [0, sink) and
                              [len - window, len))                                       */
  KVQ_LAYOUT_RING = 2      /* sink + window; position p >= sink lives in slot
                              sink + (p - sink) mod window, nothing moves                 */
} kvq_layout;

typedef enum kvq_dtype { KVQ_DTYPE_F32 = 0, KVQ_DTYPE_BF16 = 1, KVQ_DTYPE_F16 = 2 } kvq_dtype;

typedef enum kvq_evict_mode {
  KVQ_EVICT_MIDDLE = 0,    /* StreamingLLM: drop logical [sink, len - window) */
  KVQ_EVICT_KEEPSET = 1    /* SnapKV: keep an ascending index set per (b, kv head) */
} kvq_evict_mode;

/* kvq_append flags */
#define KVQ_APPEND_CALIBRATE_K 1   /* KIVI_CHAN keys: compute and freeze the per-channel
                                      scales from this call's tokens before coding them */
#define KVQ_APPEND_RECOMPUTE_K 2   /* KIVI_CHAN keys, LINEAR / COMPACT layouts ([SLK] "KIVI",
                                      "Caveats": the range is recomputed on every append):
                                      dequantise the stored keys in fp32 from the stored fp16
                                      scale and zero (u * s, then + z), take each channel's
                                      range over them and the new keys, code every stored key
                                      again and the new ones with the new scale / zero.
                                      O(stored * D) per call; excludes CALIBRATE_K. */

/* kvq_append_decode flags */
#define KVQ_STEP_EARLY_READ 1      /* the kernel just before the call writes neither this
                                      cache nor its counters (see kvq_append_decode) */

/* Device status codes (kvq_stats.device_status). */
#define KVQ_DEV_OK 0
#define KVQ_DEV_OVERFLOW 1         /* an append would pass the capacity; nothing was written */
#define KVQ_DEV_BAD_KEEPSET 2      /* keep-set not strictly ascending or beyond stored rows */
#define KVQ_DEV_TIMEOUT 3          /* a bounded wait inside a kernel ran out; outputs of that call
                                      are unspecified */

typedef struct kvq_config {
  int32_t batch;        /* B >= 1 */
  int32_t n_kv_heads;   /* Hkv >= 1 */
  int32_t head_dim;     /* D in {32, 64, 128} */
  int32_t capacity;     /* rows per (b, kv head); COMPACT needs >= sink + window + the
                           largest append, RING uses exactly sink + window */
  int32_t layout;       /* kvq_layout */
  int32_t sink;         /* StreamingLLM sink tokens (COMPACT / RING) */
  int32_t window;       /* StreamingLLM window tokens (COMPACT / RING), >= 1 */
  int32_t k_format, k_bits, k_group;   /* kvq_format, 16/8/4, channels per group */
  int32_t v_format, v_bits, v_group;   /* FP16 or AFFINE_TOKEN */
  /* device fp32 [Hkv, D] per-(kv head, channel) mean subtracted from K right before it
     is quantised ([KMC] "Summary"); NULL disables centering.  Copied into the cache
     buffer by kvq_cache_init.  Only legal with KVQ_FMT_Q4_0 keys. */
  const float* k_bias;
} kvq_config;

/* Byte offsets of the planes inside the caller's cache buffer (0 = absent).  Every
   offset is a multiple of 256.  cap_alloc = capacity rounded up to 64 rows.
     state              device counters and status (256 bytes)
     split_sem          uint32 [B*Hkv] arrival counters of decode splits
     {k,v}_codes        uint8  [B][Hkv][cap_alloc][row_bytes]: fp16 bytes, or the
                        signed 8-bit level q = u - 128, or 4-bit codes with channel
                        2j in the low nibble of byte j
     {k,v}_tok_scale    fp16   [B][Hkv][cap_alloc][n_groups] (AFFINE_TOKEN, Q4_0)
     {k,v}_tok_zero     fp16   [B][Hkv][cap_alloc][n_groups] (AFFINE_TOKEN)
     k_ch_scale/zero    fp16   [B][Hkv][D]  stored per-channel metadata (KIVI_CHAN)
     k_ch_scale32/zero32 fp32  [B][Hkv][D]  the values codes are computed from
     k_bias             fp32   [Hkv][D]     copy of kvq_config.k_bias
     k_blk_scale/zero   fp16   [B][Hkv][cap_alloc / R][D]  per-block, per-channel K
                        metadata (KIVI_BLOCK)
     {k,v}_tail         fp32   [B][Hkv][R][D]  the full-precision tail (KIVI_BLOCK)  */
typedef struct kvq_cache_layout {
  size_t total_bytes;
  int32_t cap_alloc;
  int32_t k_row_bytes, v_row_bytes;
  int32_t k_n_groups, v_n_groups;
  size_t state, split_sem;
  size_t k_codes, k_tok_scale, k_tok_zero, k_ch_scale, k_ch_zero, k_ch_scale32, k_ch_zero32, k_bias;
  size_t v_codes, v_tok_scale, v_tok_zero;
  size_t k_blk_scale, k_blk_zero, k_tail, v_tail;
} kvq_cache_layout;

typedef struct kvq_stats {
  int64_t pos;            /* absolute position of the next token (tokens ever appended;
                             SnapKV's true offset, [SKV] "RoPE position semantics") */
  int32_t stored;         /* rows currently held ([SLK] "Caveats": stored vs current length) */
  int32_t capacity;
  int32_t device_status;  /* KVQ_DEV_* */
  int32_t k_calibrated;   /* KIVI_CHAN: per-channel scales frozen */
  size_t cache_bytes;     /* size of the cache buffer */
  size_t live_bytes;      /* bytes of codes + metadata of the stored rows (and, for
                             KIVI_BLOCK, of the full-precision tail) */
  int32_t tail;           /* KIVI_BLOCK: tokens in the full-precision tail (stored counts
                             the quantised bulk only); 0 otherwise */
} kvq_stats;

typedef struct kvq_cache_s* kvq_cache;

/* Computes the plane layout for `cfg` (no device work).  Returns INVALID_ARG or
   UNSUPPORTED for configurations the library rejects, among them caches of
   2^31 - 64 rows or more (batch * n_kv_heads * capacity, with capacity rounded
   up to a multiple of 64): the decode kernels address each code plane with a
   signed 32-bit row coordinate. */
kvq_status kvq_cache_layout_query(const kvq_config* cfg, kvq_cache_layout* out);

/* Creates a cache over the caller's device buffer `dev_mem` of `bytes` bytes
   (>= layout.total_bytes, 256-byte aligned).  Zeroes the counters and copies the
   K bias on `stream`.  `*out` receives a host handle; the buffer must outlive it. */
kvq_status kvq_cache_init(const kvq_config* cfg, void* dev_mem, size_t bytes, cudaStream_t stream,
                          kvq_cache* out);

/* Frees the host handle (not the device buffer). */
void kvq_cache_release(kvq_cache cache);

/* Quantise-on-append ([SLK] "Implementation": after each per-layer append;
   [KMC] "Why this is safe": the bias costs a single subtraction when K is
   written).
   k, v: device [B, Hkv, n, D] of `in_dtype` (kvq_dtype).  Tokens take absolute
   positions pos .. pos + n - 1.  LINEAR / COMPACT write rows stored .. stored + n - 1
   (device overflow -> KVQ_DEV_OVERFLOW, nothing written); RING writes each
   surviving token into its slot and leaves stored = min(pos + n, sink + window).
   flags: KVQ_APPEND_CALIBRATE_K computes the KIVI per-channel K scales from these
   n tokens and freezes them (required once before any other append to a
   KIVI_CHAN cache; UNSUPPORTED otherwise).  Codes use fp32 scales
   scale = max(1e-5, (max - min) / (qMax - qMin)), zero = min, and
   u = clamp(rint((x - zero) / scale), 0, qMax - qMin) ([SLK] "Affine quantisation
   formula"); Q4_0 uses d = max|x - kbar| / 7, u = clamp(rint((x - kbar) / d), -8, 7) + 8
   (u = 8 when d == 0).  Stored scales and zeros are fp16.
   KIVI_BLOCK keys ([MLX] section 3): the tail (t rows) followed by the n new tokens
   is taken in order; each complete run of R is a closed block, coded (keys per
   channel over its R tokens, values per token) into bulk rows stored .. stored + R - 1,
   and the rest becomes the tail; the split into calls does not change the result.
   Device overflow of the bulk -> KVQ_DEV_OVERFLOW, nothing written; flags must be 0.
   Speed only: outside KIVI_BLOCK caches, appends of 32 or more tokens whose k
   and v start on 16-byte boundaries are staged through shared memory by bulk
   copies; other appends read the rows directly.  Both give the same bytes. */
kvq_status kvq_append(kvq_cache cache, const void* k, const void* v, int32_t n_tokens, int32_t in_dtype,
                      int32_t flags, cudaStream_t stream);

/* Bulk quantise-on-convert ([MLX] section 1: an existing full-precision cache is
   turned into a quantised one in one pass once the context is long enough).
   k, v: a dense cache the caller already holds, device f32 / bf16 / fp16 by
   in_dtype, token t of (b, kv head) at row (b*Hkv + h)*head_stride + t, rows of D
   elements (head_stride >= n_tokens: a dense cache with spare capacity).  The
   first n_tokens tokens of every (b, kv head) are coded exactly as kvq_append
   would code the same tokens given contiguously (same flags, same counters);
   the source is only read.  head_stride < n_tokens -> INVALID_ARG; other errors as
   kvq_append. */
kvq_status kvq_convert(kvq_cache cache, const void* k, const void* v, int64_t head_stride, int32_t n_tokens,
                       int32_t in_dtype, int32_t flags, cudaStream_t stream);

/* KVQ_EVICT_MIDDLE ([SLK] "Implementation"): when stored > sink + window, drop
   logical [sink, stored - window).  COMPACT moves the window rows (codes and
   per-token metadata) down; RING needs no data movement and enqueues nothing;
   LINEAR returns INVALID_ARG.  Per-channel K metadata is never touched.
   KVQ_EVICT_KEEPSET ([SKV] "How it works", step 4): keep_idx device int32
   [B, Hkv, n_keep], strictly ascending per (b, kv head), each < stored; row
   keep_idx[b,h,j] moves to row j, stored becomes n_keep, pos is unchanged (the
   true offset).  Done in place, in increasing row order. */
kvq_status kvq_evict(kvq_cache cache, int32_t mode, const int32_t* keep_idx, int32_t n_keep,
                     cudaStream_t stream);

/* Workspace bytes kvq_decode_attn needs for this cache and n_q_heads (0 when
   the call needs none).  Depends on the cache's capacity and the SM count. */
size_t kvq_decode_workspace_bytes(kvq_cache cache, int32_t n_q_heads);

/* The launch plan kvq_decode_attn uses for a cache of configuration `cfg` with
   n_q_heads query heads on a GPU of `sms` SMs (no device work; for tests and
   tuning).  *nsplit: splits per (b, kv head) sized from the capacity (about
   eight CTAs per SM in all, at least 64 rows per split, 256 from 4096 rows on,
   at most 128); the CUDA-core kernel (fp32 io, head_dim 32) uses it.
   *nsplit_tc: the tensor-core kernel's splits; *wide: 1 when that grid runs
   eight-warp CTAs in a single wave (two per SM, one for over four query heads
   per kv head) with *nsplit_tc == *nsplit; 2 when that single wave instead
   runs one sixteen-warp CTA per SM, *nsplit_tc = SMs / (B * Hkv) splits (one
   fewer for KIVI_BLOCK keys, whose tail takes one more CTA), chosen for up
   to four query heads per kv head when every split keeps at least four
   64-row tiles of the capacity and there are at least two; 0 when it runs
   smaller CTAs (four warps, four per SM; eight warps, two per SM, for over
   four query heads per kv head) over as many splits as fill two whole waves
   without starting a third.  The kernels spread the rows actually stored
   over at most that many splits.  Configuration errors as kvq_cache_layout_query; a bad n_q_heads or
   sms, or a null output, is INVALID_ARG. */
kvq_status kvq_decode_plan_query(const kvq_config* cfg, int32_t n_q_heads, int32_t sms, int32_t* nsplit,
                                 int32_t* nsplit_tc, int32_t* wide);

/* Fused decode attention over the stored rows, reading the packed codes and
   dequantising in registers ([MLX] section 5: decode reads the cache; [SLK]
   "Affine quantisation formula": attention over the dequantised K, V).
   q: device [B, Hq, D]; out: device [B, Hq, D]; both of io_dtype.
   o[b,h] = softmax(q . k_hat^T * softmax_scale) v_hat, k_hat/v_hat from the stored
   codes and fp16 metadata; softmax_scale <= 0 means 1/sqrt(D).  The rows are
   split across CTAs and merged with the online-softmax rule.  workspace: device,
   >= kvq_decode_workspace_bytes bytes (may be NULL when that is 0).  Calls on the
   same cache must not overlap on the GPU.  KIVI_BLOCK caches attend over the
   quantised bulk and then the exact fp32 tail ([MLX] section 3), with one more
   CTA per (b, kv head) for the tail.  Hq / Hkv from 1 to 8 on the tensor-core
   path (16-bit io, head_dim 64 / 128), 1 to 4 on the CUDA-core path (fp32 io,
   head_dim 32). */
kvq_status kvq_decode_attn(kvq_cache cache, const void* q, void* out, int32_t n_q_heads, int32_t io_dtype,
                           float softmax_scale, void* workspace, size_t ws_bytes, cudaStream_t stream);

/* One decode step of one layer in one call ([SLK] "Implementation": per layer
   and step, append the token, evict, then attend): the effect of kvq_append of
   one token (k, v: device [B, Hkv, 1, D] of in_dtype, no flags), then
   kvq_evict(KVQ_EVICT_MIDDLE) for COMPACT and RING caches, then
   kvq_decode_attn (arguments, workspace and errors as that call), so the
   attention sees the new token.  LINEAR and RING caches served by the
   tensor-core decode with head_dim 128 (16-bit io, not KIVI_BLOCK keys) whose
   decode grid is a single wave (kvq_decode_plan_query's *wide >= 1) do it in
   one launch: the CTA holding the last stored rows codes the token into its
   slot (bit-identical to kvq_append) and adds it to the attention from the
   dequantised row, a full ring leaves the slot it overwrites out of the
   attention, and the counters advance as kvq_append would.  Every other cache
   runs the three steps as separate launches (in a grid of several waves the
   coding would hold back its CTA for longer than a separate launch costs).
   Device overflow of a LINEAR cache sets KVQ_DEV_OVERFLOW and attends over the
   rows already stored.  flags: 0 or KVQ_STEP_EARLY_READ, the caller's promise
   that the kernel just before this call on the stream writes neither this
   cache nor its counters (another layer's step, the projection that produced
   q, k and v): the one-launch step then reads the counters and requests the
   stored rows before that kernel has finished, and waits for it only for q,
   k and v.  Breaking the promise gives wrong results (not a fault). */
kvq_status kvq_append_decode(kvq_cache cache, const void* k, const void* v, int32_t in_dtype, const void* q,
                             void* out, int32_t n_q_heads, int32_t io_dtype, float softmax_scale, void* workspace,
                             size_t ws_bytes, int32_t flags, cudaStream_t stream);

/* One decode step of n_layers layers in one call: kvq_append_decode on caches[l]
   with k[l], v[l], q[l], out[l] (and workspace[l] / ws_bytes[l] when the arrays
   are given; NULL arrays mean no workspace for every layer), layer 0 first, all
   on `stream`.  Every argument keeps kvq_append_decode's meaning and layout; the
   arrays are host arrays of n_layers device pointers, read during the call only.
   flags apply to layer 0; every later layer runs as if KVQ_STEP_EARLY_READ were
   given, since the kernel just before it is the previous layer's step, which
   writes only the previous layer's cache, so the caches must be distinct
   (KVQ_ERR_INVALID_ARG otherwise, nothing enqueued).  Stops at the first layer
   whose step fails and returns its status, with the layer named in
   kvq_last_error(); the layers before it are enqueued.  This is the same step
   as the StreamingLLM + KIVI page's per-layer loop in "Implementation"
   (append, evict, attend, layer by layer), with one crossing of this boundary
   per step instead of one per layer. */
kvq_status kvq_append_decode_layers(int32_t n_layers, const kvq_cache* caches, const void* const* k,
                                    const void* const* v, int32_t in_dtype, const void* const* q, void* const* out,
                                    int32_t n_q_heads, int32_t io_dtype, float softmax_scale,
                                    void* const* workspace, const size_t* ws_bytes, int32_t flags,
                                    cudaStream_t stream);

/* Test hook for the failure path of the tensor-core decode: while on (0 off,
   the default; process-wide, read at each launch), every CTA of the following
   decode launches arms its first tile's barrier for 16 bytes more than the
   copies bring, so that its bounded wait runs out (after 200 ms), the launch
   sets KVQ_DEV_TIMEOUT and returns with the cache untouched; the GPU stays
   usable.  Nothing faults or traps. */
void kvq_test_stall_decode_tiles(int32_t on);

/* kvq_decode_attn for callers that cannot allocate device memory.  The pages
   have no counterpart of this call; it exists for this library's users.
   Some callers may not call cudaMalloc at all: code running inside an allocator
   or memory-pool callback, plugin hosts that forbid device allocations after
   start-up, loops that must never enter the driver's allocator.  This call
   takes the same cache, q and out as kvq_decode_attn but no workspace: the
   split-KV partials go to a fixed device array inside the library of
   kvq_noalloc_scratch_bytes() bytes (4 MiB), which every GPU that loads the
   library holds until the process exits.  A cache whose
   kvq_decode_workspace_bytes exceeds that returns KVQ_ERR_CAPACITY and enqueues
   nothing.  The first call on each device looks up the array's device address
   (cudaGetSymbolAddress, that device current), and so does the first call
   after that device's context was replaced (cudaDeviceReset); make those calls
   before any stream capture.  All calls on a device share the array and leave their last
   contents in it (nothing in it needs to start at zero): calls that overlap on
   the GPU race and give wrong results, so serialise them.  Allocates nothing. */
kvq_status kvq_decode_attn_noalloc(kvq_cache cache, const void* q, void* out, int32_t n_q_heads,
                                   int32_t io_dtype, float softmax_scale, cudaStream_t stream);

/* Size in bytes of the built-in scratch array kvq_decode_attn_noalloc uses. */
size_t kvq_noalloc_scratch_bytes(void);

/* Workspace bytes snapkv_select needs. */
size_t snapkv_workspace_bytes(int32_t batch, int32_t n_kv_heads, int32_t S, int32_t head_dim,
                              int32_t obs_window);

/* SnapKV observation-window scoring and selection ([SKV] "How it works", steps 1-3;
   "Evidence": window clamped to S, min(budget, S) indices, sorted, budget >= S
   keeps all).  k: device fp16, row (b, h, s) at k + ((b*Hkv + h)*head_stride + s)*D
   elements (head_stride >= S).  score[b,h,j] = mean over the last w = min(obs_window, S)
   rows r of softmax_j(k_r . k_j / sqrt(D)), no mask.  Kept: positions [0, min(n_sink, S))
   plus the top (budget - n_sink) of the rest by score (equal scores: lower position
   first), ascending.  scores_out: device fp32 [B, Hkv, S] or NULL; idx_out: device
   int32 [B, Hkv, min(budget, S)].  n_sink > budget -> INVALID_ARG.
   obs_window in 1..64, head_dim in {32, 64, 128}, S >= 1; k 8-byte aligned
   (INVALID_ARG otherwise).  When every scoring CTA fits on the device at once
   the scores come from one cooperative launch whose CTAs of a head wait for
   one another (bounded, ~200 ms); should that wait ever run out, every index
   of that call is -1.  Calls that overlap on the GPU must not share a
   workspace. */
kvq_status snapkv_select(const void* k, int64_t head_stride, int32_t batch, int32_t n_kv_heads, int32_t S,
                         int32_t head_dim, int32_t obs_window, int32_t budget, int32_t n_sink,
                         float* scores_out, int32_t* idx_out, void* workspace, size_t ws_bytes,
                         cudaStream_t stream);

/* Max-pool smoothing of SnapKV scores, the SnapKV paper's step that [SKV] "Proxy
   limitation" says the page leaves out: pooled[b,h,j] = max of scores[b,h,i] over
   i in [j - r, j + r] clipped to [0, S), r = kernel_size / 2.  scores, pooled: device
   fp32 [B, Hkv, S], not overlapping.  Compose snapkv_select (scores_out) ->
   snapkv_pool -> snapkv_topk to select on smoothed scores (sinks still forced).
   kernel_size odd in 1..63, else INVALID_ARG. */
kvq_status snapkv_pool(const float* scores, float* pooled, int32_t batch, int32_t n_kv_heads, int32_t S,
                       int32_t kernel_size, cudaStream_t stream);

/* The selection step of snapkv_select alone, on caller-given fp32 scores
   [B, Hkv, S] (device), with the same rule.  Needs no workspace. */
kvq_status snapkv_topk(const float* scores, int32_t batch, int32_t n_kv_heads, int32_t S, int32_t budget,
                       int32_t n_sink, int32_t* idx_out, cudaStream_t stream);

/* Synchronises the device, copies `cache`'s counters to the host and fills `*out`. */
kvq_status kvq_stats_read(kvq_cache cache, kvq_stats* out);

/* Clears the device status word and the decode merge's per-(b, kv head)
   arrival counters (stream-ordered).  After a KVQ_DEV_TIMEOUT the cache is
   usable again once this has run: the stored rows and counters are intact. */
kvq_status kvq_clear_status(kvq_cache cache, cudaStream_t stream);

/* Number of kernels the last call on this thread enqueued (for launch accounting). */
int32_t kvq_last_launch_count(void);

/* Message of the last error on the calling thread ("" if none). */
const char* kvq_last_error(void);

int32_t kvq_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
