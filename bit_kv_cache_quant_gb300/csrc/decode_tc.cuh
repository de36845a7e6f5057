// Decode attention on the tensor cores (mma.sync m16n8k16, fp16 operands, fp32
// accumulators) for head_dim 64 / 128 and bf16 / fp16 queries and outputs.
//
// Same split-KV partition and online-softmax merge as decode_kernel.  A CTA of
// eight warps streams its split in 64-token tiles that TMA copies into a ring
// of NSTAGE shared-memory stages; warps 0-3 take the even tiles and warps 4-7
// the odd ones, each warp 16 tokens of a tile.  There is no CTA-wide barrier
// in the loop: every warp waits on the stage's mbarrier itself, and the last of
// the four warps to finish a stage copies the tile NSTAGE ahead into it.
// Per warp and 16-token block, both contractions are taken transposed so that
// the 16 rows of the MMA are tokens (scores) or value channels (outputs) and
// the 8 columns hold four query heads as (fp16 part, residual) pairs:
//   S^T[16 x 8] = K[16 x D] . Q^T : the key codes as A, exact small integers
//     (Q4_0 as the signed levels u - 8); column 2j of Q^T holds fp16(q) of
//     head j, column 2j + 1 the residual q - fp16(q), so the score of head j
//     is the sum of the two columns and q enters exactly.  Keys with
//     per-token groups (affine, Q4_0) get one fp32 accumulator per 32-channel
//     block and are scaled afterwards, per scale group, s * sum(q u) +
//     z * sum(q) (Q4_0: d * sum(q (u - 8))), so the scores carry no fp16
//     rounding of the keys.  Per-channel KIVI scales are folded into q; their
//     zero term is a per-row constant the softmax does not see and is dropped.
//     Each thread then holds one head's scores for two tokens, and the
//     online-softmax state of that head.
//   O^T[16 x 8] += V^T[16 x 16] . P^T : the value block as A, the
//     probabilities (again fp16 part + residual columns) as B, moved into the
//     B layout with a warp transpose (movmatrix).  Values with several scale
//     groups per token are dequantised to fp16 in registers (one HFMA2 with
//     the token's fp16 scale and zero); values with one group per token enter
//     as exact integer codes, the token's scale multiplies its probability
//     and sum(p * zero) is accumulated apart in fp32 and added to every
//     channel.  The accumulator columns of a thread belong to the same head
//     as its scores, so the softmax rescale stays inside the thread.
// With up to four query heads per kv head one column tile does it; five to
// eight take two.
// Codes become fp16 through the mantissa of 1024.0 (see nibbles_to_h2).
#pragma once

#include <type_traits>

#include "decode_tc_frag.cuh"
#include "quantize_row.cuh"

namespace kvq {

// The fused append's new token, by one warp: codes the token of (b, kv head)
// bh into cache slot `slot` with the append's rules, scores the dequantised
// key against each head (fp32), and leaves the head's (score, 1, value row)
// in m_row, l_row and newv (channel d of the value row at word
// (d % VCH) * 8 + d / VCH, the per-warp accumulator layout).
template <int D, int G, int VCH>
__device__ __forceinline__ void append_new_token(const CacheView& c, const DecodeArgs& a, int b, int kvh, size_t bh,
                                              int slot, int lane, float* newv, float* m_row, float* l_row) {
  constexpr int E = D / 32;
  float xk[E], xv[E], hk[E], hv[E], qv[G][E];
  // every input first (the cache writes below would hold back later loads)
  const size_t ro = bh * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    xk[e] = load_io(a.k_new, ro + e, a.in_dtype);
    xv[e] = load_io(a.v_new, ro + e, a.in_dtype);
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const size_t qo = ((size_t)b * a.Hq + (size_t)kvh * G + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) qv[h][e] = load_io(a.q, qo + e, a.io_dtype);
  }
  quantize_row_dq<E, true>(c.k, c.k_bias ? c.k_bias + (size_t)kvh * D : nullptr, xk, bh, c.cap_alloc, slot, lane, hk);
  quantize_row_dq<E, true>(c.v, nullptr, xv, bh, c.cap_alloc, slot, lane, hv);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int d = lane * E + e;
    newv[(d % VCH) * 8 + d / VCH] = hv[e];
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float p = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) p = fmaf(qv[h][e], hk[e], p);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
    if (lane == 0) {
      m_row[h] = p * a.qscale;
      l_row[h] = 1.0f;
    }
  }
}

template <int ROWB, int NW>
__device__ __forceinline__ void lds_row_words(uint32_t (&w)[NW], const uint8_t* plane, int r, int off) {
  static_assert(NW == 1 || NW == 2 || NW % 4 == 0, "word count");
  if constexpr (NW == 1) {
    w[0] = *reinterpret_cast<const uint32_t*>(plane + swz_off<ROWB>(r, off));
  } else if constexpr (NW == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(plane + swz_off<ROWB>(r, off));
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < NW / 4; ++i) {
      const uint4 v = *reinterpret_cast<const uint4*>(plane + swz_off<ROWB>(r, off + 16 * i));
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  }
}

// O^T += V^T . P^T for one 16-token block.  A = the value codes of the
// thread's four tokens (words A, B, C, E: logical tokens 2t, 2t + 1, 2t + 8,
// 2t + 9), paired per channel as the A fragment wants them; m-tile mt covers
// this thread's value channels 2 mt (fragment row g) and 2 mt + 1 (row g + 8).
// B = the transposed probabilities pb.  Codes are
// dequantised to fp16 in registers with each token's scale and zero when DEQ,
// else taken as exact integers (the scale then sits in pb and the zero in a
// separate sum); 8-bit codes then enter as 1024 + u, the caller's zero sum
// carrying -1024 times the scale.
// The NW words are words mo / (m-tiles per word) onward of the thread's value
// bytes; they feed m-tiles mo onward.
template <int VB, int NW, int MT, bool DEQ>
__device__ __forceinline__ void pvt_mma(float (&oacc)[MT][4], const uint32_t (&pb)[2], int mo,
                                        const uint32_t (&A)[NW], const uint32_t (&B)[NW], const uint32_t (&C)[NW],
                                        const uint32_t (&E)[NW], __half2 sAB, __half2 zAB, __half2 sCD, __half2 zCD) {
  if constexpr (VB == 4) {
    static_assert(4 * NW <= MT, "m-tiles");
#pragma unroll
    for (int wi = 0; wi < NW; ++wi) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t sel = half ? 0x7632u : 0x5410u;
        __half2 h0[4], h1[4];
        nibbles_to_h2(__byte_perm(A[wi], B[wi], sel), h0);   // h0[i]: channel 8 wi + 4 half + i of tokens A, B
        nibbles_to_h2(__byte_perm(C[wi], E[wi], sel), h1);
        if constexpr (DEQ) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            h0[i] = __hfma2(h0[i], sAB, zAB);
            h1[i] = __hfma2(h1[i], sCD, zCD);
          }
        }
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const uint32_t va[4] = {h2u(h0[2 * pp]), h2u(h0[2 * pp + 1]), h2u(h1[2 * pp]), h2u(h1[2 * pp + 1])};
          mma_f16(oacc[mo + 4 * wi + 2 * half + pp], va, pb[0], pb[1]);
        }
      }
    }
  } else if constexpr (VB == 8) {
    static_assert(2 * NW <= MT, "m-tiles");
#pragma unroll
    for (int wi = 0; wi < NW; ++wi) {
      const uint32_t a_ = A[wi] ^ 0x80808080u, b_ = B[wi] ^ 0x80808080u;
      const uint32_t c_ = C[wi] ^ 0x80808080u, e_ = E[wi] ^ 0x80808080u;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t sel = half ? 0x7362u : 0x5140u;
        __half2 l0, h0, l1, h1;
        if constexpr (DEQ) {
          bytes_to_h2(__byte_perm(a_, b_, sel), l0, h0);       // channels 4 wi + 2 half + 0 / 1
          bytes_to_h2(__byte_perm(c_, e_, sel), l1, h1);
          l0 = __hfma2(l0, sAB, zAB); h0 = __hfma2(h0, sAB, zAB);
          l1 = __hfma2(l1, sCD, zCD); h1 = __hfma2(h1, sCD, zCD);
        } else {
          // 1024 + u: the offset leaves through the zero sum (see the vfold step)
          bytes_to_h2_1024(__byte_perm(a_, b_, sel), l0, h0);
          bytes_to_h2_1024(__byte_perm(c_, e_, sel), l1, h1);
        }
        const uint32_t va[4] = {h2u(l0), h2u(h0), h2u(l1), h2u(h1)};
        mma_f16(oacc[mo + 2 * wi + half], va, pb[0], pb[1]);
      }
    }
  } else {
    static_assert(NW <= MT, "m-tiles");
#pragma unroll
    for (int wi = 0; wi < NW; ++wi) {
      const uint32_t va[4] = {__byte_perm(A[wi], B[wi], 0x5410u), __byte_perm(A[wi], B[wi], 0x7632u),
                              __byte_perm(C[wi], E[wi], 0x5410u), __byte_perm(C[wi], E[wi], 0x7632u)};
      mma_f16(oacc[mo + wi], va, pb[0], pb[1]);
    }
  }
}

// A CTA has NGRP tile groups of HG head groups of four warps.  Tile group gp
// consumes tiles gp, gp + NGRP, ...; within it, head group j computes query
// heads 4 j .. 4 j + 3 over the same stages (HG = 2 for five to eight heads per
// kv head).  Four-warp CTAs (four per SM) suit grids of several waves;
// eight-warp tile pairs (two per SM) halve the time per split when the whole
// grid fits in one wave; sixteen-warp CTAs of four tile groups (one per SM)
// give a one-wave grid of few (b, kv head) units the most warps per tile.
template <int NGRP, int HG> struct TcShape {
  static constexpr int warps = 4 * NGRP * HG;
  static constexpr int threads = 32 * warps;
  static constexpr int ctas_per_sm = NGRP * HG == 1 ? kTcCtasPerSm : 4 / (NGRP * HG);
};

template <int G> struct TcHeads {
  static constexpr int hg = (G + 3) / 4;   // head groups
};

// Pipeline depth.  Four-warp CTAs (four per SM, several waves) use two
// stages: deeper rings measured slower on the 32K and ring workloads, whose
// time is instruction issue, not latency.  Larger CTAs (one wave) take as
// many stages (a multiple of NGRP, up to 8) as fit next to the static shared
// memory, so that a short split is requested in one go.
template <int D, int G, int KF, int VF, int NGRP> struct TcStages {
  // largest stage: key scale groups of 32 channels, value groups of D / 8
  static constexpr int kng_max = D / 32;
  static constexpr int vng_max = 8;
  static constexpr int stage = ((64 * D * FmtBits<KF>::v / 8 + 64 * D * FmtBits<VF>::v / 8 +
                                 ((KF == F_AFF8 || KF == F_AFF4) ? 2 : (KF == F_Q40 ? 1 : 0)) * 64 * kng_max * 2 +
                                 ((VF == F_AFF8 || VF == F_AFF4) ? 2 : 0) * 64 * vng_max * 2 +
                                 ((KF == F_KIVIB8 || KF == F_KIVIB4) ? 2 * D * 2 : 0)) +
                                1023) / 1024 * 1024;
  using Shape = TcShape<NGRP, TcHeads<G>::hg>;
  static constexpr int warps = Shape::warps;
  // per-warp (head, channel) accumulators, written over the stages after the loop
  static constexpr int acc_bytes = warps * G * (D + 8) * 4;
  static constexpr int static_smem =
      2 * kMaxSplits * G * 4 + 2 * (warps + 1) * G * 4 + (D + 8) * 4 + (D / 32) * 32 + 1024;
  static constexpr int budget = 227 * 1024 / Shape::ctas_per_sm - 2048 - static_smem;
  static constexpr int raw = (budget / stage) / NGRP * NGRP;
  static constexpr int cap = NGRP == 1 ? kTcStagesNarrow : 8;
  static constexpr int v = raw < 2 ? 2 : (raw > cap ? cap : raw);
  // dynamic shared memory for a stage size (+ 1 KB to align the ring to 1024)
  static constexpr int dyn_bytes(int stage_bytes) {
    return (v * stage_bytes > acc_bytes ? v * stage_bytes : acc_bytes) + 1024;
  }
};

// APP: the fused append of kvq_append_decode (a.k_new set); its own
// instantiation, so that the plain decode carries none of its code.
template <int D, int G, int KF, int VF, int NGRP, bool APP>
__global__ void __launch_bounds__(TcShape<NGRP, TcHeads<G>::hg>::threads, TcShape<NGRP, TcHeads<G>::hg>::ctas_per_sm)
    decode_tc_kernel(const __grid_constant__ CacheView c, DecodeArgs a) {
  constexpr int HG = TcHeads<G>::hg;
  constexpr int NSTAGE = TcStages<D, G, KF, VF, NGRP>::v;
  constexpr int NWARP = TcShape<NGRP, HG>::warps;
  constexpr int TW = 4 * HG;       // warps reading each tile
  constexpr int KB = FmtBits<KF>::v;
  constexpr int VB = FmtBits<VF>::v;
  constexpr int KROW = D * KB / 8;
  constexpr int VROW = D * VB / 8;
  constexpr int KS = D / 16;       // k-steps of K Q^T
  constexpr int NB = D / 32;       // 32-channel key blocks
  constexpr int MT = D / 16;       // 16-channel m-tiles of O^T
  constexpr int VCH = D / 8;       // value channels owned by thread g
  constexpr int VTB = VROW / 8;    // value bytes per token owned by thread g
  constexpr bool K_AFF = (KF == F_AFF8 || KF == F_AFF4);
  constexpr bool K_KIVI = (KF == F_KIVI8 || KF == F_KIVI4);
  constexpr bool K_Q40 = (KF == F_Q40);
  constexpr bool KG = K_AFF || K_Q40;
  constexpr bool V_AFF = (VF == F_AFF8 || VF == F_AFF4);
  constexpr bool K_KIVIB = (KF == F_KIVIB8 || KF == F_KIVIB4);
  constexpr int NACC = KG ? NB : 1;
  // tiles of the split requested into L2 before the dependency wait: the
  // whole initial ring of a one-wave grid, four tiles for a CTA of several
  // waves (whose later tiles would only crowd L2)
  constexpr int PF_TILES = NGRP == 1 ? 4 : NSTAGE;
  static_assert(G >= 1 && G <= 8, "up to 8 query heads per kv head");
  static_assert(!(APP && K_KIVIB), "the fused append does not code KIVI_BLOCK keys");
  static_assert(NSTAGE % NGRP == 0, "each stage serves one tile group");

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // per-warp (max, sum) of each head; with APP, slot NWARP: the new token
  // (or nothing)
  __shared__ float sm_m[NWARP + APP][G];
  __shared__ float sm_l[NWARP + APP][G];
  __shared__ float sm_newv[APP ? D + 8 : 1];   // the new token's dequantised value row (merge slot NWARP)
  __shared__ __align__(8) uint64_t mbar[NSTAGE];
  __shared__ __align__(8) uint64_t mbar_meta;   // metadata of the initial ring (one use)
  __shared__ int s_ninit;                       // tiles of the initial ring
  __shared__ unsigned s_done[NSTAGE];     // warps done with a stage, over all its tiles (TW per tile)
  __shared__ int s_last_tile[NSTAGE];     // last tile copied into a stage, -1 if none
  __shared__ int s_T;
  __shared__ long long s_pos;             // fused append: absolute position of the new token
  __shared__ volatile int s_fail;
  __shared__ float sm_qsum[NB][8];        // sum of q of each head over each 32-channel key block
  // KIVI_BLOCK keys: the query in fp32 (the fragments are folded with each
  // block's channel scales as the tiles reach a new block) and the tail length
  __shared__ float sm_qraw[K_KIVIB ? G : 1][K_KIVIB ? D : 1];
  __shared__ int s_tail;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
  const size_t bh = (size_t)b * c.Hkv + kvh;
  const int kng = c.k.n_groups;
  const int vng = c.v.n_groups;
  // plane-major ring for the one-wave shapes, stage-major for four-warp CTAs
  using Ring = TcRing<D, KF, VF, NSTAGE, (NGRP > 1)>;
  static_assert(Ring::bytes <= NSTAGE * TcStages<D, G, KF, VF, NGRP>::stage, "the ring fits its stages");
  const Ring R(kng, vng);

  // Before the grids this launch depends on have finished (programmatic
  // dependent launch), touch only what they cannot change: the tensor maps
  // and this CTA's barriers.  Besides, request into L2 the first rows of the
  // split this CTA would read if the stored length were what the counter
  // holds now.  That read races with a producer still running, so it is only
  // a hint: the rows are clamped to this (b, kv head)'s allocation, and a
  // prefetch into L2 (the point of coherence) never serves stale data.
  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(&c.kmap) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(&c.vmap) : "memory");
    if (!K_KIVIB && !a.early) {   // (an early launch requests the rows themselves)
      const int Th = min(max(*reinterpret_cast<volatile const int*>(&c.state->stored), 0), c.cap_alloc);
      int h0, h1, hn;
      split_rows(Th, a.nsplit, split, h0, h1, hn);
      if (split < hn && h1 > h0) {
        // whole tiles (every plane offset of a 64-row boundary is 16-byte
        // aligned), at most PF_TILES of them
        const int r1 = min(min((h1 + kTileTokens - 1) / kTileTokens * kTileTokens, c.cap_alloc),
                           h0 + PF_TILES * kTileTokens);
        const size_t row0 = bh * c.cap_alloc + h0;
        const uint32_t nr = (uint32_t)(r1 - h0);
        prefetch_l2_bulk(c.k.codes + row0 * KROW, nr * KROW);
        prefetch_l2_bulk(c.v.codes + row0 * VROW, nr * VROW);
        if constexpr (KG) prefetch_l2_bulk(c.k.tok_scale + row0 * c.k.n_groups, nr * 2 * c.k.n_groups);
        if constexpr (K_AFF) prefetch_l2_bulk(c.k.tok_zero + row0 * c.k.n_groups, nr * 2 * c.k.n_groups);
        if constexpr (V_AFF) {
          prefetch_l2_bulk(c.v.tok_scale + row0 * c.v.n_groups, nr * 2 * c.v.n_groups);
          prefetch_l2_bulk(c.v.tok_zero + row0 * c.v.n_groups, nr * 2 * c.v.n_groups);
        }
      }
    }
    // the query rows of this kv head, and a fused append's new key and value
    // rows (the producer may still write them, so they are only requested
    // into L2)
    {
      const int es = a.io_dtype == KVQ_DTYPE_F32 ? 4 : 2;
      const uint8_t* q0 = reinterpret_cast<const uint8_t*>(a.q) + ((size_t)b * a.Hq + (size_t)kvh * G) * D * es;
      for (int off = 0; off < G * D * es; off += 128) prefetch_l2(q0 + off);
      if constexpr (APP) {
        const int ei = a.in_dtype == KVQ_DTYPE_F32 ? 4 : 2;
        for (int off = 0; off < D * ei; off += 128) {
          prefetch_l2(reinterpret_cast<const uint8_t*>(a.k_new) + bh * D * ei + off);
          prefetch_l2(reinterpret_cast<const uint8_t*>(a.v_new) + bh * D * ei + off);
        }
      }
    }
    s_fail = 0;
    s_ninit = 0;
    if constexpr (APP) {
#pragma unroll
      for (int h = 0; h < G; ++h) {   // merge slot NWARP stays empty unless this CTA appends
        sm_m[NWARP][h] = neg_inf();
        sm_l[NWARP][h] = 0.0f;
      }
    }
    mbar_init(&mbar_meta, 1);
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&mbar[s], 1);
      s_done[s] = 0u;
      s_last_tile[s] = -1;
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    fence_async_smem();   // the initialised barriers are visible to the copy engine
  }
  // Warp 0 reads the stored length and requests the whole initial ring of
  // tiles: lane s the code planes of stage s, lane NSTAGE the metadata of
  // all of them (one copy per plane; every copy request costs the issuing
  // SM's copy engine time, so a ring of many small copies arrives late),
  // while the other warps build their query fragments.
  auto issue_ring = [&]() {
    int T0 = 0;
    if (lane == 0) {
      T0 = c.state->stored;
      s_T = T0;
      if constexpr (APP) s_pos = c.state->pos;
      if constexpr (K_KIVIB) s_tail = c.state->tail;
    }
    T0 = __shfl_sync(0xffffffffu, T0, 0);
    int a0, a1, ns0;
    split_rows(T0, a.nsplit, split, a0, a1, ns0);
    if (split < ns0) {
      const int nt0 = min((a1 - a0 + kTileTokens - 1) / kTileTokens, NSTAGE);
      __syncwarp();   // lane 0's barrier initialisation is visible to the warp
      if (lane < nt0) {
        const int r0 = a0 + lane * kTileTokens;
        const uint32_t stall = lane == 0 ? a.stall_tx : 0u;
        if constexpr (NGRP > 1) {
          mbar_expect_tx(&mbar[lane], (uint32_t)R.tx_codes + stall);
          issue_codes<D, KF, VF>(smem, R, lane, c, bh, r0, &mbar[lane]);
        } else {
          mbar_expect_tx(&mbar[lane], (uint32_t)(R.tx_codes + R.tx_meta) + stall);
          issue_codes<D, KF, VF>(smem, R, lane, c, bh, r0, &mbar[lane]);
          if (R.tx_meta > 0) issue_meta(smem, R, lane, 1, c, bh, r0, &mbar[lane]);
        }
        s_last_tile[lane] = lane;
      } else if (NGRP > 1 && lane == NSTAGE && R.tx_meta > 0) {
        mbar_expect_tx(&mbar_meta, (uint32_t)(nt0 * R.tx_meta));
        issue_meta(smem, R, 0, nt0, c, bh, a0, &mbar_meta);
      }
      if (lane == 0) s_ninit = nt0;
    }
  };
  // With a.early the caller guarantees that the kernel before this launch
  // writes neither this cache nor its counters, so the counters and the
  // stored rows are read before the dependency wait: the whole initial ring
  // then lands while that kernel finishes.  Only the query (and a fused
  // append's new token) wait for it.
  if (a.early && warp == 0) issue_ring();
  grid_dependency_wait();
  // Once every CTA of this grid has passed this point (or exited), the next
  // launch may start its own prologue (and L2 requests) while this one runs.
  grid_launch_dependents();
  if (!a.early && warp == 0) issue_ring();
  // Warp roles: 16-row block of each tile, head group, tile group.
  const int blk = (warp & 3) * 16;
  const int hg = (warp >> 2) % HG;
  const int grp = (warp >> 2) / HG;
  const int hd = 4 * hg + t;   // the query head whose scores and outputs this thread holds
  // Column 2j + e of the warp's Q^T holds head 4 hg + j: e = 0 its fp16(q),
  // e = 1 the residual q - fp16(q), so that head's score is the sum of the two
  // columns and q enters exactly.  Thread (g, t) builds column g at the key
  // channels of its fragment slots.
  uint32_t qf[KS][2];
  {
    const int hq = 4 * hg + (g >> 1);
    const bool live = hq < G;
    const size_t qo = ((size_t)b * a.Hq + (size_t)kvh * G + (live ? hq : 0)) * D;
    // the thread's query values at its fragment channels (key_channels), in
    // 16-byte (4-bit keys) or 8-byte loads when the row is 16-byte aligned
    float xq[KS][4];
    load_query_channels<D, KB>(a.q, qo, a.io_dtype, t, live, xq);
    float qb[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) qb[i] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      int ch[4];
      key_channels<KB>(ks, t, ch);
      float x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v = xq[ks][i];
        if constexpr (K_KIVI) v *= __half2float(c.k.ch_scale[bh * D + ch[i]]);
        x[i] = v;
      }
      if constexpr (K_AFF) qb[ks >> 1] += (x[0] + x[1]) + (x[2] + x[3]);
      const __half2 h01 = __floats2half2_rn(x[0], x[1]);
      const __half2 h23 = __floats2half2_rn(x[2], x[3]);
      qf[ks][0] = h2u(h01);
      qf[ks][1] = h2u(h23);
      if (g & 1) {
        const float2 f01 = __half22float2(h01);
        const float2 f23 = __half22float2(h23);
        qf[ks][0] = h2u(__floats2half2_rn(x[0] - f01.x, x[1] - f01.y));
        qf[ks][1] = h2u(__floats2half2_rn(x[2] - f23.x, x[3] - f23.y));
      }
    }
    if constexpr (K_AFF) {
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        qb[i] += __shfl_xor_sync(0xffffffffu, qb[i], 1);
        qb[i] += __shfl_xor_sync(0xffffffffu, qb[i], 2);
      }
      if ((warp & 3) == 0 && grp == 0 && t == 0 && !(g & 1) && live) {
#pragma unroll
        for (int i = 0; i < NB; ++i) sm_qsum[i][hq] = qb[i];
      }
    }
  }
  if constexpr (K_KIVIB) {
    for (int i = threadIdx.x; i < G * D; i += blockDim.x)
      sm_qraw[i / D][i % D] = load_io(a.q, ((size_t)b * a.Hq + (size_t)kvh * G + i / D) * D + i % D, a.io_dtype);
  }
  __syncthreads();
  const int T = s_T;
  int t0, t1, nse;
  split_rows(T, a.nsplit, split, t0, t1, nse);
  // Fused append ("StreamingLLM + KIVI", "Implementation": per layer and
  // step, append the token, evict, attend): the splits attend over the T rows
  // stored before this step, and the last live split's CTA codes the new
  // token into its slot and adds it to the merge as one more state.  A full
  // ring overwrites the slot of the oldest window token, which the splits
  // therefore leave out (excl).  The counters advance as kvq_append would,
  // once every CTA has read them (merge_store's step arrival).
  int excl = -1, slot = 0;
  bool app_cta = false;
  StepUpdate step{};
  if constexpr (APP) {
    const long long p = s_pos;
    const bool ring = c.layout == KVQ_LAYOUT_RING;
    step.on = true;
    step.ok = ring || (long long)T + 1 <= c.cap;
    step.pos = p + 1;
    const long long w = (long long)c.sink + c.window;
    step.stored = ring ? (int)(p + 1 < w ? p + 1 : w) : T + 1;
    if (ring) {
      slot = p < c.sink ? (int)p : c.sink + (int)((p - c.sink) % c.window);
      if (T >= c.sink + c.window) excl = slot;
    } else {
      slot = T;
    }
    app_cta = step.ok && split == nse - 1;
  }
  // KIVI_BLOCK: CTA a.nsplit attends over the fp32 tail and merges as one
  // more split (partial slot nse, after the bulk's); a cache with no closed
  // block has no bulk splits.
  int nse_all = nse, TT = 0;
  bool is_tail = false;
  if constexpr (K_KIVIB) {
    TT = s_tail;
    is_tail = split == a.nsplit;
    if (T == 0) nse = TT > 0 ? 0 : 1;
    nse_all = nse + (TT > 0 ? 1 : 0);
  }
  // no rows for this CTA (no copy was issued); in a fused step it still
  // arrives at the merge, which counts every CTA of its (b, kv head)
  if (!APP && (is_tail ? TT == 0 : split >= nse)) return;
  const int ntiles = is_tail ? 0 : (t1 - t0 + kTileTokens - 1) / kTileTokens;

  const int vgi = V_AFF ? (g * VCH) / c.v.group : 0;

  // Values with one (scale, zero) per token: the scale multiplies the
  // probability instead of every code and the zero term is summed apart.
  const bool vfold = V_AFF && vng == 1;
  float m_run = neg_inf();
  float l_part = 0.0f;
  float zacc = 0.0f;   // sum of p * zero over this thread's tokens (vfold)
  float oacc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.0f;
  // Sum of q of head hd over each key scale group (affine keys); padding
  // heads take a live head's sums (their outputs are dropped).
  float qg[NB];
  if constexpr (K_AFF) {
    const int h = min(hd, G - 1);
#pragma unroll
    for (int i = 0; i < NB; ++i) qg[i] = sm_qsum[i][h];
    if (2 * kng == NB) {
#pragma unroll
      for (int j = 0; j < NB / 2; ++j) qg[j] = qg[2 * j] + qg[2 * j + 1];
    } else if constexpr (NB == 4) {
      if (kng != NB) qg[0] = (qg[0] + qg[1]) + (qg[2] + qg[3]);
    }
  }

  // Tile rows of the two tokens whose scores this thread holds (logical g and
  // g + 8) and of the four tokens its value fragments read (2t, 2t + 1,
  // 2t + 8, 2t + 9).
  const int rk[2] = {blk + tau<VROW>(g), blk + tau<VROW>(g + 8)};
  const int rr[4] = {blk + tau<VROW>(2 * t), blk + tau<VROW>(2 * t + 1), blk + tau<VROW>(2 * t + 8),
                     blk + tau<VROW>(2 * t + 9)};
  // KIVI_BLOCK keys: k = s u + z with a (scale, zero) per (block, channel), so
  // the score is sum((q s) u) + sum(q z); the fragments hold q s of the block
  // of the warp's current tile and zt = sum(q z) of head hd.
  int cur_blk = -1;
  float zt = 0.0f;

  // The fused append's token, coded while the first tiles are in flight.
  if constexpr (APP) {
    if (app_cta && warp == NWARP - 1)
      append_new_token<D, G, VCH>(c, a, b, kvh, bh, slot, lane, sm_newv, sm_m[NWARP], sm_l[NWARP]);
  }
  const int ninit = s_ninit;
  // the plane-major initial ring's metadata has landed (seen by this warp)
  bool meta_in = NGRP == 1 || R.tx_meta == 0;
  for (int it = grp; it < ntiles; it += NGRP) {
    const int stg = it % NSTAGE;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&mbar[stg], (it / NSTAGE) & 1))) {
      s_fail = 1;
      break;
    }
    if (it < ninit && !meta_in) {
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&mbar_meta, 0))) {
        s_fail = 1;
        break;
      }
      meta_in = true;
    }
    // this stage's planes; the metadata planes are indexed by ring row
    const uint8_t* kst = smem + R.kc(stg);
    const uint8_t* vst = smem + R.vc(stg);
    const int tok0 = t0 + it * kTileTokens + blk;
    if constexpr (K_KIVIB) {
      const int bk = (t0 + it * kTileTokens) / c.k.group;
      if (bk != cur_blk && tok0 < t1) {   // warp-uniform
        cur_blk = bk;
        const __half* bs = reinterpret_cast<const __half*>(smem + R.kbs(stg));
        const __half* bz = reinterpret_cast<const __half*>(smem + R.kbz(stg));
        const int hq = 4 * hg + (g >> 1);
        const float* qr = sm_qraw[hq < G ? hq : 0];
        const bool live = hq < G;
        float zp = 0.0f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          int ch[4];
          key_channels<KB>(ks, t, ch);
          float x[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float q = live ? qr[ch[i]] : 0.0f;
            zp = fmaf(q, __half2float(bz[ch[i]]), zp);
            x[i] = q * __half2float(bs[ch[i]]);
          }
          const __half2 h01 = __floats2half2_rn(x[0], x[1]);
          const __half2 h23 = __floats2half2_rn(x[2], x[3]);
          qf[ks][0] = h2u(h01);
          qf[ks][1] = h2u(h23);
          if (g & 1) {
            const float2 f01 = __half22float2(h01);
            const float2 f23 = __half22float2(h23);
            qf[ks][0] = h2u(__floats2half2_rn(x[0] - f01.x, x[1] - f01.y));
            qf[ks][1] = h2u(__floats2half2_rn(x[2] - f23.x, x[3] - f23.y));
          }
        }
        // quad g holds head 4 hg + g / 2 (both of its columns carry the same sum)
        zp += __shfl_xor_sync(0xffffffffu, zp, 1);
        zp += __shfl_xor_sync(0xffffffffu, zp, 2);
        zt = __shfl_sync(0xffffffffu, zp, 8 * t);
      }
    }
    // Blocks wholly inside the split skip the row masks; the last block of
    // the split (rows past its end) and a block holding the excluded ring
    // slot take them.
    auto block = [&](auto masked) {
      constexpr bool MASK = decltype(masked)::value;
      // ------------------------------------------------------ S^T = K Q^T
      // acc[.][2e + j]: token rk[e], column 2j (j = 0: fp16 part, 1: residual)
      float acc[NACC][4];
#pragma unroll
      for (int i = 0; i < NACC; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
      const uint8_t* kpl = kst;
      if constexpr (KB == 4) {
#pragma unroll
        for (int p = 0; p < NB; ++p) {
          __half2 h0[4], h1[4];
          nibbles_to_h2<K_Q40 ? 8 : 0>(*reinterpret_cast<const uint32_t*>(kpl + swz_off<KROW>(rk[0], 16 * p + 4 * t)), h0);
          nibbles_to_h2<K_Q40 ? 8 : 0>(*reinterpret_cast<const uint32_t*>(kpl + swz_off<KROW>(rk[1], 16 * p + 4 * t)), h1);
          const uint32_t ka0[4] = {h2u(h0[0]), h2u(h1[0]), h2u(h0[2]), h2u(h1[2])};
          const uint32_t ka1[4] = {h2u(h0[1]), h2u(h1[1]), h2u(h0[3]), h2u(h1[3])};
          mma_f16(acc[KG ? p : 0], ka0, qf[2 * p][0], qf[2 * p][1]);
          mma_f16(acc[KG ? p : 0], ka1, qf[2 * p + 1][0], qf[2 * p + 1][1]);
        }
      } else if constexpr (KB == 8) {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          __half2 l0, h0, l1, h1;
          bytes_to_h2(*reinterpret_cast<const uint32_t*>(kpl + swz_off<KROW>(rk[0], 16 * ks + 4 * t)) ^ 0x80808080u,
                      l0, h0);
          bytes_to_h2(*reinterpret_cast<const uint32_t*>(kpl + swz_off<KROW>(rk[1], 16 * ks + 4 * t)) ^ 0x80808080u,
                      l1, h1);
          const uint32_t ka[4] = {h2u(l0), h2u(l1), h2u(h0), h2u(h1)};
          mma_f16(acc[KG ? (ks >> 1) : 0], ka, qf[ks][0], qf[ks][1]);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint2 v0 = *reinterpret_cast<const uint2*>(kpl + swz_off<KROW>(rk[0], 32 * ks + 8 * t));
          const uint2 v1 = *reinterpret_cast<const uint2*>(kpl + swz_off<KROW>(rk[1], 32 * ks + 8 * t));
          const uint32_t ka[4] = {v0.x, v1.x, v0.y, v1.y};
          mma_f16(acc[0], ka, qf[ks][0], qf[ks][1]);
        }
      }
      bool vk[2];
      float sc[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        vk[e] = !MASK || (tok0 - blk + rk[e] < t1 && (!APP || tok0 - blk + rk[e] != excl));
        float v = 0.0f;
        if constexpr (K_Q40) {
          // codes entered as signed levels u - 8: the score is sum over blocks of d * sum(q (u - 8))
          float d[NB], x[NB];
          load_halves<NB>(smem + R.ks(stg) + rk[e] * (2 * NB), d);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) x[nb] = acc[nb][2 * e] + acc[nb][2 * e + 1];
          v = fmaf(d[1], x[1], d[0] * x[0]);
          if constexpr (NB == 4) v += fmaf(d[3], x[3], d[2] * x[2]);
        } else if constexpr (K_AFF) {
          // s * sum(q u) + z * sum(q) per scale group of 32, 64 or 128 channels
          float x[NB];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) x[nb] = acc[nb][2 * e] + acc[nb][2 * e + 1];
          const uint8_t* srow = smem + R.ks(stg) + rk[e] * (2 * kng);
          const uint8_t* zrow = smem + R.kz(stg) + rk[e] * (2 * kng);
          if (kng == NB) {
            float sg[NB], zg[NB];
            load_halves<NB>(srow, sg);
            load_halves<NB>(zrow, zg);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) v = fmaf(sg[nb], x[nb], fmaf(zg[nb], qg[nb], v));
          } else if (2 * kng == NB) {
            float sg[NB / 2], zg[NB / 2];
            load_halves<NB / 2>(srow, sg);
            load_halves<NB / 2>(zrow, zg);
#pragma unroll
            for (int j = 0; j < NB / 2; ++j) v = fmaf(sg[j], x[2 * j] + x[2 * j + 1], fmaf(zg[j], qg[j], v));
          } else if constexpr (NB == 4) {
            float sg[1], zg[1];
            load_halves<1>(srow, sg);
            load_halves<1>(zrow, zg);
            v = fmaf(sg[0], (x[0] + x[1]) + (x[2] + x[3]), zg[0] * qg[0]);
          }
        } else {
          v = acc[0][2 * e] + acc[0][2 * e + 1];
          if constexpr (K_KIVIB) v += zt;
        }
        sc[e] = vk[e] ? v * a.qscale : neg_inf();
      }

      // ------------------------------------------------- online softmax (log2)
      // The block's 16 tokens of head hd sit in the eight threads of quad
      // position t.
      // The block's scores are weighed against the running max; only when one
      // of them exceeds it (one vote for the warp's four heads) is the block
      // max reduced and the state rescaled, which gives the same result as
      // doing so every block.
      float mb = fmaxf(sc[0], sc[1]);
      if (__any_sync(0xffffffffu, mb > m_run)) {
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
        const float mn = fmaxf(m_run, mb);               // finite: row tok0 is valid
        if (mn > m_run) {
          const float alpha = fast_exp2(m_run - mn);
          l_part *= alpha;
          zacc *= alpha;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            oacc[mt][0] *= alpha; oacc[mt][1] *= alpha; oacc[mt][2] *= alpha; oacc[mt][3] *= alpha;
          }
          m_run = mn;
        }
      }
      float p[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[e] = fast_exp2(sc[e] - m_run);
        l_part += p[e];
      }
      // Rows past the split's end were copied as whatever the buffer holds
      // (the excluded slot, as whatever the fused append was writing): their
      // weight is 0, and their value scale / zero (or fp16 values) are zeroed
      // so that no NaN reaches the MMA.
      bool vok[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) vok[i] = !MASK || (tok0 - blk + rr[i] < t1 && (!APP || tok0 - blk + rr[i] != excl));
      __half2 sAB = u2h(0u), zAB = u2h(0u), sCD = u2h(0u), zCD = u2h(0u);
      if constexpr (V_AFF) {
        const __half* vs = reinterpret_cast<const __half*>(smem + R.vs(stg));
        const __half* vz = reinterpret_cast<const __half*>(smem + R.vz(stg));
        if (vfold) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float si = vk[e] ? __half2float(vs[rk[e]]) : 0.0f;
            float zi = vk[e] ? __half2float(vz[rk[e]]) : 0.0f;
            if constexpr (VB == 8) zi = fmaf(-1024.0f, si, zi);   // 8-bit codes enter as 1024 + u
            zacc = fmaf(p[e], zi, zacc);
            p[e] *= si;
          }
        } else {
          const __half h0 = __ushort_as_half(0);
          sAB = __halves2half2(vok[0] ? vs[rr[0] * vng + vgi] : h0, vok[1] ? vs[rr[1] * vng + vgi] : h0);
          zAB = __halves2half2(vok[0] ? vz[rr[0] * vng + vgi] : h0, vok[1] ? vz[rr[1] * vng + vgi] : h0);
          sCD = __halves2half2(vok[2] ? vs[rr[2] * vng + vgi] : h0, vok[3] ? vs[rr[3] * vng + vgi] : h0);
          zCD = __halves2half2(vok[2] ? vz[rr[2] * vng + vgi] : h0, vok[3] ? vz[rr[3] * vng + vgi] : h0);
        }
      }
      // ---------------------------------------------------- O^T += V^T P^T
      // P^T as the B operand: the thread holds (fp16 part, residual) of head
      // hd for tokens g and g + 8, the accumulator layout of the 16 x 8 matrix
      // P^T; one transpose per 8-row half gives the fragment layout.
      uint32_t pb[2];
      {
        const __half2 ph = __floats2half2_rn(p[0], p[1]);
        const float2 pf = __half22float2(ph);
        const __half2 pl = __floats2half2_rn(p[0] - pf.x, p[1] - pf.y);
        pb[0] = movmatrix_t(h2u(__lows2half2(ph, pl)));
        pb[1] = movmatrix_t(h2u(__highs2half2(ph, pl)));
      }
      // The thread's value bytes of its four tokens, in chunks of at most 16
      // bytes per token.
      constexpr int NWT = VTB / 4;
      constexpr int NW = NWT > 4 ? 4 : NWT;
      const uint8_t* vpl = vst;
#pragma unroll
      for (int w0 = 0; w0 < NWT; w0 += NW) {
        // keep the next chunk's loads behind this one's MMAs (register pressure)
        if (w0 > 0) asm volatile("" ::: "memory");
        uint32_t A[NW], B[NW], C[NW], E[NW];
        lds_row_words<VROW, NW>(A, vpl, rr[0], g * VTB + 4 * w0);
        lds_row_words<VROW, NW>(B, vpl, rr[1], g * VTB + 4 * w0);
        lds_row_words<VROW, NW>(C, vpl, rr[2], g * VTB + 4 * w0);
        lds_row_words<VROW, NW>(E, vpl, rr[3], g * VTB + 4 * w0);
        if constexpr (VB == 16) {
          if (MASK) {   // only the split's last block
#pragma unroll
            for (int w = 0; w < NW; ++w) {
              A[w] = vok[0] ? A[w] : 0u;
              B[w] = vok[1] ? B[w] : 0u;
              C[w] = vok[2] ? C[w] : 0u;
              E[w] = vok[3] ? E[w] : 0u;
            }
          }
        }
        const int mo = w0 * (MT / NWT);
        if (V_AFF && !vfold)
          pvt_mma<VB, NW, MT, true>(oacc, pb, mo, A, B, C, E, sAB, zAB, sCD, zCD);
        else
          pvt_mma<VB, NW, MT, false>(oacc, pb, mo, A, B, C, E, sAB, zAB, sCD, zCD);
      }
    };
    if (tok0 + 16 <= t1 && (!APP || (unsigned)(excl - tok0) >= 16u)) block(std::false_type{});
    else if (tok0 < t1) block(std::true_type{});   // warp-uniform
    // Release the stage.  The tile group's last warp to finish it copies the
    // tile NSTAGE ahead into it (the warp barrier, the acquire-release count
    // and the proxy fence order every warp's reads of the stage before the
    // copy engine's writes).  A warp whose wait ran out stops; the others' waits
    // then run out in turn.
    __syncwarp();
    if (lane == 0) {
      if ((atom_add_acq_rel_cta(&s_done[stg], 1u) % TW) == TW - 1) {
        const int nx = it + NSTAGE;
        if (nx < ntiles) {
          fence_async_smem();
          mbar_expect_tx(&mbar[stg], (uint32_t)(R.tx_codes + R.tx_meta));
          issue_codes<D, KF, VF>(smem, R, stg, c, bh, t0 + nx * kTileTokens, &mbar[stg]);
          if (R.tx_meta > 0) issue_meta(smem, R, stg, 1, c, bh, t0 + nx * kTileTokens, &mbar[stg]);
          s_last_tile[stg] = nx;
        }
      }
    }
  }
  // The fused append's new token: the appending CTA's last warp codes it
  // into its slot with the append's rules, then scores the dequantised key
  // against each head (fp32) and leaves the head's (score, 1, value row)
  // as merge slot NWARP.
  __syncthreads();
  // A stage never arrived: report it and wait (bounded) for the copies still
  // in flight into this CTA's shared memory.  The CTA still takes part in the
  // split merge with empty states (the status word marks the outputs as
  // invalid), so that the merge counter of its (b, kv head) returns to zero.
  const bool failed = s_fail != 0;
  if (failed) {
    if (threadIdx.x == 0) {
      set_status(c.state, KVQ_DEV_TIMEOUT);
      for (int s = 0; s < NSTAGE; ++s)
        if (s_last_tile[s] >= 0) mbar_wait_bounded(&mbar[s], (s_last_tile[s] / NSTAGE) & 1);
      if (NGRP > 1 && s_ninit > 0 && R.tx_meta > 0) mbar_wait_bounded(&mbar_meta, 0);
    }
    __syncthreads();
  }

  // Per-warp results to shared memory, over the stage ring (every copy has
  // landed and been read).  Thread (g, t) holds head hd at its value channels
  // d = g * VCH + 2 mt + e, stored at (d % VCH) * 8 + d / VCH.
  float(*sm_acc)[G][D + 8] = reinterpret_cast<float(*)[G][D + 8]>(smem);
  if (is_tail) {
    if constexpr (K_KIVIB) {
      // The fp32 tail rows [0, TT): the head group's 4 NGRP warps take rows in
      // turn, each for the group's heads, lane l for channels [l C, l C + C).
      // A warp loads U of its rows before using any, so that the tail costs
      // about TT / (4 NGRP U) memory round trips rather than one per row; the
      // rows are still folded in one at a time, in order.
      constexpr int C = D / 32;
      constexpr int U = 8;
      constexpr int RS = 4 * NGRP;   // row stride between a warp's rows
      const int wi = (warp & 3) + 4 * grp;
      const float* tk = c.tail_k + (bh * c.k.group) * D + lane * C;
      const float* tv = c.tail_v + (bh * c.k.group) * D + lane * C;
      float tm[4], tl[4], ta[4][C];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        tm[j] = neg_inf();
        tl[j] = 0.0f;
#pragma unroll
        for (int i = 0; i < C; ++i) ta[j][i] = 0.0f;
      }
      for (int r0 = wi; r0 < TT; r0 += RS * U) {
        float x[U][C], y[U][C];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int r = r0 + u * RS;
#pragma unroll
          for (int i = 0; i < C; ++i) {
            x[u][i] = r < TT ? tk[(size_t)r * D + i] : 0.0f;
            y[u][i] = r < TT ? tv[(size_t)r * D + i] : 0.0f;
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (r0 + u * RS >= TT) break;   // warp-uniform
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int h = 4 * hg + j;
            if (h >= G) break;   // warp-uniform
            float p = 0.0f;
#pragma unroll
            for (int i = 0; i < C; ++i) p = fmaf(sm_qraw[h][lane * C + i], x[u][i], p);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
            const float sc = p * a.qscale;
            const float mn = fmaxf(tm[j], sc);
            const float alpha = fast_exp2(tm[j] - mn);
            const float pw = fast_exp2(sc - mn);
            tl[j] = fmaf(tl[j], alpha, pw);
#pragma unroll
            for (int i = 0; i < C; ++i) ta[j][i] = fmaf(ta[j][i], alpha, pw * y[u][i]);
            tm[j] = mn;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int h = 4 * hg + j;
        if (h >= G) break;
#pragma unroll
        for (int i = 0; i < C; ++i) {
          const int d = lane * C + i;
          sm_acc[warp][h][(d % VCH) * 8 + d / VCH] = ta[j][i];
        }
        if (lane == 0) {
          sm_m[warp][h] = tm[j];
          sm_l[warp][h] = tl[j];
        }
      }
    }
  } else {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l_part += __shfl_xor_sync(0xffffffffu, l_part, o);
      zacc += __shfl_xor_sync(0xffffffffu, zacc, o);
    }
    if (hd < G) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        sm_acc[warp][hd][(2 * mt) * 8 + g] = failed ? 0.0f : (oacc[mt][0] + oacc[mt][1]) + zacc;
        sm_acc[warp][hd][(2 * mt + 1) * 8 + g] = failed ? 0.0f : (oacc[mt][2] + oacc[mt][3]) + zacc;
      }
      if (g == 0) {
        sm_m[warp][hd] = failed ? neg_inf() : m_run;
        sm_l[warp][hd] = failed ? 0.0f : l_part;
      }
    }
  }
  __syncthreads();
  if constexpr (K_KIVIB) {
    DecodeArgs am = a;
    am.nsplit = a.nsplit + 1;   // partial slots per (b, kv head): the splits and the tail
    merge_store<D, G, 8, NWARP, HG>(c, am, b, kvh, is_tail ? nse : split, nse_all, sm_m, sm_l, &sm_acc[0][0][0]);
  } else if constexpr (APP) {
    merge_store<D, G, 8, NWARP, HG, 1, true>(c, a, b, kvh, split, nse, sm_m, sm_l, &sm_acc[0][0][0], sm_newv, step);
  } else {
    merge_store<D, G, 8, NWARP, HG>(c, a, b, kvh, split, nse, sm_m, sm_l, &sm_acc[0][0][0]);
  }
}

template <int D, int G, int KF, int VF, int NGRP, bool APP>
cudaError_t launch_decode_tc_shape(const CacheView& c, const DecodeArgs& a, cudaStream_t st) {
  using S = TcStages<D, G, KF, VF, NGRP>;
  using Shape = typename S::Shape;
  auto kern = decode_tc_kernel<D, G, KF, VF, NGRP, APP>;
  const int smem = S::dyn_bytes(S::stage);
  static_assert(S::dyn_bytes(S::stage) + S::static_smem <= 227 * 1024, "shared memory per CTA");
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e = once_per_device(configured, [&]() {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (e != cudaSuccess) return e;
  // Launched as a programmatic dependent of the previous kernel in the
  // stream: its CTAs may start once that kernel's CTAs have all triggered
  // (this kernel triggers right after its own dependency wait) and wait in
  // the kernel for it to complete before reading anything.
  cudaLaunchConfig_t cfg = {};
  // KIVI_BLOCK keys: one more CTA per (b, kv head) for the full-precision tail
  cfg.gridDim = dim3(a.nsplit + ((KF == F_KIVIB8 || KF == F_KIVIB4) ? 1 : 0), c.Hkv, c.B);
  cfg.blockDim = dim3(Shape::threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, c, a);
  note_launch();
  return e;
}

template <int D, int G, int KF, int VF, bool APP>
cudaError_t launch_decode_tc_app(const CacheView& c, const DecodeArgs& at, cudaStream_t st) {
  if constexpr (G <= 4) {
    if (at.wide == 2) return launch_decode_tc_shape<D, G, KF, VF, 4, APP>(c, at, st);
  }
  if (at.wide == 2) return cudaErrorInvalidValue;   // the plan gives sixteen-warp CTAs up to four heads only
  return at.wide ? launch_decode_tc_shape<D, G, KF, VF, 2, APP>(c, at, st)
                 : launch_decode_tc_shape<D, G, KF, VF, 1, APP>(c, at, st);
}

// The fused append is instantiated for head_dim 128, every format but
// KIVI_BLOCK keys and the one-wave shapes (wide 1 and 2): there the step's
// separate append launch would cost as much as the decode's own chain, while
// in a grid of several waves the token's coding delays its CTA's pipeline by
// more than a separate launch costs (measured).  Other caches and plans report
// cudaErrorNotSupported (nothing launched) and kvq_append_decode runs the
// separate steps.
template <int D, int G, int KF, int VF>
cudaError_t launch_decode_tc_dg(const CacheView& c, const DecodeArgs& a, cudaStream_t st) {
  DecodeArgs at = a;
  at.nsplit = a.nsplit_tc;
  if (at.nsplit < 1 || at.nsplit > kMaxSplits) return cudaErrorInvalidValue;
  if (a.k_new) {
    if constexpr (D == 128 && !(KF == F_KIVIB8 || KF == F_KIVIB4)) {
      if constexpr (G <= 4) {
        if (at.wide == 2) return launch_decode_tc_shape<D, G, KF, VF, 4, true>(c, at, st);
      }
      if (at.wide == 1) return launch_decode_tc_shape<D, G, KF, VF, 2, true>(c, at, st);
    }
    return cudaErrorNotSupported;
  }
  return launch_decode_tc_app<D, G, KF, VF, false>(c, at, st);
}

template <int D, int KF, int VF>
cudaError_t launch_decode_tc_d(const CacheView& c, int G, const DecodeArgs& a, cudaStream_t st) {
  switch (G) {
    case 1: return launch_decode_tc_dg<D, 1, KF, VF>(c, a, st);
    case 2: return launch_decode_tc_dg<D, 2, KF, VF>(c, a, st);
    case 3: return launch_decode_tc_dg<D, 3, KF, VF>(c, a, st);
    case 4: return launch_decode_tc_dg<D, 4, KF, VF>(c, a, st);
    case 5: return launch_decode_tc_dg<D, 5, KF, VF>(c, a, st);
    case 6: return launch_decode_tc_dg<D, 6, KF, VF>(c, a, st);
    case 7: return launch_decode_tc_dg<D, 7, KF, VF>(c, a, st);
    case 8: return launch_decode_tc_dg<D, 8, KF, VF>(c, a, st);
    default: return cudaErrorNotSupported;
  }
}

// Tensor-core path when its preconditions hold (head_dim 64 / 128, 16-bit io,
// key groups of at least 32 channels, each thread's value channels inside one
// group); the exact CUDA-core kernel otherwise (fp32 outputs, head_dim 32).
template <int KF, int VF>
cudaError_t launch_decode(const CacheView& c, int G, const DecodeArgs& a, cudaStream_t st) {
  {
  constexpr bool K_AFF = (KF == F_AFF8 || KF == F_AFF4);
  constexpr bool V_AFF = (VF == F_AFF8 || VF == F_AFF4);
  const bool groups_ok = (!K_AFF || c.k.group >= 32) && (!V_AFF || c.v.group >= c.D / 8);
  if ((c.D == 64 || c.D == 128) && a.io_dtype != KVQ_DTYPE_F32 && groups_ok && c.has_maps) {
    if (c.D == 128) return launch_decode_tc_d<128, KF, VF>(c, G, a, st);
    return launch_decode_tc_d<64, KF, VF>(c, G, a, st);
  }
  if (a.k_new) return cudaErrorNotSupported;   // the fused append runs on the tensor-core kernel only
  return launch_decode_cc<KF, VF>(c, G, a, st);
  }
}

}  // namespace kvq
