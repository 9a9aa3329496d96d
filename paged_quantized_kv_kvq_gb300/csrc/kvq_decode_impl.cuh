// kvq_decode_impl.cuh -- paged decode attention over a quantized KV pool.
//
// Method ("KV Cache优化实战：大模型推理显存占用与加速方案详解",
// 0539edu.com/news/5800990): the decode step attends the new Q over all cached
// K/V (§1.1); Q heads are grouped and each group shares one K/V head (§2.1);
// the cache lives in fixed-size physical blocks reached through a block table
// (§2.2); K/V are INT8/FP8 codes with per-token, per-channel or per-group
// scales, or FP16 (§2.3, §3.3); dequantization is fused into the attention
// kernel instead of running as a separate pass (§4.3).
//
// GB300 design (sm_103a):
//  * Persistent, balanced ("stream-K") grid: a unit is (sequence, kv head,
//    head tile of up to 8 Q heads) and owns ceil(L/bs) pages.  All units'
//    pages form one index space (computed in-kernel from context_lens); every
//    warp of the grid streams one equal, contiguous range of it, so all SMs
//    finish together whatever the length mix.  A unit wholly inside one warp's
//    range is written straight to the output; a unit cut by range ends leaves
//    a partial (running max, sum, unnormalised output) per piece, and a small
//    merge kernel, launched as a programmatic dependent of the decode kernel
//    (its launch overlaps the decode's tail), combines the pieces by
//    log-sum-exp.  The decode kernel itself never waits on another warp.
//  * Each warp keeps NSTAGE shared-memory stages in flight: lane 0 reads the
//    block table and issues one bulk (TMA) copy of the (block, kv head) page --
//    K codes, V codes and group scales are contiguous -- completing on an
//    mbarrier; a stage goes back to the copy engine once the page's P.V is
//    done (holding V in shared memory rather than registers keeps the kernel
//    at 3 CTAs per SM for every format).  Waits are bounded; a wait that runs
//    out sets an error bit instead of hanging.
//  * The Q heads of the unit share every loaded page: Q.K^T and P.V run on the
//    tensor cores as mma.m16n8k16 with the heads on the n dimension, 32 tokens
//    (two 16-token sub-tiles) per online-softmax update.  Codes are exact in
//    fp16 (int8 in [-127,127], every e4m3 value), so dequantization is a scale
//    applied outside the contraction: per-token / per-group K scales multiply
//    the fp32 scores, per-token / per-group V scales are folded into the softmax
//    weights, per-channel scales fold into q (K) and the output columns (V).
//  * fp32 operands entering a tensor-core product (softmax weights times V
//    scale; q times a per-channel K scale) are split into an fp16 high part and
//    an fp16 low part (two MMAs), after scaling by a power of two that keeps
//    them away from fp16 overflow and underflow; the power of two is undone
//    exactly at the end.  Softmax runs in base 2 (scores times log2 e).
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "kvq_common.cuh"
#include "kvq_context.h"

namespace kvq {

constexpr int kDecodeWarps = 4;
constexpr int kDecodeStages = 8;     // shared-memory stages per warp (at most; 80 KB per CTA)
constexpr int kDecodeCtasPerSm = 3;  // resident CTAs per SM the grid is sized for
constexpr int kDecodeThreads = kDecodeWarps * 32;
constexpr int kPartRows = 8;       // partial rows per (warp, slot): one per Q head of a tile
constexpr int kMergeThreads = 256;

struct DecodeParams {
  PoolView pool;
  const __half* q;     // [S][Hq][D], rows q_stride elements apart
  const int* table;    // [S][max_blocks]
  const int* lens;     // [S]
  float* out;          // [S][Hq][D], rows out_stride elements apart
  int64_t q_stride, out_stride;
  int* ps;             // [S + 1] page prefix over sequences (written by CTA 0 for the merge)
  float* part;         // [warps][2][kPartRows][D + 2]: m, l, O of cut units
  // Shared-prefix cascade: the first `skip` blocks of every sequence are the
  // shared prefix, already attended by the prefix kernel, whose partial rows
  // (m, l, O in true units) are in pre[S][Hq][D + 2]; skip = 0, pre = null
  // otherwise.
  const float* pre;
  int skip;
  int S, Hq, G, n_ht, max_blocks, max_ctx;
  int ppw_fixed;       // pages per warp; 0 = balance the pages over all warps
  int nstage;          // shared-memory stages per warp
  int wait_tries;      // bound of every pipeline wait (tries of ~1 ms each)
  // Self-test of the bounded waits: warp 0 arms the barrier of its copy
  // number `fault_issue` but issues no copy, so that wait runs out; -1 = off.
  int fault_issue;
  int stage_bytes;
  int grid;            // decode CTAs (the merge kernel derives the warp ranges from it)
  float sm_scale_log2;  // sm_scale * log2(e)
};

__device__ __forceinline__ float pow2f(int e) {  // 2^e for e in [-126, 127]
  return __int_as_float((e + 127) << 23);
}

__device__ __forceinline__ int exponent_of(float x) {  // floor(log2 x) for normal x > 0
  return ((__float_as_int(x) >> 23) & 0xFF) - 127;
}

__device__ __forceinline__ float warp_max_over_rows(float v) {  // reduce over lane>>2
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  return v;
}

__device__ __forceinline__ float warp_sum_over_rows(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// Split an fp32 pair into fp16 hi and lo pairs: (a, b) ~= hi + lo.
__device__ __forceinline__ void split_h2(float a, float b, uint32_t& hi, uint32_t& lo) {
  __half2 h = __floats2half2_rn(a, b);
  __half2 r = __floats2half2_rn(a - __low2float(h), b - __high2float(h));
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&r);
}

template <int FMT>
struct FmtTraits {
  static constexpr bool one_byte = FMT != FMT_FP16;
  static constexpr bool group_scales = FMT == FMT_INT8_GROUP || FMT == FMT_INT4_GROUP;
  static constexpr bool token_scales = FMT == FMT_INT8_TOKEN || FMT == FMT_FP8_TOKEN;
  static constexpr bool row_scales = group_scales || token_scales;  // per-(token[,group]) K/V scales
  static constexpr bool channel = FMT == FMT_INT8_CHANNEL;
  static constexpr bool maybe_nan = FMT == FMT_FP16 || FMT == FMT_FP8_TOKEN || FMT == FMT_FP8_E5M2;
};

// 32-bit words a lane holds of one 16-token sub-tile of K (or V).
template <int FMT, int D>
__host__ __device__ constexpr int lane_words() {
  return FMT == FMT_FP16 ? D / 4 : (FMT == FMT_INT4_GROUP ? D / 16 : D / 8);
}

// Word w (4 elements) of a lane's sub-tile -> (lo, hi) fp16x2 pairs.
template <int FMT>
__device__ __forceinline__ void word_to_h2(const uint32_t* words, int w, uint32_t& lo, uint32_t& hi) {
  if constexpr (FMT == FMT_FP16) {
    lo = words[2 * w];
    hi = words[2 * w + 1];
  } else if constexpr (FMT == FMT_FP8_TOKEN) {
    e4m3x4_to_h2x2(words[w], lo, hi);
  } else if constexpr (FMT == FMT_FP8_E5M2) {
    e5m2x4_to_h2x2(words[w], lo, hi);
  } else {
    i8x4_to_h2x2(words[w], lo, hi);
  }
}

// A-fragment words of k-step kk of a K sub-tile (rows = tokens g, g+8; k =
// channels 16kk + 4j..+3 in the layout's order).
template <int FMT, int D>
__device__ __forceinline__ void k_frag(const uint32_t* w, int kk, uint32_t& a0, uint32_t& a1,
                                       uint32_t& a2, uint32_t& a3) {
  if constexpr (FMT == FMT_INT4_GROUP) {
    i4x8_to_h2x4(w[kk], a0, a2, a1, a3);
  } else {
    word_to_h2<FMT>(w, kk, a0, a2);           // row g   : channels e=0,1 | e=2,3
    word_to_h2<FMT>(w, D / 16 + kk, a1, a3);  // row g+8
  }
}

// A-fragment words of m-tile mt of a V sub-tile read as V^T (rows = channels
// 16mt + g, +8; k = tokens 2j, 2j+1 | 2j+8, 2j+9).
template <int FMT>
__device__ __forceinline__ void v_frag(const uint32_t* w, int mt, uint32_t& a0, uint32_t& a1,
                                       uint32_t& a2, uint32_t& a3) {
  if constexpr (FMT == FMT_INT4_GROUP) {
    i4x8_to_h2x4(w[mt], a0, a2, a1, a3);
  } else {
    word_to_h2<FMT>(w, 2 * mt, a0, a2);      // channel 16mt+g
    word_to_h2<FMT>(w, 2 * mt + 1, a1, a3);  // channel 16mt+g+8
  }
}

// The same fragment from the V words of two 8-token pages (block size 8),
// interleaved per m-tile by load_v8: page A's word gives channels 16mt+g and
// +8 at tokens 2j, 2j+1, page B's word the same at tokens 8+2j, 8+2j+1.
template <int FMT>
__device__ __forceinline__ void v_frag8(const uint32_t* w, int mt, uint32_t& a0, uint32_t& a1,
                                        uint32_t& a2, uint32_t& a3) {
  word_to_h2<FMT>(w, 2 * mt, a0, a1);
  word_to_h2<FMT>(w, 2 * mt + 1, a2, a3);
}

// Copy a lane's share of a sub-tile from shared memory (16-byte chunks).
template <int FMT, int D>
__device__ __forceinline__ void load_lane_words(const char* tile, int lane, uint32_t* words) {
  constexpr int chunks = lane_words<FMT, D>() / 4;
#pragma unroll
  for (int c = 0; c < chunks; ++c) {
    uint4 v = *reinterpret_cast<const uint4*>(tile + c * 512 + lane * 16);
    words[4 * c + 0] = v.x;
    words[4 * c + 1] = v.y;
    words[4 * c + 2] = v.z;
    words[4 * c + 3] = v.w;
  }
}

// A lane's words of one 8-token page (half of lane_words), or zeros when the
// page is absent.
template <int FMT, int D>
__device__ __forceinline__ void load_half_words(const char* page, int lane, uint32_t* words) {
  constexpr int chunks = lane_words<FMT, D>() / 8;
#pragma unroll
  for (int c = 0; c < chunks; ++c) {
    const uint4 v = page != nullptr ? *reinterpret_cast<const uint4*>(page + c * 512 + lane * 16)
                                    : make_uint4(0u, 0u, 0u, 0u);
    words[4 * c + 0] = v.x;
    words[4 * c + 1] = v.y;
    words[4 * c + 2] = v.z;
    words[4 * c + 3] = v.w;
  }
}

// V words of a 16-token tile made of two 8-token pages, interleaved per m-tile
// (A's 4-element group, then B's) for v_frag8.
template <int FMT, int D>
__device__ __forceinline__ void load_v8(const char* a, const char* b, int lane, uint32_t* words) {
  constexpr int HALF = lane_words<FMT, D>() / 2;
  constexpr int PER = FMT == FMT_FP16 ? 2 : 1;  // 32-bit words per 4-element group
  uint32_t wa[HALF], wb[HALF];
  load_half_words<FMT, D>(a, lane, wa);
  load_half_words<FMT, D>(b, lane, wb);
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int x = 0; x < PER; ++x) {
      words[2 * PER * mt + x] = wa[PER * mt + x];
      words[2 * PER * mt + PER + x] = wb[PER * mt + x];
    }
}

// Position of a warp in the unit-major page index space.
struct Cursor {
  int s, lu, pi, Ps;  // sequence, unit within the sequence, page within the unit, pages per unit
};

// Everything one online-softmax update needs from two 16-token sub-tiles,
// held in registers: K fragment words, the scales of the two rows this lane
// owns (tokens g and g+8), where the V codes sit in shared memory, the valid
// rows.
template <int FMT, int D, int NG>
struct PairRegs {
  using T = FmtTraits<FMT>;
  static constexpr int NU32 = lane_words<FMT, D>();
  static constexpr int NS = T::group_scales ? NG : 1;
  uint32_t kw[2][NU32];
  float ks[2][2][NS];  // [tile][row g | g+8][group]
  float vs[2][2][NS];
  const char* vtile[2];  // V codes in shared memory
  const char* vtile_b[2];  // block size 8: V codes of the tile's second page (or null)
  int rows[2];
};

// Fill tile t of `r` from sub-tile `sub` of a staged page.
template <int FMT, int D, int NG>
__device__ __forceinline__ void load_tile(PairRegs<FMT, D, NG>& r, int t, const char* stage,
                                          int sub, int rows, const PoolView& pool, int lane) {
  using T = FmtTraits<FMT>;
  constexpr int NS = PairRegs<FMT, D, NG>::NS;
  const int g = lane >> 2;
  load_lane_words<FMT, D>(stage + sub * pool.sub_bytes, lane, r.kw[t]);
  r.vtile[t] = stage + pool.code_bytes + sub * pool.sub_bytes;
  if constexpr (T::row_scales) {
    const float* ks;
    const float* vs;
    if constexpr (T::group_scales) {
      ks = reinterpret_cast<const float*>(stage + 2 * pool.code_bytes) + sub * 16 * NG;
      vs = ks + pool.bs * NG;
    } else {
      ks = reinterpret_cast<const float*>(stage + pool.page_bytes) + sub * 16;
      vs = ks + pool.bs;
    }
#pragma unroll
    for (int gi = 0; gi < NS; ++gi) {
      r.ks[t][0][gi] = ks[g * NS + gi];
      r.ks[t][1][gi] = ks[(g + 8) * NS + gi];
      r.vs[t][0][gi] = vs[g * NS + gi];
      r.vs[t][1][gi] = vs[(g + 8) * NS + gi];
    }
  }
  r.rows[t] = rows;
}

// Fill tile t of `r` from two 8-token pages (block size 8): page A gives rows
// 0..7, page B (null if absent) rows 8..15.  Rows valid: 0 .. rows-1.
template <int FMT, int D, int NG>
__device__ __forceinline__ void load_tile8(PairRegs<FMT, D, NG>& r, int t, const char* A,
                                           const char* B, int rows, const PoolView& pool,
                                           int lane) {
  using T = FmtTraits<FMT>;
  constexpr int NS = PairRegs<FMT, D, NG>::NS;
  constexpr int HALF = PairRegs<FMT, D, NG>::NU32 / 2;
  const int g = lane >> 2;
  uint32_t wa[HALF], wb[HALF];
  load_half_words<FMT, D>(A, lane, wa);
  load_half_words<FMT, D>(B, lane, wb);
#pragma unroll
  for (int x = 0; x < HALF; ++x) {
    r.kw[t][x] = wa[x];
    r.kw[t][HALF + x] = wb[x];
  }
  r.vtile[t] = A + pool.code_bytes;
  r.vtile_b[t] = B != nullptr ? B + pool.code_bytes : nullptr;
  if constexpr (T::row_scales) {
    // scales of token g of each page: [bs][NS] per group, [2][bs] per token
    const int ko = T::group_scales ? 2 * pool.code_bytes : pool.page_bytes;
    const int vo = T::group_scales ? 8 * NG * 4 : 8 * 4;
    const float* ka = reinterpret_cast<const float*>(A + ko) + g * NS;
    const float* va = reinterpret_cast<const float*>(A + ko + vo) + g * NS;
#pragma unroll
    for (int gi = 0; gi < NS; ++gi) {
      r.ks[t][0][gi] = ka[gi];
      r.vs[t][0][gi] = va[gi];
    }
    if (B != nullptr) {
      const float* kb = reinterpret_cast<const float*>(B + ko) + g * NS;
      const float* vb = reinterpret_cast<const float*>(B + ko + vo) + g * NS;
#pragma unroll
      for (int gi = 0; gi < NS; ++gi) {
        r.ks[t][1][gi] = kb[gi];
        r.vs[t][1][gi] = vb[gi];
      }
    } else {
#pragma unroll
      for (int gi = 0; gi < NS; ++gi) r.ks[t][1][gi] = r.vs[t][1][gi] = 0.f;
    }
  }
  r.rows[t] = rows;
}

// One online-softmax update over two sub-tiles (32 tokens) for the up-to-8 Q
// heads of a unit.  Lane (g = lane/4, j = lane%4) holds the scores of tokens g
// and g+8 of each tile for heads 2j and 2j+1, and O^T rows 16mt+g, 16mt+g+8
// for the same two heads.  Tile 1 may be empty (rows = 0).
template <int FMT, int D, int NG, bool BS8 = false>
__device__ __forceinline__ void compute_pair(PairRegs<FMT, D, NG>& r, int lane,
                                             const uint32_t (&qb)[D / 16][2],
                                             const uint32_t (&ql)[FmtTraits<FMT>::channel ? D / 16 : 1][2],
                                             float csc, float (&m)[2], float (&l)[2], int& E,
                                             float (&o)[D / 16][4]) {
  using T = FmtTraits<FMT>;
  constexpr int KS = D / 16;
  constexpr int NU32 = PairRegs<FMT, D, NG>::NU32;
  constexpr int NS = PairRegs<FMT, D, NG>::NS;
  constexpr int KPG = KS / NG;
  constexpr int SUB = KPG >= 2 ? 2 : 1;  // independent accumulators per scale group
  const float kNegInf = __int_as_float(0xff800000u);
  const int g = lane >> 2, j = lane & 3;

  // ---- scores: S[t][r] = sum_d code_K[t][d] q'[r][d], per scale group
  float z[2][4];
  {
    float acc[2][NG * SUB][4];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int a = 0; a < NG * SUB; ++a) acc[t][a][0] = acc[t][a][1] = acc[t][a][2] = acc[t][a][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int ai = (kk / KPG) * SUB + (SUB == 2 ? (kk & 1) : 0);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        uint32_t a0, a1, a2, a3;
        k_frag<FMT, D>(r.kw[t], kk, a0, a1, a2, a3);
        mma_16816(acc[t][ai], a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        if constexpr (T::channel) mma_16816(acc[t][ai], a0, a1, a2, a3, ql[kk][0], ql[kk][1]);
      }
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      float zz[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        float s4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          s4[e] = SUB == 2 ? acc[t][gi * SUB][e] + acc[t][gi * SUB + 1][e] : acc[t][gi * SUB][e];
        float sA = csc, sB = csc;
        if constexpr (T::row_scales) {
          sA *= r.ks[t][0][T::group_scales ? gi : 0];
          sB *= r.ks[t][1][T::group_scales ? gi : 0];
        }
        zz[0] = fmaf(s4[0], sA, zz[0]);
        zz[1] = fmaf(s4[1], sA, zz[1]);
        zz[2] = fmaf(s4[2], sB, zz[2]);
        zz[3] = fmaf(s4[3], sB, zz[3]);
      }
      const bool vA = g < r.rows[t], vB = g + 8 < r.rows[t];
      z[t][0] = vA ? zz[0] : kNegInf;
      z[t][1] = vA ? zz[1] : kNegInf;
      z[t][2] = vB ? zz[2] : kNegInf;
      z[t][3] = vB ? zz[3] : kNegInf;
    }
  }

  // ---- online softmax (base 2) over the 32 tokens
  float pr[2][4];
  {
    float t0 = fmaxf(fmaxf(z[0][0], z[0][2]), fmaxf(z[1][0], z[1][2]));
    float t1 = fmaxf(fmaxf(z[0][1], z[0][3]), fmaxf(z[1][1], z[1][3]));
    t0 = warp_max_over_rows(t0);
    t1 = warp_max_over_rows(t1);
    const float mn0 = fmaxf(m[0], t0), mn1 = fmaxf(m[1], t1);
    const float ms0 = mn0 == kNegInf ? 0.f : mn0;
    const float ms1 = mn1 == kNegInf ? 0.f : mn1;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      pr[t][0] = fast_exp2(z[t][0] - ms0);
      pr[t][1] = fast_exp2(z[t][1] - ms1);
      pr[t][2] = fast_exp2(z[t][2] - ms0);
      pr[t][3] = fast_exp2(z[t][3] - ms1);
    }
    int dE = 0;
    if constexpr (T::row_scales) {
      float vmax = 0.f;
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int gi = 0; gi < NS; ++gi) {
          if (g < r.rows[t]) vmax = fmaxf(vmax, r.vs[t][0][gi]);
          if (g + 8 < r.rows[t]) vmax = fmaxf(vmax, r.vs[t][1][gi]);
        }
      vmax = warp_max_over_rows(vmax);
      if (vmax > 0.f) {
        const int En = min(E, 13 - exponent_of(vmax));
        dE = En - E;
        E = En;
      }
    }
    const float al0 = fast_exp2(m[0] - ms0), al1 = fast_exp2(m[1] - ms1);
    l[0] = fmaf(l[0], al0, (pr[0][0] + pr[0][2]) + (pr[1][0] + pr[1][2]));
    l[1] = fmaf(l[1], al1, (pr[0][1] + pr[0][3]) + (pr[1][1] + pr[1][3]));
    m[0] = mn0;
    m[1] = mn1;
    const float f2 = pow2f(dE);
    const float ao0 = al0 * f2, ao1 = al1 * f2;
    if (__any_sync(0xffffffffu, ao0 != 1.f || ao1 != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        o[mt][0] *= ao0;
        o[mt][1] *= ao1;
        o[mt][2] *= ao0;
        o[mt][3] *= ao1;
      }
    }
  }

  // ---- P.V: B operand = p * s_V * 2^E split into fp16 hi + lo, transposed so
  // that k runs over the tile's tokens
  constexpr int NB = T::group_scales ? NG : 1;
  uint32_t bh0[2][NB], bh1[2][NB], bl0[2][NB], bl1[2][NB];
  {
    const float sc = pow2f(E);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const bool vA = g < r.rows[t], vB = g + 8 < r.rows[t];
#pragma unroll
      for (int gi = 0; gi < NB; ++gi) {
        float fA = sc, fB = sc;
        if constexpr (T::row_scales) {
          fA *= r.vs[t][0][gi];
          fB *= r.vs[t][1][gi];
        }
        const float p0 = vA ? pr[t][0] * fA : 0.f, p1 = vA ? pr[t][1] * fA : 0.f;
        const float p2 = vB ? pr[t][2] * fB : 0.f, p3 = vB ? pr[t][3] * fB : 0.f;
        uint32_t hA, lA, hB, lB;
        split_h2(p0, p1, hA, lA);
        split_h2(p2, p3, hB, lB);
        bh0[t][gi] = movmatrix_t(hA);
        bh1[t][gi] = movmatrix_t(hB);
        bl0[t][gi] = movmatrix_t(lA);
        bl1[t][gi] = movmatrix_t(lB);
      }
    }
  }
  {
    uint32_t vwp[2][NU32];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if constexpr (BS8)
        load_v8<FMT, D>(r.vtile[t], r.vtile_b[t], lane, vwp[t]);
      else
        load_lane_words<FMT, D>(r.vtile[t], lane, vwp[t]);
    }
    if constexpr (T::maybe_nan && BS8) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int rows = r.rows[t];
        if (rows < 16) {
          // page A's words hold tokens 2j, 2j+1 (rows of the tile), page B's
          // tokens 8+2j, 8+2j+1; zero the ones past the context
          const int t0 = 2 * j;
          if constexpr (FMT == FMT_FP16) {
            const uint32_t mlo = (t0 < rows ? 0xFFFFu : 0u) | (t0 + 1 < rows ? 0xFFFF0000u : 0u);
            const uint32_t mhi = (t0 + 8 < rows ? 0xFFFFu : 0u) | (t0 + 9 < rows ? 0xFFFF0000u : 0u);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              vwp[t][4 * mt] &= mlo;
              vwp[t][4 * mt + 1] &= mlo;
              vwp[t][4 * mt + 2] &= mhi;
              vwp[t][4 * mt + 3] &= mhi;
            }
          } else {
            const uint32_t mlo = (t0 < rows ? 0x00FF00FFu : 0u) | (t0 + 1 < rows ? 0xFF00FF00u : 0u);
            const uint32_t mhi = (t0 + 8 < rows ? 0x00FF00FFu : 0u) | (t0 + 9 < rows ? 0xFF00FF00u : 0u);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              vwp[t][2 * mt] &= mlo;
              vwp[t][2 * mt + 1] &= mhi;
            }
          }
        }
      }
    } else if constexpr (T::maybe_nan) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int rows = r.rows[t];
        if (rows < 16) {
          // tokens of this lane's V bytes: 2j, 2j+1, 2j+8, 2j+9; zero the ones
          // past the context so that 0 * NaN cannot reach the sum
          const int t0 = 2 * j;
          if constexpr (FMT == FMT_FP16) {
            const uint32_t mlo = (t0 < rows ? 0xFFFFu : 0u) | (t0 + 1 < rows ? 0xFFFF0000u : 0u);
            const uint32_t mhi = (t0 + 8 < rows ? 0xFFFFu : 0u) | (t0 + 9 < rows ? 0xFFFF0000u : 0u);
#pragma unroll
            for (int w = 0; w < NU32 / 2; ++w) {
              vwp[t][2 * w] &= mlo;
              vwp[t][2 * w + 1] &= mhi;
            }
          } else {
            const uint32_t msk = (t0 < rows ? 0xFFu : 0u) | (t0 + 1 < rows ? 0xFF00u : 0u) |
                                 (t0 + 8 < rows ? 0xFF0000u : 0u) |
                                 (t0 + 9 < rows ? 0xFF000000u : 0u);
#pragma unroll
            for (int w = 0; w < NU32; ++w) vwp[t][w] &= msk;
          }
        }
      }
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const int gi = T::group_scales ? (mt / KPG) : 0;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        uint32_t a0, a1, a2, a3;
        if constexpr (BS8)
          v_frag8<FMT>(vwp[t], mt, a0, a1, a2, a3);
        else
          v_frag<FMT>(vwp[t], mt, a0, a1, a2, a3);
        mma_16816(o[mt], a0, a1, a2, a3, bh0[t][gi], bh1[t][gi]);
        mma_16816(o[mt], a0, a1, a2, a3, bl0[t][gi], bl1[t][gi]);
      }
    }
  }
}

// Q fragments of a unit: head n = g of the tile, channels 16kk + 4j .. +3.
// Per-channel pools fold the K channel scale into q (fp32), scale the result by
// 2^eq so that max|q'| lies in [2^13, 2^14), and split it into fp16 hi + lo;
// csc then carries 2^-eq.
template <int FMT, int D>
__device__ __forceinline__ void load_q(const DecodeParams& p, int s, int h, int ht, int lane,
                                       uint32_t (&qb)[D / 16][2],
                                       uint32_t (&ql)[FmtTraits<FMT>::channel ? D / 16 : 1][2],
                                       float& csc) {
  constexpr int KS = D / 16;
  const int g = lane >> 2, j = lane & 3;
  const int Gt = min(8, p.G - 8 * ht);
  const bool hv = g < Gt;
  const int hq = h * p.G + 8 * ht + (hv ? g : 0);
  const __half* qp = p.q + (int64_t)s * p.q_stride + (int64_t)hq * D;
  csc = p.sm_scale_log2;
  if constexpr (!FmtTraits<FMT>::channel) {
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint2 v = hv ? *reinterpret_cast<const uint2*>(qp + 16 * kk + 4 * j) : make_uint2(0, 0);
      qb[kk][0] = v.x;
      qb[kk][1] = v.y;
    }
  } else {
    const float* ksc = p.pool.chan_scales + (int64_t)h * D;
    float qf[KS][4];
    float amax = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint2 v = hv ? *reinterpret_cast<const uint2*>(qp + 16 * kk + 4 * j) : make_uint2(0, 0);
      __half2 a = *reinterpret_cast<__half2*>(&v.x), b = *reinterpret_cast<__half2*>(&v.y);
      const int d0 = 16 * kk + 4 * j;
      qf[kk][0] = __low2float(a) * ksc[d0 + 0];
      qf[kk][1] = __high2float(a) * ksc[d0 + 1];
      qf[kk][2] = __low2float(b) * ksc[d0 + 2];
      qf[kk][3] = __high2float(b) * ksc[d0 + 3];
#pragma unroll
      for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qf[kk][e]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const int eq = amax > 0.f ? 13 - exponent_of(amax) : 0;
    const float up = ldexpf(1.f, eq);
    csc = ldexpf(csc, -eq);
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      split_h2(qf[kk][0] * up, qf[kk][1] * up, qb[kk][0], ql[kk][0]);
      split_h2(qf[kk][2] * up, qf[kk][3] * up, qb[kk][1], ql[kk][1]);
    }
  }
}

template <int FMT, int D, int NG, bool BS8>
__global__ void __launch_bounds__(kDecodeThreads, kDecodeCtasPerSm)
    kvq_decode_kernel(const DecodeParams p) {
  using T = FmtTraits<FMT>;
  constexpr int KS = D / 16;
  const float kNegInf = __int_as_float(0xff800000u);

  extern __shared__ __align__(128) char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, j = lane & 3;
  const PoolView& pool = p.pool;
  const int bs = pool.bs;
  const int nstage = p.nstage;
  const int U = pool.Hkv * p.n_ht;  // units per sequence

  // The merge grid may launch now: every CTA of this (persistent) grid is
  // resident once all have passed this point, and the merge reads nothing of
  // ours before its griddepcontrol.wait returns on this grid's completion.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  char* stages = smem + warp * nstage * p.stage_bytes;
  uint64_t* bars_base = reinterpret_cast<uint64_t*>(smem + kDecodeWarps * nstage * p.stage_bytes);
  uint64_t* bars = bars_base + warp * nstage;
  // block size 8: a stage holds two consecutive pages of the range (slots 0
  // and 1, stage_bytes / 2 apart) completing on one barrier
  constexpr int SPS = BS8 ? 2 : 1;  // pages per stage
  int* phys_base = reinterpret_cast<int*>(bars_base + kDecodeWarps * nstage);
  int* stage_phys = phys_base + warp * nstage * SPS;
  int* wtot = phys_base + kDecodeWarps * nstage * SPS;  // [kDecodeWarps]
  int* PS = wtot + kDecodeWarps;                  // [S + 1] page prefix over sequences

  // ---- pages per sequence and their prefix (every CTA computes the same)
  {
    int carry = 0;
    for (int base = 0; base < p.S; base += kDecodeThreads) {
      const int s = base + threadIdx.x;
      int v = 0;
      if (s < p.S) {
        int L = p.lens[s];
        if (L > p.max_ctx) {
          if (blockIdx.x == 0) set_error(pool.err, ERR_RANGE);
          L = p.max_ctx;
        }
        v = L > 0 ? max((L + bs - 1) / bs - p.skip, 0) * U : 0;
      }
      int x = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      if (lane == 31) wtot[warp] = x;
      __syncthreads();
      int before = 0, all = 0;
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) {
        before += w < warp ? wtot[w] : 0;
        all += wtot[w];
      }
      if (s < p.S) PS[s + 1] = carry + before + x;
      carry += all;
      __syncthreads();
    }
    if (threadIdx.x == 0) PS[0] = 0;
    __syncthreads();
  }

  const int Ttot = PS[p.S];
  const int nwarps = gridDim.x * kDecodeWarps;
  const int gw = blockIdx.x * kDecodeWarps + warp;
  const int ppw = p.ppw_fixed > 0 ? p.ppw_fixed : (Ttot + nwarps - 1) / nwarps;
  const int a0 = (int)min((int64_t)gw * ppw, (int64_t)Ttot);
  const int b0 = (int)min((int64_t)a0 + ppw, (int64_t)Ttot);
  const int n_w = b0 - a0;

  // Writes to the output and the workspace come only after
  // griddepcontrol.wait: when this grid is a programmatic dependent (of the
  // decode-step append, itself a dependent of whatever ran before), the
  // previous merge may still be reading them until then.
  auto after_wait = [&]() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (gw == 0)  // the page prefix, for the merge kernel
      for (int s = lane; s <= p.S; s += 32) p.ps[s] = PS[s];
    // sequences with nothing (left) to attend get zeros, or in the cascade
    // the normalised prefix result
    for (int s = gw; s < p.S; s += nwarps) {
      if (PS[s + 1] != PS[s]) continue;
      float* o = p.out + (int64_t)s * p.out_stride;
      if (p.pre == nullptr) {
        for (int i = lane; i < p.Hq * D; i += 32) o[i] = 0.f;
      } else {
        for (int hq = 0; hq < p.Hq; ++hq) {
          const float* pr = p.pre + ((int64_t)s * p.Hq + hq) * (D + 2);
          const float lp = pr[1];
          const float f = lp > 0.f ? 1.f / lp : 0.f;
          for (int d = lane; d < D; d += 32) o[(int64_t)hq * D + d] = pr[2 + d] * f;
        }
      }
    }
  };
  if (n_w <= 0) {
    after_wait();
    return;
  }

  auto locate = [&](int x) -> Cursor {
    int lo = 0, hi = p.S;  // PS[lo] <= x < PS[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (PS[mid] <= x) lo = mid; else hi = mid;
    }
    Cursor c;
    c.s = lo;
    c.Ps = (PS[lo + 1] - PS[lo]) / U;
    const int r = x - PS[lo];
    c.lu = r / c.Ps;
    c.pi = r - c.lu * c.Ps;
    return c;
  };
  auto advance = [&](Cursor& c) {
    if (++c.pi < c.Ps) return;
    c.pi = 0;
    if (++c.lu < U) return;
    c.lu = 0;
    do { ++c.s; } while (c.s < p.S && PS[c.s + 1] == PS[c.s]);
    c.Ps = c.s < p.S ? (PS[c.s + 1] - PS[c.s]) / U : 1;
  };

  // ---- pipeline set-up
  if (lane == 0) {
    for (int st = 0; st < nstage; ++st) mbar_init(&bars[st], 1);
    fence_barrier_init();
  }
  __syncwarp();

  const uint32_t page_tx = pool.page_bytes + (T::token_scales ? 2 * bs * 4 : 0);
  // Block-table entries of the pages to issue, cached one per lane and loaded
  // 32 to 64 pages ahead: tcur covers issue indices [tbase, tbase+32), tnext
  // the 32 after, so a table load never stalls a copy issue.
  auto table_entry = [&](int n) -> int {  // page n of this warp's range
    if (n >= n_w) return -1;
    const Cursor c = locate(a0 + n);
    return p.table[(int64_t)c.s * p.max_blocks + p.skip + c.pi];
  };
  int tbase = 0;
  int tcur = table_entry(lane), tnext = table_entry(32 + lane);
  Cursor ic = locate(a0);  // next page to issue (lane 0 tracks it)
  int n_issued = 0;
  int pst = 0;  // stage of the next issue (n_issued mod nstage)
  auto issue_one = [&](int phys) {  // lane 0 only: page at the issue cursor
    const int st = pst;
    char* dst = stages + st * p.stage_bytes;
    const bool ok = phys >= 0 && (int64_t)phys < pool.num_blocks;
    stage_phys[st] = ok ? phys : -1;
    if (ok && p.fault_issue >= 0 && gw == 0 && n_issued == p.fault_issue) {
      mbar_arrive_expect_tx(&bars[st], page_tx);  // bytes that never come
    } else if (ok) {
      const int h = p.n_ht == 1 ? ic.lu : ic.lu / p.n_ht;  // (no division for G <= 8)
      mbar_arrive_expect_tx(&bars[st], page_tx);
      bulk_g2s(dst, pool.pages + ((int64_t)phys * pool.Hkv + h) * pool.page_bytes, pool.page_bytes,
               &bars[st]);
      if constexpr (T::token_scales)
        bulk_g2s(dst + pool.page_bytes, pool.tok_scales + (int64_t)phys * 2 * bs, 2 * bs * 4,
                 &bars[st]);
    } else {
      set_error(pool.err, ERR_RANGE);
      mbar_arrive(&bars[st]);
    }
  };
  // All lanes call this (the table cache is spread over the lanes); lane 0 issues.
  auto issue_next = [&]() {
    if (n_issued - tbase == 32) {
      tcur = tnext;
      tbase += 32;
      tnext = table_entry(tbase + 32 + lane);
    }
    const int phys = __shfl_sync(0xffffffffu, tcur, n_issued - tbase);
    if (lane == 0) {
      issue_one(phys);
      advance(ic);
    }
    ++n_issued;
    if (++pst == nstage) pst = 0;
  };
  // Block size 8: issue pages n_issued and n_issued + 1 (when in the range)
  // into the next stage, their copies completing on its one barrier.  All
  // lanes call this; lane 0 issues.  n_issued is even here, so both table
  // entries sit in tcur.
  const int slot_bytes = p.stage_bytes / 2;
  auto issue_pair = [&]() {
    if (n_issued - tbase == 32) {
      tcur = tnext;
      tbase += 32;
      tnext = table_entry(tbase + 32 + lane);
    }
    const bool two = n_issued + 1 < n_w;
    const int ph0 = __shfl_sync(0xffffffffu, tcur, n_issued - tbase);
    const int ph1 = __shfl_sync(0xffffffffu, tcur, (n_issued + 1 - tbase) & 31);
    if (lane == 0) {
      const int st = pst;
      int phys[2] = {ph0, ph1}, hh[2] = {0, 0};
      bool ok[2] = {false, false};
      uint32_t tx = 0;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (k == 1 && !two) {
          stage_phys[2 * st + 1] = -1;
          continue;
        }
        ok[k] = phys[k] >= 0 && (int64_t)phys[k] < pool.num_blocks;
        stage_phys[2 * st + k] = ok[k] ? phys[k] : -1;
        hh[k] = p.n_ht == 1 ? ic.lu : ic.lu / p.n_ht;
        if (ok[k]) tx += page_tx; else set_error(pool.err, ERR_RANGE);
        advance(ic);
      }
      if (tx == 0) {
        mbar_arrive(&bars[st]);
      } else {
        mbar_arrive_expect_tx(&bars[st], tx);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          if (!ok[k]) continue;
          if (p.fault_issue >= 0 && gw == 0 && n_issued + k == p.fault_issue) continue;  // never comes
          char* dst = stages + st * p.stage_bytes + k * slot_bytes;
          bulk_g2s(dst, pool.pages + ((int64_t)phys[k] * pool.Hkv + hh[k]) * pool.page_bytes,
                   pool.page_bytes, &bars[st]);
          if constexpr (T::token_scales)
            bulk_g2s(dst + pool.page_bytes, pool.tok_scales + (int64_t)phys[k] * 2 * bs, 2 * bs * 4,
                     &bars[st]);
        }
      }
    }
    n_issued += two ? 2 : 1;
    if (++pst == nstage) pst = 0;
  };
  // Everything above reads only inputs (lengths, block table).  When the
  // decode is a programmatic dependent of the decode-step append (directly or
  // through the prefix kernel), that append launched this grid only after
  // everything before it on the stream had completed, and it writes one page
  // per sequence: the one holding position L-1, the sequence's last page.  So
  // the first stages are filled before griddepcontrol.wait up to the first
  // last page, and the rest after it; without a dependency the wait returns
  // at once.
  if constexpr (BS8) {
    int k = 0;
    for (; k < nstage && n_issued < n_w; ++k) {
      Cursor c2 = ic;
      advance(c2);
      const bool last = __shfl_sync(
          0xffffffffu, ic.pi + 1 == ic.Ps || (n_issued + 1 < n_w && c2.pi + 1 == c2.Ps), 0);
      if (last) break;
      issue_pair();
    }
    after_wait();
    for (; k < nstage && n_issued < n_w; ++k) issue_pair();
  } else {
    const int npre = min(n_w, nstage);
    int k = 0;
    for (; k < npre; ++k) {
      const bool last = __shfl_sync(0xffffffffu, ic.pi + 1 == ic.Ps, 0);  // lane 0's cursor
      if (last) break;
      issue_next();
    }
    after_wait();
    for (; k < npre; ++k) issue_next();
  }

  // Consumer position: page i sits in stage cst; cph is the parity of that
  // stage's current fill.
  int cst = 0;
  uint32_t cph = 0;
  auto wait_stage = [&](int st, uint32_t parity) -> bool {
    const bool ok = mbar_wait_bounded(&bars[st], parity, p.wait_tries);
    return __all_sync(0xffffffffu, ok);
  };

  // ---- per-unit state (heads 2j, 2j+1 of the tile)
  uint32_t qb[KS][2];
  uint32_t ql[T::channel ? KS : 1][2];
  float csc = 0.f;
  float m[2], l[2], o[KS][4];
  int E = 0;
  Cursor cc = locate(a0);     // page being consumed
  const Cursor first = cc;    // the unit this warp's range starts in
  int seg_pi0 = cc.pi;        // first page of the current unit in this range
  int L = 0;                  // context length of the current unit's sequence
  auto start_unit = [&]() {
    L = min(p.lens[cc.s], p.max_ctx) - p.skip * bs;  // tokens after the skipped prefix
    load_q<FMT, D>(p, cc.s, cc.lu / p.n_ht, cc.lu % p.n_ht, lane, qb, ql, csc);
    m[0] = m[1] = kNegInf;
    l[0] = l[1] = 0.f;
    E = T::row_scales ? 100 : 14;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    seg_pi0 = cc.pi;
  };

  // Write the unit's result (whole unit in this range) or its partial, and
  // merge the partials if this piece is the unit's last to finish.
  auto finish_unit = [&](const Cursor& u, int seg_end) {
    const int h = u.lu / p.n_ht, ht = u.lu % p.n_ht;
    const int Gt = min(8, p.G - 8 * ht);
    const float lt0 = warp_sum_over_rows(l[0]), lt1 = warp_sum_over_rows(l[1]);
    const float inv2E = pow2f(-E);
    const float* vch = T::channel ? pool.chan_scales + ((int64_t)pool.Hkv + h) * D : nullptr;
    const int64_t row0 = (int64_t)u.s * p.Hq + h * p.G + 8 * ht;  // (prefix partial rows)
    float* obase = p.out + (int64_t)u.s * p.out_stride + (int64_t)(h * p.G + 8 * ht) * D;
    if (seg_pi0 == 0 && seg_end == u.Ps) {
      if (p.pre == nullptr) {
        const float f0 = lt0 > 0.f ? inv2E / lt0 : 0.f, f1 = lt1 > 0.f ? inv2E / lt1 : 0.f;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d0 = 16 * mt + g;
          const float c0 = T::channel ? vch[d0] : 1.f, c8 = T::channel ? vch[d0 + 8] : 1.f;
          if (2 * j < Gt) {
            float* dst = obase + (2 * j) * D;
            dst[d0] = o[mt][0] * f0 * c0;
            dst[d0 + 8] = o[mt][2] * f0 * c8;
          }
          if (2 * j + 1 < Gt) {
            float* dst = obase + (2 * j + 1) * D;
            dst[d0] = o[mt][1] * f1 * c0;
            dst[d0 + 8] = o[mt][3] * f1 * c8;
          }
        }
        return;
      }
      // cascade: log-sum-exp with the row's prefix partial
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (2 * j + c >= Gt) continue;
        const float* pr = p.pre + (row0 + 2 * j + c) * (D + 2);
        const float mp = pr[0], lp = pr[1];
        const float mu = m[c], lu = c ? lt1 : lt0;
        const float M = fmaxf(mu, mp);
        const float wu = mu == kNegInf ? 0.f : fast_exp2(mu - M);
        const float wp = mp == kNegInf ? 0.f : fast_exp2(mp - M);
        const float den = fmaf(lu, wu, lp * wp);
        const float inv = den > 0.f ? 1.f / den : 0.f;
        const float fu = wu * inv2E * inv, fp = wp * inv;
        float* dst = obase + (2 * j + c) * D;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d0 = 16 * mt + g;
          const float c0 = T::channel ? vch[d0] : 1.f, c8 = T::channel ? vch[d0 + 8] : 1.f;
          dst[d0] = fmaf(o[mt][c] * c0, fu, pr[2 + d0] * fp);
          dst[d0 + 8] = fmaf(o[mt][2 + c] * c8, fu, pr[2 + d0 + 8] * fp);
        }
      }
      return;
    }
    // -- partial: rows (m, l, O) in true units, for the tile's valid heads
    const int slot = (u.s == first.s && u.lu == first.lu) ? 0 : 1;
    float* base = p.part + ((int64_t)gw * 2 + slot) * kPartRows * (D + 2);
    const bool v0 = 2 * j < Gt, v1 = 2 * j + 1 < Gt;
    float* r0 = base + (2 * j) * (D + 2);
    float* r1 = base + (2 * j + 1) * (D + 2);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const int d0 = 16 * mt + g;
      const float c0 = T::channel ? vch[d0] : 1.f, c8 = T::channel ? vch[d0 + 8] : 1.f;
      if (v0) {
        r0[2 + d0] = o[mt][0] * inv2E * c0;
        r0[2 + d0 + 8] = o[mt][2] * inv2E * c8;
      }
      if (v1) {
        r1[2 + d0] = o[mt][1] * inv2E * c0;
        r1[2 + d0 + 8] = o[mt][3] * inv2E * c8;
      }
    }
    if (g == 0) {
      if (v0) {
        r0[0] = m[0];
        r0[1] = lt0;
      }
      if (v1) {
        r1[0] = m[1];
        r1[1] = lt1;
      }
    }
  };

  // ---- main loop: pages of this warp's range, two 16-token sub-tiles at a time
  start_unit();
  PairRegs<FMT, D, NG> R;
  int i = 0;
  bool failed = false;
  while (i < n_w) {
    // pages consumed this step: a pair of one-sub-tile pages of the same unit,
    // or one page of two or more sub-tiles; block size 8: up to four pages
    // (two 16-token tiles of two pages each), all of the same unit
    int npg;
    if constexpr (BS8)
      npg = min(4, min(n_w - i, cc.Ps - cc.pi));
    else
      npg = (bs == 16 && i + 1 < n_w && cc.pi + 1 < cc.Ps) ? 2 : 1;
    auto issue_after = [&]() {
      if constexpr (BS8) {
        // a pair's stage is free once both its pages are consumed
        while (n_issued < n_w && i + npg >= n_issued + 2 - 2 * nstage) issue_pair();
      } else {
        for (int k = 0; k < npg && n_issued < n_w; ++k) issue_next();
      }
    };
    // Block size 8, the common case: four whole pages, i.e. two whole pairs
    // (16 tokens each) in consecutive stages, taken without the per-page
    // bookkeeping of the general path below (which handles a pair split by
    // the range, short or absent pages and unit ends).
    bool pairs_whole = false;
    if constexpr (BS8) {
      if (npg == 4 && (i & 1) == 0 && (cc.pi + 4) * 8 <= L) {
        const bool wrap1 = cst + 1 == nstage;
        const int st1 = wrap1 ? 0 : cst + 1;
        const int2 ph0 = *reinterpret_cast<const int2*>(stage_phys + 2 * cst);
        const int2 ph1 = *reinterpret_cast<const int2*>(stage_phys + 2 * st1);
        if ((ph0.x | ph0.y | ph1.x | ph1.y) >= 0) {  // all four pages in the pool
          pairs_whole = true;
          if (!wait_stage(cst, cph) || !wait_stage(st1, wrap1 ? cph ^ 1u : cph)) {
            failed = true;
            break;
          }
          const char* s0 = stages + cst * p.stage_bytes;
          const char* s1 = stages + st1 * p.stage_bytes;
          load_tile8<FMT, D, NG>(R, 0, s0, s0 + slot_bytes, 16, pool, lane);
          load_tile8<FMT, D, NG>(R, 1, s1, s1 + slot_bytes, 16, pool, lane);
          compute_pair<FMT, D, NG, true>(R, lane, qb, ql, csc, m, l, E, o);
        }
      }
    }
    if (pairs_whole) {
      // done above
    } else if constexpr (BS8) {
      bool ok = true;
      const char* pg[4];
      int rp[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pg[k] = nullptr;
        rp[k] = 0;
        if (k < npg && ok) {
          // page q = i + k is slot q % 2 of pair q / 2; cst is the stage of
          // pair i / 2 (nstage >= 3 pairs for block size 8); a slot-1 page's
          // pair was waited with its slot 0, in this update or the one before
          const int q = i + k, po = (q >> 1) - (i >> 1);
          const bool wrap = cst + po >= nstage;
          const int st = wrap ? cst + po - nstage : cst + po;
          if ((q & 1) == 0) ok = wait_stage(st, wrap ? cph ^ 1u : cph);
          pg[k] = stages + st * p.stage_bytes + (q & 1) * slot_bytes;
          rp[k] = stage_phys[2 * st + (q & 1)] >= 0 ? max(0, min(8, L - (cc.pi + k) * 8)) : 0;
        }
      }
      if (!ok) {
        failed = true;
        break;
      }
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const char* A = pg[2 * t];
        const char* B = pg[2 * t + 1];
        int ra = rp[2 * t], rb = rp[2 * t + 1];
        if (ra == 0) {  // an absent page contributes nothing: the tile is page B alone
          A = B;
          ra = rb;
          B = nullptr;
          rb = 0;
        }
        if (ra < 8) {  // a short first page ends its unit: no second page
          B = nullptr;
          rb = 0;
        }
        if (A == nullptr) A = pg[0];  // an empty tile reads any staged page, all rows masked
        load_tile8<FMT, D, NG>(R, t, A, B, ra + rb, pool, lane);
      }
      compute_pair<FMT, D, NG, true>(R, lane, qb, ql, csc, m, l, E, o);
    } else {
      const bool two = npg == 2;
      const bool wrap1 = cst + 1 == nstage;
      const int st0 = cst, st1 = wrap1 ? 0 : cst + 1;
      if (!wait_stage(st0, cph) || (two && !wait_stage(st1, wrap1 ? cph ^ 1u : cph))) {
        failed = true;
        break;
      }
      if (two) {
        const int r0 = stage_phys[st0] >= 0 ? min(16, L - cc.pi * 16) : 0;
        const int r1 = stage_phys[st1] >= 0 ? min(16, L - (cc.pi + 1) * 16) : 0;
        // an absent page (rows = 0) contributes nothing; keep the valid one in tile 0
        const int sA = r0 > 0 ? st0 : st1;
        load_tile<FMT, D, NG>(R, 0, stages + sA * p.stage_bytes, 0, r0 > 0 ? r0 : r1, pool, lane);
        load_tile<FMT, D, NG>(R, 1, stages + st1 * p.stage_bytes, 0, r0 > 0 ? r1 : 0, pool, lane);
        compute_pair<FMT, D, NG>(R, lane, qb, ql, csc, m, l, E, o);
      } else {
        const char* stage = stages + st0 * p.stage_bytes;
        const int nvalid = stage_phys[st0] >= 0 ? min(bs, L - cc.pi * bs) : 0;
        const int nsub = (nvalid + 15) >> 4;
        for (int sp = 0; sp < nsub; sp += 2) {
          const int rA = min(16, nvalid - sp * 16);
          const int rB = sp + 1 < nsub ? min(16, nvalid - (sp + 1) * 16) : 0;
          load_tile<FMT, D, NG>(R, 0, stage, sp, rA, pool, lane);
          load_tile<FMT, D, NG>(R, 1, stage, sp + 1 < nsub ? sp + 1 : sp, rB, pool, lane);
          compute_pair<FMT, D, NG>(R, lane, qb, ql, csc, m, l, E, o);
        }
      }
    }
    // every lane is done with the stage(s): hand them back to the copy engine
    __syncwarp();
    issue_after();
    // advance the consumer; close the unit at its last page or at the range end
    {
      const int nst = BS8 ? ((i + npg) >> 1) - (i >> 1) : npg;  // stages passed
      for (int k = 0; k < nst; ++k)
        if (++cst == nstage) {
          cst = 0;
          cph ^= 1u;
        }
    }
    i += npg;
    const Cursor done = cc;
    const int end_pi = cc.pi + npg;
    for (int k = 0; k < npg; ++k) advance(cc);
    if (end_pi == done.Ps || i == n_w) {
      finish_unit(done, end_pi);
      if (i < n_w) start_unit();
    }
  }
  if (failed) {
    // A wait ran out: flag it, mark this warp's partial rows empty (m = -inf,
    // l = 0) so that the merge does not fold in an earlier call's leftovers,
    // then wait (bounded again) for this warp's copies still in flight so that
    // none lands after the CTA has exited.
    if (lane == 0) set_error(pool.err, ERR_TIMEOUT);
    if (lane < 2 * kPartRows) {
      float* r = p.part + ((int64_t)gw * 2 * kPartRows + lane) * (D + 2);
      r[0] = kNegInf;
      r[1] = 0.f;
    }
    int st = cst;
    uint32_t ph = cph;
    // stages issued and not yet consumed (block size 8: pairs, from the one
    // holding page i)
    const int nst = BS8 ? ((n_issued + 1) >> 1) - (i >> 1) : n_issued - i;
    for (int k = 0; k < nst; ++k) {
      wait_stage(st, ph);
      if (++st == nstage) {
        st = 0;
        ph ^= 1u;
      }
    }
  }
}

// Log-sum-exp merge of the units that the decode kernel's warp ranges cut:
// unit u's pieces are the partials of warps wf..wl (slot 1 of wf when its range
// started before the unit, slot 0 otherwise).  Launched as a programmatic
// dependent of the decode kernel: griddepcontrol.wait returns once the decode
// grid has completed and its writes are visible.  CH: pieces loaded together
// (one round trip), 8 or 16 as the plan chooses.
template <int D, int CH>
__global__ void __launch_bounds__(kMergeThreads) kvq_merge_kernel(const DecodeParams p) {
  // A kernel launched after this one as a programmatic dependent (the next
  // decode-step append) may launch now; it waits for this grid's completion
  // before touching anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float kNegInf = __int_as_float(0xff800000u);
  constexpr int NW = kMergeThreads / 32;
  constexpr int NE = D / 32;   // output elements per lane
  const int lane = threadIdx.x & 31;
  const int U = p.pool.Hkv * p.n_ht;
  const int* PS = p.ps;
  const int Ttot = __ldcg(PS + p.S);
  const int nwarps = p.grid * kDecodeWarps;
  const int ppw = p.ppw_fixed > 0 ? p.ppw_fixed : (Ttot + nwarps - 1) / nwarps;
  if (ppw <= 0) return;
  // one task per (unit, Q-head row of its tile) that a Q head fills: rows
  // 0 .. min(8, G) - 1 of each tile (fewer in a ragged last tile); one warp
  // per task
  const int rpu = min(kPartRows, p.G);
  const int64_t ntasks = (int64_t)p.S * U * rpu;
  for (int64_t task = (int64_t)blockIdx.x * NW + (threadIdx.x >> 5); task < ntasks;
       task += (int64_t)gridDim.x * NW) {
    const int64_t u = task / rpu;
    const int rr = (int)(task % rpu);
    const int s = (int)(u / U), lu = (int)(u % U);
    const int ht = lu % p.n_ht;
    if (rr >= min(8, p.G - 8 * ht)) continue;
    const int ps0 = __ldcg(PS + s), ps1 = __ldcg(PS + s + 1);
    const int Ps = (ps1 - ps0) / U;
    if (Ps == 0) continue;
    const int U0 = ps0 + lu * Ps;
    const int wf = U0 / ppw, wl = (U0 + Ps - 1) / ppw;
    if (wf == wl) continue;  // written directly by its warp
    const int n_u = wl - wf + 1;
    const int h = lu / p.n_ht;
    const int64_t orow = (int64_t)s * p.Hq + h * p.G + 8 * ht + rr;
    float M = kNegInf, Lsum = 0.f, acc[NE];
#pragma unroll
    for (int i = 0; i < NE; ++i) acc[i] = 0.f;
    if (p.pre != nullptr) {  // cascade: the prefix partial is one more piece
      const float* pr = p.pre + orow * (D + 2);
      M = pr[0];
      Lsum = pr[1];
#pragma unroll
      for (int i = 0; i < NE; ++i) acc[i] = pr[2 + lane + 32 * i];
    }
    for (int k0 = 0; k0 < n_u; k0 += CH) {
      float mk[CH], lk[CH], ok[CH][NE];
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int k = k0 + c;
        if (k < n_u) {
          const int w = wf + k;
          const int sl = (k == 0 && (int64_t)w * ppw < U0) ? 1 : 0;
          const float* pr = p.part + (((int64_t)w * 2 + sl) * kPartRows + rr) * (D + 2);
          mk[c] = __ldcg(pr);
          lk[c] = __ldcg(pr + 1);
#pragma unroll
          for (int i = 0; i < NE; ++i) ok[c][i] = __ldcg(pr + 2 + lane + 32 * i);
        } else {
          mk[c] = kNegInf;
          lk[c] = 0.f;
#pragma unroll
          for (int i = 0; i < NE; ++i) ok[c][i] = 0.f;
        }
      }
      float cm = M;
#pragma unroll
      for (int c = 0; c < CH; ++c) cm = fmaxf(cm, mk[c]);
      if (cm == kNegInf) continue;
      const float fo = M == kNegInf ? 0.f : fast_exp2(M - cm);
      Lsum *= fo;
#pragma unroll
      for (int i = 0; i < NE; ++i) acc[i] *= fo;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const float wgt = mk[c] == kNegInf ? 0.f : fast_exp2(mk[c] - cm);
        Lsum = fmaf(wgt, lk[c], Lsum);
#pragma unroll
        for (int i = 0; i < NE; ++i) acc[i] = fmaf(wgt, ok[c][i], acc[i]);
      }
      M = cm;
    }
    float* dst = p.out + (int64_t)s * p.out_stride + (int64_t)(h * p.G + 8 * ht + rr) * D;
#pragma unroll
    for (int i = 0; i < NE; ++i) dst[lane + 32 * i] = Lsum > 0.f ? acc[i] / Lsum : 0.f;
  }
}

struct DecodeLaunch {
  DecodeParams p;
  dim3 grid;
  unsigned merge_grid;
  int merge_chunk;  // kvq_merge_kernel's CH
  int smem;
  cudaStream_t st;
  bool dependent;  // launch as a programmatic dependent of the previous kernel
};

template <int FMT, int D, int NG, bool BS8 = false>
cudaError_t run_decode(const DecodeLaunch& l) {
  cudaError_t e = allow_big_smem<kvq_decode_kernel<FMT, D, NG, BS8>>();
  if (e != cudaSuccess) return e;
  {
    cudaLaunchConfig_t dc = {};
    dc.gridDim = l.grid;
    dc.blockDim = dim3(kDecodeThreads);
    dc.dynamicSmemBytes = l.smem;
    dc.stream = l.st;
    cudaLaunchAttribute da[1];
    da[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    da[0].val.programmaticStreamSerializationAllowed = 1;
    dc.attrs = da;
    dc.numAttrs = l.dependent ? 1 : 0;
    e = phase_mark(l.st, cudaLaunchKernelEx(&dc, kvq_decode_kernel<FMT, D, NG, BS8>, l.p));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(l.merge_grid);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = l.st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return phase_mark(l.st, l.merge_chunk == 16
                              ? cudaLaunchKernelEx(&cfg, kvq_merge_kernel<D, 16>, l.p)
                              : cudaLaunchKernelEx(&cfg, kvq_merge_kernel<D, 8>, l.p));
}

template <int FMT, bool BS8 = false>
cudaError_t run_decode_d(const DecodeLaunch& l) {
  switch (l.p.pool.D) {
    case 64: return run_decode<FMT, 64, 1, BS8>(l);
    case 128: return run_decode<FMT, 128, 1, BS8>(l);
    default: return cudaErrorInvalidValue;
  }
}

// Per-group formats: NG = head_dim / group scale groups per head.
template <int FMT, bool BS8 = false>
cudaError_t run_decode_group(const DecodeLaunch& l) {
  const int D = l.p.pool.D, ng = l.p.pool.ng;
  if (D == 64) {
    switch (ng) {
      case 1: return run_decode<FMT, 64, 1, BS8>(l);
      case 2: return run_decode<FMT, 64, 2, BS8>(l);
      case 4: return run_decode<FMT, 64, 4, BS8>(l);
    }
  } else if (D == 128) {
    switch (ng) {
      case 1: return run_decode<FMT, 128, 1, BS8>(l);
      case 2: return run_decode<FMT, 128, 2, BS8>(l);
      case 4: return run_decode<FMT, 128, 4, BS8>(l);
      case 8: return run_decode<FMT, 128, 8, BS8>(l);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
