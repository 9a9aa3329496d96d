// kvq_decode_impl.cuh -- paged decode attention over a quantized KV pool.
//
// Method ("KV Cache优化实战：大模型推理显存占用与加速方案详解",
// 0539edu.com/news/5800990): decode step attends the new Q over all cached K/V
// (§1.1); Q heads are grouped and each group shares one K/V head (§2.1);
// the cache lives in fixed-size physical blocks reached through a block
// table (§2.2); K/V are INT8/FP8 codes with per-token, per-channel or
// per-group scales, or FP16 (§2.3, §3.3); dequantization is fused into the
// attention kernel instead of running as a separate pass (§4.3).
//
// GB300 design (sm_103a):
//  * grid = (split, kv_head x head_tile, sequence); 4 warps per CTA.  A split
//    is a contiguous run of a sequence's blocks (split-K over the context);
//    warps take the split's blocks round-robin.
//  * Each warp streams its blocks through NSTAGE shared-memory stages: lane 0
//    looks the block up in the block table and issues one bulk (TMA) copy of
//    the (block, kv head) page -- K codes, V codes and their group scales are
//    contiguous -- completing on an mbarrier.  Waits are bounded; a wait that
//    runs out sets an error bit instead of hanging.
//  * The Q heads of the kv head (up to 8 per head tile) share every loaded
//    page: Q.K^T and P.V run on the tensor cores as mma.m16n8k16 with the
//    heads on the n dimension.  Codes are exact in fp16 (int8 in [-127,127],
//    every e4m3 value), so dequantization is a scale applied outside the
//    contraction: per-token / per-group K scales multiply the fp32 scores,
//    per-token / per-group V scales are folded into the softmax weights, and
//    per-channel scales fold into q (K) and the output columns (V).
//  * fp32 operands that enter a tensor-core product (softmax weights times V
//    scale; q times a per-channel K scale) are split into an fp16 high part and
//    an fp16 low part (two MMAs), after scaling by a power of two that keeps
//    them away from fp16 overflow and underflow; that power of two is undone
//    exactly at the end.
//  * Online softmax in base 2 (scores pre-multiplied by log2 e); the warps of a
//    CTA merge through shared memory; splits merge by log-sum-exp in a second
//    small kernel.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "kvq_common.cuh"

namespace kvq {

constexpr int kDecodeWarps = 4;
constexpr int kDecodeThreads = kDecodeWarps * 32;
constexpr int kWaitTries = 4000;  // x 1 ms suspend hint per try: ~4 s upper bound

struct DecodeParams {
  PoolView pool;
  const __half* q;     // [S][Hq][D]
  const int* table;    // [S][max_blocks]
  const int* lens;     // [S]
  float* out;          // [S][Hq][D]
  float* part_o;       // [S][Hq][nsplit][D]
  float* part_ml;      // [S][Hq][nsplit][2]
  int S, Hq, G, n_ht, max_blocks, max_ctx;
  int pps;             // blocks per split
  int nsplit;
  int nstage_log2;
  int stage_bytes;
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
  static constexpr bool group_scales = FMT == FMT_INT8_GROUP;
  static constexpr bool token_scales = FMT == FMT_INT8_TOKEN || FMT == FMT_FP8_TOKEN;
  static constexpr bool row_scales = group_scales || token_scales;  // per-(token[,group]) K/V scales
  static constexpr bool channel = FMT == FMT_INT8_CHANNEL;
  static constexpr bool maybe_nan = FMT == FMT_FP16 || FMT == FMT_FP8_TOKEN;
};

// Word w (4 elements) of a lane's sub-tile -> (lo, hi) fp16x2 pairs.
template <int FMT>
__device__ __forceinline__ void word_to_h2(const uint32_t* words, int w, uint32_t& lo, uint32_t& hi) {
  if constexpr (FMT == FMT_FP16) {
    lo = words[2 * w];
    hi = words[2 * w + 1];
  } else if constexpr (FMT == FMT_FP8_TOKEN) {
    e4m3x4_to_h2x2(words[w], lo, hi);
  } else {
    i8x4_to_h2x2(words[w], lo, hi);
  }
}

// Copy a lane's share of a sub-tile from shared memory: esize*D/2 bytes.
template <int FMT, int D>
__device__ __forceinline__ void load_lane_words(const char* tile, int lane, uint32_t* words) {
  constexpr int esize = FMT == FMT_FP16 ? 2 : 1;
  constexpr int chunks = D * esize / 32;
#pragma unroll
  for (int c = 0; c < chunks; ++c) {
    uint4 v = *reinterpret_cast<const uint4*>(tile + c * 512 + lane * 16);
    words[4 * c + 0] = v.x;
    words[4 * c + 1] = v.y;
    words[4 * c + 2] = v.z;
    words[4 * c + 3] = v.w;
  }
}

// A 16-token sub-tile in shared memory: K and V codes in fragment order and the
// per-row K / V scales (group or token formats); rows = valid tokens (0..16).
struct TileRef {
  const char* k;
  const char* v;
  const float* ks;
  const float* vs;
  int rows;
};

// One online-softmax update over two sub-tiles (32 tokens) for the up-to-8 Q
// heads of a kv head.  Lane (g = lane/4, j = lane%4) holds scores of tokens
// g and g+8 of each tile for heads 2j and 2j+1, and O^T rows 16mt+g, 16mt+g+8
// for the same two heads.  B may be an empty tile (rows = 0; pointers valid).
template <int FMT, int D, int NG>
__device__ __forceinline__ void process_pair(const TileRef& A, const TileRef& B, int lane,
                                             const uint32_t (&qb)[D / 16][2],
                                             const uint32_t (&ql)[FmtTraits<FMT>::channel ? D / 16 : 1][2],
                                             float csc, float (&m)[2], float (&l)[2], int& E,
                                             float (&o)[D / 16][4]) {
  using T = FmtTraits<FMT>;
  constexpr int KS = D / 16;
  constexpr int NU32 = (FMT == FMT_FP16 ? 2 : 1) * D / 8;
  constexpr int KPG = KS / NG;
  constexpr int SUB = KPG >= 2 ? 2 : 1;  // independent accumulators per scale group
  const float kNegInf = __int_as_float(0xff800000u);
  const int g = lane >> 2, j = lane & 3;
  const TileRef* tl[2] = {&A, &B};

  // ---- scores: S[t][r] = sum_d code_K[t][d] q'[r][d], per scale group
  float z[2][4];
  {
    uint32_t kw[2][NU32];
    load_lane_words<FMT, D>(A.k, lane, kw[0]);
    load_lane_words<FMT, D>(B.k, lane, kw[1]);
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
        word_to_h2<FMT>(kw[t], kk, a0, a2);       // row g   : channels e=0,1 | e=2,3
        word_to_h2<FMT>(kw[t], KS + kk, a1, a3);  // row g+8
        mma_16816(acc[t][ai], a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        if constexpr (T::channel) mma_16816(acc[t][ai], a0, a1, a2, a3, ql[kk][0], ql[kk][1]);
      }
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const TileRef& tr = *tl[t];
      float zz[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        float s4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) s4[e] = SUB == 2 ? acc[t][gi * SUB][e] + acc[t][gi * SUB + 1][e]
                                                     : acc[t][gi * SUB][e];
        float sA = csc, sB = csc;
        if constexpr (T::group_scales) {
          sA *= tr.ks[g * NG + gi];
          sB *= tr.ks[(g + 8) * NG + gi];
        } else if constexpr (T::token_scales) {
          sA *= tr.ks[g];
          sB *= tr.ks[g + 8];
        }
        zz[0] = fmaf(s4[0], sA, zz[0]);
        zz[1] = fmaf(s4[1], sA, zz[1]);
        zz[2] = fmaf(s4[2], sB, zz[2]);
        zz[3] = fmaf(s4[3], sB, zz[3]);
      }
      const bool vA = g < tr.rows, vB = g + 8 < tr.rows;
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
      constexpr int NS = T::group_scales ? NG : 1;
      float vmax = 0.f;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const TileRef& tr = *tl[t];
#pragma unroll
        for (int gi = 0; gi < NS; ++gi) {
          if (g < tr.rows) vmax = fmaxf(vmax, tr.vs[g * NS + gi]);
          if (g + 8 < tr.rows) vmax = fmaxf(vmax, tr.vs[(g + 8) * NS + gi]);
        }
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
      const TileRef& tr = *tl[t];
      const bool vA = g < tr.rows, vB = g + 8 < tr.rows;
#pragma unroll
      for (int gi = 0; gi < NB; ++gi) {
        float fA = sc, fB = sc;
        if constexpr (T::group_scales) {
          fA *= tr.vs[g * NG + gi];
          fB *= tr.vs[(g + 8) * NG + gi];
        } else if constexpr (T::token_scales) {
          fA *= tr.vs[g];
          fB *= tr.vs[g + 8];
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
    uint32_t vw[2][NU32];
    load_lane_words<FMT, D>(A.v, lane, vw[0]);
    load_lane_words<FMT, D>(B.v, lane, vw[1]);
    if constexpr (T::maybe_nan) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int rows = tl[t]->rows;
        if (rows < 16) {
          // tokens of this lane's V bytes: 2j, 2j+1, 2j+8, 2j+9; zero the ones
          // past the context so that 0 * NaN cannot reach the sum
          const int t0 = 2 * j;
          if constexpr (FMT == FMT_FP16) {
            const uint32_t mlo = (t0 < rows ? 0xFFFFu : 0u) | (t0 + 1 < rows ? 0xFFFF0000u : 0u);
            const uint32_t mhi = (t0 + 8 < rows ? 0xFFFFu : 0u) | (t0 + 9 < rows ? 0xFFFF0000u : 0u);
#pragma unroll
            for (int w = 0; w < NU32 / 2; ++w) {
              vw[t][2 * w] &= mlo;
              vw[t][2 * w + 1] &= mhi;
            }
          } else {
            const uint32_t msk = (t0 < rows ? 0xFFu : 0u) | (t0 + 1 < rows ? 0xFF00u : 0u) |
                                 (t0 + 8 < rows ? 0xFF0000u : 0u) |
                                 (t0 + 9 < rows ? 0xFF000000u : 0u);
#pragma unroll
            for (int w = 0; w < NU32; ++w) vw[t][w] &= msk;
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
        word_to_h2<FMT>(vw[t], 2 * mt, a0, a2);      // channel 16mt+g   : tokens 2j,2j+1 | 2j+8,2j+9
        word_to_h2<FMT>(vw[t], 2 * mt + 1, a1, a3);  // channel 16mt+g+8
        mma_16816(o[mt], a0, a1, a2, a3, bh0[t][gi], bh1[t][gi]);
        mma_16816(o[mt], a0, a1, a2, a3, bl0[t][gi], bl1[t][gi]);
      }
    }
  }
}

template <int FMT, int D, int NG>
__global__ void __launch_bounds__(kDecodeThreads)
    kvq_decode_kernel(const DecodeParams p) {
  using T = FmtTraits<FMT>;
  constexpr int KS = D / 16;                  // k-steps of Q.K = m-tiles of P.V
  constexpr int NU32 = (FMT == FMT_FP16 ? 2 : 1) * D / 8;  // u32 per lane per sub-tile
  constexpr int KPG = KS / NG;                // k-steps per scale group
  const float kNegInf = __int_as_float(0xff800000u);

  extern __shared__ __align__(128) char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, j = lane & 3;
  const int split = blockIdx.x;
  const int h = blockIdx.y / p.n_ht, ht = blockIdx.y % p.n_ht;
  const int s = blockIdx.z;
  const PoolView& pool = p.pool;
  const int bs = pool.bs;
  const int nstage = 1 << p.nstage_log2;

  int L = p.lens[s];
  if (L > p.max_ctx) {
    if (threadIdx.x == 0) set_error(pool.err, ERR_RANGE);
    L = p.max_ctx;
  }
  if (L < 0) L = 0;
  const int npages = (L + bs - 1) / bs;
  const int pg0 = split * p.pps;
  const int Gt = min(8, p.G - 8 * ht);  // q heads handled by this CTA
  if (pg0 >= npages && !(split == 0 && p.nsplit == 1)) return;  // empty split: merge skips it
  const int pg1 = min(npages, pg0 + p.pps);

  char* stages = smem + warp * nstage * p.stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDecodeWarps * nstage * p.stage_bytes) +
                   warp * nstage;
  int* stage_phys = reinterpret_cast<int*>(
                        reinterpret_cast<uint64_t*>(smem + kDecodeWarps * nstage * p.stage_bytes) +
                        kDecodeWarps * nstage) +
                    warp * nstage;

  const int span = pg1 - pg0;
  const int n_w = span > warp ? (span - warp + kDecodeWarps - 1) / kDecodeWarps : 0;

  // ---- Q fragments: head n = g of this tile, channels 16kk + 4j .. +3.
  uint32_t qb[KS][2];
  uint32_t ql[T::channel ? KS : 1][2];
  float csc = p.sm_scale_log2;
  {
    const bool hv = g < Gt;
    const int hq = h * p.G + 8 * ht + (hv ? g : 0);
    const __half* qp = p.q + ((int64_t)s * p.Hq + hq) * D;
    if constexpr (!T::channel) {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint2 v = hv ? *reinterpret_cast<const uint2*>(qp + 16 * kk + 4 * j) : make_uint2(0, 0);
        qb[kk][0] = v.x;
        qb[kk][1] = v.y;
      }
    } else {
      // q' = q * s_K[h][d] (fp32), scaled by 2^Eq so that max|q'| lies in
      // [2^13, 2^14), then split into fp16 hi + lo.
      const float* ksc = pool.chan_scales + (int64_t)h * D;
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

  // ---- pipeline set-up
  if (lane == 0) {
    for (int st = 0; st < nstage; ++st) mbar_init(&bars[st], 1);
    fence_barrier_init();
  }
  __syncwarp();

  const int64_t trow = (int64_t)s * p.max_blocks;
  int tbl = (lane < n_w) ? p.table[trow + pg0 + warp + lane * kDecodeWarps] : 0;
  const uint32_t page_tx = pool.page_bytes + (T::token_scales ? 2 * bs * 4 : 0);

  auto issue = [&](int i) {
    if ((i & 31) == 0 && i > 0)
      tbl = (i + lane < n_w) ? p.table[trow + pg0 + warp + (i + lane) * kDecodeWarps] : 0;
    const int phys = __shfl_sync(0xffffffffu, tbl, i & 31);
    if (lane == 0) {
      const int st = i & (nstage - 1);
      char* dst = stages + st * p.stage_bytes;
      const bool ok = phys >= 0 && (int64_t)phys < pool.num_blocks;
      stage_phys[st] = ok ? phys : -1;
      if (ok) {
        mbar_arrive_expect_tx(&bars[st], page_tx);
        bulk_g2s(dst, pool.pages + ((int64_t)phys * pool.Hkv + h) * pool.page_bytes,
                 pool.page_bytes, &bars[st]);
        if constexpr (T::token_scales)
          bulk_g2s(dst + pool.page_bytes, pool.tok_scales + (int64_t)phys * 2 * bs, 2 * bs * 4,
                   &bars[st]);
      } else {
        set_error(pool.err, ERR_RANGE);
        mbar_arrive(&bars[st]);
      }
    }
  };

  const int npre = min(n_w, nstage);
  for (int i = 0; i < npre; ++i) issue(i);

  // ---- per-warp online-softmax state (heads 2j, 2j+1 of the tile)
  float m[2] = {kNegInf, kNegInf};
  float l[2] = {0.f, 0.f};
  int E = (T::row_scales) ? 100 : 14;  // power-of-two prescale of the P.V operand
  float o[KS][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  // Bounded wait for stage i; false (and the timeout bit set) if it gave up.
  auto wait_stage = [&](int i) -> bool {
    const int st = i & (nstage - 1);
    const uint32_t parity = (i >> p.nstage_log2) & 1;
    bool ok = false;
    for (int tries = 0; tries < kWaitTries && !ok; ++tries) ok = mbar_try_wait(&bars[st], parity);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) set_error(pool.err, ERR_TIMEOUT);
      return false;
    }
    return true;
  };
  // Sub-tile `sub` of the warp's i-th page as a tile reference (rows = 0 when
  // the page is absent, out of range or the sub-tile lies past the context).
  auto tile_of = [&](int i, int sub) -> TileRef {
    TileRef t;
    const int st = i & (nstage - 1);
    const char* stage = stages + st * p.stage_bytes;
    t.k = stage + sub * pool.sub_bytes;
    t.v = stage + pool.code_bytes + sub * pool.sub_bytes;
    t.ks = nullptr;
    t.vs = nullptr;
    if constexpr (T::group_scales) {
      t.ks = reinterpret_cast<const float*>(stage + 2 * pool.code_bytes) + sub * 16 * NG;
      t.vs = t.ks + bs * NG;
    } else if constexpr (T::token_scales) {
      t.ks = reinterpret_cast<const float*>(stage + pool.page_bytes) + sub * 16;
      t.vs = t.ks + bs;
    }
    const int page = pg0 + warp + i * kDecodeWarps;
    const int nvalid = min(bs, L - page * bs) - sub * 16;
    t.rows = (i < n_w && stage_phys[st] >= 0) ? max(0, min(16, nvalid)) : 0;
    return t;
  };

  const bool pair_pages = bs == 16;  // one 16-token sub-tile per page: pages go in pairs
  for (int i = 0; i < n_w; i += pair_pages ? 2 : 1) {
    const bool two = pair_pages && i + 1 < n_w;
    if (!wait_stage(i) || (two && !wait_stage(i + 1))) break;
    if (pair_pages) {
      TileRef A = tile_of(i, 0);
      TileRef B = two ? tile_of(i + 1, 0) : A;
      if (!two) B.rows = 0;
      if (A.rows == 0 && B.rows > 0) { TileRef t = A; A = B; B = t; }
      if (B.rows == 0) { const int r = B.rows; B = A; B.rows = r; }
      process_pair<FMT, D, NG>(A, B, lane, qb, ql, csc, m, l, E, o);
    } else {
      const int page = pg0 + warp + i * kDecodeWarps;
      const int nsub = (min(bs, L - page * bs) + 15) >> 4;
      for (int sp = 0; sp < nsub; sp += 2) {
        TileRef A = tile_of(i, sp);
        TileRef B = tile_of(i, sp + 1 < nsub ? sp + 1 : sp);
        if (sp + 1 >= nsub) B.rows = 0;
        if (A.rows == 0) break;  // page skipped (out-of-range block id)
        process_pair<FMT, D, NG>(A, B, lane, qb, ql, csc, m, l, E, o);
      }
    }
    __syncwarp();
    if (i + nstage < n_w) issue(i + nstage);
    if (two && i + 1 + nstage < n_w) issue(i + 1 + nstage);
  }

  // ---- per-warp totals, then merge the warps through shared memory
  l[0] = warp_sum_over_rows(l[0]);
  l[1] = warp_sum_over_rows(l[1]);
  __syncthreads();  // every warp is done with its stages
  constexpr int OST = D + 4;  // padded row stride (conflict-free stores)
  float* Os = reinterpret_cast<float*>(smem);            // [W][8][OST]
  float* Ms = Os + kDecodeWarps * 8 * OST;               // [W][8]
  float* Ls = Ms + kDecodeWarps * 8;                     // [W][8]
  int* Es = reinterpret_cast<int*>(Ls + kDecodeWarps * 8);  // [W]
  {
    float* ow = Os + warp * 8 * OST;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const int d0 = 16 * mt + g;
      ow[(2 * j) * OST + d0] = o[mt][0];
      ow[(2 * j + 1) * OST + d0] = o[mt][1];
      ow[(2 * j) * OST + d0 + 8] = o[mt][2];
      ow[(2 * j + 1) * OST + d0 + 8] = o[mt][3];
    }
    if (g == 0) {
      Ms[warp * 8 + 2 * j] = m[0];
      Ms[warp * 8 + 2 * j + 1] = m[1];
      Ls[warp * 8 + 2 * j] = l[0];
      Ls[warp * 8 + 2 * j + 1] = l[1];
    }
    if (lane == 0) Es[warp] = E;
  }
  __syncthreads();
  const bool direct = p.nsplit == 1;
  for (int idx = threadIdx.x; idx < Gt * D; idx += kDecodeThreads) {
    const int r = idx / D, d = idx - r * D;
    float mstar = kNegInf;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) mstar = fmaxf(mstar, Ms[w * 8 + r]);
    float acc = 0.f, wsum = 0.f;
    if (mstar != kNegInf) {
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) {
        const float mw = Ms[w * 8 + r];
        if (mw == kNegInf) continue;
        const float f = fast_exp2(mw - mstar);
        wsum = fmaf(f, Ls[w * 8 + r], wsum);
        acc = fmaf(f * pow2f(-Es[w]), Os[(w * 8 + r) * OST + d], acc);
      }
      if constexpr (T::channel) acc *= pool.chan_scales[((int64_t)pool.Hkv + h) * D + d];
    }
    const int hq = h * p.G + 8 * ht + r;
    const int64_t row = (int64_t)s * p.Hq + hq;
    if (direct) {
      p.out[row * D + d] = wsum > 0.f ? acc / wsum : 0.f;
    } else {
      p.part_o[(row * p.nsplit + split) * D + d] = acc;
      if (d == 0) {
        p.part_ml[(row * p.nsplit + split) * 2 + 0] = mstar;
        p.part_ml[(row * p.nsplit + split) * 2 + 1] = wsum;
      }
    }
  }
}

// Log-sum-exp merge of the split partials: one CTA of D threads per (seq, q head).
template <int D>
__global__ void __launch_bounds__(D) kvq_merge_kernel(const DecodeParams p) {
  const float kNegInf = __int_as_float(0xff800000u);
  const int row = blockIdx.x;  // s * Hq + hq
  const int s = row / p.Hq;
  const int d = threadIdx.x;
  int L = min(max(p.lens[s], 0), p.max_ctx);
  const int npages = (L + p.pool.bs - 1) / p.pool.bs;
  const int n = (npages + p.pps - 1) / p.pps;
  const float* ml = p.part_ml + (int64_t)row * p.nsplit * 2;
  const float* po = p.part_o + (int64_t)row * p.nsplit * D;
  float mstar = kNegInf;
  for (int i = 0; i < n; ++i) mstar = fmaxf(mstar, ml[2 * i]);
  float acc = 0.f, wsum = 0.f;
  if (mstar != kNegInf) {
    for (int i = 0; i < n; ++i) {
      const float mi = ml[2 * i];
      if (mi == kNegInf) continue;
      const float f = fast_exp2(mi - mstar);
      wsum = fmaf(f, ml[2 * i + 1], wsum);
      acc = fmaf(f, po[(int64_t)i * D + d], acc);
    }
  }
  p.out[(int64_t)row * D + d] = wsum > 0.f ? acc / wsum : 0.f;
}

}  // namespace kvq

namespace kvq {

struct DecodeLaunch {
  DecodeParams p;
  dim3 grid;
  int smem;
  cudaStream_t st;
};

constexpr int kMaxDevices = 64;

template <int FMT, int D, int NG>
cudaError_t run_decode(const DecodeLaunch& l) {
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDevices && !attr_set[dev]) {
    e = cudaFuncSetAttribute(kvq_decode_kernel<FMT, D, NG>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  kvq_decode_kernel<FMT, D, NG><<<l.grid, kDecodeThreads, l.smem, l.st>>>(l.p);
  if (l.p.nsplit > 1)
    kvq_merge_kernel<D><<<static_cast<unsigned>(l.p.S * l.p.Hq), D, 0, l.st>>>(l.p);
  return cudaGetLastError();
}

template <int FMT>
cudaError_t run_decode_d(const DecodeLaunch& l) {
  switch (l.p.pool.D) {
    case 64: return run_decode<FMT, 64, 1>(l);
    case 128: return run_decode<FMT, 128, 1>(l);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
