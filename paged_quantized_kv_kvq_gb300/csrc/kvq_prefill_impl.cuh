// kvq_prefill_impl.cuh -- prefill / chunked-prefill attention over a
// quantized paged KV pool.
//
// Method ("KV Cache优化实战：大模型推理显存占用与加速方案详解",
// 0539edu.com/news/5800990, §1.1): the prompt's tokens are processed together,
// each attending causally to the tokens up to itself; a long prompt may be
// processed in chunks, each chunk attending to the cache the earlier chunks
// wrote.  Query token i of a chunk of n tokens of a sequence whose cache holds
// L tokens (the chunk included) sits at position L - n + i.
//
// GB300 design: a CTA takes one (sequence, kv head) and 64 Q rows -- 16 query
// tokens x 4 Q heads of the group for GQA 4:1 -- 16 rows per warp.  The CTA
// streams the sequence's pages once through bulk-copy stages; for each 16-token
// sub-tile its 128 threads turn the codes into exact fp16 values once, in
// shared memory (K row-major, V channel-major, rows padded so that ldmatrix is
// conflict-free), and every warp then runs Q.K^T and P.V for its rows on
// mma.m16n8k16 with B fragments from ldmatrix.  Scales stay outside the
// contraction (K scales on the scores, V scales folded into the weights,
// per-channel scales into q and the output), as in the decode kernel.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "kvq_decode_impl.cuh"

namespace kvq {

constexpr int kPfWarps = 4;
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kPfRows = kPfWarps * 16;  // Q rows per CTA
constexpr int kKhStride = 8;            // fp16 padding of a K row (bank spread)
constexpr int kVtStride = 24;           // fp16 per V channel row (16 tokens + 8 padding)

struct PrefillParams {
  PoolView pool;
  const __half* q;      // [Tq][Hq][D]
  const int* table;     // [S][max_blocks]
  const int* lens;      // [S] tokens in the cache, the chunk included
  const int* q_start;   // [S + 1]
  float* out;           // [Tq][Hq][D]
  int S, Hq, G, max_blocks, max_ctx;
  int ntiles;           // 64-row tiles per (sequence, kv head)
  int nstage, stage_bytes;
  int kh_off, vt_off, sc_off, bar_off;  // shared-memory offsets
  float sm_scale_log2;
};

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        const void* row_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(row_addr)));
}

// One 16-token sub-tile of codes (fragment-native layout) -> exact fp16 in
// shared memory: Kh[t][d] (row stride D + kKhStride) and Vt[d][t] (row stride
// kVtStride).  Tokens at or past `nvalid` get V = 0 (they may never have been
// written; their scores are masked).
template <int FMT, int D>
__device__ __forceinline__ void dequant_subtile(const char* ktile, const char* vtile, __half* Kh,
                                                __half* Vt, int nvalid) {
  constexpr int KSt = D + kKhStride;
  constexpr int W = lane_words<FMT, D>();  // words per lane of a sub-tile
  constexpr int WPC = 4;                   // words per 16-byte chunk
  constexpr int NCH = W / WPC * 32;        // 16-byte chunks per sub-tile
  for (int ch = threadIdx.x; ch < 2 * NCH; ch += kPfThreads) {
    const bool isv = ch >= NCH;
    const int cc = isv ? ch - NCH : ch;
    const int c = cc >> 5, ln = cc & 31;
    const uint4 raw = *reinterpret_cast<const uint4*>((isv ? vtile : ktile) + c * 512 + ln * 16);
    const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
    const int g = ln >> 2, j = ln & 3;
#pragma unroll
    for (int i = 0; i < WPC; ++i) {
      if constexpr (FMT == FMT_INT4_GROUP) {
        const int w = c * WPC + i;  // 16-channel step
        uint32_t p01, p23, p45, p67;
        i4x8_to_h2x4(wv[i], p01, p23, p45, p67);
        if (!isv) {  // tokens g, g+8; channels 16w + 4j .. +3
          uint2* a = reinterpret_cast<uint2*>(Kh + g * KSt + 16 * w + 4 * j);
          uint2* b = reinterpret_cast<uint2*>(Kh + (g + 8) * KSt + 16 * w + 4 * j);
          *a = make_uint2(p01, p23);
          *b = make_uint2(p45, p67);
        } else {  // channels 16w + g, +8; tokens 2j, 2j+1 | 2j+8, 2j+9
          const uint32_t m0 = (2 * j < nvalid ? 0xFFFFu : 0u) | (2 * j + 1 < nvalid ? 0xFFFF0000u : 0u);
          const uint32_t m1 = (2 * j + 8 < nvalid ? 0xFFFFu : 0u) | (2 * j + 9 < nvalid ? 0xFFFF0000u : 0u);
          uint32_t* r0 = reinterpret_cast<uint32_t*>(Vt + (16 * w + g) * kVtStride);
          uint32_t* r1 = reinterpret_cast<uint32_t*>(Vt + (16 * w + 8 + g) * kVtStride);
          r0[j] = p01 & m0;
          r0[4 + j] = p23 & m1;
          r1[j] = p45 & m0;
          r1[4 + j] = p67 & m1;
        }
      } else {
        constexpr int es = FMT == FMT_FP16 ? 2 : 1;
        // one-byte words hold 4 codes; fp16 "words" here are the 4-element
        // groups of the layout, two 32-bit words each
        if constexpr (es == 2) {
          if (i & 1) continue;
        }
        const int w = es == 2 ? (c * 2 + (i >> 1)) : (c * WPC + i);
        uint32_t lo, hi;
        if constexpr (es == 2) {
          lo = wv[i];
          hi = wv[i + 1];
        } else {
          const uint32_t one[1] = {wv[i]};
          word_to_h2<FMT>(one, 0, lo, hi);
        }
        if (!isv) {  // token (w / (D/16)) * 8 + g, channels 16 (w % (D/16)) + 4j .. +3
          const int t = (w / (D / 16)) * 8 + g, d = 16 * (w % (D / 16)) + 4 * j;
          *reinterpret_cast<uint2*>(Kh + t * KSt + d) = make_uint2(lo, hi);
        } else {  // channel 8w + g; tokens 2j, 2j+1 (lo) and 2j+8, 2j+9 (hi)
          const int d = 8 * w + g;
          const uint32_t m0 = (2 * j < nvalid ? 0xFFFFu : 0u) | (2 * j + 1 < nvalid ? 0xFFFF0000u : 0u);
          const uint32_t m1 = (2 * j + 8 < nvalid ? 0xFFFFu : 0u) | (2 * j + 9 < nvalid ? 0xFFFF0000u : 0u);
          uint32_t* r = reinterpret_cast<uint32_t*>(Vt + d * kVtStride);
          r[j] = lo & m0;
          r[4 + j] = hi & m1;
        }
      }
    }
  }
}

template <int FMT, int D, int NG>
__global__ void __launch_bounds__(kPfThreads) kvq_prefill_kernel(const PrefillParams p) {
  using T = FmtTraits<FMT>;
  constexpr int KS = D / 16;
  constexpr int NW = D / 8;
  constexpr int NS = T::group_scales ? NG : 1;
  constexpr int NB = T::group_scales ? NG : 1;
  constexpr int CH = D / NG;
  constexpr int KSt = D + kKhStride;
  const float kNegInf = __int_as_float(0xff800000u);

  extern __shared__ __align__(128) char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, j = lane & 3;
  const PoolView& pool = p.pool;
  const int bs = pool.bs;
  const int nstage = p.nstage;
  const int tile = blockIdx.x % p.ntiles;
  const int seq = (blockIdx.x / p.ntiles) % p.S;
  const int h = blockIdx.x / (p.ntiles * p.S);

  __half* Kh = reinterpret_cast<__half*>(smem + p.kh_off);
  __half* Vt = reinterpret_cast<__half*>(smem + p.vt_off);
  float* ks_s = reinterpret_cast<float*>(smem + p.sc_off);  // [16][NS]
  float* vs_s = ks_s + 16 * NS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  int* stage_phys = reinterpret_cast<int*>(bars + nstage);

  const int qbase = p.q_start[seq];
  const int nq = p.q_start[seq + 1] - qbase;
  int ctx = p.lens[seq];
  if (ctx > p.max_ctx || ctx < nq) {
    if (tile == 0 && h == 0 && threadIdx.x == 0) set_error(pool.err, ERR_RANGE);
    ctx = min(ctx, p.max_ctx);
  }
  const int rows_total = nq * p.G;
  if (tile * kPfRows >= rows_total) return;  // past this sequence's chunk (CTA-uniform)

  // ---- this lane's two rows (g and g+8 of the warp's 16)
  int lim[2];
  const __half* qrow[2];
  int64_t orow[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int rr = tile * kPfRows + warp * 16 + g + 8 * c;
    lim[c] = 0;
    qrow[c] = nullptr;
    orow[c] = -1;
    if (rr < rows_total) {
      const int i = rr / p.G, hq = h * p.G + rr % p.G;
      lim[c] = max(0, ctx - nq + i + 1);
      orow[c] = (int64_t)(qbase + i) * p.Hq + hq;
      qrow[c] = p.q + orow[c] * D;
    }
  }
  // the CTA's widest limit: that of its last valid row
  const int last = min(rows_total, (tile + 1) * kPfRows) - 1;
  const int cta_lim = max(0, ctx - nq + last / p.G + 1);
  const int np = min(p.max_blocks, (cta_lim + bs - 1) / bs);

  // ---- Q as A fragments, channels in natural order: a0/a2 = row g,
  // channels 16kk + 2j, +1 | 16kk + 8 + 2j, +1; a1/a3 = row g+8
  uint32_t qa[KS][4];
  uint32_t qal[T::channel ? KS : 1][4];
  float csc = p.sm_scale_log2;
  if constexpr (!T::channel) {
#pragma unroll
    for (int kk = 0; kk < KS; ++kk)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        qa[kk][c] = qrow[c] ? *reinterpret_cast<const uint32_t*>(qrow[c] + 16 * kk + 2 * j) : 0u;
        qa[kk][2 + c] = qrow[c] ? *reinterpret_cast<const uint32_t*>(qrow[c] + 16 * kk + 8 + 2 * j) : 0u;
      }
  } else {
    const float* ksc = pool.chan_scales + (int64_t)h * D;
    float qf[KS][2][4];
    float amax = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk)
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = 16 * kk + 2 * j + (e & 1) + 8 * (e >> 1);
          const float x = qrow[c] ? __half2float(qrow[c][d]) : 0.f;
          qf[kk][c][e] = x * ksc[d];
          amax = fmaxf(amax, fabsf(qf[kk][c][e]));
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const int eq = amax > 0.f ? 13 - exponent_of(amax) : 0;
    const float up = ldexpf(1.f, eq);
    csc = ldexpf(csc, -eq);
#pragma unroll
    for (int kk = 0; kk < KS; ++kk)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        split_h2(qf[kk][c][0] * up, qf[kk][c][1] * up, qa[kk][c], qal[kk][c]);
        split_h2(qf[kk][c][2] * up, qf[kk][c][3] * up, qa[kk][2 + c], qal[kk][2 + c]);
      }
  }

  if (threadIdx.x == 0) {
    for (int st = 0; st < nstage; ++st) mbar_init(&bars[st], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // ---- page pipeline: thread 0 issues, every thread waits
  const uint32_t page_tx = pool.page_bytes + (T::token_scales ? 2 * bs * 4 : 0);
  const int* trow = p.table + (int64_t)seq * p.max_blocks;
  auto issue = [&](int n) {  // thread 0: page n into stage n % nstage
    const int st = n % nstage;
    const int phys = trow[n];
    const bool ok = phys >= 0 && (int64_t)phys < pool.num_blocks;
    stage_phys[st] = ok ? phys : -1;
    char* dst = smem + st * p.stage_bytes;
    if (ok) {
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
  if (threadIdx.x == 0)
    for (int n = 0; n < min(np, nstage); ++n) issue(n);

  float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
  float o[NW][4];
#pragma unroll
  for (int w = 0; w < NW; ++w) o[w][0] = o[w][1] = o[w][2] = o[w][3] = 0.f;
  int E = T::row_scales ? 100 : 14;
  int waited = 0;  // pages whose barrier this thread has seen complete
  bool failed = false;

  for (int n = 0; n < np; ++n) {
    const int st = n % nstage;
    const uint32_t parity = (n / nstage) & 1;
    bool ok = false;
    for (int tries = 0; tries < kWaitTries && !ok; ++tries) ok = mbar_try_wait(&bars[st], parity);
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    waited = n + 1;
    const char* stage = smem + st * p.stage_bytes;
    const bool present = stage_phys[st] >= 0;
    for (int sp = 0; sp < bs / 16; ++sp) {
      const int t0 = n * bs + sp * 16;
      const int nvalid = present ? max(0, min(16, ctx - t0)) : 0;
      __syncthreads();  // every warp is done with the previous sub-tile's fp16 copy
      if (nvalid > 0) {
        dequant_subtile<FMT, D>(stage + sp * pool.sub_bytes, stage + pool.code_bytes + sp * pool.sub_bytes,
                                Kh, Vt, nvalid);
        if constexpr (T::row_scales) {
          for (int x = threadIdx.x; x < 16 * NS; x += kPfThreads) {
            const int tk = x / NS, gi = x % NS;
            const float* ksp;
            const float* vsp;
            if constexpr (T::group_scales) {
              ksp = reinterpret_cast<const float*>(stage + 2 * pool.code_bytes) + (sp * 16 + tk) * NG;
              vsp = ksp + bs * NG;
            } else {
              ksp = reinterpret_cast<const float*>(stage + pool.page_bytes) + sp * 16 + tk;
              vsp = ksp + bs;
            }
            ks_s[x] = tk < nvalid ? ksp[T::group_scales ? gi : 0] : 0.f;
            vs_s[x] = tk < nvalid ? vsp[T::group_scales ? gi : 0] : 0.f;
          }
        }
      }
      __syncthreads();  // the fp16 copy is complete; the stage is no longer read
      if (sp + 1 == bs / 16 && threadIdx.x == 0 && n + nstage < np) issue(n + nstage);
      if (nvalid == 0) continue;

      // ---- scores: S[row][token], n-tile 0 = tokens 0..7, 1 = 8..15
      float z[2][4];
      {
        float acc[2][NG][4];
#pragma unroll
        for (int nn = 0; nn < 2; ++nn)
#pragma unroll
          for (int gi = 0; gi < NG; ++gi) acc[nn][gi][0] = acc[nn][gi][1] = acc[nn][gi][2] = acc[nn][gi][3] = 0.f;
        const int mrow = ((lane >> 4) << 3) + (lane & 7);  // token row this lane addresses
        const int mcol = ((lane >> 3) & 1) << 3;           // channel half
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t b00, b01, b10, b11;
          ldsm_x4(b00, b01, b10, b11, Kh + mrow * KSt + 16 * kk + mcol);
          const int gi = kk / (KS / NG);
          mma_16816(acc[0][gi], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b00, b01);
          mma_16816(acc[1][gi], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b10, b11);
          if constexpr (T::channel) {
            mma_16816(acc[0][gi], qal[kk][0], qal[kk][1], qal[kk][2], qal[kk][3], b00, b01);
            mma_16816(acc[1][gi], qal[kk][0], qal[kk][1], qal[kk][2], qal[kk][3], b10, b11);
          }
        }
#pragma unroll
        for (int nn = 0; nn < 2; ++nn)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tk = 8 * nn + 2 * j + (e & 1);
            float zz = 0.f;
#pragma unroll
            for (int gi = 0; gi < NG; ++gi)
              zz = fmaf(acc[nn][gi][e], T::row_scales ? ks_s[tk * NS + (T::group_scales ? gi : 0)] : 1.f, zz);
            z[nn][e] = t0 + tk < lim[e >> 1] ? zz * csc : kNegInf;
          }
      }
      // ---- online softmax (base 2), rows g and g+8
      float pr[2][4];
      float al[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float t = fmaxf(fmaxf(z[0][2 * c], z[0][2 * c + 1]), fmaxf(z[1][2 * c], z[1][2 * c + 1]));
        t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 1));
        t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 2));
        const float mn = fmaxf(m[c], t);
        const float ms = mn == kNegInf ? 0.f : mn;
#pragma unroll
        for (int nn = 0; nn < 2; ++nn) {
          pr[nn][2 * c] = fast_exp2(z[nn][2 * c] - ms);
          pr[nn][2 * c + 1] = fast_exp2(z[nn][2 * c + 1] - ms);
        }
        al[c] = fast_exp2(m[c] - ms);
        l[c] = fmaf(l[c], al[c], (pr[0][2 * c] + pr[0][2 * c + 1]) + (pr[1][2 * c] + pr[1][2 * c + 1]));
        m[c] = mn;
      }
      int dE = 0;
      if constexpr (T::row_scales) {
        float vmax = 0.f;
        for (int x = lane; x < 16 * NS; x += 32) vmax = fmaxf(vmax, vs_s[x]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
        if (vmax > 0.f) {
          const int En = min(E, 13 - exponent_of(vmax));
          dE = En - E;
          E = En;
        }
      }
      {
        const float f2 = pow2f(dE);
        const float a0 = al[0] * f2, a1 = al[1] * f2;
        if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
          for (int w = 0; w < NW; ++w) {
            o[w][0] *= a0;
            o[w][1] *= a0;
            o[w][2] *= a1;
            o[w][3] *= a1;
          }
        }
      }
      // ---- weights as A fragments (hi + lo), one set per V scale group
      uint32_t ah[NB][4], alo[NB][4];
      {
        const float sc = pow2f(E);
#pragma unroll
        for (int gi = 0; gi < NB; ++gi) {
          float wv[2][4];
#pragma unroll
          for (int nn = 0; nn < 2; ++nn)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tk = 8 * nn + 2 * j + (e & 1);
              wv[nn][e] = pr[nn][e] * (T::row_scales ? sc * vs_s[tk * NS + gi] : sc);
            }
          split_h2(wv[0][0], wv[0][1], ah[gi][0], alo[gi][0]);
          split_h2(wv[0][2], wv[0][3], ah[gi][1], alo[gi][1]);
          split_h2(wv[1][0], wv[1][1], ah[gi][2], alo[gi][2]);
          split_h2(wv[1][2], wv[1][3], ah[gi][3], alo[gi][3]);
        }
      }
      // ---- P.V: B fragments of channel n-tiles from the channel-major copy
      {
        const int vrow = ((lane >> 4) << 3) + (lane & 7);  // channel within a 16-channel pair
        const int vcol = ((lane >> 3) & 1) << 3;           // token half
#pragma unroll
        for (int pp = 0; pp < NW / 2; ++pp) {
          uint32_t b00, b01, b10, b11;
          ldsm_x4(b00, b01, b10, b11, Vt + (16 * pp + vrow) * kVtStride + vcol);
#pragma unroll
          for (int nn = 0; nn < 2; ++nn) {
            const int w = 2 * pp + nn;
            const int gi = T::group_scales ? (8 * w) / CH : 0;
            const uint32_t c0 = nn ? b10 : b00, c1 = nn ? b11 : b01;
            mma_16816(o[w], ah[gi][0], ah[gi][1], ah[gi][2], ah[gi][3], c0, c1);
            mma_16816(o[w], alo[gi][0], alo[gi][1], alo[gi][2], alo[gi][3], c0, c1);
          }
        }
      }
    }
  }

  if (failed) {
    // a wait ran out: flag it, then wait (bounded) for the copies still in
    // flight so that none lands after the CTA has exited
    if (threadIdx.x == 0) set_error(pool.err, ERR_TIMEOUT);
    for (int n = waited; n < min(np, waited + nstage); ++n) {
      bool ok = false;
      for (int tries = 0; tries < kWaitTries && !ok; ++tries)
        ok = mbar_try_wait(&bars[n % nstage], (n / nstage) & 1);
    }
    return;
  }

  // ---- normalised output of this warp's rows
  {
    const float inv2E = pow2f(-E);
    const float* vch = T::channel ? pool.chan_scales + ((int64_t)pool.Hkv + h) * D : nullptr;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float lt = l[c];
      lt += __shfl_xor_sync(0xffffffffu, lt, 1);
      lt += __shfl_xor_sync(0xffffffffu, lt, 2);
      if (orow[c] < 0) continue;
      const float f = lt > 0.f ? inv2E / lt : 0.f;
      float* dst = p.out + orow[c] * D;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const int d = 8 * w + 2 * j;
        const float c0 = T::channel ? vch[d] : 1.f, c1 = T::channel ? vch[d + 1] : 1.f;
        dst[d] = o[w][2 * c] * f * c0;
        dst[d + 1] = o[w][2 * c + 1] * f * c1;
      }
    }
  }
}

struct PrefillLaunch {
  PrefillParams p;
  dim3 grid;
  int smem;
  cudaStream_t st;
};

template <int FMT, int D, int NG>
cudaError_t run_prefill(const PrefillLaunch& l) {
  cudaError_t e = allow_big_smem<kvq_prefill_kernel<FMT, D, NG>>();
  if (e != cudaSuccess) return e;
  kvq_prefill_kernel<FMT, D, NG><<<l.grid, kPfThreads, l.smem, l.st>>>(l.p);
  return phase_mark(l.st, cudaGetLastError());
}

}  // namespace kvq
