// kvq_rows_impl.cuh -- shared-prefix ("cascade") attention over a quantized
// paged KV pool: many sequences' Q rows against the blocks they share.
//
// Method ("KV Cache优化实战：大模型推理显存占用与加速方案详解",
// 0539edu.com/news/5800990, §2.2 and §4.4: PagedAttention lets requests with
// a common prefix -- a system prompt, a fixed history -- share its physical
// blocks): when every sequence's first P blocks are the same physical
// blocks, those blocks are attended once for all sequences' Q rows instead of
// once per sequence.  The result is a partial (running max m, sum l,
// unnormalised output O, base-2 softmax) per (sequence, Q head) that the paged
// decode over the remaining blocks folds in by log-sum-exp.
//
// GB300 design: a CTA takes one kv head and a tile of 16 Q rows -- a row is a
// (sequence, Q head) pair, so a tile usually spans several sequences -- and
// its 4 warps split the shared blocks between them.  Each
// warp streams its blocks through bulk-copy stages (as the decode kernel does)
// and computes with the rows on the M dimension of mma.m16n8k16: Q.K^T takes
// the K codes of the fragment-native page layout directly as B fragments
// (token g's word of a lane is the B fragment of the 8-token n-tile), and
// because the score accumulator of two n-tiles is laid out as the A fragment
// of the next product, the softmax weights feed P.V without any shuffle; the V
// word of a lane is the B fragment of an 8-channel n-tile.  Per-token/group V
// scales fold into the weights (split fp16 hi + lo), per-token/group K scales
// multiply the scores, per-channel scales fold into q and the output.  The 4
// warps' partials merge in shared memory; one row of (m, l, O) per (sequence,
// Q head) goes to global memory.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "kvq_decode_impl.cuh"

namespace kvq {

constexpr int kRowsWarps = 4;
constexpr int kRowsThreads = kRowsWarps * 32;
constexpr int kRowsTile = 16;  // Q rows per CTA: one mma M tile

struct RowsParams {
  PoolView pool;
  const __half* q;      // [S][Hq][D]
  const int* table;     // [S][max_blocks]; row 0's first P entries are the shared blocks
  const int* lens;      // [S]
  float* out;           // [S][Hq][D + 2] partial rows (m, l, O)
  int S, Hq, G, max_blocks, max_ctx;
  int P;                // shared blocks
  int ntiles;           // row tiles per kv head
  int nstage, stage_bytes;
  int bar_off;          // shared-memory offset of the barriers (past stages and merge rows)
  float sm_scale_log2;
};

template <int FMT, int D, int NG>
__global__ void __launch_bounds__(kRowsThreads) kvq_rows_kernel(const RowsParams p) {
  using T = FmtTraits<FMT>;
  constexpr int KS = D / 16;  // k-steps of Q.K^T
  constexpr int NW = D / 8;   // 8-channel n-tiles of P.V
  constexpr int NU32 = lane_words<FMT, D>();
  constexpr int KPG = KS / NG;
  constexpr int NS = T::group_scales ? NG : 1;
  constexpr int NB = T::group_scales ? NG : 1;
  constexpr int CH = D / NG;  // channels per scale group
  const float kNegInf = __int_as_float(0xff800000u);

  extern __shared__ __align__(128) char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, j = lane & 3;
  const PoolView& pool = p.pool;
  const int bs = pool.bs;
  const int nstage = p.nstage;
  const int tile = blockIdx.x % p.ntiles;  // grid: (kv head, tile)
  const int h = blockIdx.x / p.ntiles;

  // A kernel launched after this one as a programmatic dependent reads our
  // output only after its griddepcontrol.wait on this grid's completion.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  char* stages = smem + warp * nstage * p.stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off) + warp * nstage;
  int* stage_phys =
      reinterpret_cast<int*>(smem + p.bar_off + kRowsWarps * nstage * 8) + warp * nstage;

  // ---- rows of the tile: row rr is (sequence rr / G, Q head rr % G) of kv
  // head h; its token limit is its own context length, at most the prefix
  const int rows_total = p.S * p.G;
  auto row_of = [&](int rr, int& lim, const __half*& qp, int64_t& orow) {
    lim = 0;
    qp = nullptr;
    orow = -1;
    if (rr >= rows_total) return;
    const int s = rr / p.G;
    lim = max(0, min(min(p.lens[s], p.max_ctx), p.P * bs));
    orow = (int64_t)s * p.Hq + h * p.G + rr % p.G;
    qp = p.q + orow * D;
  };
  int lim[2];
  const __half* qrow[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    int64_t orow;
    row_of(tile * kRowsTile + g + 8 * c, lim[c], qrow[c], orow);
  }

  // ---- Q as A fragments: a0/a2 = row g, channels 16kk+4j..+3; a1/a3 = row g+8
  uint32_t qa[KS][4];
  uint32_t qal[T::channel ? KS : 1][4];
  float csc = p.sm_scale_log2;
  if constexpr (!T::channel) {
#pragma unroll
    for (int kk = 0; kk < KS; ++kk)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint2 v = qrow[c] ? *reinterpret_cast<const uint2*>(qrow[c] + 16 * kk + 4 * j)
                                : make_uint2(0u, 0u);
        qa[kk][c] = v.x;
        qa[kk][2 + c] = v.y;
      }
  } else {
    // fold the K channel scale into q, scale by 2^eq into [2^13, 2^14), split
    const float* ksc = pool.chan_scales + (int64_t)h * D;
    float qf[KS][2][4];
    float amax = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint2 v = qrow[c] ? *reinterpret_cast<const uint2*>(qrow[c] + 16 * kk + 4 * j)
                                : make_uint2(0u, 0u);
        const __half2 a = *reinterpret_cast<const __half2*>(&v.x);
        const __half2 b = *reinterpret_cast<const __half2*>(&v.y);
        const int d0 = 16 * kk + 4 * j;
        qf[kk][c][0] = __low2float(a) * ksc[d0 + 0];
        qf[kk][c][1] = __high2float(a) * ksc[d0 + 1];
        qf[kk][c][2] = __low2float(b) * ksc[d0 + 2];
        qf[kk][c][3] = __high2float(b) * ksc[d0 + 3];
#pragma unroll
        for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qf[kk][c][e]));
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

  // ---- this warp's blocks: the tile needs blocks [0, np), split in 4 runs
  // (every warp holds all 16 rows, so wlim is the tile's widest limit)
  int wlim = max(lim[0], lim[1]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wlim = max(wlim, __shfl_xor_sync(0xffffffffu, wlim, off));
  const int np = min(p.P, (wlim + bs - 1) / bs);
  const int chunk = (np + kRowsWarps - 1) / kRowsWarps;
  const int p0 = warp * chunk;
  const int p1 = min(np, p0 + chunk);
  const int n_w = max(p1 - p0, 0);
  const int* trow = p.table;  // table row 0 names the shared blocks

  if (lane == 0) {
    for (int st = 0; st < nstage; ++st) mbar_init(&bars[st], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // The pool may be written by the kernel this one depends on (the
  // decode-step append); read it only after that kernel has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const uint32_t page_tx = pool.page_bytes + (T::token_scales ? 2 * bs * 4 : 0);
  const int tcache = lane < n_w ? trow[p0 + lane] : -1;
  int n_issued = 0, pst = 0;
  auto issue_next = [&]() {  // all lanes call; lane 0 issues
    const int cached = __shfl_sync(0xffffffffu, tcache, n_issued & 31);
    if (lane == 0) {
      const int phys = n_issued < 32 ? cached : trow[p0 + n_issued];
      const int st = pst;
      const bool ok = phys >= 0 && (int64_t)phys < pool.num_blocks;
      stage_phys[st] = ok ? phys : -1;
      if (ok) {
        char* dst = stages + st * p.stage_bytes;
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
    ++n_issued;
    if (++pst == nstage) pst = 0;
  };
  for (int i = 0; i < min(n_w, nstage); ++i) issue_next();

  int cst = 0;
  uint32_t cph = 0;
  auto wait_stage = [&](int st, uint32_t parity) -> bool {
    bool ok = false;
    for (int tries = 0; tries < kWaitTries && !ok; ++tries) ok = mbar_try_wait(&bars[st], parity);
    return __all_sync(0xffffffffu, ok);
  };

  // ---- online softmax state of rows g (index 0) and g+8 (index 1)
  float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
  float o[NW][4];
#pragma unroll
  for (int w = 0; w < NW; ++w) o[w][0] = o[w][1] = o[w][2] = o[w][3] = 0.f;
  int E = T::row_scales ? 100 : 14;
  bool failed = false;

  int i = 0;
  for (; i < n_w; ++i) {
    if (!wait_stage(cst, cph)) {
      if (lane == 0) set_error(pool.err, ERR_TIMEOUT);
      failed = true;
      break;
    }
    const char* stage = stages + cst * p.stage_bytes;
    const bool present = stage_phys[cst] >= 0;
    const int pg = p0 + i;
    for (int sub = 0; present && sub < bs / 16; ++sub) {
      const int t0 = pg * bs + sub * 16;
      if (t0 >= wlim) break;
      const int nvalid = min(16, wlim - t0);
      // ---- scales of this lane's tokens 2j, 2j+1, 8+2j, 9+2j
      float ks[4][NS], vs[4][NS];
      if constexpr (T::row_scales) {
        const float* ksp;
        const float* vsp;
        if constexpr (T::group_scales) {
          ksp = reinterpret_cast<const float*>(stage + 2 * pool.code_bytes) + sub * 16 * NG;
          vsp = ksp + bs * NG;
        } else {
          ksp = reinterpret_cast<const float*>(stage + pool.page_bytes) + sub * 16;
          vsp = ksp + bs;
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          // the scales of tokens no row reads may never have been written
          const int tk = 8 * (x >> 1) + 2 * j + (x & 1);
          const bool w = tk < nvalid;
#pragma unroll
          for (int gi = 0; gi < NS; ++gi) {
            ks[x][gi] = w ? ksp[tk * NS + gi] : 0.f;
            vs[x][gi] = w ? vsp[tk * NS + gi] : 0.f;
          }
        }
      }
      // ---- scores S[row][token] per scale group: n-tile 0 = tokens 0..7, 1 = 8..15
      float z[2][4];
      {
        uint32_t kw[NU32];
        load_lane_words<FMT, D>(stage + sub * pool.sub_bytes, lane, kw);
        constexpr int SUB = KPG >= 2 ? 2 : 1;  // independent accumulators per group
        float acc[2][NG * SUB][4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int a = 0; a < NG * SUB; ++a) acc[n][a][0] = acc[n][a][1] = acc[n][a][2] = acc[n][a][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int ai = (kk / KPG) * SUB + (SUB == 2 ? (kk & 1) : 0);
          // k_frag's A-fragment words of token rows g / g+8 are the B
          // fragments of the n-tiles of tokens 0..7 / 8..15
          uint32_t b[2][2];
          k_frag<FMT, D>(kw, kk, b[0][0], b[1][0], b[0][1], b[1][1]);
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            mma_16816(acc[n][ai], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b[n][0], b[n][1]);
            if constexpr (T::channel)
              mma_16816(acc[n][ai], qal[kk][0], qal[kk][1], qal[kk][2], qal[kk][3], b[n][0],
                        b[n][1]);
          }
        }
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int x = 2 * n + (e & 1);
            float zz = 0.f;
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
              const float sg = SUB == 2 ? acc[n][gi * SUB][e] + acc[n][gi * SUB + 1][e] : acc[n][gi][e];
              zz = fmaf(sg, T::row_scales ? ks[x][T::group_scales ? gi : 0] : 1.f, zz);
            }
            const int tabs = t0 + 8 * n + 2 * j + (e & 1);
            z[n][e] = tabs < lim[e >> 1] ? zz * csc : kNegInf;
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
        for (int n = 0; n < 2; ++n) {
          pr[n][2 * c] = fast_exp2(z[n][2 * c] - ms);
          pr[n][2 * c + 1] = fast_exp2(z[n][2 * c + 1] - ms);
        }
        al[c] = fast_exp2(m[c] - ms);
        l[c] = fmaf(l[c], al[c], (pr[0][2 * c] + pr[0][2 * c + 1]) + (pr[1][2 * c] + pr[1][2 * c + 1]));
        m[c] = mn;
      }
      int dE = 0;
      if constexpr (T::row_scales) {
        float vmax = 0.f;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int tk = 8 * (x >> 1) + 2 * j + (x & 1);
          if (tk < nvalid)
#pragma unroll
            for (int gi = 0; gi < NS; ++gi) vmax = fmaxf(vmax, vs[x][gi]);
        }
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
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              wv[n][e] = pr[n][e] * (T::row_scales ? sc * vs[2 * n + (e & 1)][gi] : sc);
          split_h2(wv[0][0], wv[0][1], ah[gi][0], alo[gi][0]);  // row g,   tokens 2j, 2j+1
          split_h2(wv[0][2], wv[0][3], ah[gi][1], alo[gi][1]);  // row g+8, tokens 2j, 2j+1
          split_h2(wv[1][0], wv[1][1], ah[gi][2], alo[gi][2]);  // row g,   tokens 8+2j, 9+2j
          split_h2(wv[1][2], wv[1][3], ah[gi][3], alo[gi][3]);  // row g+8, tokens 8+2j, 9+2j
        }
      }
      // ---- P.V: lane word w of the V sub-tile is the B fragment of channels 8w..8w+7
      {
        uint32_t vw[NU32];
        load_lane_words<FMT, D>(stage + pool.code_bytes + sub * pool.sub_bytes, lane, vw);
        if constexpr (T::maybe_nan) {
          if (nvalid < 16) {
            // zero the V of tokens that no row of this warp attends (they may
            // never have been written), so that 0 * NaN cannot reach O
            const int t0l = 2 * j;
            if constexpr (FMT == FMT_FP16) {
              const uint32_t mlo = (t0l < nvalid ? 0xFFFFu : 0u) | (t0l + 1 < nvalid ? 0xFFFF0000u : 0u);
              const uint32_t mhi = (t0l + 8 < nvalid ? 0xFFFFu : 0u) | (t0l + 9 < nvalid ? 0xFFFF0000u : 0u);
#pragma unroll
              for (int w = 0; w < NU32 / 2; ++w) {
                vw[2 * w] &= mlo;
                vw[2 * w + 1] &= mhi;
              }
            } else {
              const uint32_t msk = (t0l < nvalid ? 0xFFu : 0u) | (t0l + 1 < nvalid ? 0xFF00u : 0u) |
                                   (t0l + 8 < nvalid ? 0xFF0000u : 0u) |
                                   (t0l + 9 < nvalid ? 0xFF000000u : 0u);
#pragma unroll
              for (int w = 0; w < NU32; ++w) vw[w] &= msk;
            }
          }
        }
        // v_frag's A-fragment words of channel rows g / g+8 of m-tile mt are
        // the B fragments of the n-tiles of channels 16mt.. / 16mt+8..
#pragma unroll
        for (int mt = 0; mt < NW / 2; ++mt) {
          uint32_t b[2][2];
          v_frag<FMT>(vw, mt, b[0][0], b[1][0], b[0][1], b[1][1]);
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            const int w = 2 * mt + n;
            const int gi = T::group_scales ? (8 * w) / CH : 0;
            mma_16816(o[w], ah[gi][0], ah[gi][1], ah[gi][2], ah[gi][3], b[n][0], b[n][1]);
            mma_16816(o[w], alo[gi][0], alo[gi][1], alo[gi][2], alo[gi][3], b[n][0], b[n][1]);
          }
        }
      }
    }
    __syncwarp();
    if (n_issued < n_w) issue_next();
    if (++cst == nstage) {
      cst = 0;
      cph ^= 1u;
    }
  }

  // ---- a wait ran out: wait (bounded) for this warp's copies still in flight
  // before the stages are reused or the CTA exits
  if (failed) {
    int st = cst;
    uint32_t ph = cph;
    for (int k = i; k < n_issued; ++k) {
      wait_stage(st, ph);
      if (++st == nstage) {
        st = 0;
        ph ^= 1u;
      }
    }
  }

  // ---- merge the 4 warps' partials in shared memory (over the stages)
  __syncthreads();
  float* mb = reinterpret_cast<float*>(smem);  // [warp][16 rows][D + 2]
  {
    const float inv2E = pow2f(-E);
    const float* vch = T::channel ? pool.chan_scales + ((int64_t)pool.Hkv + h) * D : nullptr;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float lt = l[c];
      lt += __shfl_xor_sync(0xffffffffu, lt, 1);
      lt += __shfl_xor_sync(0xffffffffu, lt, 2);
      float* row = mb + ((int64_t)warp * kRowsTile + g + 8 * c) * (D + 2);
      if (j == 0) {
        row[0] = failed ? kNegInf : m[c];
        row[1] = failed ? 0.f : lt;
      }
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const int d = 8 * w + 2 * j;
        const float c0 = T::channel ? vch[d] : 1.f, c1 = T::channel ? vch[d + 1] : 1.f;
        row[2 + d] = failed ? 0.f : o[w][2 * c] * inv2E * c0;
        row[2 + d + 1] = failed ? 0.f : o[w][2 * c + 1] * inv2E * c1;
      }
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kRowsTile * D; idx += kRowsThreads) {
    const int rr = idx / D, d = idx % D;
    int rlim;
    const __half* rq;
    int64_t orow;
    row_of(tile * kRowsTile + rr, rlim, rq, orow);
    if (orow < 0) continue;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kRowsWarps; ++w) M = fmaxf(M, mb[(w * kRowsTile + rr) * (D + 2)]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kRowsWarps; ++w) {
      const float* row = mb + (w * kRowsTile + rr) * (D + 2);
      const float wt = row[0] == kNegInf ? 0.f : fast_exp2(row[0] - M);
      Ls = fmaf(wt, row[1], Ls);
      O = fmaf(wt, row[2 + d], O);
    }
    float* dst = p.out + orow * (D + 2);
    dst[2 + d] = O;
    if (d == 0) {
      dst[0] = M;
      dst[1] = Ls;
    }
  }
}

struct RowsLaunch {
  RowsParams p;
  dim3 grid;
  int smem;
  cudaStream_t st;
  bool dependent;
};

template <int FMT, int D, int NG>
cudaError_t run_rows(const RowsLaunch& l) {
  cudaError_t e = allow_big_smem<kvq_rows_kernel<FMT, D, NG>>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = l.grid;
  cfg.blockDim = dim3(kRowsThreads);
  cfg.dynamicSmemBytes = l.smem;
  cfg.stream = l.st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = l.dependent ? 1 : 0;
  return phase_mark(l.st, cudaLaunchKernelEx(&cfg, kvq_rows_kernel<FMT, D, NG>, l.p));
}

}  // namespace kvq
