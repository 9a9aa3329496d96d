// kvq_prefill_tc_impl.cuh -- prefill / chunked-prefill attention over a
// quantized paged KV pool on the 5th-generation tensor cores (tcgen05, TMEM).
//
// Method ("KV Cache优化实战：大模型推理显存占用与加速方案详解",
// 0539edu.com/news/5800990, §1.1): the prompt's tokens are processed together,
// each attending causally to the tokens up to itself; a chunk of n tokens of a
// sequence whose cache holds L tokens (the chunk included) has its token i at
// position L - n + i.  K/V are read from the block-paged cache (§2.2) in their
// stored format (§2.3, §3.3) and dequantized inside the kernel (§4.3).
//
// GB300 design.  A CTA of 12 warps takes one (sequence, kv head) and two
// tiles of 128 Q rows -- the (query token, Q head of the group) pairs, 32
// query tokens x 4 heads per tile for GQA 4:1 -- and walks the keys in steps
// of 64 tokens, with the work split by role:
//   * 4 converter warps load the next step's code pages into registers while
//     the current step is being used, then turn them into exact fp16 values
//     in shared memory -- K as a 64 x D tile, V transposed as a D x 64 tile,
//     both K-major with the 128-byte swizzle, two buffers -- and publish the
//     step's per-token scales and valid-token mask;
//   * each tile's 4 softmax warps own its 128 rows (one row per thread, one
//     TMEM lane each): they read the row's 64 scores S = Q.K^T from tensor
//     memory, apply the K scales, the causal limit and the online softmax
//     (base 2), and write the weights p * s_V * 2^E as an fp16 high part and
//     an fp16 low part (K-major 128 x 64 tiles); the row's exponent reference
//     moves only when a score passes it by more than 2^8, and only then (or
//     when E drops) is its row of the output accumulator in TMEM rescaled;
//   * one thread of each tile issues that tile's tensor-core work: O +=
//     P_hi.V + P_lo.V (M 128, N D, K 64), then, once the next step is
//     converted, S = Q.K^T (M 128, N 64, K D), both tcgen05.mma kind::f16
//     with fp32 accumulators in TMEM.
// While one tile runs its softmax the tensor cores run the other tile's
// products, and the conversion of a step is shared by both tiles.  Codes are
// exact in fp16, so dequantization is a scale outside the contraction, as in
// the decode kernel; the hi + lo split keeps the weights exact to ~2^-22.
// Every wait is bounded and gives up early once another role has given up;
// the CTA then flags a timeout in the pool's error word, waits (bounded) for
// its MMAs in flight and frees TMEM.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "kvq_decode_impl.cuh"
#include "kvq_tc.cuh"

namespace kvq {

constexpr int kTcRows = 128;      // Q rows per tile = TMEM lanes
constexpr int kTcStep = 64;       // key tokens per step
constexpr int kTcSlack = 8;       // log2 of how far a row may exceed its reference maximum
constexpr int kTcConv = 128;      // converter threads

struct PrefillTcParams {
  PoolView pool;
  const __half* q;      // [Tq][Hq][D]
  const int* table;     // [S][max_blocks]
  const int* lens;      // [S]
  const int* q_start;   // [S + 1]
  float* out;           // [Tq][Hq][D]
  int S, Hq, G, max_blocks, max_ctx;
  int ntiles;           // 128-row tiles per (sequence, kv head)
  int ngroups;          // CTAs per (sequence, kv head): ceil(ntiles / NT)
  float sm_scale_log2;
};

// Shared-memory plan of a CTA with NT tiles (byte offsets from a 1024-byte
// aligned base): Q tiles (and their low parts for per-channel pools), the two
// K and V^T buffers, each tile's weight tiles, the misc block.
template <int D, int NT, bool CH>
struct TcPlan {
  static constexpr int QB = kTcRows * D * 2, KB = kTcStep * D * 2, VB = D * kTcStep * 2,
                       PB = kTcRows * kTcStep * 2;
  static constexpr int q = 0;                              // [NT][QB] (+ [NT][QB] low parts)
  static constexpr int kh = NT * QB * (CH ? 2 : 1);        // [2][KB]
  static constexpr int vt = kh + 2 * KB;                   // [2][VB]
  static constexpr int pw = vt + 2 * VB;                   // [NT][hi, lo][PB]
  static constexpr int misc = pw + NT * 2 * PB;
  // misc: float ks[2][64], vs[2][64]; float vmax[2][2]; uint32 mask[2][2];
  // int abort; uint64 kv_full[2], kv_empty[2], s_full[NT], o_full[NT], drain[NT]; uint32 tslot
  static constexpr int ks = misc, vs = misc + 512, vmax = misc + 1024, mask = misc + 1040,
                       abort = misc + 1056, bars = misc + 1064, tslot = bars + 8 * (4 + 3 * NT);
  static constexpr int bytes = tslot + 16;
  static constexpr int request = bytes + 1024;             // alignment slack
  static constexpr int threads = kTcRows * NT + kTcConv;
  static constexpr int cols = NT == 2 ? 512 : 256;          // TMEM: O at 128X, S at 256 + 64X (NT 2)
  static constexpr int s_col(int x) { return NT == 2 ? 256 + 64 * x : 128; }
};

template <int FMT>
__device__ __forceinline__ void tc_word_to_h2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t one[1] = {w};
  word_to_h2<FMT>(one, 0, lo, hi);
}

// Convert one 16-byte chunk (lane L, chunk c) of a K or V code sub-tile into
// the fp16 tiles.  `s` is the sub-tile's slot in the step (tokens 16s..16s+15
// of the tile); V tokens at or past `nv` are written as zero.
template <int FMT, int D>
__device__ __forceinline__ void tc_convert_chunk(uint4 raw, int L, int c, bool isv, int s, int nv,
                                                 char* kh, char* vt) {
  const int g = L >> 2, j = L & 3;
  const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
  const uint32_t m0 = (2 * j < nv ? 0xFFFFu : 0u) | (2 * j + 1 < nv ? 0xFFFF0000u : 0u);
  const uint32_t m1 = (2 * j + 8 < nv ? 0xFFFFu : 0u) | (2 * j + 9 < nv ? 0xFFFF0000u : 0u);
  if constexpr (FMT == FMT_INT4_GROUP) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int w = 4 * c + i;  // 16-channel step
      uint32_t p01, p23, p45, p67;
      i4x8_to_h2x4(wv[i], p01, p23, p45, p67);
      if (!isv) {  // tokens g, g+8; channels 16w + 4j .. +3
        *reinterpret_cast<uint2*>(kh + sw128_offset(16 * s + g, 16 * w + 4 * j, kTcStep)) =
            make_uint2(p01, p23);
        *reinterpret_cast<uint2*>(kh + sw128_offset(16 * s + g + 8, 16 * w + 4 * j, kTcStep)) =
            make_uint2(p45, p67);
      } else {  // channels 16w + g, +8; tokens 2j, 2j+1 | 2j+8, 2j+9
        const int d0 = 16 * w + g;
        *reinterpret_cast<uint32_t*>(vt + sw128_offset(d0, 16 * s + 2 * j, D)) = p01 & m0;
        *reinterpret_cast<uint32_t*>(vt + sw128_offset(d0, 16 * s + 2 * j + 8, D)) = p23 & m1;
        *reinterpret_cast<uint32_t*>(vt + sw128_offset(d0 + 8, 16 * s + 2 * j, D)) = p45 & m0;
        *reinterpret_cast<uint32_t*>(vt + sw128_offset(d0 + 8, 16 * s + 2 * j + 8, D)) = p67 & m1;
      }
    }
  } else if constexpr (FMT == FMT_FP16) {
    // a chunk holds two 4-element groups (two 32-bit words each)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int w = 2 * c + i;
      const uint32_t lo = wv[2 * i], hi = wv[2 * i + 1];
      if (!isv) {  // token (w / (D/16)) * 8 + g, channels 16 (w % (D/16)) + 4j .. +3
        const int t = (w / (D / 16)) * 8 + g, d = 16 * (w % (D / 16)) + 4 * j;
        *reinterpret_cast<uint2*>(kh + sw128_offset(16 * s + t, d, kTcStep)) = make_uint2(lo, hi);
      } else {  // channel 8w + g; tokens 2j, 2j+1 (lo) and 2j+8, 2j+9 (hi)
        const int d = 8 * w + g;
        *reinterpret_cast<uint32_t*>(vt + sw128_offset(d, 16 * s + 2 * j, D)) = lo & m0;
        *reinterpret_cast<uint32_t*>(vt + sw128_offset(d, 16 * s + 2 * j + 8, D)) = hi & m1;
      }
    }
  } else {  // one-byte codes: four per 32-bit word
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int w = 4 * c + i;
      uint32_t lo, hi;
      tc_word_to_h2<FMT>(wv[i], lo, hi);
      if (!isv) {
        const int t = (w / (D / 16)) * 8 + g, d = 16 * (w % (D / 16)) + 4 * j;
        *reinterpret_cast<uint2*>(kh + sw128_offset(16 * s + t, d, kTcStep)) = make_uint2(lo, hi);
      } else {
        const int d = 8 * w + g;
        *reinterpret_cast<uint32_t*>(vt + sw128_offset(d, 16 * s + 2 * j, D)) = lo & m0;
        *reinterpret_cast<uint32_t*>(vt + sw128_offset(d, 16 * s + 2 * j + 8, D)) = hi & m1;
      }
    }
  }
}

// Bounded wait that gives up early once another role has set *abort; a wait
// that runs out sets it.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  // spin first: a suspended thread is not always resumed the moment the
  // phase completes, and these waits are on the critical path
  for (int i = 0; i < kSpinPolls; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort) return false;
  }
  for (int tries = 0; tries < kWaitTries; ++tries) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
  }
  *abort = 1;
  return false;
}

// The same bound without the spinning phase, for a thread off the critical
// path (its polls would take issue slots from the warps sharing its
// scheduler): suspending tries only.
__device__ __forceinline__ bool tc_wait_suspend(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (int tries = 0; tries < kWaitTries; ++tries) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
  }
  *abort = 1;
  return false;
}

// Named barrier ID over `count` threads with an OR of `pred` (the id is an
// immediate: a barrier id held in a register makes the compiler reserve all
// sixteen barriers and lowers the register budget of the kernel).
template <int ID>
__device__ __forceinline__ bool bar_or_n(int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(ID), "r"(count)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ bool bar_or(int id, int count, bool pred) {
  switch (id) {
    case 1: return bar_or_n<1>(count, pred);
    case 2: return bar_or_n<2>(count, pred);
    default: return bar_or_n<3>(count, pred);
  }
}

// Split two fp32 weights into fp16 high and low pairs: (a, b) ~= hi + lo.
__device__ __forceinline__ void tc_split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  float ra, rb;
  f2_unpack(f2_sub(f2_pack(a, b), f2_pack(hf.x, hf.y)), ra, rb);
  const __half2 r = __floats2half2_rn(ra, rb);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

template <int FMT, int D, int NT>
__global__ void __launch_bounds__(TcPlan<D, NT, FmtTraits<FMT>::channel>::threads, 1)
    kvq_prefill_tc_kernel(const PrefillTcParams p) {
  using T = FmtTraits<FMT>;
  constexpr bool CH = T::channel;
  using PL = TcPlan<D, NT, CH>;
  constexpr int ES = FMT == FMT_FP16 ? 2 : 1;
  constexpr int SUB_BYTES = FMT == FMT_INT4_GROUP ? 8 * D : 16 * D * ES;
  constexpr int CPS = SUB_BYTES / 16;                 // 16-byte chunks per K (or V) sub-tile
  constexpr int NCH = (CPS + kTcConv - 1) / kTcConv;  // chunks per converter thread and sub-tile
  const float kNegInf = __int_as_float(0xff800000u);

  extern __shared__ __align__(1024) char smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  char* sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PoolView& pool = p.pool;
  const int bs = pool.bs;
  // heaviest tile groups (longest causal ranges) first
  const int per = p.S * pool.Hkv;
  const int grp = p.ngroups - 1 - static_cast<int>(blockIdx.x / per);
  const int seq = static_cast<int>(blockIdx.x % per) % p.S;
  const int h = static_cast<int>(blockIdx.x % per) / p.S;

  const int qbase = p.q_start[seq];
  const int nq = p.q_start[seq + 1] - qbase;
  int ctx = p.lens[seq];
  if (ctx > p.max_ctx || ctx < nq) {
    if (grp == 0 && h == 0 && tid == 0) set_error(pool.err, ERR_RANGE);
    ctx = min(ctx, p.max_ctx);
  }
  const int rows_total = nq * p.G;
  const int row0 = grp * NT * kTcRows;  // first row of the CTA
  if (row0 >= rows_total) return;       // CTA-uniform
  const int last = min(rows_total, row0 + NT * kTcRows) - 1;
  const int kv_end = max(0, min(ctx, ctx - nq + last / p.G + 1));
  const int nsteps = (kv_end + kTcStep - 1) / kTcStep;

  // softmax threads: tile X, row r (= TMEM lane)
  const bool is_sm = tid < NT * kTcRows;
  const int X = is_sm ? warp >> 2 : 0;
  const int r = (warp & 3) * 32 + lane;
  const int rr = row0 + X * kTcRows + r;
  const bool row_ok = is_sm && rr < rows_total;
  const int lim = row_ok ? max(0, ctx - nq + rr / p.G + 1) : 0;
  const int64_t orow = row_ok ? (int64_t)(qbase + rr / p.G) * p.Hq + h * p.G + rr % p.G : -1;
  if (nsteps == 0) {  // nothing to attend: zeros (CTA-uniform)
    if (row_ok)
      for (int d = 0; d < D; ++d) p.out[orow * D + d] = 0.f;
    return;
  }

  float* ks_s = reinterpret_cast<float*>(sm + PL::ks);      // [2][64]
  float* vs_s = reinterpret_cast<float*>(sm + PL::vs);      // [2][64]
  float* vmax_s = reinterpret_cast<float*>(sm + PL::vmax);  // [2][2]
  uint32_t* mask_s = reinterpret_cast<uint32_t*>(sm + PL::mask);  // [2][2]
  volatile int* abort_f = reinterpret_cast<volatile int*>(sm + PL::abort);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + PL::bars);
  uint64_t* kv_full = bars;           // [2]: converted K/V of a step (128 arrivals)
  uint64_t* kv_empty = bars + 2;      // [2]: every tile's MMAs of that step done (NT commits)
  uint64_t* s_full = bars + 4;        // [NT]: S of the tile's current step
  uint64_t* o_full = bars + 4 + NT;   // [NT]: the tile's last P.V done
  uint64_t* drain = bars + 4 + 2 * NT;  // [NT]: clean-up
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + PL::tslot);

  if (tid == 0) {
    mbar_init(&kv_full[0], kTcConv);
    mbar_init(&kv_full[1], kTcConv);
    mbar_init(&kv_empty[0], NT);
    mbar_init(&kv_empty[1], NT);
    for (int x = 0; x < NT; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&o_full[x], 1);
      mbar_init(&drain[x], 1);
    }
    *abort_f = 0;
    fence_barrier_init();
  }
  if (warp == 0) tc_alloc(tslot, PL::cols);

  // ---- softmax threads: their own Q row into the tile (K-major, swizzled)
  float csc = p.sm_scale_log2;
  if (is_sm) {
    const __half* src = row_ok ? p.q + orow * D : nullptr;
    char* qx = sm + PL::q + X * PL::QB;
    if constexpr (!CH) {
      // the warp loads its 32 rows together: one instruction covers 256 / D
      // whole rows (each row's source address comes from its owner lane); a
      // batch of loads is issued before any of its shared-memory stores,
      // which the compiler may not move loads past
      constexpr int CPR = D / 8, RPI = 32 / CPR, NI = 32 / RPI, QBATCH = 8;
      const int cj = lane % CPR, rj = lane / CPR;
#pragma unroll
      for (int k0 = 0; k0 < NI; k0 += QBATCH) {
        uint4 v[QBATCH];
#pragma unroll
        for (int b = 0; b < QBATCH; ++b) {
          const __half* sj = reinterpret_cast<const __half*>(__shfl_sync(
              0xffffffffu, reinterpret_cast<unsigned long long>(src), (k0 + b) * RPI + rj));
          v[b] = sj ? *reinterpret_cast<const uint4*>(sj + 8 * cj) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int b = 0; b < QBATCH; ++b)
          *reinterpret_cast<uint4*>(qx + sw128_offset(r - lane + (k0 + b) * RPI + rj, 8 * cj,
                                                      kTcRows)) = v[b];
      }
    } else {
      // fold the K channel scale into the row, scale it by 2^eq so that its
      // largest magnitude lies in [2^13, 2^14), split into fp16 hi + lo
      const float* ksc = pool.chan_scales + (int64_t)h * D;
      char* ql = sm + PL::q + (NT + X) * PL::QB;
      float amax = 0.f;
      if (src)
        for (int d = 0; d < D; ++d) amax = fmaxf(amax, fabsf(__half2float(src[d]) * ksc[d]));
      const int eq = amax > 0.f ? 13 - exponent_of(amax) : 0;
      const float up = ldexpf(1.f, eq);
      csc = ldexpf(csc, -eq);
      for (int c = 0; c < D / 8; ++c) {
        uint4 hv4 = make_uint4(0, 0, 0, 0), lv4 = make_uint4(0, 0, 0, 0);
        if (src) {
          uint32_t* ho = reinterpret_cast<uint32_t*>(&hv4);
          uint32_t* lo = reinterpret_cast<uint32_t*>(&lv4);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int d = 8 * c + 2 * e;
            split_h2(__half2float(src[d]) * ksc[d] * up, __half2float(src[d + 1]) * ksc[d + 1] * up,
                     ho[e], lo[e]);
          }
        }
        *reinterpret_cast<uint4*>(qx + sw128_offset(r, 8 * c, kTcRows)) = hv4;
        *reinterpret_cast<uint4*>(ql + sw128_offset(r, 8 * c, kTcRows)) = lv4;
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const int* trow = p.table + (int64_t)seq * p.max_blocks;

  if (!is_sm) {
    // ======================= converters =======================
    const int cid = tid - NT * kTcRows;
    const int npg = kTcStep / bs;
    // raw codes of one step: [sub-tile][K|V][chunk] for this thread's chunks
    uint4 rv[4][2][NCH];
    float sk = 0.f, sv = 0.f;  // this thread's token scales (cid < 64)
    bool tok_ok = false;       // and whether that token is present
    int tphys[4];              // block ids of the step being loaded
    auto load_table = [&](int j, int (&ph)[4]) {
#pragma unroll
      for (int pg = 0; pg < 4; ++pg) {
        const int tb = j * kTcStep + pg * bs;
        const int n = tb / bs;
        ph[pg] = (pg < npg && tb < kv_end && n < p.max_blocks) ? trow[n] : -1;
      }
    };
    auto page_of = [&](int phys) -> const char* {
      return pool.pages + ((int64_t)phys * pool.Hkv + h) * pool.page_bytes;
    };
    auto phys_ok = [&](int phys) { return phys >= 0 && (int64_t)phys < pool.num_blocks; };
    auto load_step = [&](int j, const int (&ph)[4]) {
      const int t0 = j * kTcStep;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int pg = (16 * s) / bs, sub = ((16 * s) % bs) >> 4;
        const bool ok = phys_ok(ph[pg]) && t0 + 16 * s < kv_end;
        const char* base = ok ? page_of(ph[pg]) + sub * SUB_BYTES : nullptr;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv)
#pragma unroll
          for (int i = 0; i < NCH; ++i) {
            const int ch = cid + i * kTcConv;
            rv[s][kv][i] = (ok && ch < CPS)
                               ? *reinterpret_cast<const uint4*>(base + (kv ? pool.code_bytes : 0) +
                                                                 (ch >> 5) * 512 + (ch & 31) * 16)
                               : make_uint4(0, 0, 0, 0);
          }
      }
      if (cid < kTcStep) {
        const int pg = cid / bs, off = cid - (cid / bs) * bs;
        const bool ok = phys_ok(ph[pg]) && t0 + cid < kv_end;
        tok_ok = ok;
        sk = 0.f;
        sv = ok ? 1.f : 0.f;
        if constexpr (T::group_scales) {
          if (ok) {
            const float* sc = reinterpret_cast<const float*>(page_of(ph[pg]) + 2 * pool.code_bytes);
            sk = sc[off];
            sv = sc[bs + off];
          }
        } else if constexpr (T::token_scales) {
          if (ok) {
            sk = pool.tok_scales[((int64_t)ph[pg] * 2) * bs + off];
            sv = pool.tok_scales[((int64_t)ph[pg] * 2 + 1) * bs + off];
          }
        }
      }
    };
    load_table(0, tphys);
    load_step(0, tphys);
    load_table(1, tphys);
    for (int j = 0; j < nsteps; ++j) {
      const int b = j & 1;
      if (j >= 2 && !tc_wait(&kv_empty[b], ((j >> 1) - 1) & 1, abort_f)) break;
      const int t0 = j * kTcStep;
      char* khb = sm + PL::kh + b * PL::KB;
      char* vtb = sm + PL::vt + b * PL::VB;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int nvalid = min(max(kv_end - (t0 + 16 * s), 0), 16);
#pragma unroll
        for (int kv = 0; kv < 2; ++kv)
#pragma unroll
          for (int i = 0; i < NCH; ++i) {
            const int ch = cid + i * kTcConv;
            if (ch < CPS) tc_convert_chunk<FMT, D>(rv[s][kv][i], ch & 31, ch >> 5, kv == 1, s,
                                                   nvalid, khb, vtb);
          }
      }
      if (cid < kTcStep) {
        // token t0 + cid: its K and V scale (0 for a token that is absent or
        // past the end), and its bit of the step's valid-token mask
        ks_s[b * 64 + cid] = sk;
        vs_s[b * 64 + cid] = sv;
        const uint32_t bits = __ballot_sync(0xffffffffu, tok_ok);
        float vm = sv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
        if (lane == 0) {
          mask_s[b * 2 + (cid >> 5)] = bits;
          vmax_s[b * 2 + (cid >> 5)] = vm;
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&kv_full[b]);
      if (j + 1 < nsteps) {
        int nx[4];
#pragma unroll
        for (int pg = 0; pg < 4; ++pg) nx[pg] = tphys[pg];
        load_step(j + 1, nx);
        load_table(j + 2, tphys);
      }
    }
  } else {
    // ======================= softmax + MMA issue, tile X =======================
    const uint32_t tO = tmem + X * 128, tS = tmem + PL::s_col(X);
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t qa = smem_u32(sm + PL::q + X * PL::QB);
    const uint32_t qla = smem_u32(sm + PL::q + (NT + X) * PL::QB);
    const uint32_t pha = smem_u32(sm + PL::pw + X * 2 * PL::PB);
    const uint32_t pla = pha + PL::PB;
    char* p_hi = sm + PL::pw + X * 2 * PL::PB;
    char* p_lo = p_hi + PL::PB;
    constexpr uint32_t id_s = tc_idesc_f16(128, kTcStep);
    constexpr uint32_t id_o = tc_idesc_f16(128, D);
    const bool issuer = r == 0;  // thread 0 of the tile
    const int bar_id = 1 + X;
    auto issue_s = [&](int j) {  // S = Q K^T of step j (issuer)
      const uint32_t kha = smem_u32(sm + PL::kh + (j & 1) * PL::KB);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * (kTcStep * 128) + (kk & 3) * 32;
        const uint32_t qo = (kk >> 2) * (kTcRows * 128) + (kk & 3) * 32;
        tc_mma_f16(tS, sw128_desc(qa + qo), sw128_desc(kha + ko), id_s, kk > 0);
        if constexpr (CH) tc_mma_f16(tS, sw128_desc(qla + qo), sw128_desc(kha + ko), id_s, 1);
      }
      tc_commit(&s_full[X]);
    };
    bool failed = false;
    if (issuer) {
      if (tc_wait(&kv_full[0], 0, abort_f)) {
        tc_fence_after();
        issue_s(0);
      }
    }
    float m = kNegInf, l = 0.f;
    int E = T::row_scales ? 100 : 14 - kTcSlack;
    for (int j = 0; j < nsteps; ++j) {
      const int b = j & 1;
      bool ok = tc_wait(&s_full[X], j & 1, abort_f);
      // the step's scales and mask were published with kv_full (already
      // complete: S of this step was computed from them)
      ok = ok && tc_wait(&kv_full[b], (j >> 1) & 1, abort_f);
      if (bar_or(bar_id, kTcRows, !ok)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const int t0 = j * kTcStep;
      float z[kTcStep];
      {
        float a[32];
        tc_ld32(tS + lane_base, a);
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = a[i];
        tc_ld32(tS + lane_base + 32, a);
#pragma unroll
        for (int i = 0; i < 32; ++i) z[32 + i] = a[i];
      }
      const float* ksb = ks_s + b * 64;
      const float* vsb = vs_s + b * 64;
      const uint32_t mk0 = mask_s[b * 2], mk1 = mask_s[b * 2 + 1];
      const int lr = lim - t0;  // tokens [0, lr) of this step are attended by this row
      float mx = kNegInf;
      if (lr >= kTcStep && (mk0 & mk1) == 0xffffffffu) {
#pragma unroll
        for (int t = 0; t < kTcStep; t += 4) {
          float a0 = z[t], a1 = z[t + 1], a2 = z[t + 2], a3 = z[t + 3];
          if constexpr (T::row_scales) {
            const float4 k4 = *reinterpret_cast<const float4*>(ksb + t);
            f2_unpack(f2_mul(f2_pack(a0, a1), f2_pack(k4.x, k4.y)), a0, a1);
            f2_unpack(f2_mul(f2_pack(a2, a3), f2_pack(k4.z, k4.w)), a2, a3);
          }
          z[t] = a0;
          z[t + 1] = a1;
          z[t + 2] = a2;
          z[t + 3] = a3;
          mx = fmaxf(mx, fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)));
        }
      } else {
#pragma unroll
        for (int t = 0; t < kTcStep; ++t) {
          const bool okt = t < lr && (((t < 32 ? mk0 : mk1) >> (t & 31)) & 1u);
          z[t] = okt ? (T::row_scales ? z[t] * ksb[t] : z[t]) : kNegInf;
          mx = fmaxf(mx, z[t]);
        }
      }
      // scores in log2 units are z * csc (csc > 0).  The reference maximum m
      // moves only when the step's maximum passes it by more than kTcSlack,
      // so the TMEM accumulator is rescaled only then (or when E drops).
      const float mxz = mx == kNegInf ? kNegInf : mx * csc;
      const float mn = (m == kNegInf || mxz > m + kTcSlack) ? mxz : m;
      const float ms = mn == kNegInf ? 0.f : mn;
      int dE = 0;
      if constexpr (T::row_scales) {
        const float vmax = fmaxf(vmax_s[b * 2], vmax_s[b * 2 + 1]);
        if (vmax > 0.f) {
          const int En = min(E, 13 - kTcSlack - exponent_of(vmax));
          dE = En - E;
          E = En;
        }
      }
      // p' = 2^(z csc - ms + E), the weight before the V scale
      const float nbias = static_cast<float>(E) - ms;
      uint64_t rs2 = f2_pack(0.f, 0.f);
      {
        const uint64_t c2 = f2_pack(csc, csc), b2 = f2_pack(nbias, nbias);
#pragma unroll
        for (int t = 0; t < kTcStep; t += 2) {
          float a0, a1;
          f2_unpack(f2_fma(f2_pack(z[t], z[t + 1]), c2, b2), a0, a1);
          z[t] = fast_exp2(a0);  // 0 for masked tokens
          z[t + 1] = fast_exp2(a1);
          rs2 = f2_add(rs2, f2_pack(z[t], z[t + 1]));
        }
      }
      float rsa, rsb;
      f2_unpack(rs2, rsa, rsb);
      const float alpha = fast_exp2(m - ms);
      l = fmaf(l, alpha, (rsa + rsb) * pow2f(-E));
      m = mn;
      if (j > 0) {
        // O holds steps 0..j-1: the P.V of step j-1 completed before S of
        // step j (one issuing thread, in order)
        const float f = alpha * pow2f(dE);
        if (__any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tc_ld32(tO + lane_base + 32 * c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= f;
            tc_st32(tO + lane_base + 32 * c, o);
          }
          tc_wait_st();
        }
      }
#pragma unroll
      for (int c = 0; c < kTcStep / 8; ++c) {
        uint32_t hv[4], lv[4];
        float vv[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
        if constexpr (T::row_scales) {
          const float4 v0 = *reinterpret_cast<const float4*>(vsb + 8 * c);
          const float4 v1 = *reinterpret_cast<const float4*>(vsb + 8 * c + 4);
          vv[0] = v0.x, vv[1] = v0.y, vv[2] = v0.z, vv[3] = v0.w;
          vv[4] = v1.x, vv[5] = v1.y, vv[6] = v1.z, vv[7] = v1.w;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float w0 = z[8 * c + 2 * e], w1 = z[8 * c + 2 * e + 1];
          // masked tokens (absent, past the end, or causally later) have p' = 0;
          // their V scale is 0 too
          if constexpr (T::row_scales)
            f2_unpack(f2_mul(f2_pack(w0, w1), f2_pack(vv[2 * e], vv[2 * e + 1])), w0, w1);
          tc_split2(w0, w1, hv[e], lv[e]);
        }
        const uint32_t o = sw128_offset(r, 8 * c, kTcRows);
        *reinterpret_cast<uint4*>(p_hi + o) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4*>(p_lo + o) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      bar_or(bar_id, kTcRows, false);  // the tile's weights are written, S is read
      if (issuer) {
        tc_fence_after();
        const uint32_t vta = smem_u32(sm + PL::vt + b * PL::VB);
#pragma unroll
        for (int kk = 0; kk < kTcStep / 16; ++kk)
          tc_mma_f16(tO, sw128_desc(pha + kk * 32), sw128_desc(vta + kk * 32), id_o,
                     (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kTcStep / 16; ++kk)
          tc_mma_f16(tO, sw128_desc(pla + kk * 32), sw128_desc(vta + kk * 32), id_o, 1u);
        tc_commit(&kv_empty[b]);
        if (j + 1 < nsteps) {
          if (tc_wait(&kv_full[(j + 1) & 1], ((j + 1) >> 1) & 1, abort_f)) {
            tc_fence_after();
            issue_s(j + 1);
          }
        } else {
          tc_commit(&o_full[X]);
        }
      }
      __syncwarp();
    }
    if (!failed) {
      // ---- normalised output rows once the tile's last P.V is done
      bool ok = tc_wait(&o_full[X], 0, abort_f);
      if (bar_or(bar_id, kTcRows, !ok)) {
        failed = true;
      } else {
        tc_fence_after();
        const float f = l > 0.f ? pow2f(-E) / l : 0.f;
        const float* vch = CH ? pool.chan_scales + ((int64_t)pool.Hkv + h) * D : nullptr;
        // Each warp passes 16-column blocks of its 32 rows through shared
        // memory (the tile's weight buffer, free once its last P.V is done),
        // so that a store instruction covers 8 rows x 64 contiguous bytes
        // instead of 32 rows x 16 bytes.  Writer: lane = row, chunk q4 at
        // position q4 ^ ((row / 2) % 4); reader: row 8k + lane / 4, chunk
        // lane % 4 (both conflict-free).
        float* scr = reinterpret_cast<float*>(sm + PL::pw + X * 2 * PL::PB) + (warp & 3) * (32 * 16);
        const int rb = lane >> 2, cb = lane & 3;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tc_ld32(tO + lane_base + 32 * c, o);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const float* oo = o + 16 * hh + 4 * q4;
              float4 v = make_float4(oo[0] * f, oo[1] * f, oo[2] * f, oo[3] * f);
              if constexpr (CH) {
                const float* cs = vch + 32 * c + 16 * hh + 4 * q4;
                v.x *= cs[0];
                v.y *= cs[1];
                v.z *= cs[2];
                v.w *= cs[3];
              }
              *reinterpret_cast<float4*>(scr + lane * 16 + 4 * (q4 ^ ((lane >> 1) & 3))) = v;
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int rw = 8 * k + rb;
              const long long orow_k = __shfl_sync(0xffffffffu, static_cast<long long>(orow), rw);
              const float4 v = *reinterpret_cast<const float4*>(scr + rw * 16 + 4 * (cb ^ ((rw >> 1) & 3)));
              if (orow_k >= 0)
                *reinterpret_cast<float4*>(p.out + orow_k * D + 32 * c + 16 * hh + 4 * cb) = v;
            }
            __syncwarp();
          }
        }
      }
    }
    if (issuer) {
      // every MMA this thread issued has completed before TMEM is freed
      tc_commit(&drain[X]);
      bool ok = false;
      for (int tries = 0; tries < kWaitTries && !ok; ++tries) ok = mbar_try_wait(&drain[X], 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_f) set_error(pool.err, ERR_TIMEOUT);
  if (warp == 0) tc_dealloc(tmem, PL::cols);
}

struct PrefillTcLaunch {
  PrefillTcParams p;
  dim3 grid;
  cudaStream_t st;
};

template <int FMT, int D, int NT>
cudaError_t run_prefill_tc(const PrefillTcLaunch& l) {
  using PL = TcPlan<D, NT, FmtTraits<FMT>::channel>;
  static_assert(PL::request <= 227 * 1024, "shared memory plan too large");
  cudaError_t e = allow_big_smem<kvq_prefill_tc_kernel<FMT, D, NT>>();
  if (e != cudaSuccess) return e;
  kvq_prefill_tc_kernel<FMT, D, NT><<<l.grid, PL::threads, PL::request, l.st>>>(l.p);
  return phase_mark(l.st, cudaGetLastError());
}

}  // namespace kvq
