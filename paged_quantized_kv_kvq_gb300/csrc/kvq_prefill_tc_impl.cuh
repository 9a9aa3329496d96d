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
// GB300 design.  A CTA takes one (sequence, kv head) and 128 Q rows -- the
// (query token, Q head of the group) pairs, 32 query tokens x 4 heads for GQA
// 4:1 -- and walks the keys in steps of 64 tokens:
//   1. the step's pages, brought into a shared-memory stage by bulk copies
//      issued one step ahead, are turned by the 128 threads into exact fp16
//      values: K as a 64 x D tile, V transposed as a D x 64 tile, both K-major
//      with the 128-byte swizzle; the step's per-token scales go to shared
//      memory;
//   2. one thread issues S = Q.K^T (M 128, N 64, K = D) into tensor memory;
//   3. each thread owns one row: it reads its 64 scores from TMEM, applies
//      the K scales, the causal limit and the online softmax (base 2), and
//      writes the weights p * s_V * 2^E as an fp16 high part and an fp16 low
//      part (one K-major 128 x 64 tile each; the low part reuses the K tile,
//      which S no longer needs); its exponent reference moves only when a
//      score passes it by more than 2^8, and only then (or when E drops) is
//      its row of the output accumulator in TMEM rescaled;
//   4. one thread issues O += P_hi.V + P_lo.V (M 128, N D, K 64) into TMEM.
// Codes are exact in fp16, so dequantization is a scale outside the
// contraction, as in the decode kernel; the hi + lo split keeps the weights
// exact to ~2^-22.  The output row is normalised once at the end.  Two CTAs
// share an SM (at most ~113 KB of shared memory and 256 TMEM columns each),
// so one CTA's tensor work overlaps the other's conversion and softmax.  Every
// wait on the MMA barrier is bounded; a wait that runs out sets the pool's
// timeout bit, waits (bounded) for the MMAs in flight and frees TMEM.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "kvq_decode_impl.cuh"
#include "kvq_tc.cuh"

namespace kvq {

constexpr int kTcThreads = 128;   // = Q rows per CTA = TMEM lanes
constexpr int kTcStep = 64;       // key tokens per step
constexpr int kTcCols = 256;      // TMEM columns: O at [0, D), S at [128, 192)
constexpr int kTcSCol = 128;
constexpr int kTcSlack = 8;       // log2 of how far a row may exceed its reference maximum

struct PrefillTcParams {
  PoolView pool;
  const __half* q;      // [Tq][Hq][D]
  const int* table;     // [S][max_blocks]
  const int* lens;      // [S]
  const int* q_start;   // [S + 1]
  float* out;           // [Tq][Hq][D]
  int S, Hq, G, max_blocks, max_ctx;
  int ntiles;           // 128-row tiles per (sequence, kv head)
  float sm_scale_log2;
  // shared-memory plan (byte offsets from a 1024-byte aligned base)
  int off_qlo, off_kh, off_vt, off_phi, off_plo, off_raw, off_misc;
  int npg;              // pages per key step (64 / block size)
  int pstride;          // bytes of one page slot of the raw stage
  int tok_bytes;        // per-token scale bytes copied after each page (0 otherwise)
};

// The misc block: float ks[64], vs[64], vmax[2]; uint32 tmask[2]; float
// red[4]; int stage_ok[4]; uint64 bar_mma, bar_raw; uint32 tslot.
constexpr int kMiscKs = 0, kMiscVs = 256, kMiscVmax = 512, kMiscMask = 520, kMiscRed = 528,
              kMiscOk = 544, kMiscBarMma = 560, kMiscBarRaw = 568, kMiscSlot = 576,
              kMiscBytes = 640;

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

// Bounded wait on an mbarrier by every thread; CTA-uniform result.
__device__ __forceinline__ bool tc_wait_bar(uint64_t* bar, uint32_t parity) {
  bool ok = false;
  for (int tries = 0; tries < kWaitTries && !ok; ++tries) ok = mbar_try_wait(bar, parity);
  return !__syncthreads_or(!ok);
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

template <int FMT, int D>
__global__ void __launch_bounds__(kTcThreads, 2) kvq_prefill_tc_kernel(const PrefillTcParams p) {
  using T = FmtTraits<FMT>;
  constexpr bool CH = T::channel;
  const float kNegInf = __int_as_float(0xff800000u);

  extern __shared__ __align__(1024) char smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  char* sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PoolView& pool = p.pool;
  const int bs = pool.bs;
  // heaviest tiles (longest causal ranges) first
  const int per_tile = p.S * pool.Hkv;
  const int tile = p.ntiles - 1 - static_cast<int>(blockIdx.x / per_tile);
  const int seq = static_cast<int>(blockIdx.x % per_tile) % p.S;
  const int h = static_cast<int>(blockIdx.x % per_tile) / p.S;

  const int qbase = p.q_start[seq];
  const int nq = p.q_start[seq + 1] - qbase;
  int ctx = p.lens[seq];
  if (ctx > p.max_ctx || ctx < nq) {
    if (tile == 0 && h == 0 && tid == 0) set_error(pool.err, ERR_RANGE);
    ctx = min(ctx, p.max_ctx);
  }
  const int rows_total = nq * p.G;
  if (tile * kTcThreads >= rows_total) return;  // CTA-uniform

  // ---- this thread's row and the CTA's key range
  const int rr = tile * kTcThreads + tid;
  const bool row_ok = rr < rows_total;
  const int lim = row_ok ? max(0, ctx - nq + rr / p.G + 1) : 0;
  int64_t orow = -1;
  if (row_ok) orow = (int64_t)(qbase + rr / p.G) * p.Hq + h * p.G + rr % p.G;
  const int last = min(rows_total, (tile + 1) * kTcThreads) - 1;
  const int kv_end = max(0, min(ctx, ctx - nq + last / p.G + 1));
  const int nsteps = (kv_end + kTcStep - 1) / kTcStep;
  if (nsteps == 0) {  // nothing to attend: zeros (CTA-uniform)
    if (row_ok)
      for (int d = 0; d < D; ++d) p.out[orow * D + d] = 0.f;
    return;
  }

  char* q_hi = sm;
  char* q_lo = sm + p.off_qlo;
  char* kh = sm + p.off_kh;
  char* vt = sm + p.off_vt;
  char* p_hi = sm + p.off_phi;
  char* p_lo = sm + p.off_plo;  // may be the K tile: free once S is computed
  char* raw = sm + p.off_raw;
  char* misc = sm + p.off_misc;
  float* ks_s = reinterpret_cast<float*>(misc + kMiscKs);
  float* vs_s = reinterpret_cast<float*>(misc + kMiscVs);
  float* vmax_s = reinterpret_cast<float*>(misc + kMiscVmax);
  uint32_t* tmask_s = reinterpret_cast<uint32_t*>(misc + kMiscMask);
  float* red = reinterpret_cast<float*>(misc + kMiscRed);
  int* stage_ok = reinterpret_cast<int*>(misc + kMiscOk);
  uint64_t* bar_mma = reinterpret_cast<uint64_t*>(misc + kMiscBarMma);
  uint64_t* bar_raw = reinterpret_cast<uint64_t*>(misc + kMiscBarRaw);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(misc + kMiscSlot);
  const int* trow = p.table + (int64_t)seq * p.max_blocks;

  // Thread 0: bulk-copy the pages of key step j into the raw stage, one
  // transaction count on bar_raw (a plain arrival when no page is present).
  auto issue_step = [&](int j) {
    uint32_t total = 0;
    int phys[4];
    for (int pg = 0; pg < p.npg; ++pg) {
      const int tb = j * kTcStep + pg * bs;
      const int n = tb / bs;
      phys[pg] = (tb < kv_end && n < p.max_blocks) ? trow[n] : -1;
      const bool ok = phys[pg] >= 0 && (int64_t)phys[pg] < pool.num_blocks;
      if (tb < kv_end && !ok) set_error(pool.err, ERR_RANGE);
      if (!ok) phys[pg] = -1;
      stage_ok[pg] = ok ? 1 : 0;
      if (ok) total += pool.page_bytes + p.tok_bytes;
    }
    if (total == 0) {
      mbar_arrive(bar_raw);
      return;
    }
    mbar_arrive_expect_tx(bar_raw, total);
    for (int pg = 0; pg < p.npg; ++pg) {
      if (phys[pg] < 0) continue;
      char* dst = raw + pg * p.pstride;
      bulk_g2s(dst, pool.pages + ((int64_t)phys[pg] * pool.Hkv + h) * pool.page_bytes,
               pool.page_bytes, bar_raw);
      if (p.tok_bytes)
        bulk_g2s(dst + pool.page_bytes, pool.tok_scales + (int64_t)phys[pg] * 2 * bs, p.tok_bytes,
                 bar_raw);
    }
  };

  // ---- barriers, the first step's pages, TMEM (warp 0 allocates)
  if (tid == 0) {
    mbar_init(bar_mma, 1);
    mbar_init(bar_raw, 1);
    fence_barrier_init();
    issue_step(0);
  }
  if (warp == 0) tc_alloc(tslot, kTcCols);

  // ---- Q tile (rows of this CTA, zero past the chunk), K-major swizzled
  float csc = p.sm_scale_log2;
  auto q_row_ptr = [&](int r) -> const __half* {
    const int x = tile * kTcThreads + r;
    if (x >= rows_total) return nullptr;
    return p.q + ((int64_t)(qbase + x / p.G) * p.Hq + h * p.G + x % p.G) * D;
  };
  if constexpr (!CH) {
    for (int it = tid; it < kTcThreads * (D / 8); it += kTcThreads) {
      const int r = it / (D / 8), c = it % (D / 8);
      const __half* src = q_row_ptr(r);
      const uint4 v = src ? *reinterpret_cast<const uint4*>(src + 8 * c) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(q_hi + sw128_offset(r, 8 * c, kTcThreads)) = v;
    }
  } else {
    // fold the K channel scale into q, scale the tile by 2^eq so that its
    // largest magnitude lies in [2^13, 2^14), split into fp16 hi + lo
    const float* ksc = pool.chan_scales + (int64_t)h * D;
    float amax = 0.f;
    for (int it = tid; it < kTcThreads * (D / 8); it += kTcThreads) {
      const int r = it / (D / 8), c = it % (D / 8);
      const __half* src = q_row_ptr(r);
      if (src == nullptr) continue;
      const uint4 v = *reinterpret_cast<const uint4*>(src + 8 * c);
      const __half* hv = reinterpret_cast<const __half*>(&v);
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(__half2float(hv[e]) * ksc[8 * c + e]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const int eq = amax > 0.f ? 13 - exponent_of(amax) : 0;
    const float up = ldexpf(1.f, eq);
    csc = ldexpf(csc, -eq);
    for (int it = tid; it < kTcThreads * (D / 8); it += kTcThreads) {
      const int r = it / (D / 8), c = it % (D / 8);
      const __half* src = q_row_ptr(r);
      uint4 hv4 = make_uint4(0, 0, 0, 0), lv4 = make_uint4(0, 0, 0, 0);
      if (src != nullptr) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + 8 * c);
        const __half* hv = reinterpret_cast<const __half*>(&v);
        uint32_t* ho = reinterpret_cast<uint32_t*>(&hv4);
        uint32_t* lo = reinterpret_cast<uint32_t*>(&lv4);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          split_h2(__half2float(hv[2 * e]) * ksc[8 * c + 2 * e] * up,
                   __half2float(hv[2 * e + 1]) * ksc[8 * c + 2 * e + 1] * up, ho[e], lo[e]);
      }
      *reinterpret_cast<uint4*>(q_hi + sw128_offset(r, 8 * c, kTcThreads)) = hv4;
      *reinterpret_cast<uint4*>(q_lo + sw128_offset(r, 8 * c, kTcThreads)) = lv4;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tO = tmem, tS = tmem + kTcSCol;
  const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;

  const uint32_t qhi_a = smem_u32(q_hi), qlo_a = smem_u32(q_lo), kh_a = smem_u32(kh),
                 vt_a = smem_u32(vt), phi_a = smem_u32(p_hi), plo_a = smem_u32(p_lo);
  constexpr uint32_t id_s = tc_idesc_f16(128, kTcStep);
  constexpr uint32_t id_o = tc_idesc_f16(128, D);

  float m = kNegInf, l = 0.f;
  int E = T::row_scales ? 100 : 14 - kTcSlack;
  uint32_t ph_mma = 0, ph_raw = 0;
  bool failed = false;

  for (int jstep = 0; jstep < nsteps; ++jstep) {
    const int t0 = jstep * kTcStep;
    // ---- 1. this step's pages have landed: codes -> fp16 tiles, scales
    if (!tc_wait_bar(bar_raw, ph_raw)) {
      failed = true;
      break;
    }
    ph_raw ^= 1u;
    if (tid < kTcStep) {
      const int t = t0 + tid;
      const int pg = tid / bs, off = tid - pg * bs;
      const bool ok = stage_ok[pg] != 0 && t < kv_end;
      const char* page = raw + pg * p.pstride;
      float k_s = 1.f, v_s = 1.f;
      if constexpr (T::group_scales) {
        const float* sc = reinterpret_cast<const float*>(page + 2 * pool.code_bytes);
        k_s = ok ? sc[off] : 0.f;
        v_s = ok ? sc[bs + off] : 0.f;
      } else if constexpr (T::token_scales) {
        const float* sc = reinterpret_cast<const float*>(page + pool.page_bytes);
        k_s = ok ? sc[off] : 0.f;
        v_s = ok ? sc[bs + off] : 0.f;
      } else {
        v_s = ok ? 1.f : 0.f;
      }
      ks_s[tid] = k_s * csc;
      vs_s[tid] = v_s;
      const uint32_t bits = __ballot_sync(0xffffffffu, ok);
      float vm = v_s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
      if (lane == 0) {
        tmask_s[warp] = bits;
        vmax_s[warp] = vm;
      }
    }
    {
      constexpr int ES = FMT == FMT_FP16 ? 2 : 1;
      constexpr int SUB_BYTES = FMT == FMT_INT4_GROUP ? 8 * D : 16 * D * ES;
      constexpr int CPS = SUB_BYTES / 16;  // 16-byte chunks per K (or V) sub-tile
      for (int it = tid; it < 8 * CPS; it += kTcThreads) {
        const int s = it / (2 * CPS), rem = it - s * (2 * CPS);
        const bool isv = rem >= CPS;
        const int ch = isv ? rem - CPS : rem;
        const int pg = (16 * s) / bs, sub = ((16 * s) % bs) >> 4;
        const int nvalid = min(max(kv_end - (t0 + 16 * s), 0), 16);
        const bool ok = stage_ok[pg] != 0 && nvalid > 0;
        uint4 rv = make_uint4(0, 0, 0, 0);
        if (ok)
          rv = *reinterpret_cast<const uint4*>(raw + pg * p.pstride + (isv ? pool.code_bytes : 0) +
                                               sub * SUB_BYTES + (ch >> 5) * 512 + (ch & 31) * 16);
        tc_convert_chunk<FMT, D>(rv, ch & 31, ch >> 5, isv, s, ok ? nvalid : 0, kh, vt);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 2. the raw stage is free: fetch the next step; S = Q K^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * (kTcStep * 128) + (kk & 3) * 32;
        const uint32_t qo = (kk >> 2) * (kTcThreads * 128) + (kk & 3) * 32;
        tc_mma_f16(tS, sw128_desc(qhi_a + qo), sw128_desc(kh_a + ko), id_s, kk > 0);
        if constexpr (CH) tc_mma_f16(tS, sw128_desc(qlo_a + qo), sw128_desc(kh_a + ko), id_s, 1);
      }
      tc_commit(bar_mma);
      if (jstep + 1 < nsteps) issue_step(jstep + 1);
    }
    if (!tc_wait_bar(bar_mma, ph_mma)) {
      failed = true;
      break;
    }
    ph_mma ^= 1u;
    tc_fence_after();

    // ---- 3. online softmax of this thread's row (base 2); the weights carry
    // the V scale and 2^E, which is folded into the exponent
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
    const uint32_t mk0 = tmask_s[0], mk1 = tmask_s[1];
    const int lr = lim - t0;  // tokens [0, lr) of this step are attended by this row
    float mx = kNegInf;
    if (lr >= kTcStep && (mk0 & mk1) == 0xffffffffu) {
#pragma unroll
      for (int t = 0; t < kTcStep; t += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(ks_s + t);
        float a0, a1, a2, a3;
        f2_unpack(f2_mul(f2_pack(z[t], z[t + 1]), f2_pack(k4.x, k4.y)), a0, a1);
        f2_unpack(f2_mul(f2_pack(z[t + 2], z[t + 3]), f2_pack(k4.z, k4.w)), a2, a3);
        z[t] = a0;
        z[t + 1] = a1;
        z[t + 2] = a2;
        z[t + 3] = a3;
        mx = fmaxf(mx, fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)));
      }
    } else {
#pragma unroll
      for (int t = 0; t < kTcStep; ++t) {
        const bool ok = t < lr && (((t < 32 ? mk0 : mk1) >> (t & 31)) & 1u);
        z[t] = ok ? z[t] * ks_s[t] : kNegInf;
        mx = fmaxf(mx, z[t]);
      }
    }
    // The row's reference maximum m moves only when the step's maximum passes
    // it by more than kTcSlack (weights then stay below 2^kTcSlack, and the
    // 2^E prescale leaves that much headroom below the fp16 range), so the
    // accumulator in TMEM is rescaled only on such a jump or when E drops.
    const float mn = (m == kNegInf || mx > m + kTcSlack) ? mx : m;
    const float ms = mn == kNegInf ? 0.f : mn;
    int dE = 0;
    if constexpr (T::row_scales) {
      const float vmax = fmaxf(vmax_s[0], vmax_s[1]);
      if (vmax > 0.f) {
        const int En = min(E, 13 - kTcSlack - exponent_of(vmax));
        dE = En - E;
        E = En;
      }
    }
    // p' = 2^(z - ms + E): the weights before the V scale
    const float bias = ms - static_cast<float>(E);
    uint64_t rs2 = f2_pack(0.f, 0.f);
    {
      const uint64_t b2 = f2_pack(bias, bias);
#pragma unroll
      for (int t = 0; t < kTcStep; t += 2) {
        float a0, a1;
        f2_unpack(f2_sub(f2_pack(z[t], z[t + 1]), b2), a0, a1);
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
    if (jstep > 0) {
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
      if constexpr (T::row_scales) {
        const float4 v0 = *reinterpret_cast<const float4*>(vs_s + 8 * c);
        const float4 v1 = *reinterpret_cast<const float4*>(vs_s + 8 * c + 4);
        const float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float w0, w1;
          f2_unpack(f2_mul(f2_pack(z[8 * c + 2 * e], z[8 * c + 2 * e + 1]),
                           f2_pack(vv[2 * e], vv[2 * e + 1])), w0, w1);
          tc_split2(w0, w1, hv[e], lv[e]);
        }
      } else {
        // no V scale: masked tokens already have p' = 0; a token of an absent
        // page has vs = 0
        const float4 v0 = *reinterpret_cast<const float4*>(vs_s + 8 * c);
        const float4 v1 = *reinterpret_cast<const float4*>(vs_s + 8 * c + 4);
        const float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          tc_split2(vv[2 * e] != 0.f ? z[8 * c + 2 * e] : 0.f,
                    vv[2 * e + 1] != 0.f ? z[8 * c + 2 * e + 1] : 0.f, hv[e], lv[e]);
      }
      const uint32_t o = sw128_offset(tid, 8 * c, kTcThreads);
      *reinterpret_cast<uint4*>(p_hi + o) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
      *reinterpret_cast<uint4*>(p_lo + o) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 4. O += P_hi V + P_lo V
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTcStep / 16; ++kk)
        tc_mma_f16(tO, sw128_desc(phi_a + kk * 32), sw128_desc(vt_a + kk * 32), id_o,
                   (jstep > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < kTcStep / 16; ++kk)
        tc_mma_f16(tO, sw128_desc(plo_a + kk * 32), sw128_desc(vt_a + kk * 32), id_o, 1u);
      tc_commit(bar_mma);
    }
    if (!tc_wait_bar(bar_mma, ph_mma)) {
      failed = true;
      break;
    }
    ph_mma ^= 1u;
    tc_fence_after();
  }

  if (failed) {
    // a wait ran out: flag it, wait (bounded) for the MMAs and copies in
    // flight, free TMEM
    if (tid == 0) set_error(pool.err, ERR_TIMEOUT);
    tc_wait_bar(bar_mma, ph_mma);
    tc_wait_bar(bar_raw, ph_raw);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, kTcCols);
    return;
  }

  // ---- normalised output row
  {
    const float f = l > 0.f ? pow2f(-E) / l : 0.f;
    const float* vch = CH ? pool.chan_scales + ((int64_t)pool.Hkv + h) * D : nullptr;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float o[32];
      tc_ld32(tO + lane_base + 32 * c, o);
      if (row_ok) {
        float4* dst = reinterpret_cast<float4*>(p.out + orow * D + 32 * c);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 v = make_float4(o[4 * i] * f, o[4 * i + 1] * f, o[4 * i + 2] * f, o[4 * i + 3] * f);
          if constexpr (CH) {
            const float* cs = vch + 32 * c + 4 * i;
            v.x *= cs[0];
            v.y *= cs[1];
            v.z *= cs[2];
            v.w *= cs[3];
          }
          dst[i] = v;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, kTcCols);
}

struct PrefillTcLaunch {
  PrefillTcParams p;
  dim3 grid;
  int smem;
  cudaStream_t st;
};

template <int FMT, int D>
cudaError_t run_prefill_tc(const PrefillTcLaunch& l) {
  cudaError_t e = allow_big_smem<kvq_prefill_tc_kernel<FMT, D>>();
  if (e != cudaSuccess) return e;
  kvq_prefill_tc_kernel<FMT, D><<<l.grid, kTcThreads, l.smem, l.st>>>(l.p);
  return cudaGetLastError();
}

}  // namespace kvq
