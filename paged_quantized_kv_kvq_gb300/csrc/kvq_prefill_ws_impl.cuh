// kvq_prefill_ws_impl.cuh -- prefill / chunked-prefill attention over a
// quantized paged KV pool in two passes through a caller workspace, on the
// 5th-generation tensor cores.
//
// Method ("KV Cache优化实战：大模型推理显存占用与加速方案详解",
// 0539edu.com/news/5800990, §1.1): query token i of a chunk of n tokens of a
// sequence whose cache holds L tokens (the chunk included) sits at position
// L - n + i and attends to positions 0 .. L - n + i of the block-paged cache
// (§2.2), whose K/V are stored as codes with scales (§2.3, §3.3).
//
// Why two passes.  Every 64-token key step of a (sequence, kv head) is read
// by every CTA whose query rows come after it -- 16 of them on average for a
// 2048-token prompt -- and in the one-pass kernel each of those CTAs turns
// the codes into fp16 again, on the same SM issue slots the softmax needs.
// Here a staging pass does that once per step: it writes the step's codes as
// exact fp16 values, already in the layout the tensor core reads from shared
// memory (K as a 64 x D tile, V transposed as a D x 64 tile, both K-major
// with the 128-byte swizzle), plus the step's per-token K and V scales, its
// valid-token mask and its largest V scale, into one record of the
// workspace.  The scales stay outside the contraction exactly as in the
// one-pass kernel, so the arithmetic is the same; only where the fp16 copy
// of the codes is made differs.
//
// The attention pass: a work item is one (sequence, kv head) and two tiles
// of 128 Q rows (one tile for per-channel pools, whose Q has a low part too);
// the grid is persistent, one CTA per SM taking every grid-th item, longest
// items first.  The CTA's eight softmax warps own the rows (one row per
// thread, one TMEM lane each); a copier thread bulk-copies the step records
// into four shared-memory stages the moment each is free, running ahead
// across items, and one control thread per tile issues that tile's
// tcgen05.mma.  Per tile, tensor memory holds the output accumulator O, the
// step's scores S and the step's weights P:
//   * the control thread issues S = Q.K^T (M 128, N 64, K D, A and B from
//     shared memory) for every tile once the step's record has landed and the
//     tile has read its previous S;
//   * each softmax thread reads its row of S, signals that S may be
//     overwritten, applies the K scales, the causal limit and the online
//     softmax (base 2), and writes the weights p * s_V * 2^E as fp16 high and
//     low parts into P with tcgen05.st; the row's exponent reference moves
//     only when a score passes it by more than 2^8, and only then (or when E
//     drops) is its row of O rescaled;
//   * the control thread then issues O += P_hi.V + P_lo.V (M 128, N D, K 64,
//     A from tensor memory, V^T from shared memory).
// So the next step's S is computed while the softmax of the current one runs,
// and the two tiles' softmax and tensor work interleave.  The next item's Q
// rows are loaded before the current item's epilogue, whose output rows go
// out through a per-warp shared-memory transpose.  The threads meet
// only at mbarriers; every wait is bounded and gives up early once another
// role has given up; the CTA then flags a timeout, waits (bounded) for its
// copies and MMAs in flight, and frees TMEM.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "kvq_prefill_tc_impl.cuh"

namespace kvq {

// One staged key step of one (sequence, kv head) in the workspace.
template <int D>
struct StepRec {
  static constexpr int KB = kTcStep * D * 2, VB = D * kTcStep * 2;
  static constexpr int kh = 0, vt = KB;             // fp16 tiles, swizzled K-major
  static constexpr int ks = KB + VB;                // float[64] K scales (0: absent token)
  static constexpr int vs = ks + 256;               // float[64] V scales (0: absent token)
  static constexpr int mask = vs + 256;             // uint32[2] valid tokens
  static constexpr int vmax = mask + 8;             // float[2] largest V scale per half
  static constexpr int copy = vmax + 8;             // bytes the attention pass copies
  static constexpr int bytes = (copy + 1023) / 1024 * 1024;  // record stride
};

struct StageParams {
  PoolView pool;
  const int* table;  // [S][max_blocks]
  const int* lens;   // [S]
  char* ws;          // records [S][max_steps][Hkv]
  int S, max_blocks, max_ctx, max_steps;
};

// Staging pass: one CTA of 128 threads per (sequence, key step, kv head).
template <int FMT, int D>
__global__ void __launch_bounds__(128) kvq_prefill_stage_kernel(const StageParams p) {
  using T = FmtTraits<FMT>;
  using R = StepRec<D>;
  constexpr int SUB_BYTES = FMT == FMT_INT4_GROUP ? 8 * D : 16 * D * (FMT == FMT_FP16 ? 2 : 1);
  constexpr int CPS = SUB_BYTES / 16;
  const PoolView& pool = p.pool;
  const int bs = pool.bs;
  const int h = blockIdx.x % pool.Hkv;
  const int j = (blockIdx.x / pool.Hkv) % p.max_steps;
  const int s = blockIdx.x / (pool.Hkv * p.max_steps);
  const int ctx = min(p.lens[s], p.max_ctx);
  const int t0 = j * kTcStep;
  if (t0 >= ctx) return;
  char* rec = p.ws + ((int64_t)(s * p.max_steps + j) * pool.Hkv + h) * R::bytes;
  const int* trow = p.table + (int64_t)s * p.max_blocks;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto page_of = [&](int t, int& off) -> const char* {  // the page of token t, or null
    const int n = t / bs;
    off = t - n * bs;
    const int phys = n < p.max_blocks ? trow[n] : -1;
    if (phys < 0 || (int64_t)phys >= pool.num_blocks) return nullptr;
    return pool.pages + ((int64_t)phys * pool.Hkv + h) * pool.page_bytes;
  };
  // codes -> fp16 tiles
  for (int it = tid; it < 8 * CPS; it += 128) {
    const int s4 = it / (2 * CPS), rem = it - s4 * (2 * CPS);
    const bool isv = rem >= CPS;
    const int ch = isv ? rem - CPS : rem;
    int off;
    const char* page = page_of(t0 + 16 * s4, off);
    const int nvalid = page ? min(max(ctx - (t0 + 16 * s4), 0), 16) : 0;
    uint4 rv = make_uint4(0, 0, 0, 0);
    if (nvalid > 0)
      rv = *reinterpret_cast<const uint4*>(page + (isv ? pool.code_bytes : 0) + (off >> 4) * SUB_BYTES +
                                           (ch >> 5) * 512 + (ch & 31) * 16);
    tc_convert_chunk<FMT, D>(rv, ch & 31, ch >> 5, isv, s4, nvalid, rec + R::kh, rec + R::vt);
  }
  // per-token scales, the valid-token mask, the largest V scale
  if (tid < kTcStep) {
    const int t = t0 + tid;
    int off;
    const char* page = t < ctx ? page_of(t, off) : nullptr;
    if (t < ctx && page == nullptr && (off == 0 || tid == 0)) set_error(pool.err, ERR_RANGE);
    const bool ok = page != nullptr;
    float sk = 0.f, sv = ok ? 1.f : 0.f;
    if (ok) {
      if constexpr (T::group_scales) {
        const float* sc = reinterpret_cast<const float*>(page + 2 * pool.code_bytes);
        sk = sc[off];
        sv = sc[bs + off];
      } else if constexpr (T::token_scales) {
        const int64_t blk = (page - pool.pages) / ((int64_t)pool.Hkv * pool.page_bytes);
        sk = pool.tok_scales[(blk * 2) * bs + off];
        sv = pool.tok_scales[(blk * 2 + 1) * bs + off];
      }
    }
    reinterpret_cast<float*>(rec + R::ks)[tid] = sk;
    reinterpret_cast<float*>(rec + R::vs)[tid] = sv;
    const uint32_t bits = __ballot_sync(0xffffffffu, ok);
    float vm = sv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
    if (lane == 0) {
      reinterpret_cast<uint32_t*>(rec + R::mask)[warp] = bits;
      reinterpret_cast<float*>(rec + R::vmax)[warp] = vm;
    }
  }
}

struct PrefillWsParams {
  PoolView pool;
  const __half* q;      // [Tq][Hq][D]
  const int* lens;      // [S]
  const int* q_start;   // [S + 1]
  float* out;           // [Tq][Hq][D]
  const char* ws;       // staged records
  int S, Hq, G, max_ctx, max_steps;
  int ngroups;          // CTAs per (sequence, kv head): ceil(tiles / NT)
  float sm_scale_log2;
};

constexpr int kWsStages = 4;  // record stages in shared memory

template <int FMT>
struct WsShape {
  static constexpr int NT = FMT == FMT_INT8_CHANNEL ? 1 : 2;
};

// Wait on an mbarrier phase with one lane of the warp spinning (bounded, see
// tc_wait); the warp barrier then orders the other lanes' later accesses
// after that lane's acquire (one test per lane instead would be 32 atomic
// reads of the same word).  Warp-uniform result.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = tc_wait(bar, parity, abort);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok;
}

// One arrival for the whole warp, after every lane's prior work (a warp-wide
// arrive would be 32 atomic updates of the same word).  The lanes' shared
// memory writes, tensor memory accesses (each lane fenced with
// tcgen05.fence::before_thread_sync) and proxy fences are ordered before the
// arrival by the warp barrier.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Shared-memory plan of the attention pass (offsets from a 1024-byte aligned
// base): Q tiles (and low parts), kWsStages record stages, misc (flags and
// mbarriers), the softmax warps' output transpose blocks.
template <int D, int NT, bool CH>
struct WsPlan {
  using R = StepRec<D>;
  static constexpr int QB = kTcRows * D * 2;
  static constexpr int q = 0;
  static constexpr int stage = NT * QB * (CH ? 2 : 1);     // [kWsStages][R::bytes]
  static constexpr int misc = stage + kWsStages * R::bytes;
  // misc: int abort; uint64 kv_full[S], kv_empty[S], s_full[NT], s_read[NT],
  // p_full[NT], pv_done[NT], o_full[NT], q_full[NT], drain; uint32 tslot
  static constexpr int abort = misc, bars = misc + 8;
  static constexpr int nbars = 2 * kWsStages + 6 * NT + 1;
  static constexpr int tslot = bars + 8 * nbars;
  // per softmax warp, a 32-row x 16-float block of its output rows on their
  // way to global memory (rows 64 bytes apart, 16-byte chunks swizzled)
  static constexpr int oscr = misc + 256;
  static constexpr int OSCR_WARP = 32 * 16 * 4;
  static constexpr int request = oscr + 4 * NT * OSCR_WARP + 1024;  // + alignment slack
  static_assert(tslot + 16 <= oscr, "mbarriers overlap the output blocks");
  // the softmax warps, one control warp per tile (its lane 0 issues that
  // tile's MMAs) and a copier warp (its lane 0 issues the record copies)
  static constexpr int threads = kTcRows * NT + 32 * NT + 32;
  // TMEM: per tile x, O at 128x (D columns), S at 256 + 128x (64), P at S + 64
  // (32 columns of fp16 pairs for the high part, 32 for the low part); one
  // tile: O 0, S 128, P 192
  static constexpr int cols = NT == 2 ? 512 : 256;
  static constexpr int s_col(int x) { return NT == 2 ? 256 + 128 * x : 128; }
};

// One work item of the attention pass: NT tiles of 128 Q rows of one
// (sequence, kv head).  Items are numbered heaviest (longest causal range)
// first; a CTA takes items blockIdx.x, blockIdx.x + gridDim.x, ...
struct WsItem {
  int seq, h, qbase, nq, ctx, rows_total, row0, kv_end, nsteps;
  bool bad_ctx;
};

template <int NT>
__device__ __forceinline__ WsItem ws_item(const PrefillWsParams& p, int i) {
  const int per = p.S * p.pool.Hkv;
  WsItem it;
  const int grp = p.ngroups - 1 - i / per;
  it.seq = (i % per) % p.S;
  it.h = (i % per) / p.S;
  it.qbase = p.q_start[it.seq];
  it.nq = p.q_start[it.seq + 1] - it.qbase;
  int ctx = p.lens[it.seq];
  it.bad_ctx = ctx > p.max_ctx || ctx < it.nq;
  it.ctx = min(ctx, p.max_ctx);
  it.rows_total = it.nq * p.G;
  it.row0 = grp * NT * kTcRows;
  if (it.row0 >= it.rows_total) {
    it.kv_end = it.nsteps = -1;  // nothing in this item
    return it;
  }
  const int last = min(it.rows_total, it.row0 + NT * kTcRows) - 1;
  it.kv_end = max(0, min(it.ctx, it.ctx - it.nq + last / p.G + 1));
  it.nsteps = (it.kv_end + kTcStep - 1) / kTcStep;
  return it;
}

template <int FMT, int D>
__global__ void __launch_bounds__(WsPlan<D, WsShape<FMT>::NT, FmtTraits<FMT>::channel>::threads, 1)
    kvq_prefill_ws_kernel(const PrefillWsParams p) {
  using T = FmtTraits<FMT>;
  constexpr bool CH = T::channel;
  constexpr int NT = WsShape<FMT>::NT;
  constexpr int NS = kWsStages;
  using PL = WsPlan<D, NT, CH>;
  using R = StepRec<D>;
  const float kNegInf = __int_as_float(0xff800000u);

  extern __shared__ __align__(1024) char smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  char* sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PoolView& pool = p.pool;
  const int n_items = p.ngroups * p.S * pool.Hkv;

  volatile int* abort_f = reinterpret_cast<volatile int*>(sm + PL::abort);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + PL::bars);
  uint64_t* kv_full = bars;                // [NS]: the step's record landed
  uint64_t* kv_empty = bars + NS;          // [NS]: every tile's MMAs of the step in that stage done
  uint64_t* s_full = bars + 2 * NS;        // [NT]: S of the tile's current step
  uint64_t* s_read = s_full + NT;          // [NT]: the tile's 4 warps have read S
  uint64_t* p_full = s_read + NT;          // [NT]: the tile's 4 warps have written P
  uint64_t* pv_done = p_full + NT;         // [NT]: the tile's last issued P.V done
  uint64_t* o_full = pv_done + NT;         // [NT]: the tile's final P.V of an item done
  uint64_t* q_full = o_full + NT;          // [NT]: the tile's Q rows of an item written
  uint64_t* drain = q_full + NT;           // clean-up
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + PL::tslot);
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], NT);
    }
    for (int x = 0; x < NT; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&s_read[x], kTcRows / 32);  // one arrival per warp
      mbar_init(&p_full[x], kTcRows / 32);  // one arrival per warp
      mbar_init(&pv_done[x], 1);
      mbar_init(&o_full[x], 1);
      mbar_init(&q_full[x], kTcRows / 32);  // one arrival per warp
    }
    mbar_init(drain, NT);
    *abort_f = 0;
    fence_barrier_init();
  }
  if (warp == 0) tc_alloc(tslot, PL::cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  auto stage_of = [&](int g) { return sm + PL::stage + (g % NS) * R::bytes; };
  const bool is_sm = tid < NT * kTcRows;

  if (!is_sm && warp == 5 * NT) {
    // ============ copier: the step records into the stages, as soon as each
    // stage is free, over the global step sequence of this CTA ============
    if (lane == 0) {
      int copied = 0;
      for (int item = blockIdx.x; item < n_items && !*abort_f; item += gridDim.x) {
        const WsItem it = ws_item<NT>(p, item);
        bool ok = true;
        for (int j = 0; j < it.nsteps; ++j) {
          if (copied >= NS &&
              !tc_wait_suspend(&kv_empty[copied % NS], ((copied / NS) - 1) & 1, abort_f)) {
            ok = false;
            break;
          }
          const char* rec = p.ws + (((int64_t)it.seq * p.max_steps + j) * pool.Hkv + it.h) * R::bytes;
          mbar_arrive_expect_tx(&kv_full[copied % NS], R::copy);
          bulk_g2s(stage_of(copied), rec, R::copy, &kv_full[copied % NS]);
          ++copied;
        }
        if (!ok) break;
      }
      // every copy has landed before the CTA exits
      for (int g = copied > NS ? copied - NS : 0; g < copied; ++g) {
        bool ok = false;
        for (int tries = 0; tries < kWaitTries && !ok; ++tries)
          ok = mbar_try_wait(&kv_full[g % NS], (g / NS) & 1);
      }
    }
  } else if (!is_sm) {
    // ============ control: tile C's MMAs ============
    const int C = warp - 4 * NT;
    if (lane == 0) {
      constexpr uint32_t id_s = tc_idesc_f16(128, kTcStep);
      constexpr uint32_t id_o = tc_idesc_f16(128, D);
      const uint32_t qa = smem_u32(sm + PL::q + C * PL::QB);
      const uint32_t qla = smem_u32(sm + PL::q + (NT + C) * PL::QB);
      const uint32_t ts = tmem + PL::s_col(C);
      const uint32_t tp = ts + 64;
      const uint32_t to = tmem + C * 128;
      auto issue_s = [&](int g) {  // S = Q K^T of global step g
        const uint32_t kha = smem_u32(stage_of(g) + R::kh);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * (kTcStep * 128) + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * (kTcRows * 128) + (kk & 3) * 32;
          tc_mma_f16(ts, sw128_desc(qa + qo), sw128_desc(kha + ko), id_s, kk > 0);
          if constexpr (CH) tc_mma_f16(ts, sw128_desc(qla + qo), sw128_desc(kha + ko), id_s, 1);
        }
        tc_commit(&s_full[C]);
      };
      auto issue_pv = [&](int g, bool first) {  // O += P V of global step g (P in TMEM)
        const uint32_t vta = smem_u32(stage_of(g) + R::vt);
#pragma unroll
        for (int kk = 0; kk < kTcStep / 16; ++kk)
          tc_mma_f16_ts(to, tp + 8 * kk, sw128_desc(vta + kk * 32), id_o, (!first || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kTcStep / 16; ++kk)
          tc_mma_f16_ts(to, tp + 32 + 8 * kk, sw128_desc(vta + kk * 32), id_o, 1u);
        tc_commit(&pv_done[C]);
      };
      int gbase = 0, n_done = 0;  // global steps before the item, items with steps done
      for (int item = blockIdx.x; item < n_items && !*abort_f; item += gridDim.x) {
        const WsItem it = ws_item<NT>(p, item);
        if (it.nsteps <= 0) continue;
        // this item's Q rows are in shared memory
        if (!tc_wait(&q_full[C], n_done & 1, abort_f)) break;
        bool ok = true;
        for (int j = 0; j <= it.nsteps && ok; ++j) {
          const int g = gbase + j;
          if (j < it.nsteps) {
            // S of step j, once its record has landed and the tile has read
            // its previous S
            ok = tc_wait(&kv_full[g % NS], (g / NS) & 1, abort_f) &&
                 (g == 0 || tc_wait(&s_read[C], (g - 1) & 1, abort_f));
            if (!ok) break;
            tc_fence_after();
            issue_s(g);
          }
          if (j > 0) {
            // P.V of step j-1, once the tile's weights are written
            ok = tc_wait(&p_full[C], (g - 1) & 1, abort_f);
            if (!ok) break;
            tc_fence_after();
            issue_pv(g - 1, j == 1);
            if (j == it.nsteps) tc_commit(&o_full[C]);
            tc_commit(&kv_empty[(g - 1) % NS]);  // this tile's MMAs reading that stage are issued
          }
        }
        if (!ok) break;
        gbase += it.nsteps;
        ++n_done;
      }
      // every MMA has completed before the CTA exits
      tc_commit(drain);
      bool ok = false;
      for (int tries = 0; tries < kWaitTries && !ok; ++tries) ok = mbar_try_wait(drain, 0);
    }
  } else {
    // ======================= softmax rows of tile X =======================
    const int X = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t tO = tmem + X * 128;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + PL::s_col(X) + lane_base;
    const uint32_t tP = tS + 64;
    char* qx = sm + PL::q + X * PL::QB;
    char* ql = sm + PL::q + (NT + X) * PL::QB;
    bool failed = false;
    int gbase = 0, n_done = 0;
    // The next item with key steps, from `from` on; items without any write
    // zeros for their rows here.
    auto next_item = [&](int from, WsItem& it) -> int {
      for (int i = from; i < n_items; i += gridDim.x) {
        it = ws_item<NT>(p, i);
        if (it.nsteps < 0) continue;  // no rows in this item
        if (it.bad_ctx && it.row0 == 0 && it.h == 0 && tid == 0) set_error(pool.err, ERR_RANGE);
        if (it.nsteps > 0) return i;
        const int rr = it.row0 + X * kTcRows + r;
        if (rr < it.rows_total) {
          float* o = p.out + ((int64_t)(it.qbase + rr / p.G) * p.Hq + it.h * p.G + rr % p.G) * D;
          for (int d = 0; d < D; ++d) o[d] = 0.f;
        }
      }
      return n_items;
    };
    // This row of an item's Q into the tile (K-major, swizzled), then the
    // tile's q_full arrival; returns the row's score scale (per-channel pools
    // fold the K channel scale into the row and scale it by a power of two).
    auto load_q = [&](const WsItem& it) -> float {
      const int rr = it.row0 + X * kTcRows + r;
      const __half* src =
          rr < it.rows_total
              ? p.q + ((int64_t)(it.qbase + rr / p.G) * p.Hq + it.h * p.G + rr % p.G) * D
              : nullptr;
      float csc = p.sm_scale_log2;
      if constexpr (!CH) {
        // the warp loads its 32 rows together: one instruction covers 256 / D
        // whole rows (each row's source address comes from its owner lane);
        // a batch of loads is issued before any of its shared-memory stores,
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
        // largest magnitude of the scaled row into [2^13, 2^14), fp16 hi + lo
        const float* ksc = pool.chan_scales + (int64_t)it.h * D;
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
      warp_arrive(&q_full[X]);
      return csc;
    };
    WsItem it;
    int item = next_item(blockIdx.x, it);
    float csc = item < n_items ? load_q(it) : 0.f;
    for (; item < n_items && !failed;) {
      const int rr = it.row0 + X * kTcRows + r;
      const bool row_ok = rr < it.rows_total;
      const int lim = row_ok ? max(0, it.ctx - it.nq + rr / p.G + 1) : 0;
      const int64_t orow =
          row_ok ? (int64_t)(it.qbase + rr / p.G) * p.Hq + it.h * p.G + rr % p.G : -1;
      float m = kNegInf, l = 0.f;
      int E = T::row_scales ? 100 : 14 - kTcSlack;
      for (int j = 0; j < it.nsteps; ++j) {
        const int g = gbase + j;
        const char* st = stage_of(g);
        // S of this step (its record's scales and mask landed before it)
        if (!warp_wait(&s_full[X], g & 1, abort_f) ||
            !warp_wait(&kv_full[g % NS], (g / NS) & 1, abort_f)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const int t0 = j * kTcStep;
        float z[kTcStep];
        {
          float a[32];
          tc_ld32(tS, a);
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = a[i];
          tc_ld32(tS + 32, a);
#pragma unroll
          for (int i = 0; i < 32; ++i) z[32 + i] = a[i];
        }
        tc_fence_before();
        warp_arrive(&s_read[X]);  // the next S may go into this buffer
        const float* ksb = reinterpret_cast<const float*>(st + R::ks);
        const float* vsb = reinterpret_cast<const float*>(st + R::vs);
        const uint32_t mk0 = reinterpret_cast<const uint32_t*>(st + R::mask)[0];
        const uint32_t mk1 = reinterpret_cast<const uint32_t*>(st + R::mask)[1];
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
            mx = fmax3(fmax3(mx, a0, a1), a2, a3);
          }
        } else {
#pragma unroll
          for (int t = 0; t < kTcStep; ++t) {
            const bool okt = t < lr && (((t < 32 ? mk0 : mk1) >> (t & 31)) & 1u);
            z[t] = okt ? (T::row_scales ? z[t] * ksb[t] : z[t]) : kNegInf;
            mx = fmaxf(mx, z[t]);
          }
        }
        // scores in log2 units are z * csc (csc > 0); the reference maximum m
        // moves only when the step's maximum passes it by more than kTcSlack
        const float mxz = mx == kNegInf ? kNegInf : mx * csc;
        const float mn = (m == kNegInf || mxz > m + kTcSlack) ? mxz : m;
        const float ms = mn == kNegInf ? 0.f : mn;
        int dE = 0;
        if constexpr (T::row_scales) {
          const float* vm = reinterpret_cast<const float*>(st + R::vmax);
          const float vmax = fmaxf(vm[0], vm[1]);
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
        if (g > 0) {
          // the previous P.V must be done before P is overwritten (and, within
          // an item, before O is rescaled)
          if (!warp_wait(&pv_done[X], (g - 1) & 1, abort_f)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const float f = alpha * pow2f(dE);
          if (j > 0 && __any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              float o[32];
              tc_ld32(tO + lane_base + 32 * c, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= f;
              tc_st32(tO + lane_base + 32 * c, o);
            }
          }
        }
        // the weights w = p' * s_V as fp16 hi + lo pairs into P (two halves of
        // 32 tokens: 16 columns of the high part, 16 of the low part each)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t hv[16], lv[16];
#pragma unroll
          for (int c = 0; c < 16; c += 2) {
            const int t = 32 * hf + 2 * c;
            float w0 = z[t], w1 = z[t + 1], w2 = z[t + 2], w3 = z[t + 3];
            // masked tokens (absent, past the end, or causally later) have
            // p' = 0; an absent token's V scale is 0 too
            if constexpr (T::row_scales) {
              const float4 v4 = *reinterpret_cast<const float4*>(vsb + t);
              f2_unpack(f2_mul(f2_pack(w0, w1), f2_pack(v4.x, v4.y)), w0, w1);
              f2_unpack(f2_mul(f2_pack(w2, w3), f2_pack(v4.z, v4.w)), w2, w3);
            }
            tc_split2(w0, w1, hv[c], lv[c]);
            tc_split2(w2, w3, hv[c + 1], lv[c + 1]);
          }
          tc_st16(tP + 16 * hf, hv);
          tc_st16(tP + 32 + 16 * hf, lv);
        }
        tc_wait_st();
        tc_fence_before();
        warp_arrive(&p_full[X]);
      }
      if (failed) break;
      // ---- the next item's Q now (the S products of this item, the last
      // readers of the tile, are done: this thread has read their results),
      // so that its first S overlaps this item's epilogue
      WsItem nit;
      const int nitem = next_item(item + gridDim.x, nit);
      const float ncsc = nitem < n_items ? load_q(nit) : 0.f;
      // ---- normalised output rows once the item's last P.V is done
      if (!warp_wait(&o_full[X], n_done & 1, abort_f)) {
        failed = true;
        break;
      }
      tc_fence_after();
      {
        const float f = l > 0.f ? pow2f(-E) / l : 0.f;
        const float* vch = CH ? pool.chan_scales + ((int64_t)pool.Hkv + it.h) * D : nullptr;
        // Each warp passes 16-column blocks of its 32 rows through shared
        // memory, so that a store instruction covers 8 rows x 64 contiguous
        // bytes instead of 32 rows x 16 bytes.  Writer: lane = row, chunk q4
        // at position q4 ^ ((row / 2) % 4); reader: row 8k + lane / 4, chunk
        // lane % 4 (both conflict-free).
        float* scr = reinterpret_cast<float*>(sm + PL::oscr) + warp * (32 * 16);
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
      // the next item's first P.V overwrites O: it is issued only after this
      // tile's next p_full, which comes after these reads
      tc_fence_before();
      gbase += it.nsteps;
      ++n_done;
      item = nitem;
      it = nit;
      csc = ncsc;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_f) set_error(pool.err, ERR_TIMEOUT);
  if (warp == 0) tc_dealloc(tmem, PL::cols);
}

}  // namespace kvq
