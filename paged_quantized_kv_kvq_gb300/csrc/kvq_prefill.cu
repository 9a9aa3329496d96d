// kvq_prefill.cu -- launch planning and format dispatch of the prefill kernel
// (kvq_prefill_impl.cuh).
#include <algorithm>

#include "kvq_internal.h"
#include "kvq_prefill_impl.cuh"

namespace kvq {

namespace {

int round_up(int x, int m) { return (x + m - 1) / m * m; }

template <int FMT>
cudaError_t run_prefill_d(const PrefillLaunch& l) {
  const int D = l.p.pool.D, ng = l.p.pool.ng;
  if constexpr (FMT == FMT_INT8_GROUP || FMT == FMT_INT4_GROUP) {
    if (D == 64) {
      switch (ng) {
        case 1: return run_prefill<FMT, 64, 1>(l);
        case 2: return run_prefill<FMT, 64, 2>(l);
        case 4: return run_prefill<FMT, 64, 4>(l);
      }
    } else if (D == 128) {
      switch (ng) {
        case 1: return run_prefill<FMT, 128, 1>(l);
        case 2: return run_prefill<FMT, 128, 2>(l);
        case 4: return run_prefill<FMT, 128, 4>(l);
        case 8: return run_prefill<FMT, 128, 8>(l);
      }
    }
    return cudaErrorInvalidValue;
  } else {
    switch (D) {
      case 64: return run_prefill<FMT, 64, 1>(l);
      case 128: return run_prefill<FMT, 128, 1>(l);
    }
    return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill(const PoolView& pool, const __half* q, int S, int Hq, const int* q_start,
                           int max_q_len, const int* table, int max_blocks, const int* lens,
                           int max_ctx, float sm_scale, float* out, cudaStream_t st) {
  // tcgen05 kernel where the format allows; per-group formats with several
  // scale groups per head take the mma.sync kernel below
  if (prefill_tc_supported(pool)) {
    const cudaError_t e = launch_prefill_tc(pool, q, S, Hq, q_start, max_q_len, table, max_blocks,
                                            lens, max_ctx, sm_scale, out, st);
    if (e != cudaErrorInvalidValue) return e;  // else: no room for its tiles, use the kernel below
  }
  const bool tok = pool.fmt == FMT_INT8_TOKEN || pool.fmt == FMT_FP8_TOKEN;
  const int stage_bytes = round_up(pool.page_bytes + (tok ? 2 * pool.bs * 4 : 0), 128);
  int nstage = 4;
  while (nstage > 2 && nstage * stage_bytes > 64 * 1024) --nstage;
  const int G = Hq / pool.Hkv;
  const int64_t ntiles = ((int64_t)max_q_len * G + kPfRows - 1) / kPfRows;
  const int64_t grid = (int64_t)pool.Hkv * S * ntiles;
  if (grid < 1 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  PrefillLaunch l;
  PrefillParams& p = l.p;
  p.kh_off = nstage * stage_bytes;
  p.vt_off = round_up(p.kh_off + 16 * (pool.D + kKhStride) * 2, 128);
  p.sc_off = round_up(p.vt_off + pool.D * kVtStride * 2, 128);
  p.bar_off = round_up(p.sc_off + 2 * 16 * std::max(pool.ng, 1) * 4, 128);
  l.smem = round_up(p.bar_off + nstage * (8 + 4), 128);
  if (l.smem > 227 * 1024) return cudaErrorInvalidValue;
  p.pool = pool;
  p.q = q;
  p.table = table;
  p.lens = lens;
  p.q_start = q_start;
  p.out = out;
  p.S = S;
  p.Hq = Hq;
  p.G = G;
  p.max_blocks = max_blocks;
  p.max_ctx = max_ctx;
  p.ntiles = static_cast<int>(ntiles);
  p.nstage = nstage;
  p.stage_bytes = stage_bytes;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  l.grid = dim3(static_cast<unsigned>(grid));
  l.st = st;
  switch (pool.fmt) {
    case FMT_FP16: return run_prefill_d<FMT_FP16>(l);
    case FMT_INT8_TOKEN: return run_prefill_d<FMT_INT8_TOKEN>(l);
    case FMT_INT8_CHANNEL: return run_prefill_d<FMT_INT8_CHANNEL>(l);
    case FMT_INT8_GROUP: return run_prefill_d<FMT_INT8_GROUP>(l);
    case FMT_FP8_TOKEN: return run_prefill_d<FMT_FP8_TOKEN>(l);
    case FMT_INT4_GROUP: return run_prefill_d<FMT_INT4_GROUP>(l);
    case FMT_FP8_E5M2: return run_prefill_d<FMT_FP8_E5M2>(l);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
