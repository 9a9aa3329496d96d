// kvq_rows.cu -- launch planning and format dispatch of the shared-prefix
// attention kernel (kvq_rows_impl.cuh).
#include <algorithm>

#include "kvq_internal.h"
#include "kvq_rows_impl.cuh"

namespace kvq {

namespace {

int round_up(int x, int m) { return (x + m - 1) / m * m; }

template <int FMT>
cudaError_t run_rows_d(const RowsLaunch& l) {
  const int D = l.p.pool.D, ng = l.p.pool.ng;
  if constexpr (FMT == FMT_INT8_GROUP || FMT == FMT_INT4_GROUP) {
    if (D == 64) {
      switch (ng) {
        case 1: return run_rows<FMT, 64, 1>(l);
        case 2: return run_rows<FMT, 64, 2>(l);
        case 4: return run_rows<FMT, 64, 4>(l);
      }
    } else if (D == 128) {
      switch (ng) {
        case 1: return run_rows<FMT, 128, 1>(l);
        case 2: return run_rows<FMT, 128, 2>(l);
        case 4: return run_rows<FMT, 128, 4>(l);
        case 8: return run_rows<FMT, 128, 8>(l);
      }
    }
    return cudaErrorInvalidValue;
  } else {
    switch (D) {
      case 64: return run_rows<FMT, 64, 1>(l);
      case 128: return run_rows<FMT, 128, 1>(l);
    }
    return cudaErrorInvalidValue;
  }
}

}  // namespace

bool plan_rows(const PoolView& pool, int S, int Hq, RowsPlan* plan) {
  constexpr int W = kRowsWarps;
  const bool tok = pool.fmt == FMT_INT8_TOKEN || pool.fmt == FMT_FP8_TOKEN;
  const int stage_bytes = round_up(pool.page_bytes + (tok ? 2 * pool.bs * 4 : 0), 128);
  const int G = Hq / pool.Hkv;
  const int64_t ntiles = ((int64_t)S * G + kRowsTile - 1) / kRowsTile;  // per kv head
  int nstage = 4;
  while (nstage > 2 && W * nstage * stage_bytes > 80 * 1024) --nstage;
  const int merge_bytes = W * kRowsTile * (pool.D + 2) * 4;
  const int bar_off = round_up(std::max(W * nstage * stage_bytes, merge_bytes), 128);
  const int smem = round_up(bar_off + W * nstage * (8 + 4), 128);
  if (smem > 227 * 1024 || ntiles < 1) return false;
  const int64_t grid = (int64_t)pool.Hkv * ntiles;
  if (grid > 0x7fffffffLL) return false;
  plan->grid = static_cast<int>(grid);
  plan->ntiles = static_cast<int>(ntiles);
  plan->nstage = nstage;
  plan->stage_bytes = stage_bytes;
  plan->bar_off = bar_off;
  plan->smem_bytes = smem;
  return true;
}

cudaError_t launch_rows(const RowsArgs& a, const RowsPlan& plan, cudaStream_t st, bool dependent) {
  RowsLaunch l;
  RowsParams& p = l.p;
  p.pool = a.pool;
  p.q = a.q;
  p.table = a.table;
  p.lens = a.lens;
  p.out = a.out;
  p.S = a.S;
  p.Hq = a.Hq;
  p.G = a.Hq / a.pool.Hkv;
  p.max_blocks = a.max_blocks;
  p.max_ctx = a.max_ctx;
  p.P = a.P;
  p.ntiles = plan.ntiles;
  p.nstage = plan.nstage;
  p.stage_bytes = plan.stage_bytes;
  p.bar_off = plan.bar_off;
  p.sm_scale_log2 = a.sm_scale * 1.4426950408889634f;
  l.grid = dim3(static_cast<unsigned>(plan.grid));
  l.smem = plan.smem_bytes;
  l.st = st;
  l.dependent = dependent;
  switch (a.pool.fmt) {
    case FMT_FP16: return run_rows_d<FMT_FP16>(l);
    case FMT_INT8_TOKEN: return run_rows_d<FMT_INT8_TOKEN>(l);
    case FMT_INT8_CHANNEL: return run_rows_d<FMT_INT8_CHANNEL>(l);
    case FMT_INT8_GROUP: return run_rows_d<FMT_INT8_GROUP>(l);
    case FMT_FP8_TOKEN: return run_rows_d<FMT_FP8_TOKEN>(l);
    case FMT_INT4_GROUP: return run_rows_d<FMT_INT4_GROUP>(l);
    case FMT_FP8_E5M2: return run_rows_d<FMT_FP8_E5M2>(l);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
