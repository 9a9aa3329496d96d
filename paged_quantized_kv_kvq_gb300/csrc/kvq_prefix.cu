// kvq_prefix.cu -- launch planning and format dispatch of the shared-prefix
// attention kernel (kvq_prefix_impl.cuh).
#include <algorithm>

#include "kvq_internal.h"
#include "kvq_prefix_impl.cuh"

namespace kvq {

namespace {

int round_up(int x, int m) { return (x + m - 1) / m * m; }

template <int FMT>
cudaError_t run_prefix_d(const PrefixLaunch& l) {
  const int D = l.p.pool.D, ng = l.p.pool.ng;
  if constexpr (FMT == FMT_INT8_GROUP) {
    if (D == 64) {
      switch (ng) {
        case 1: return run_prefix<FMT, 64, 1>(l);
        case 2: return run_prefix<FMT, 64, 2>(l);
        case 4: return run_prefix<FMT, 64, 4>(l);
      }
    } else if (D == 128) {
      switch (ng) {
        case 1: return run_prefix<FMT, 128, 1>(l);
        case 2: return run_prefix<FMT, 128, 2>(l);
        case 4: return run_prefix<FMT, 128, 4>(l);
        case 8: return run_prefix<FMT, 128, 8>(l);
      }
    }
    return cudaErrorInvalidValue;
  } else {
    switch (D) {
      case 64: return run_prefix<FMT, 64, 1>(l);
      case 128: return run_prefix<FMT, 128, 1>(l);
    }
    return cudaErrorInvalidValue;
  }
}

}  // namespace

bool plan_prefix(const PoolView& pool, int S, int Hq, int P, PrefixPlan* plan) {
  constexpr int W = kPrefixWarps;
  const bool tok = pool.fmt == FMT_INT8_TOKEN || pool.fmt == FMT_FP8_TOKEN;
  const int stage_bytes = round_up(pool.page_bytes + (tok ? 2 * pool.bs * 4 : 0), 128);
  const int G = Hq / pool.Hkv;
  const int64_t rows = (int64_t)S * G;
  const int64_t ntiles = (rows + kPrefixRows - 1) / kPrefixRows;
  const int chunk = (P + W - 1) / W;
  int nstage = 4;
  while (nstage > 2 && W * nstage * stage_bytes > 80 * 1024) --nstage;
  nstage = std::max(1, std::min(nstage, chunk));
  const int merge_bytes = W * kPrefixRows * (pool.D + 2) * 4;
  const int bar_off = round_up(std::max(W * nstage * stage_bytes, merge_bytes), 128);
  const int smem = round_up(bar_off + W * nstage * (8 + 4), 128);
  if (smem > 227 * 1024 || P < 1) return false;
  if ((int64_t)pool.Hkv * ntiles > 0x7fffffffLL) return false;
  plan->grid = static_cast<int>(pool.Hkv * ntiles);
  plan->ntiles = static_cast<int>(ntiles);
  plan->chunk = chunk;
  plan->nstage = nstage;
  plan->stage_bytes = stage_bytes;
  plan->bar_off = bar_off;
  plan->smem_bytes = smem;
  return true;
}

cudaError_t launch_prefix(const PrefixArgs& a, const PrefixPlan& plan, cudaStream_t st,
                          bool dependent) {
  PrefixLaunch l;
  PrefixParams& p = l.p;
  p.pool = a.pool;
  p.q = a.q;
  p.table = a.table;
  p.lens = a.lens;
  p.pre = a.pre;
  p.S = a.S;
  p.Hq = a.Hq;
  p.G = a.Hq / a.pool.Hkv;
  p.max_ctx = a.max_ctx;
  p.P = a.P;
  p.ntiles = plan.ntiles;
  p.chunk = plan.chunk;
  p.nstage = plan.nstage;
  p.stage_bytes = plan.stage_bytes;
  p.bar_off = plan.bar_off;
  p.sm_scale_log2 = a.sm_scale * 1.4426950408889634f;
  l.grid = dim3(static_cast<unsigned>(plan.grid));
  l.smem = plan.smem_bytes;
  l.st = st;
  l.dependent = dependent;
  switch (a.pool.fmt) {
    case FMT_FP16: return run_prefix_d<FMT_FP16>(l);
    case FMT_INT8_TOKEN: return run_prefix_d<FMT_INT8_TOKEN>(l);
    case FMT_INT8_CHANNEL: return run_prefix_d<FMT_INT8_CHANNEL>(l);
    case FMT_INT8_GROUP: return run_prefix_d<FMT_INT8_GROUP>(l);
    case FMT_FP8_TOKEN: return run_prefix_d<FMT_FP8_TOKEN>(l);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
