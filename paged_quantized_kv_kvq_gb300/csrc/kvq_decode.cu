// kvq_decode.cu -- launch planning for the paged decode kernel: pipeline
// depth, split-K over the context, workspace layout, format dispatch.
#include <algorithm>

#include "kvq_decode_impl.cuh"
#include "kvq_internal.h"

namespace kvq {

static int round_up(int x, int m) { return (x + m - 1) / m * m; }

bool plan_decode(const PoolView& pool, int S, int Hq, int max_ctx, int split_blocks, int sms,
                 DecodePlan* plan) {
  constexpr int W = kDecodeWarps;
  const bool tok = pool.fmt == FMT_INT8_TOKEN || pool.fmt == FMT_FP8_TOKEN;
  const int stage_bytes = round_up(pool.page_bytes + (tok ? 2 * pool.bs * 4 : 0), 128);
  int nstage_log2 = 3;  // 8 stages per warp at most
  while (nstage_log2 > 1 && W * (1 << nstage_log2) * stage_bytes > 96 * 1024) --nstage_log2;
  const int nstage = 1 << nstage_log2;
  const int stage_area = W * nstage * stage_bytes + W * nstage * (8 + 4);
  const int merge_area = W * (8 * (pool.D + 4) + 16) * 4 + 16;
  const int smem = round_up(std::max(stage_area, merge_area), 128);
  if (smem > 227 * 1024) return false;
  const int G = Hq / pool.Hkv;
  const int n_ht = (G + 7) / 8;
  const int ctas_per_sm = std::max(1, std::min(4, (228 * 1024) / (smem + 1024)));
  const int max_pages = (std::max(max_ctx, 0) + pool.bs - 1) / pool.bs;
  int pps;
  if (split_blocks > 0) {
    pps = split_blocks;
  } else {
    const int64_t units = (int64_t)S * pool.Hkv * n_ht;
    const int64_t target = 4LL * std::max(sms, 1) * ctas_per_sm;  // ~4 waves of CTAs
    const int64_t total = units * max_pages;
    int64_t want = total / std::max<int64_t>(target, 1);
    want = std::max<int64_t>(want, 2 * W);  // at least two blocks per warp
    pps = static_cast<int>(std::min<int64_t>(want, std::max(max_pages, 1)));
  }
  pps = std::max(pps, 1);
  const int nsplit = std::max(1, (max_pages + pps - 1) / pps);
  plan->pps = pps;
  plan->nsplit = nsplit;
  plan->n_ht = n_ht;
  plan->nstage_log2 = nstage_log2;
  plan->stage_bytes = stage_bytes;
  plan->smem_bytes = smem;
  plan->ws_bytes = 0;
  if (nsplit > 1) {
    const size_t rows = (size_t)S * Hq * nsplit;
    const size_t ml = (rows * 2 * sizeof(float) + 255) / 256 * 256;
    plan->ws_bytes = ml + rows * pool.D * sizeof(float);
  }
  return true;
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t st) {
  DecodeLaunch l;
  DecodeParams& p = l.p;
  p.pool = a.pool;
  p.q = a.q;
  p.table = a.table;
  p.lens = a.lens;
  p.out = a.out;
  p.part_ml = nullptr;
  p.part_o = nullptr;
  if (plan.nsplit > 1) {
    const size_t rows = (size_t)a.S * a.Hq * plan.nsplit;
    const size_t ml = (rows * 2 * sizeof(float) + 255) / 256 * 256;
    p.part_ml = static_cast<float*>(a.workspace);
    p.part_o = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + ml);
  }
  p.S = a.S;
  p.Hq = a.Hq;
  p.G = a.Hq / a.pool.Hkv;
  p.n_ht = plan.n_ht;
  p.max_blocks = a.max_blocks;
  p.max_ctx = a.max_ctx;
  p.pps = plan.pps;
  p.nsplit = plan.nsplit;
  p.nstage_log2 = plan.nstage_log2;
  p.stage_bytes = plan.stage_bytes;
  p.sm_scale_log2 = a.sm_scale * 1.4426950408889634f;
  l.grid = dim3(static_cast<unsigned>(plan.nsplit), static_cast<unsigned>(a.pool.Hkv * plan.n_ht),
                static_cast<unsigned>(a.S));
  l.smem = plan.smem_bytes;
  l.st = st;
  switch (a.pool.fmt) {
    case FMT_INT8_GROUP: return launch_decode_int8_group(l);
    case FMT_FP16: return launch_decode_fp16(l);
    case FMT_INT8_TOKEN:
    case FMT_FP8_TOKEN: return launch_decode_token(l);
    case FMT_INT8_CHANNEL: return launch_decode_channel(l);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
