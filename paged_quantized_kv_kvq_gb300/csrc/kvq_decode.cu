// kvq_decode.cu -- launch planning for the paged decode kernel: pipeline
// depth, the persistent grid, the workspace (page prefix + partials), format
// dispatch.
#include <algorithm>

#include "kvq_decode_impl.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

int round_up(int x, int m) { return (x + m - 1) / m * m; }
size_t round_up_sz(size_t x, size_t m) { return (x + m - 1) / m * m; }

}  // namespace

bool plan_decode(const PoolView& pool, int S, int Hq, int max_ctx, int split_blocks, int sms,
                 DecodePlan* plan) {
  constexpr int W = kDecodeWarps;
  const bool tok = pool.fmt == FMT_INT8_TOKEN || pool.fmt == FMT_FP8_TOKEN;
  // Block size 8: a stage holds a pair of pages (two page slots) completing
  // on one barrier.
  const int sps = pool.bs == 8 ? 2 : 1;
  const int stage_bytes = sps * round_up(pool.page_bytes + (tok ? 2 * pool.bs * 4 : 0), 128);
  // Pages in flight per SM = CTAs per SM x W x stages; 3 CTAs x 4 warps x 4
  // stages keeps ~200 KB of copies in flight, above what HBM latency needs.
  // Block size 8 consumes up to four pages (three pairs) per update, so keeps
  // at least three stages.  The stages are cut to what lets kDecodeCtasPerSm
  // CTAs share an SM (228 KB, 1 KB of it reserved per CTA): a fourth stage of
  // 4 KB pages that left room for only two CTAs (8 warps) cost more in
  // latency hiding than it gave.
  const int min_stage = pool.bs == 8 ? 3 : 2;
  auto smem_of = [&](int ns) {
    return round_up(W * ns * stage_bytes + W * ns * (8 + 4 * sps) + W * 4 + (S + 1) * 4, 128);
  };
  const int budget = std::min(80 * 1024, 228 * 1024 / kDecodeCtasPerSm - 1024);
  int nstage = kDecodeStages;
  while (nstage > min_stage && smem_of(nstage) > budget) --nstage;
  const int smem = smem_of(nstage);
  if (smem > 227 * 1024) return false;
  const int G = Hq / pool.Hkv;
  const int n_ht = (G + 7) / 8;
  const int ctas_per_sm = std::max(1, std::min(kDecodeCtasPerSm, (228 * 1024) / (smem + 1024)));
  const int64_t units = (int64_t)S * pool.Hkv * n_ht;
  const int64_t max_pages = (std::max(max_ctx, 0) + pool.bs - 1) / pool.bs;
  const int64_t tmax = std::max<int64_t>(units * max_pages, 1);
  int64_t grid;
  int ppw_fixed = 0;
  if (split_blocks > 0) {
    ppw_fixed = split_blocks;
    grid = ((tmax + split_blocks - 1) / split_blocks + W - 1) / W;
  } else {
    grid = (int64_t)std::max(sms, 1) * ctas_per_sm;
    grid = std::min<int64_t>(grid, (tmax + W - 1) / W);  // at least one page per warp
  }
  grid = std::max<int64_t>(grid, 1);
  if (grid > 0x7fffffff / W) return false;
  plan->grid = static_cast<int>(grid);
  plan->ppw_fixed = ppw_fixed;
  plan->n_ht = n_ht;
  plan->nstage = nstage;
  plan->stage_bytes = stage_bytes;
  plan->smem_bytes = smem;
  plan->ps_bytes = round_up_sz((size_t)(S + 1) * sizeof(int), 256);
  // one warp per (unit, head row that a Q head fills); enough CTAs to cover
  // every task once
  const int64_t merge_tasks = units * std::min(kPartRows, G);
  plan->merge_grid = static_cast<int>(std::max<int64_t>(
      1, std::min<int64_t>((merge_tasks + kMergeThreads / 32 - 1) / (kMergeThreads / 32),
                           16LL * std::max(sms, 1))));
  // Pieces per merge round trip: 16 once a warp's range spans 1024 tokens or
  // more (long layers: long_8x32k 3.30 -> 3.20 ms per step, the MHA fp16
  // layers of 100 x ~1152 tokens 10.16 -> 9.92), 8 below that (64 x 2048
  // GQA: 1.806 ms with 8 against 1.819 with 16); measured, the range bound
  // taken from max_ctx since the lengths live on the device.
  const int64_t warps_total = grid * W;
  const int64_t tok_per_warp = (int64_t)units * std::max(max_ctx, 0) / std::max<int64_t>(warps_total, 1);
  plan->merge_chunk = tok_per_warp >= 1024 ? 16 : 8;
  plan->ws_bytes = plan->ps_bytes +
                   (size_t)grid * W * 2 * kPartRows * (pool.D + 2) * sizeof(float);
  return true;
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t st,
                          bool dependent) {
  DecodeLaunch l;
  DecodeParams& p = l.p;
  p.pool = a.pool;
  p.q = a.q;
  p.table = a.table;
  p.lens = a.lens;
  p.out = a.out;
  p.q_stride = a.q_stride > 0 ? a.q_stride : (int64_t)a.Hq * a.pool.D;
  p.out_stride = a.out_stride > 0 ? a.out_stride : (int64_t)a.Hq * a.pool.D;
  p.ps = static_cast<int*>(a.workspace);
  p.part = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + plan.ps_bytes);
  p.S = a.S;
  p.Hq = a.Hq;
  p.G = a.Hq / a.pool.Hkv;
  p.n_ht = plan.n_ht;
  p.max_blocks = a.max_blocks;
  p.max_ctx = a.max_ctx;
  p.ppw_fixed = plan.ppw_fixed;
  p.nstage = plan.nstage;
  p.stage_bytes = plan.stage_bytes;
  p.grid = plan.grid;
  p.sm_scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.skip = a.skip;
  p.pre = a.pre;
  p.wait_tries = a.wait_tries;
  p.fault_issue = a.fault_issue;
  l.grid = dim3(static_cast<unsigned>(plan.grid));
  l.merge_grid = static_cast<unsigned>(plan.merge_grid);
  l.merge_chunk = plan.merge_chunk;
  l.smem = plan.smem_bytes;
  l.st = st;
  l.dependent = dependent;
  if (a.pool.bs == 8)
    return a.pool.fmt == FMT_INT8_GROUP ? launch_decode_bs8_group(l) : launch_decode_bs8_misc(l);
  switch (a.pool.fmt) {
    case FMT_INT8_GROUP: return launch_decode_int8_group(l);
    case FMT_INT4_GROUP: return launch_decode_int4_group(l);
    case FMT_FP16: return launch_decode_fp16(l);
    case FMT_INT8_TOKEN:
    case FMT_FP8_TOKEN: return launch_decode_token(l);
    case FMT_INT8_CHANNEL: return launch_decode_channel(l);
    case FMT_FP8_E5M2: return launch_decode_e5m2(l);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
