// kvq_prefill_tc.cu -- launch of the tcgen05 prefill kernel
// (kvq_prefill_tc_impl.cuh) and its format dispatch.
#include "kvq_internal.h"
#include "kvq_prefill_tc_impl.cuh"

namespace kvq {

bool prefill_tc_supported(const PoolView& pool) {
  const bool grouped = pool.fmt == FMT_INT8_GROUP || pool.fmt == FMT_INT4_GROUP;
  return (!grouped || pool.ng == 1) && (pool.D == 64 || pool.D == 128) && pool.bs % 16 == 0;
}

namespace {

template <int FMT>
cudaError_t run_tc_d(const PrefillTcLaunch& l) {
  switch (l.p.pool.D) {
    case 64: return run_prefill_tc<FMT, 64>(l);
    case 128: return run_prefill_tc<FMT, 128>(l);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill_tc(const PoolView& pool, const __half* q, int S, int Hq,
                              const int* q_start, int max_q_len, const int* table, int max_blocks,
                              const int* lens, int max_ctx, float sm_scale, float* out,
                              cudaStream_t st) {
  if (!prefill_tc_supported(pool)) return cudaErrorInvalidValue;
  const int G = Hq / pool.Hkv;
  const int64_t ntiles = ((int64_t)max_q_len * G + kTcThreads - 1) / kTcThreads;
  const int64_t grid = ntiles * S * pool.Hkv;
  if (grid < 1 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  PrefillTcLaunch l;
  PrefillTcParams& p = l.p;
  // shared-memory plan: Q (hi, and lo for per-channel), the K tile, the V^T
  // tile, the weight tiles (the low part reuses the K tile when it is as
  // large), the raw page stage of one key step, the misc block
  const bool ch = pool.fmt == FMT_INT8_CHANNEL;
  const bool tok = pool.fmt == FMT_INT8_TOKEN || pool.fmt == FMT_FP8_TOKEN;
  const int D = pool.D;
  const int qb = kTcThreads * D * 2, kb = kTcStep * D * 2, vb = D * kTcStep * 2,
            pb = kTcThreads * kTcStep * 2;
  p.off_qlo = qb;
  p.off_kh = ch ? 2 * qb : qb;
  p.off_vt = p.off_kh + kb;
  p.off_phi = p.off_vt + vb;
  int next = p.off_phi + pb;
  if (kb >= pb) {
    p.off_plo = p.off_kh;
  } else {
    p.off_plo = next;
    next += pb;
  }
  p.npg = kTcStep / pool.bs;
  p.tok_bytes = tok ? 2 * pool.bs * 4 : 0;
  p.pstride = (pool.page_bytes + p.tok_bytes + 127) / 128 * 128;
  p.off_raw = next;
  next += p.npg * p.pstride;
  p.off_misc = (next + 127) / 128 * 128;
  // 1024 bytes of alignment slack; at least 80 KB so that no more than two
  // CTAs (2 x 256 TMEM columns) share an SM
  l.smem = p.off_misc + kMiscBytes + 1024;
  if (l.smem < 80 * 1024) l.smem = 80 * 1024;
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
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  l.grid = dim3(static_cast<unsigned>(grid));
  l.st = st;
  switch (pool.fmt) {
    case FMT_FP16: return run_tc_d<FMT_FP16>(l);
    case FMT_INT8_TOKEN: return run_tc_d<FMT_INT8_TOKEN>(l);
    case FMT_INT8_CHANNEL: return run_tc_d<FMT_INT8_CHANNEL>(l);
    case FMT_INT8_GROUP: return run_tc_d<FMT_INT8_GROUP>(l);
    case FMT_FP8_TOKEN: return run_tc_d<FMT_FP8_TOKEN>(l);
    case FMT_INT4_GROUP: return run_tc_d<FMT_INT4_GROUP>(l);
    case FMT_FP8_E5M2: return run_tc_d<FMT_FP8_E5M2>(l);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
