// kvq_prefill_tc.cu -- launch of the tcgen05 prefill kernel
// (kvq_prefill_tc_impl.cuh) and its format dispatch.
#include "kvq_internal.h"
#include "kvq_prefill_tc_impl.cuh"
#include "kvq_prefill_ws_impl.cuh"

namespace kvq {

bool prefill_tc_supported(const PoolView& pool) {
  const bool grouped = pool.fmt == FMT_INT8_GROUP || pool.fmt == FMT_INT4_GROUP;
  return (!grouped || pool.ng == 1) && (pool.D == 64 || pool.D == 128) && pool.bs % 16 == 0;
}

namespace {

template <int FMT, int NT>
cudaError_t run_tc_d(const PrefillTcLaunch& l) {
  switch (l.p.pool.D) {
    case 64: return run_prefill_tc<FMT, 64, NT>(l);
    case 128: return run_prefill_tc<FMT, 128, NT>(l);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill_tc(const PoolView& pool, const __half* q, int S, int Hq,
                              const int* q_start, int max_q_len, const int* table, int max_blocks,
                              const int* lens, int max_ctx, float sm_scale, float* out,
                              cudaStream_t st) {
  if (!prefill_tc_supported(pool)) return cudaErrorInvalidValue;
  // two Q tiles per CTA share each converted key step; per-channel pools keep
  // a low part of Q as well and take one tile per CTA
  const int NT = pool.fmt == FMT_INT8_CHANNEL ? 1 : 2;
  const int G = Hq / pool.Hkv;
  const int64_t ntiles = ((int64_t)max_q_len * G + kTcRows - 1) / kTcRows;
  const int64_t ngroups = (ntiles + NT - 1) / NT;
  const int64_t grid = ngroups * S * pool.Hkv;
  if (grid < 1 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  PrefillTcLaunch l;
  PrefillTcParams& p = l.p;
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
  p.ngroups = static_cast<int>(ngroups);
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  l.grid = dim3(static_cast<unsigned>(grid));
  l.st = st;
  switch (pool.fmt) {
    case FMT_FP16: return run_tc_d<FMT_FP16, 2>(l);
    case FMT_INT8_TOKEN: return run_tc_d<FMT_INT8_TOKEN, 2>(l);
    case FMT_INT8_CHANNEL: return run_tc_d<FMT_INT8_CHANNEL, 1>(l);
    case FMT_INT8_GROUP: return run_tc_d<FMT_INT8_GROUP, 2>(l);
    case FMT_FP8_TOKEN: return run_tc_d<FMT_FP8_TOKEN, 2>(l);
    case FMT_INT4_GROUP: return run_tc_d<FMT_INT4_GROUP, 2>(l);
    case FMT_FP8_E5M2: return run_tc_d<FMT_FP8_E5M2, 2>(l);
  }
  return cudaErrorInvalidValue;
}

size_t prefill_ws_bytes(const PoolView& pool, int S, int max_ctx) {
  if (!prefill_tc_supported(pool) || S < 1 || max_ctx < 1) return 0;
  const int64_t steps = (max_ctx + kTcStep - 1) / kTcStep;
  const int64_t rec = pool.D == 64 ? StepRec<64>::bytes : StepRec<128>::bytes;
  return static_cast<size_t>(S * steps * pool.Hkv * rec);
}

namespace {

template <int FMT, int D>
cudaError_t run_ws(const StageParams& sp, const PrefillWsParams& ap, int64_t ntiles,
                   cudaStream_t st) {
  constexpr int NT = WsShape<FMT>::NT;
  using PL = WsPlan<D, NT, FmtTraits<FMT>::channel>;
  static_assert(PL::request <= 227 * 1024, "shared memory plan too large");
  const int64_t sgrid = (int64_t)sp.S * sp.max_steps * sp.pool.Hkv;
  if (sgrid > 0x7fffffffLL) return cudaErrorInvalidValue;
  kvq_prefill_stage_kernel<FMT, D><<<static_cast<unsigned>(sgrid), 128, 0, st>>>(sp);
  cudaError_t e = phase_mark(st, cudaGetLastError());
  if (e != cudaSuccess) return e;
  PrefillWsParams a = ap;
  const int64_t ngroups = (ntiles + NT - 1) / NT;
  const int64_t items = ngroups * a.S * a.pool.Hkv;
  if (items < 1 || items > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.ngroups = static_cast<int>(ngroups);
  // persistent: one CTA per SM (its shared memory allows no more), each
  // taking every grid-th item
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    sms = 152;
  const int64_t grid = items < sms ? items : sms;
  e = allow_big_smem<kvq_prefill_ws_kernel<FMT, D>>();
  if (e != cudaSuccess) return e;
  kvq_prefill_ws_kernel<FMT, D><<<static_cast<unsigned>(grid), PL::threads, PL::request, st>>>(a);
  return phase_mark(st, cudaGetLastError());
}

template <int FMT>
cudaError_t run_ws_d(const StageParams& sp, const PrefillWsParams& ap, int64_t ntiles,
                     cudaStream_t st) {
  switch (sp.pool.D) {
    case 64: return run_ws<FMT, 64>(sp, ap, ntiles, st);
    case 128: return run_ws<FMT, 128>(sp, ap, ntiles, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill_ws(const PoolView& pool, const __half* q, int S, int Hq,
                              const int* q_start, int max_q_len, const int* table, int max_blocks,
                              const int* lens, int max_ctx, float sm_scale, float* out, void* ws,
                              cudaStream_t st) {
  if (!prefill_tc_supported(pool)) return cudaErrorInvalidValue;
  const int G = Hq / pool.Hkv;
  const int64_t ntiles = ((int64_t)max_q_len * G + kTcRows - 1) / kTcRows;
  const int max_steps = (max_ctx + kTcStep - 1) / kTcStep;
  if (ntiles > 0x7fffffffLL || max_steps < 1) return cudaErrorInvalidValue;
  StageParams sp{pool, table, lens, static_cast<char*>(ws), S, max_blocks, max_ctx, max_steps};
  PrefillWsParams ap{};
  ap.pool = pool;
  ap.q = q;
  ap.lens = lens;
  ap.q_start = q_start;
  ap.out = out;
  ap.ws = static_cast<const char*>(ws);
  ap.S = S;
  ap.Hq = Hq;
  ap.G = G;
  ap.max_ctx = max_ctx;
  ap.max_steps = max_steps;
  ap.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  switch (pool.fmt) {
    case FMT_FP16: return run_ws_d<FMT_FP16>(sp, ap, ntiles, st);
    case FMT_INT8_TOKEN: return run_ws_d<FMT_INT8_TOKEN>(sp, ap, ntiles, st);
    case FMT_INT8_CHANNEL: return run_ws_d<FMT_INT8_CHANNEL>(sp, ap, ntiles, st);
    case FMT_INT8_GROUP: return run_ws_d<FMT_INT8_GROUP>(sp, ap, ntiles, st);
    case FMT_FP8_TOKEN: return run_ws_d<FMT_FP8_TOKEN>(sp, ap, ntiles, st);
    case FMT_INT4_GROUP: return run_ws_d<FMT_INT4_GROUP>(sp, ap, ntiles, st);
    case FMT_FP8_E5M2: return run_ws_d<FMT_FP8_E5M2>(sp, ap, ntiles, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
