// kvq_internal.h -- host-side declarations shared by the C ABI and the kernel
// translation units.  Not part of the public interface.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime_api.h>

#include "kvq_common.cuh"

namespace kvq {

cudaError_t launch_append(const PoolView& pool, const __half* k, const __half* v,
                          const int64_t* slots, int64_t T, cudaStream_t st);
// Append with slots from `slots`, or -- when slots is null -- the decode-step
// form: token t is sequence t's new token, stored at position lens[t]-1.
// `dependent`: launch as a programmatic dependent of the previous kernel (the
// kernel waits for its completion before reading anything).  `x_stride`:
// elements between consecutive tokens of k and v (0 = kv_heads * head_dim).
cudaError_t launch_step_append(const PoolView& pool, const __half* k, const __half* v,
                               const int64_t* slots, int64_t T, const int* table, const int* lens,
                               int max_blocks, int max_ctx, cudaStream_t st, bool dependent,
                               int64_t x_stride = 0);
cudaError_t launch_copy_blocks(const PoolView& pool, const int* src, const int* dst, int n,
                               cudaStream_t st);
cudaError_t launch_calibrate(const PoolView& pool, const __half* k, const __half* v, int64_t T,
                             cudaStream_t st);
cudaError_t launch_read_slots(const PoolView& pool, const int64_t* slots, int64_t n,
                              void* codes_out, float* scales_out, cudaStream_t st);

// Launch geometry of one decode call.
struct DecodePlan {
  int grid = 0;         // persistent CTAs
  int ppw_fixed = 0;    // pages per warp when forced; 0 = balanced
  int n_ht = 0;         // head tiles of 8 Q heads per kv head
  int nstage = 0;  // pipeline stages per warp
  int stage_bytes = 0;  // bytes of one stage
  int smem_bytes = 0;   // dynamic shared memory per CTA
  int merge_grid = 0;   // CTAs of the merge kernel
  int merge_chunk = 8;  // pieces the merge loads per round trip
  size_t ps_bytes = 0;  // page prefix at the start of the workspace
  size_t ws_bytes = 0;  // page prefix + split partials
};

// Plan a decode call; `sms` is the device's SM count.  Returns false for an
// unsupported geometry.
bool plan_decode(const PoolView& pool, int S, int Hq, int max_ctx, int split_blocks, int sms,
                 DecodePlan* plan);

struct DecodeArgs {
  PoolView pool;
  const __half* q;
  const int* table;
  const int* lens;
  float* out;
  void* workspace;
  int S, Hq, max_blocks, max_ctx;
  float sm_scale;
  // shared-prefix cascade: skip the first `skip` blocks of every sequence and
  // fold in the prefix partials `pre` ([S][Hq][D+2]); 0 / null otherwise
  int skip = 0;
  const float* pre = nullptr;
  int64_t q_stride = 0, out_stride = 0;  // elements between sequences' rows; 0 = Hq * D
  int wait_tries = kWaitTries;  // bound of each pipeline wait, in ~1 ms tries
  int fault_issue = -1;   // self-test only: withhold warp 0's copy of this index
};

// `dependent`: launch the decode as a programmatic dependent of the kernel
// just before it on the stream (the decode-step append).
cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t st,
                          bool dependent = false);

// Shared-prefix attention (kvq_rows_impl.cuh): the first P blocks of every
// sequence (those of table row 0) attended once per kv head for all
// sequences' Q rows, writing the partial rows out[S][Hq][D+2] (m, l, O) that
// a decode with skip = P folds in.
struct RowsPlan {
  int grid = 0, ntiles = 0, nstage = 0, stage_bytes = 0, bar_off = 0, smem_bytes = 0;
};
bool plan_rows(const PoolView& pool, int S, int Hq, RowsPlan* plan);
struct RowsArgs {
  PoolView pool;
  const __half* q;
  const int* table;
  const int* lens;
  float* out;
  int S, Hq, max_blocks, max_ctx;
  int P = 0;
  float sm_scale;
};
cudaError_t launch_rows(const RowsArgs& a, const RowsPlan& plan, cudaStream_t st, bool dependent);

// Prefill / chunked prefill (kvq_prefill_impl.cuh): the query tokens
// q_start[s]..q_start[s+1]-1 of each sequence attend causally to its cache.
cudaError_t launch_prefill(const PoolView& pool, const __half* q, int S, int Hq, const int* q_start,
                           int max_q_len, const int* table, int max_blocks, const int* lens,
                           int max_ctx, float sm_scale, float* out, cudaStream_t st);

// The same on the 5th-generation tensor cores (kvq_prefill_tc_impl.cuh): for
// formats with at most one scale per token and K|V (per-group only when the
// group is the whole head), head_dim 64 or 128, blocks of 16 tokens or more.
bool prefill_tc_supported(const PoolView& pool);
cudaError_t launch_prefill_tc(const PoolView& pool, const __half* q, int S, int Hq,
                              const int* q_start, int max_q_len, const int* table, int max_blocks,
                              const int* lens, int max_ctx, float sm_scale, float* out,
                              cudaStream_t st);

// Prefill in two passes through a workspace (kvq_prefill_ws_impl.cuh): the
// codes of every 64-token key step staged once as fp16 tiles, then the
// attention pass.  Same formats as launch_prefill_tc; 0 bytes otherwise.
size_t prefill_ws_bytes(const PoolView& pool, int S, int max_ctx);
cudaError_t launch_prefill_ws(const PoolView& pool, const __half* q, int S, int Hq,
                              const int* q_start, int max_q_len, const int* table, int max_blocks,
                              const int* lens, int max_ctx, float sm_scale, float* out, void* ws,
                              cudaStream_t st);

// Per-format kernel launchers (one translation unit each, compiled in parallel).
struct DecodeLaunch;
cudaError_t launch_decode_int8_group(const DecodeLaunch& l);
cudaError_t launch_decode_int4_group(const DecodeLaunch& l);
cudaError_t launch_decode_fp16(const DecodeLaunch& l);
cudaError_t launch_decode_token(const DecodeLaunch& l);
cudaError_t launch_decode_channel(const DecodeLaunch& l);
cudaError_t launch_decode_e5m2(const DecodeLaunch& l);
cudaError_t launch_decode_bs8_group(const DecodeLaunch& l);  // block size 8, INT8 per-group
cudaError_t launch_decode_bs8_misc(const DecodeLaunch& l);   // block size 8, the other formats

}  // namespace kvq
