// kvq_api.cu -- the C ABI (include/kvq.h): pool creation and byte accounting,
// host-side argument checks, and dispatch to the kernels.
#include <cstdlib>
#include <cstring>
#include <new>

#include "kvq.h"
#include "kvq_common.cuh"
#include "kvq_context.h"
#include "kvq_internal.h"

using kvq::PoolView;

namespace {

// Events handed to this host thread's next kernel launches
// (kvq_set_phase_events).
struct PhaseEvents {
  cudaEvent_t ev[KVQ_MAX_PHASE_EVENTS] = {};
  int n = 0;     // registered
  int next = 0;  // the next launch records ev[next] while next < n
};
thread_local PhaseEvents t_phase;

}  // namespace

cudaError_t kvq::phase_mark(cudaStream_t st, cudaError_t launched) {
  if (launched != cudaSuccess || t_phase.next >= t_phase.n) return launched;
  return cudaEventRecord(t_phase.ev[t_phase.next++], st);
}

struct kvq_pool {
  PoolView view;
  void* base = nullptr;
  size_t total_bytes = 0;
  bool owned = false;
  int device = 0;
  kvq_pool_layout layout{};
};

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool valid_dtype(int d) { return d >= KVQ_FP16 && d <= KVQ_FP8_E5M2; }

// Geometry check + byte accounting.  Fills `view` offsets relative to base 0.
kvq_status layout_for(int64_t num_blocks, int bs, int Hkv, int D, int dtype, int group,
                      kvq_pool_layout* lay, PoolView* view, size_t* off_pages, size_t* off_tok,
                      size_t* off_chan) {
  if (num_blocks < 1 || bs < 1 || Hkv < 1 || D < 1 || !valid_dtype(dtype) || lay == nullptr)
    return KVQ_ERR_INVALID_ARG;
  if (D % 16 != 0) return KVQ_ERR_INVALID_ARG;
  // blocks of 8 tokens (half a sub-tile per page), 16, 32 or 64 -- the sizes
  // the kernels have been run and checked at (others are refused until they
  // have); INT4's words pack tokens t and t+8 together and take 16 or more
  if (bs != 8 && bs != 16 && bs != 32 && bs != 64) return KVQ_ERR_UNSUPPORTED;
  if (bs == 8 && dtype == KVQ_INT4_PER_GROUP) return KVQ_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  int ng = 1;
  const bool grouped = dtype == KVQ_INT8_PER_GROUP || dtype == KVQ_INT4_PER_GROUP;
  if (grouped) {
    if (group <= 0 || D % group != 0) return KVQ_ERR_INVALID_ARG;
    if (group % 16 != 0) return KVQ_ERR_UNSUPPORTED;
    ng = D / group;
  } else {
    group = 0;
  }
  const int esize = dtype == KVQ_FP16 ? 2 : 1;
  // bytes of one 16-token sub-tile of K (or V) codes: INT4 packs two per byte
  const int sub_bytes = dtype == KVQ_INT4_PER_GROUP ? 8 * D : 16 * D * esize;
  const size_t code_bytes = (size_t)bs * sub_bytes / 16;  // K (or V) codes of one page
  const size_t page_scale = grouped ? 2 * (size_t)bs * ng * 4 : 0;
  const size_t page_bytes = 2 * code_bytes + page_scale;
  const size_t n_pages = (size_t)num_blocks * Hkv;
  size_t off = kvq::kHeaderBytes;
  const size_t op = off;
  off = align_up(off + n_pages * page_bytes, 256);
  const size_t ot = off;
  const bool tok = dtype == KVQ_INT8_PER_TOKEN || dtype == KVQ_FP8_E4M3_PER_TOKEN;
  const size_t tok_bytes = tok ? (size_t)num_blocks * 2 * bs * 4 : 0;
  off = align_up(off + tok_bytes, 256);
  const size_t oc = off;
  const size_t chan_bytes = dtype == KVQ_INT8_PER_CHANNEL ? 2 * (size_t)Hkv * D * 4 : 0;
  off = align_up(off + chan_bytes, 256);

  lay->total_bytes = off;
  lay->code_bytes = 2 * (size_t)num_blocks * Hkv * code_bytes;
  lay->scale_bytes = n_pages * page_scale + tok_bytes + chan_bytes;
  lay->header_bytes = off - lay->code_bytes - lay->scale_bytes;
  lay->page_bytes = page_bytes;
  if (view) {
    view->num_blocks = num_blocks;
    view->bs = bs;
    view->Hkv = Hkv;
    view->D = D;
    view->fmt = dtype;
    view->group = group;
    view->ng = ng;
    view->esize = esize;
    view->sub_bytes = sub_bytes;
    view->code_bytes = static_cast<int>(code_bytes);
    view->page_bytes = static_cast<int>(page_bytes);
  }
  if (off_pages) *off_pages = op;
  if (off_tok) *off_tok = ot;
  if (off_chan) *off_chan = oc;
  return KVQ_OK;
}

int device_sms() {
  static int cached[kvq::kMaxDevicesApi] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (dev >= 0 && dev < kvq::kMaxDevicesApi && cached[dev] > 0) return cached[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 152;
  if (dev >= 0 && dev < kvq::kMaxDevicesApi) cached[dev] = sms;
  return sms;
}

kvq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

}  // namespace

extern "C" {

kvq_status kvq_pool_layout_query(int64_t num_blocks, int block_size, int kv_heads, int head_dim,
                                 kvq_dtype dtype, int group, kvq_pool_layout* out) {
  return layout_for(num_blocks, block_size, kv_heads, head_dim, dtype, group, out, nullptr,
                    nullptr, nullptr, nullptr);
}

size_t kvq_pool_bytes(int64_t num_blocks, int block_size, int kv_heads, int head_dim,
                      kvq_dtype dtype, int group) {
  kvq_pool_layout lay{};
  if (layout_for(num_blocks, block_size, kv_heads, head_dim, dtype, group, &lay, nullptr, nullptr,
                 nullptr, nullptr) != KVQ_OK)
    return 0;
  return lay.total_bytes;
}

kvq_status kvq_alloc_pool(int64_t num_blocks, int block_size, int kv_heads, int head_dim,
                          kvq_dtype dtype, int group, void* device_buf, size_t buf_bytes,
                          kvq_pool** out) {
  if (out == nullptr) return KVQ_ERR_INVALID_ARG;
  *out = nullptr;
  kvq_pool_layout lay{};
  PoolView view{};
  size_t op = 0, ot = 0, oc = 0;
  kvq_status st = layout_for(num_blocks, block_size, kv_heads, head_dim, dtype, group, &lay, &view,
                             &op, &ot, &oc);
  if (st != KVQ_OK) return st;
  if (view.page_bytes <= 0 || (size_t)view.page_bytes != lay.page_bytes) return KVQ_ERR_UNSUPPORTED;
  void* base = device_buf;
  bool owned = false;
  if (base == nullptr) {
    if (cudaMalloc(&base, lay.total_bytes) != cudaSuccess) return KVQ_ERR_CUDA;
    owned = true;
  } else {
    if (buf_bytes < lay.total_bytes || (reinterpret_cast<uintptr_t>(base) & 255) != 0)
      return KVQ_ERR_INVALID_ARG;
  }
  // Clear the header (error word) and the per-channel scales.
  cudaError_t e = cudaMemset(base, 0, kvq::kHeaderBytes);
  if (e == cudaSuccess && dtype == KVQ_INT8_PER_CHANNEL)
    e = cudaMemset(static_cast<char*>(base) + oc, 0, 2 * (size_t)kv_heads * head_dim * 4);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    if (owned) cudaFree(base);
    return KVQ_ERR_CUDA;
  }
  kvq_pool* p = new (std::nothrow) kvq_pool;
  if (p == nullptr) {
    if (owned) cudaFree(base);
    return KVQ_ERR_INVALID_ARG;
  }
  char* b = static_cast<char*>(base);
  view.err = reinterpret_cast<int*>(b);
  view.pages = b + op;
  view.tok_scales = reinterpret_cast<float*>(b + ot);
  view.chan_scales = reinterpret_cast<float*>(b + oc);
  p->view = view;
  p->base = base;
  p->total_bytes = lay.total_bytes;
  p->owned = owned;
  p->layout = lay;
  cudaGetDevice(&p->device);
  *out = p;
  return KVQ_OK;
}

kvq_status kvq_free_pool(kvq_pool* pool) {
  if (pool == nullptr) return KVQ_OK;
  kvq_status st = KVQ_OK;
  if (pool->owned) {
    if (cudaDeviceSynchronize() != cudaSuccess) st = KVQ_ERR_CUDA;
    if (cudaFree(pool->base) != cudaSuccess) st = KVQ_ERR_CUDA;
  }
  delete pool;
  return st;
}

kvq_status kvq_set_channel_scales(kvq_pool* pool, const float* k_scale, const float* v_scale,
                                  cudaStream_t stream) {
  if (pool == nullptr || k_scale == nullptr || v_scale == nullptr) return KVQ_ERR_INVALID_ARG;
  if (pool->view.fmt != KVQ_INT8_PER_CHANNEL) return KVQ_ERR_INVALID_ARG;
  const size_t n = (size_t)pool->view.Hkv * pool->view.D * sizeof(float);
  cudaError_t e = cudaMemcpyAsync(pool->view.chan_scales, k_scale, n, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(reinterpret_cast<char*>(pool->view.chan_scales) + n, v_scale, n,
                        cudaMemcpyDeviceToDevice, stream);
  return from_cuda(e);
}

kvq_status kvq_calibrate_channel_scales(kvq_pool* pool, const kvq_half* k, const kvq_half* v,
                                        int64_t T, cudaStream_t stream) {
  if (pool == nullptr || k == nullptr || v == nullptr || T < 1) return KVQ_ERR_INVALID_ARG;
  if (pool->view.fmt != KVQ_INT8_PER_CHANNEL) return KVQ_ERR_INVALID_ARG;
  return from_cuda(kvq::launch_calibrate(pool->view, reinterpret_cast<const __half*>(k),
                                         reinterpret_cast<const __half*>(v), T, stream));
}

kvq_status kvq_append(kvq_pool* pool, const kvq_half* k, const kvq_half* v,
                      const int64_t* slot_mapping, int64_t T, cudaStream_t stream) {
  if (pool == nullptr || T < 0) return KVQ_ERR_INVALID_ARG;
  if (T == 0) return KVQ_OK;
  if (k == nullptr || v == nullptr || slot_mapping == nullptr) return KVQ_ERR_INVALID_ARG;
  if (T > 0x7fffffffLL) return KVQ_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) return KVQ_ERR_INVALID_ARG;
  return from_cuda(kvq::launch_append(pool->view, reinterpret_cast<const __half*>(k),
                                      reinterpret_cast<const __half*>(v), slot_mapping, T, stream));
}

kvq_status kvq_copy_blocks(kvq_pool* pool, const int32_t* src_blocks, const int32_t* dst_blocks,
                           int n, cudaStream_t stream) {
  if (pool == nullptr || n < 0) return KVQ_ERR_INVALID_ARG;
  if (n == 0) return KVQ_OK;
  if (src_blocks == nullptr || dst_blocks == nullptr || n > 0x7fffffff) return KVQ_ERR_INVALID_ARG;
  return from_cuda(kvq::launch_copy_blocks(pool->view, src_blocks, dst_blocks, n, stream));
}

kvq_status kvq_append_strided(kvq_pool* pool, const kvq_half* k, const kvq_half* v,
                              int64_t row_stride, const int64_t* slot_mapping, int64_t T,
                              cudaStream_t stream) {
  if (pool == nullptr || T < 0) return KVQ_ERR_INVALID_ARG;
  if (T == 0) return KVQ_OK;
  if (k == nullptr || v == nullptr || slot_mapping == nullptr) return KVQ_ERR_INVALID_ARG;
  if (T > 0x7fffffffLL) return KVQ_ERR_UNSUPPORTED;
  if (row_stride < (int64_t)pool->view.Hkv * pool->view.D || row_stride % 8 != 0)
    return KVQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) return KVQ_ERR_INVALID_ARG;
  return from_cuda(kvq::launch_step_append(pool->view, reinterpret_cast<const __half*>(k),
                                           reinterpret_cast<const __half*>(v), slot_mapping, T,
                                           nullptr, nullptr, 0, 0, stream, false, row_stride));
}

size_t kvq_decode_workspace_bytes_ex(const kvq_pool* pool, int num_seqs, int num_q_heads,
                                     int max_context_len, int split_blocks) {
  if (pool == nullptr || num_seqs < 0 || num_q_heads < 1 || num_q_heads % pool->view.Hkv != 0)
    return 0;
  kvq::DecodePlan plan;
  if (!kvq::plan_decode(pool->view, num_seqs, num_q_heads, max_context_len, split_blocks,
                        device_sms(), &plan))
    return 0;
  return plan.ws_bytes;
}

size_t kvq_decode_workspace_bytes(const kvq_pool* pool, int num_seqs, int num_q_heads,
                                  int max_context_len) {
  return kvq_decode_workspace_bytes_ex(pool, num_seqs, num_q_heads, max_context_len, 0);
}

}  // extern "C"

// Argument checks and plan shared by the decode entry points.
static kvq_status prepare_decode(const kvq_pool* pool, const kvq_half* q, int num_seqs,
                                 int num_q_heads, const int32_t* block_table,
                                 int max_blocks_per_seq, const int32_t* context_lens,
                                 int max_context_len, float sm_scale, float* out, void* workspace,
                                 size_t ws_bytes, int split_blocks, kvq::DecodeArgs* a,
                                 kvq::DecodePlan* plan) {
  if (pool == nullptr || num_seqs < 0 || num_q_heads < 1 || max_blocks_per_seq < 1 ||
      max_context_len < 0 || split_blocks < 0)
    return KVQ_ERR_INVALID_ARG;
  if (num_seqs == 0) return KVQ_OK;
  if (q == nullptr || block_table == nullptr || context_lens == nullptr || out == nullptr)
    return KVQ_ERR_INVALID_ARG;
  if (num_q_heads % pool->view.Hkv != 0) return KVQ_ERR_INVALID_ARG;
  if ((int64_t)max_context_len > (int64_t)max_blocks_per_seq * pool->view.bs) return KVQ_ERR_INVALID_ARG;
  if (num_seqs > 65535) return KVQ_ERR_UNSUPPORTED;
  if (!(sm_scale == sm_scale)) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(q) & 15) return KVQ_ERR_INVALID_ARG;
  if (!kvq::plan_decode(pool->view, num_seqs, num_q_heads, max_context_len, split_blocks,
                        device_sms(), plan))
    return KVQ_ERR_UNSUPPORTED;
  if (plan->ws_bytes > 0) {
    if (workspace == nullptr || ws_bytes < plan->ws_bytes) return KVQ_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return KVQ_ERR_INVALID_ARG;
  }
  a->pool = pool->view;
  a->q = reinterpret_cast<const __half*>(q);
  a->table = block_table;
  a->lens = context_lens;
  a->out = out;
  a->workspace = workspace;
  a->S = num_seqs;
  a->Hq = num_q_heads;
  a->max_blocks = max_blocks_per_seq;
  a->max_ctx = max_context_len;
  a->sm_scale = sm_scale;
  return KVQ_OK;
}

extern "C" {

kvq_status kvq_paged_decode_ex(const kvq_pool* pool, const kvq_half* q, int num_seqs,
                               int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                               const int32_t* context_lens, int max_context_len, float sm_scale,
                               float* out, void* workspace, size_t ws_bytes, int split_blocks,
                               cudaStream_t stream) {
  kvq::DecodeArgs a;
  kvq::DecodePlan plan;
  const kvq_status st =
      prepare_decode(pool, q, num_seqs, num_q_heads, block_table, max_blocks_per_seq, context_lens,
                     max_context_len, sm_scale, out, workspace, ws_bytes, split_blocks, &a, &plan);
  if (st != KVQ_OK || num_seqs == 0) return st;
  return from_cuda(kvq::launch_decode(a, plan, stream));
}

kvq_status kvq_selftest_decode_timeout(const kvq_pool* pool, const kvq_half* q, int num_seqs,
                                       int num_q_heads, const int32_t* block_table,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int max_context_len, float* out, void* workspace,
                                       size_t ws_bytes, int wait_tries, cudaStream_t stream) {
  if (wait_tries < 1 || wait_tries > 1000) return KVQ_ERR_INVALID_ARG;
  kvq::DecodeArgs a;
  kvq::DecodePlan plan;
  const kvq_status st =
      prepare_decode(pool, q, num_seqs, num_q_heads, block_table, max_blocks_per_seq, context_lens,
                     max_context_len, 1.0f, out, workspace, ws_bytes, 0, &a, &plan);
  if (st != KVQ_OK || num_seqs == 0) return st;
  a.wait_tries = wait_tries;
  a.fault_issue = 0;  // warp 0's first copy is armed but never issued
  return from_cuda(kvq::launch_decode(a, plan, stream));
}

kvq_status kvq_paged_decode_strided(const kvq_pool* pool, const kvq_half* q,
                                    int64_t q_row_stride, int num_seqs, int num_q_heads,
                                    const int32_t* block_table, int max_blocks_per_seq,
                                    const int32_t* context_lens, int max_context_len,
                                    float sm_scale, float* out, int64_t out_row_stride,
                                    void* workspace, size_t ws_bytes, cudaStream_t stream) {
  kvq::DecodeArgs a;
  kvq::DecodePlan plan;
  const kvq_status st =
      prepare_decode(pool, q, num_seqs, num_q_heads, block_table, max_blocks_per_seq, context_lens,
                     max_context_len, sm_scale, out, workspace, ws_bytes, 0, &a, &plan);
  if (st != KVQ_OK || num_seqs == 0) return st;
  const int64_t row = (int64_t)num_q_heads * pool->view.D;
  if (q_row_stride < row || q_row_stride % 8 != 0 || out_row_stride < row) return KVQ_ERR_INVALID_ARG;
  a.q_stride = q_row_stride;
  a.out_stride = out_row_stride;
  return from_cuda(kvq::launch_decode(a, plan, stream));
}

kvq_status kvq_decode_step(kvq_pool* pool, const kvq_half* k_new, const kvq_half* v_new,
                           const kvq_half* q, int num_seqs, int num_q_heads,
                           const int32_t* block_table, int max_blocks_per_seq,
                           const int32_t* context_lens, int max_context_len, float sm_scale,
                           float* out, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  kvq::DecodeArgs a;
  kvq::DecodePlan plan;
  const kvq_status st =
      prepare_decode(pool, q, num_seqs, num_q_heads, block_table, max_blocks_per_seq, context_lens,
                     max_context_len, sm_scale, out, workspace, ws_bytes, 0, &a, &plan);
  if (st != KVQ_OK || num_seqs == 0) return st;
  if (k_new == nullptr || v_new == nullptr) return KVQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return KVQ_ERR_INVALID_ARG;
  cudaError_t e = kvq::launch_step_append(pool->view, reinterpret_cast<const __half*>(k_new),
                                          reinterpret_cast<const __half*>(v_new), nullptr, num_seqs,
                                          block_table, context_lens, max_blocks_per_seq,
                                          max_context_len, stream, /*dependent=*/true);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(kvq::launch_decode(a, plan, stream, /*dependent=*/true));
}

}  // extern "C"

// Prefix-partial bytes at the start of a cascade workspace.
static size_t cascade_pre_bytes(const kvq_pool* pool, int num_seqs, int num_q_heads) {
  const size_t b = (size_t)num_seqs * num_q_heads * (pool->view.D + 2) * sizeof(float);
  return (b + 255) / 256 * 256;
}

// Checks, plans and launches of the cascade; k_new/v_new non-null adds the
// decode-step append in front.
static kvq_status cascade(kvq_pool* pool, const kvq_half* k_new, const kvq_half* v_new,
                          const kvq_half* q, int num_seqs, int num_q_heads,
                          const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* context_lens, int max_context_len, int prefix_blocks,
                          float sm_scale, float* out, void* workspace, size_t ws_bytes,
                          cudaStream_t stream) {
  if (pool == nullptr || prefix_blocks < 0 || prefix_blocks > max_blocks_per_seq)
    return KVQ_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_q_heads < 1 || num_q_heads % pool->view.Hkv != 0)
    return KVQ_ERR_INVALID_ARG;
  const size_t pre_bytes = cascade_pre_bytes(pool, num_seqs, num_q_heads);
  const bool casc = prefix_blocks > 0;
  // the prefix kernel reads whole 16-token sub-tiles from one page
  if (casc && pool->view.bs == 8) return KVQ_ERR_UNSUPPORTED;
  if (casc && (workspace == nullptr || ws_bytes < pre_bytes)) return KVQ_ERR_WORKSPACE;
  void* dws = casc ? static_cast<char*>(workspace) + pre_bytes : workspace;
  const size_t dws_bytes = casc ? ws_bytes - pre_bytes : ws_bytes;
  kvq::DecodeArgs a;
  kvq::DecodePlan plan;
  kvq_status st = prepare_decode(pool, q, num_seqs, num_q_heads, block_table, max_blocks_per_seq,
                                 context_lens, max_context_len, sm_scale, out, dws, dws_bytes, 0,
                                 &a, &plan);
  if (st != KVQ_OK || num_seqs == 0) return st;
  kvq::RowsPlan pplan;
  if (casc && !kvq::plan_rows(pool->view, num_seqs, num_q_heads, &pplan))
    return KVQ_ERR_UNSUPPORTED;
  const bool step = k_new != nullptr || v_new != nullptr;
  if (step) {
    if (k_new == nullptr || v_new == nullptr) return KVQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
      return KVQ_ERR_INVALID_ARG;
    cudaError_t e = kvq::launch_step_append(pool->view, reinterpret_cast<const __half*>(k_new),
                                            reinterpret_cast<const __half*>(v_new), nullptr,
                                            num_seqs, block_table, context_lens,
                                            max_blocks_per_seq, max_context_len, stream, true);
    if (e != cudaSuccess) return from_cuda(e);
  }
  if (casc) {
    kvq::RowsArgs pa;
    pa.pool = pool->view;
    pa.q = reinterpret_cast<const __half*>(q);
    pa.table = block_table;
    pa.lens = context_lens;
    pa.out = static_cast<float*>(workspace);
    pa.S = num_seqs;
    pa.Hq = num_q_heads;
    pa.max_blocks = max_blocks_per_seq;
    pa.max_ctx = max_context_len;
    pa.P = prefix_blocks;
    pa.sm_scale = sm_scale;
    cudaError_t e = kvq::launch_rows(pa, pplan, stream, step);
    if (e != cudaSuccess) return from_cuda(e);
    a.skip = prefix_blocks;
    a.pre = pa.out;
  }
  return from_cuda(kvq::launch_decode(a, plan, stream, step || casc));
}

extern "C" {

size_t kvq_cascade_workspace_bytes(const kvq_pool* pool, int num_seqs, int num_q_heads,
                                   int max_context_len) {
  if (pool == nullptr || num_seqs < 0 || num_q_heads < 1 || num_q_heads % pool->view.Hkv != 0)
    return 0;
  return cascade_pre_bytes(pool, num_seqs, num_q_heads) +
         kvq_decode_workspace_bytes_ex(pool, num_seqs, num_q_heads, max_context_len, 0);
}

kvq_status kvq_cascade_decode(const kvq_pool* pool, const kvq_half* q, int num_seqs,
                              int num_q_heads, const int32_t* block_table, int max_blocks_per_seq,
                              const int32_t* context_lens, int max_context_len,
                              int prefix_blocks, float sm_scale, float* out, void* workspace,
                              size_t ws_bytes, cudaStream_t stream) {
  return cascade(const_cast<kvq_pool*>(pool), nullptr, nullptr, q, num_seqs, num_q_heads,
                 block_table, max_blocks_per_seq, context_lens, max_context_len, prefix_blocks,
                 sm_scale, out, workspace, ws_bytes, stream);
}

kvq_status kvq_cascade_decode_step(kvq_pool* pool, const kvq_half* k_new, const kvq_half* v_new,
                                   const kvq_half* q, int num_seqs, int num_q_heads,
                                   const int32_t* block_table, int max_blocks_per_seq,
                                   const int32_t* context_lens, int max_context_len,
                                   int prefix_blocks, float sm_scale, float* out, void* workspace,
                                   size_t ws_bytes, cudaStream_t stream) {
  if (k_new == nullptr || v_new == nullptr) return KVQ_ERR_INVALID_ARG;
  return cascade(pool, k_new, v_new, q, num_seqs, num_q_heads, block_table, max_blocks_per_seq,
                 context_lens, max_context_len, prefix_blocks, sm_scale, out, workspace, ws_bytes,
                 stream);
}

kvq_status kvq_prefill(const kvq_pool* pool, const kvq_half* q, int num_seqs, int num_q_heads,
                       const int32_t* q_start, int max_q_len, const int32_t* block_table,
                       int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                       float sm_scale, float* out, cudaStream_t stream) {
  if (pool == nullptr || num_seqs < 0 || num_q_heads < 1 || max_q_len < 0 ||
      max_blocks_per_seq < 1 || max_context_len < 0)
    return KVQ_ERR_INVALID_ARG;
  // the prefill kernel converts whole 16-token sub-tiles of one page
  if (pool->view.bs == 8) return KVQ_ERR_UNSUPPORTED;
  if (num_seqs == 0 || max_q_len == 0) return KVQ_OK;
  if (q == nullptr || q_start == nullptr || block_table == nullptr || context_lens == nullptr ||
      out == nullptr)
    return KVQ_ERR_INVALID_ARG;
  if (num_q_heads % pool->view.Hkv != 0) return KVQ_ERR_INVALID_ARG;
  if ((int64_t)max_context_len > (int64_t)max_blocks_per_seq * pool->view.bs) return KVQ_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(q) & 15) return KVQ_ERR_INVALID_ARG;
  const cudaError_t e = kvq::launch_prefill(
      pool->view, reinterpret_cast<const __half*>(q), num_seqs, num_q_heads, q_start, max_q_len,
      block_table, max_blocks_per_seq, context_lens, max_context_len, sm_scale, out, stream);
  return e == cudaErrorInvalidValue ? KVQ_ERR_UNSUPPORTED : from_cuda(e);
}

size_t kvq_prefill_workspace_bytes(const kvq_pool* pool, int num_seqs, int max_context_len) {
  if (pool == nullptr || num_seqs < 1 || max_context_len < 1) return 0;
  return kvq::prefill_ws_bytes(pool->view, num_seqs, max_context_len);
}

kvq_status kvq_prefill_ex(const kvq_pool* pool, const kvq_half* q, int num_seqs, int num_q_heads,
                          const int32_t* q_start, int max_q_len, const int32_t* block_table,
                          int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                          float sm_scale, float* out, void* workspace, size_t ws_bytes,
                          cudaStream_t stream) {
  if (pool == nullptr) return KVQ_ERR_INVALID_ARG;
  const size_t need = kvq_prefill_workspace_bytes(pool, num_seqs, max_context_len);
  if (need == 0)  // a format or geometry the two-pass path does not take
    return kvq_prefill(pool, q, num_seqs, num_q_heads, q_start, max_q_len, block_table,
                       max_blocks_per_seq, context_lens, max_context_len, sm_scale, out, stream);
  if (num_seqs < 0 || num_q_heads < 1 || max_q_len < 0 || max_blocks_per_seq < 1 ||
      max_context_len < 0)
    return KVQ_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_q_len == 0) return KVQ_OK;
  if (q == nullptr || q_start == nullptr || block_table == nullptr || context_lens == nullptr ||
      out == nullptr)
    return KVQ_ERR_INVALID_ARG;
  if (num_q_heads % pool->view.Hkv != 0) return KVQ_ERR_INVALID_ARG;
  if ((int64_t)max_context_len > (int64_t)max_blocks_per_seq * pool->view.bs) return KVQ_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return KVQ_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(q) & 15) return KVQ_ERR_INVALID_ARG;
  if (workspace == nullptr || ws_bytes < need) return KVQ_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return KVQ_ERR_INVALID_ARG;
  const cudaError_t e = kvq::launch_prefill_ws(
      pool->view, reinterpret_cast<const __half*>(q), num_seqs, num_q_heads, q_start, max_q_len,
      block_table, max_blocks_per_seq, context_lens, max_context_len, sm_scale, out, workspace,
      stream);
  return e == cudaErrorInvalidValue ? KVQ_ERR_UNSUPPORTED : from_cuda(e);
}

kvq_status kvq_paged_decode(const kvq_pool* pool, const kvq_half* q, int num_seqs, int num_q_heads,
                            const int32_t* block_table, int max_blocks_per_seq,
                            const int32_t* context_lens, int max_context_len, float sm_scale,
                            float* out, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return kvq_paged_decode_ex(pool, q, num_seqs, num_q_heads, block_table, max_blocks_per_seq,
                             context_lens, max_context_len, sm_scale, out, workspace, ws_bytes, 0,
                             stream);
}

kvq_status kvq_read_slots(const kvq_pool* pool, const int64_t* slots, int64_t n, void* codes_out,
                          float* scales_out, cudaStream_t stream) {
  if (pool == nullptr || n < 0) return KVQ_ERR_INVALID_ARG;
  if (n == 0) return KVQ_OK;
  if (slots == nullptr || codes_out == nullptr || n > 0x7fffffffLL) return KVQ_ERR_INVALID_ARG;
  const int f = pool->view.fmt;
  const bool has_scales = f == KVQ_INT8_PER_GROUP || f == KVQ_INT4_PER_GROUP ||
                          f == KVQ_INT8_PER_TOKEN || f == KVQ_FP8_E4M3_PER_TOKEN;
  return from_cuda(kvq::launch_read_slots(pool->view, slots, n, codes_out,
                                          has_scales ? scales_out : nullptr, stream));
}

kvq_status kvq_get_error(kvq_pool* pool, cudaStream_t stream) {
  if (pool == nullptr) return KVQ_ERR_INVALID_ARG;
  int host = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpy(&host, pool->view.err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(pool->view.err, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  if (host & kvq::ERR_RANGE) return KVQ_ERR_OUT_OF_RANGE;
  if (host & kvq::ERR_TIMEOUT) return KVQ_ERR_TIMEOUT;
  return KVQ_OK;
}

kvq_status kvq_set_phase_events(const cudaEvent_t* events, int n) {
  if (n < 0 || n > KVQ_MAX_PHASE_EVENTS || (n > 0 && events == nullptr)) return KVQ_ERR_INVALID_ARG;
  for (int k = 0; k < n; ++k) t_phase.ev[k] = events[k];
  t_phase.n = n;
  t_phase.next = 0;
  return KVQ_OK;
}

const char* kvq_status_string(kvq_status status) {
  switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported geometry";
    case KVQ_ERR_CUDA: return "CUDA runtime error";
    case KVQ_ERR_OUT_OF_RANGE: return "slot, block id or context length out of range";
    case KVQ_ERR_WORKSPACE: return "decode workspace too small";
    case KVQ_ERR_TIMEOUT: return "a bounded device wait gave up";
  }
  return "unknown status";
}

}  // extern "C"
