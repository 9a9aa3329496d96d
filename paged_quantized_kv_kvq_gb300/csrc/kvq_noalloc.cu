// kvq_noalloc.cu -- kvq_paged_decode_noalloc: paged decode whose split-K
// scratch is a fixed device array owned by the library, for callers that
// cannot allocate device memory (see include/kvq.h).
#include "kvq.h"
#include "kvq_context.h"

namespace {

// The scratch: one copy per GPU that loads this library, kept until exit.
static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

// Device address of the array in the current CUDA context, looked up on the
// first call in that context (with it current) and remembered per context, so
// that a device reset or another driver context gets a fresh lookup.  Host
// code cannot use the symbol itself: on the host it names a stand-in, not
// device memory.
kvq::PerContext<void*> g_addr;

cudaError_t scratch_address(void** out) {
  return g_addr.get(out, [](void** p) { return cudaGetSymbolAddress(p, g_decode_scratch); });
}

}  // namespace

extern "C" kvq_status kvq_paged_decode_noalloc(const kvq_pool* pool, const kvq_half* q,
                                               int num_seqs, int num_q_heads,
                                               const int32_t* block_table, int max_blocks_per_seq,
                                               const int32_t* context_lens, int max_context_len,
                                               float sm_scale, float* out, int split_blocks,
                                               cudaStream_t stream) {
  if (pool == nullptr) return KVQ_ERR_INVALID_ARG;
  const size_t need = kvq_decode_workspace_bytes_ex(pool, num_seqs, num_q_heads, max_context_len,
                                                    split_blocks);
  if (need > KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KVQ_ERR_CUDA;
  // The split partials are written before they are read; nothing needs clearing.
  return kvq_paged_decode_ex(pool, q, num_seqs, num_q_heads, block_table, max_blocks_per_seq,
                             context_lens, max_context_len, sm_scale, out, scratch,
                             KVQ_NOALLOC_SCRATCH_BYTES, split_blocks, stream);
}
