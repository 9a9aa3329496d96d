// kvq_context.h -- host-side bookkeeping of per-CUDA-context set-up, and the
// per-thread hook that records timing events after kernel launches.
//
// Some set-up is done once and then remembered: a kernel's opt-in to more
// than 48 KB of dynamic shared memory (cudaFuncSetAttribute), and the device
// address of a file-scope __device__ array (cudaGetSymbolAddress).  Both
// belong to a CUDA context, not to a device number: after cudaDeviceReset,
// or in another driver context on the same device, the remembered state is
// gone or points at memory that is no longer mapped.  So the caches below are
// keyed on the id of the context current on the calling thread (cuCtxGetId,
// a per-process unique number), looked up through the runtime's driver entry
// points (no link against libcuda), and guarded by a mutex because any host
// thread may call the library.
#pragma once
#include <cuda.h>
#include <cuda_runtime_api.h>

#include <mutex>

namespace kvq {

// Id of the CUDA context current on this thread; 0 if there is none yet or
// the driver cannot tell (callers then do their set-up without caching).
inline unsigned long long current_context_id() {
  using GetCur = CUresult(CUDAAPI*)(CUcontext*);
  using GetId = CUresult(CUDAAPI*)(CUcontext, unsigned long long*);
  static GetCur get_cur = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      return static_cast<GetCur>(nullptr);
    return reinterpret_cast<GetCur>(f);
  }();
  static GetId get_id = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      return static_cast<GetId>(nullptr);
    return reinterpret_cast<GetId>(f);
  }();
  if (get_cur == nullptr || get_id == nullptr) return 0;
  CUcontext c = nullptr;
  if (get_cur(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// A value computed once per CUDA context (up to kSlots contexts remembered;
// the oldest is forgotten first, which only costs a repeated set-up).
template <class V>
class PerContext {
 public:
  static constexpr int kSlots = 64;

  // The value for the current context: the cached one, or make(&v) run now.
  template <class Make>
  cudaError_t get(V* out, Make&& make) {
    unsigned long long id = current_context_id();
    {
      std::lock_guard<std::mutex> lock(mu_);
      for (int i = 0; id != 0 && i < kSlots; ++i)
        if (ids_[i] == id) {
          *out = vals_[i];
          return cudaSuccess;
        }
    }
    V v{};
    const cudaError_t e = make(&v);  // may make the context current
    if (e != cudaSuccess) return e;
    if (id == 0) id = current_context_id();
    if (id != 0) {
      std::lock_guard<std::mutex> lock(mu_);
      ids_[next_] = id;
      vals_[next_] = v;
      next_ = (next_ + 1) % kSlots;
    }
    *out = v;
    return cudaSuccess;
  }

 private:
  std::mutex mu_;
  unsigned long long ids_[kSlots] = {};
  V vals_[kSlots] = {};
  int next_ = 0;
};

// Per-kernel timing events (kvq_set_phase_events): every kernel launch of the
// library passes its launch status through this, right after the launch, on
// the kernel's stream.  On success it records the calling thread's next
// registered event, if one is left; the launch's error otherwise.  Defined in
// kvq_api.cu.
cudaError_t phase_mark(cudaStream_t st, cudaError_t launched);

// Opt a kernel in to up to 227 KB of dynamic shared memory, once per
// context (one cache per kernel: the kernel is a template argument).
template <auto Kernel>
cudaError_t allow_big_smem() {
  static PerContext<char> done;
  char v = 0;
  return done.get(&v, [](char*) {
    return cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
}

}  // namespace kvq
