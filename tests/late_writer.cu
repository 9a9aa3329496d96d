// Test helper, built by the test that uses it: a kernel standing for a
// caller's kernel that produces the context lengths of the next decode step
// and, as kernels written for programmatic dependent launch do, lets its
// dependents launch at its start.  It copies n int32 values after a bounded
// delay (at most ~0.1 s whatever the clock), so that a dependent which reads
// them before waiting for this grid's completion sees the old values.
#include <cuda_runtime.h>

__global__ void late_write_kernel(int* dst, const int* src, int n, unsigned long long delay_ns) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int i = 0; i < 100000; ++i) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 >= delay_ns) break;
    __nanosleep(1000);
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}

extern "C" int late_write(int* dst, const int* src, int n, unsigned long long delay_ns,
                          void* stream) {
  late_write_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(dst, src, n, delay_ns);
  return static_cast<int>(cudaGetLastError());
}
