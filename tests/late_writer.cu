// Test helper: a one-block kernel that lets the next grid on its stream start at once
// (programmatic dependent launch), waits about delay_ns, then copies up to two int32 arrays.  A
// decode call launched right after it starts while the old values are still in place and must see
// only the new ones after its grid-dependency wait.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__global__ void late_copy_kernel(const int32_t* src0, int32_t* dst0, int n0, const int32_t* src1, int32_t* dst1,
                                 int n1, long long delay_ns) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  // bounded: at most ~2e5 sleeps of ~1 us, whatever the timer does
  for (int i = 0; i < 200000; ++i) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (static_cast<long long>(t - t0) >= delay_ns) break;
    __nanosleep(1000);
  }
  for (int i = threadIdx.x; i < n0; i += blockDim.x) dst0[i] = src0[i];
  for (int i = threadIdx.x; i < n1; i += blockDim.x) dst1[i] = src1[i];
}

}  // namespace

// Returns the CUDA error code of the launch (0 on success).
extern "C" int late_copy(const int32_t* src0, int32_t* dst0, int n0, const int32_t* src1, int32_t* dst1, int n1,
                         long long delay_ns, void* stream) {
  if (n0 < 0 || n1 < 0 || (n0 > 0 && (!src0 || !dst0)) || (n1 > 0 && (!src1 || !dst1))) return -1;
  late_copy_kernel<<<1, 256, 0, static_cast<cudaStream_t>(stream)>>>(src0, dst0, n0, src1, dst1, n1, delay_ns);
  return static_cast<int>(cudaGetLastError());
}
