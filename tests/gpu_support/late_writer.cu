// late_writer.cu -- test support: a kernel that lets its programmatic dependents start at
// once and writes its output only after a short delay.
//
// The packed-sequence kernels of libcconv.so are launched as programmatic dependents of
// whatever kernel precedes them on the stream.  They may start while that kernel still
// runs, and must not read anything it writes (cu_seqlens here) before their
// griddepcontrol.wait.  This kernel executes griddepcontrol.launch_dependents first, then
// waits `delay_ns` nanoseconds (measured on %globaltimer, so the wait always ends), then
// copies n int32 values from src to dst.  A dependent that read dst before its wait would
// see the old contents.
#include <cuda_runtime.h>
#include <stdint.h>

__global__ void late_copy_kernel(int32_t* dst, const int32_t* src, int n,
                                 unsigned long long delay_ns) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  do {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < delay_ns);
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}

extern "C" int late_copy(int32_t* dst, const int32_t* src, int n, unsigned long long delay_ns,
                         cudaStream_t stream) {
  if (delay_ns > 10000000ull) return -1;  // at most 10 ms
  late_copy_kernel<<<1, 256, 0, stream>>>(dst, src, n, delay_ns);
  return static_cast<int>(cudaGetLastError());
}
