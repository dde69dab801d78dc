// common.cuh -- device helpers shared by the cconv kernels (sm_103a only).
//
// Inline PTX for the pieces the kernels are built from: mbarrier-tracked TMA tile loads,
// packed f32x2 arithmetic, the hardware tanh approximation and bf16 pack / unpack.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/cconv.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "cconv kernels are written for sm_103a (Blackwell) only"
#endif

namespace cconv {

// ------------------------------------------------------------------------------------
// fault word: set by a kernel that gave up a bounded wait (never expected to happen)
// ------------------------------------------------------------------------------------
enum FaultCode : unsigned {
  kFaultFwdWait = 1u,
  kFaultBwdWait = 2u,
  kFaultSeqlens = 4u,  // an ill-formed cu_seqlens was passed (results unspecified)
};

// Nanoseconds a kernel waits on one TMA tile before it reports a fault and returns.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------------------------
// shared memory, mbarrier, TMA
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later async-proxy ones.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for phase `parity` of `bar` to complete, giving up after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Nanoseconds the thread that issued a CTA's tile copies waits, per stage, for them to land
// before it returns.
constexpr unsigned long long kDrainLimitNs = 100000000ull;

// The thread that issued `issued` tile copies into stages 0, 1, ..., S-1, 0, ... (each
// completing on its stage's full barrier) waits until every one of them has landed before it
// returns.  A CTA's shared memory stays allocated until its last thread exits, so with this
// wait at the end of the issuing thread no copy can land in the shared memory of a CTA that
// has exited, whichever of its threads gave up a bounded wait first.  In a run where nothing
// gave up, it only waits for the last few stages, which the consumers are waiting for too.
template <int S>
__device__ __forceinline__ void drain_issued(uint64_t* full, int issued) {
  for (int s = 0; s < S && s < issued; ++s) {
    const int armed = (issued - 1 - s) / S + 1;  // phases of stage s that were armed
    (void)mbar_wait_bounded(&full[s], static_cast<uint32_t>(armed - 1) & 1u, kDrainLimitNs);
  }
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
// Coordinates are (innermost, middle, outermost) = (channel, row, batch).  Rows outside
// [0, T) and channels outside [0, D) are filled with zeros by the copy engine.  No L2 cache
// hint: with an evict_first policy the lockstep kernels were slower (backward 70.2 against
// 67.0 us, forward 43.4 against 42.0 us at B=2 T=8192 D=4096, with streaming row stores in
// both; an evict_normal policy gave 67.3 and 43.0 us).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c, int r, int b) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c), "r"(r), "r"(b), "r"(smem_addr(bar))
      : "memory");
}

// The same with an L2 cache-policy operand.  The independent-pipeline backward (rows under
// 2048 channels) is faster with evict_first loads: D=512 17.9 against 18.6 us, D=1024 25.5
// against 25.9 us, D=1536 34.2 against 35.1 us (B=2 T=8192), while the lockstep kernels
// are faster without a hint.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c, int r, int b, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c), "r"(r), "r"(b), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

// L2 eviction policy for data read exactly once.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

__device__ __forceinline__ uint2 lds64(const void* p) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_addr(p)));
  return v;
}

// Programmatic dependent launch: wait for the preceding grid / let the next one start.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------------------------
// packed f32x2 arithmetic (one instruction for two lanes of fp32 work)
// ------------------------------------------------------------------------------------
typedef unsigned long long f2;  // {lo, hi} fp32 pair in one 64-bit register

__device__ __forceinline__ f2 f2_pack(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 f2_splat(float v) { return f2_pack(v, v); }

// Hardware tanh approximation (MUFU), relative error about 2^-11.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ f2 f2_tanh(f2 v) {
  float lo, hi;
  f2_unpack(v, lo, hi);
  return f2_pack(tanh_approx(lo), tanh_approx(hi));
}

// bf16x2 word -> fp32 pair: a bf16 is the upper half of a binary32, so each half is moved
// into the top 16 bits of a zeroed word (one byte permute each).
__device__ __forceinline__ f2 bf16x2_to_f2(uint32_t u) {
  return f2_pack(__uint_as_float(__byte_perm(u, 0u, 0x1044)),
                 __uint_as_float(__byte_perm(u, 0u, 0x3244)));
}

// fp32 pair -> bf16x2 word, round to nearest even.
__device__ __forceinline__ uint32_t f2_to_bf16x2(f2 v) {
  float lo, hi;
  f2_unpack(v, lo, hi);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16(float v) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}


// ------------------------------------------------------------------------------------
// host: launch with programmatic stream serialisation.  The kernel may be scheduled
// before the previous kernel on the stream has finished (once that kernel's CTAs have all
// triggered or exited); every cconv kernel executes griddepcontrol.wait before its first
// global-memory read or write, so it still reads and writes only after the previous kernel
// has completed and flushed.  (The packed backward prefetches cu_seqlens into L2 before the
// wait: a prefetch returns no data, and L2 is where device memory is coherent.)  Without a
// trigger in the previous kernel this is an ordinary stream-ordered launch.
// ------------------------------------------------------------------------------------
// With CCONV_DEBUG set in the environment, failing CUDA calls are reported on stderr.
cudaError_t report_cuda(const char* what, cudaError_t e);

// Launch recording (cconv_describe_begin / cconv_describe_end, host.cu): while the calling
// thread records, a launch is described instead of enqueued.
bool recording_launches();
void record_launch(const void* func, dim3 grid, dim3 block, size_t smem);

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  if (recording_launches()) {
    record_launch(reinterpret_cast<const void*>(kernel), grid, block, smem);
    return cudaSuccess;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return report_cuda("kernel launch", cudaLaunchKernelEx(&lc, kernel, args...));
}

// ------------------------------------------------------------------------------------
// host side helpers (defined in host.cu)
// ------------------------------------------------------------------------------------
int sm_count_current_device(int* sms, int* device);
int encode_rows_map(CUtensorMap* map, const void* base, int64_t B, int64_t T, int64_t D,
                    int64_t sb, int64_t st, int box_c, int box_r);
int set_max_dynamic_smem(const void* func, int bytes);
// Validates n state indices against a pool of S slots (negative, >= S, repeated), as the
// decode update does, and writes status[0..1]; nothing else (fwd.cu).
int launch_index_check(const int32_t* idx, int64_t n, int64_t S, int32_t* status,
                       cudaStream_t stream);

}  // namespace cconv

