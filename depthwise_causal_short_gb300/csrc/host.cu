// host.cu -- host-side pieces shared by the cconv entry points: status names, device SM
// count, TMA descriptor encoding, the fault-word reader.
#include <cudaTypedefs.h>

#include <cxxabi.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace cconv {

// Per-TU fault readers (each kernel file owns its own device fault word).
int read_clear_fault_fwd(unsigned* out);
int read_clear_fault_bwd(unsigned* out);

cudaError_t report_cuda(const char* what, cudaError_t e) {
  static const bool debug = getenv("CCONV_DEBUG") != nullptr;
  if (e != cudaSuccess && debug)
    fprintf(stderr, "cconv: %s failed: %s (%d)\n", what, cudaGetErrorString(e), static_cast<int>(e));
  return e;
}

static PFN_cuCtxGetCurrent_v4000 ctx_get_current_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  return fn;
}

// The driver call made here (cuTensorMapEncodeTiled) needs a context current on the
// calling thread.  A thread that has so far made only runtime calls that bind none
// (cudaGetDevice, cudaDeviceGetAttribute, stream-ordered allocator hits) has none:
// autograd's per-device worker thread, for example, can reach a backward call before any
// kernel launch of its own.  If no context is current, cudaSetDevice on the device already
// current binds that device's primary context (the runtime creates it there since CUDA
// 12) without changing which device is current; a context the caller made current itself,
// primary or not, is left alone.  Checked once per thread and device.
static int bind_current_context(int* device) {
  thread_local int checked = -1;
  int dev = 0;
  if (report_cuda("cudaGetDevice", cudaGetDevice(&dev)) != cudaSuccess) return CCONV_ERR_CUDA;
  if (checked != dev) {
    PFN_cuCtxGetCurrent_v4000 get = ctx_get_current_fn();
    CUcontext ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
      if (report_cuda("cudaSetDevice", cudaSetDevice(dev)) != cudaSuccess)
        return CCONV_ERR_CUDA;
    }
    checked = dev;
  }
  if (device) *device = dev;
  return CCONV_OK;
}

int sm_count_current_device(int* sms, int* device) {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (bind_current_context(&dev) != CCONV_OK) return CCONV_ERR_CUDA;
  if (device) *device = dev;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *sms = c;
      return CCONV_OK;
    }
  }
  int n = 0;
  if (report_cuda("cudaDeviceGetAttribute",
                  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) !=
          cudaSuccess ||
      n <= 0)
    return CCONV_ERR_CUDA;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  *sms = n;
  return CCONV_OK;
}

int smem_per_sm_current_device(int* per_sm, int* reserved_per_block) {
  static std::atomic<int> cache_sm[64], cache_res[64];
  int dev = 0;
  if (bind_current_context(&dev) != CCONV_OK) return CCONV_ERR_CUDA;
  if (dev >= 0 && dev < 64) {
    const int a = cache_sm[dev].load(std::memory_order_relaxed);
    const int b = cache_res[dev].load(std::memory_order_relaxed);
    if (a > 0 && b > 0) {
      *per_sm = a;
      *reserved_per_block = b - 1;
      return CCONV_OK;
    }
  }
  int a = 0, b = 0;
  if (report_cuda("cudaDeviceGetAttribute",
                  cudaDeviceGetAttribute(&a, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
          cudaSuccess ||
      report_cuda("cudaDeviceGetAttribute",
                  cudaDeviceGetAttribute(&b, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
          cudaSuccess ||
      a <= 0 || b < 0)
    return CCONV_ERR_CUDA;
  if (dev >= 0 && dev < 64) {
    cache_res[dev].store(b + 1, std::memory_order_relaxed);  // 0 marks "not cached"
    cache_sm[dev].store(a, std::memory_order_relaxed);
  }
  *per_sm = a;
  *reserved_per_block = b;
  return CCONV_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map of a [B, T, D] bf16 tensor (channel stride 1) read in boxes of
// box_c channels x box_r rows x 1 batch.  Zero fill outside the tensor.
int encode_rows_map(CUtensorMap* map, const void* base, int64_t B, int64_t T, int64_t D,
                    int64_t sb, int64_t st, int box_c, int box_r) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) {
    report_cuda("cuTensorMapEncodeTiled lookup", cudaErrorSymbolNotFound);
    return CCONV_ERR_CUDA;
  }
  if (bind_current_context(nullptr) != CCONV_OK) return CCONV_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)st * 2u, (cuuint64_t)sb * 2u};
  cuuint32_t box[3] = {(cuuint32_t)box_c, (cuuint32_t)box_r, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    static const bool debug = getenv("CCONV_DEBUG") != nullptr;
    if (debug) fprintf(stderr, "cconv: cuTensorMapEncodeTiled failed: CUresult %d\n", (int)r);
    return CCONV_ERR_CUDA;
  }
  return CCONV_OK;
}

// ------------------------------------------------------------------------------------
// launch recording: what each entry point would launch, with the kernels' attributes
// ------------------------------------------------------------------------------------
struct LaunchRecord {
  const void* func;
  dim3 grid, block;
  size_t smem;
};

static thread_local bool t_recording = false;
static thread_local std::vector<LaunchRecord> t_records;

bool recording_launches() { return t_recording; }

void record_launch(const void* func, dim3 grid, dim3 block, size_t smem) {
  t_records.push_back(LaunchRecord{func, grid, block, smem});
}

static void copy_name(char* dst, size_t n, const char* src) {
  size_t k = 0;
  for (; src && src[k] && k + 1 < n; ++k) dst[k] = src[k];
  dst[k] = 0;
}

int set_max_dynamic_smem(const void* func, int bytes) {
  // Per device and cheap; repeated on every launch rather than cached.
  return report_cuda("cudaFuncSetAttribute",
                     cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          bytes)) == cudaSuccess
             ? CCONV_OK
             : CCONV_ERR_CUDA;
}

}  // namespace cconv

extern "C" {

CCONV_API const char* cconv_status_str(int status) {
  switch (status) {
    case CCONV_OK: return "CCONV_OK";
    case CCONV_ERR_NULL: return "CCONV_ERR_NULL: a required pointer is NULL";
    case CCONV_ERR_SHAPE: return "CCONV_ERR_SHAPE: a size is out of range";
    case CCONV_ERR_WIDTH: return "CCONV_ERR_WIDTH: W must be in [1, 4]";
    case CCONV_ERR_ALIGN: return "CCONV_ERR_ALIGN: pointer, row stride or D breaks the 16-byte rule";
    case CCONV_ERR_STRIDE: return "CCONV_ERR_STRIDE: a stride is not positive (or ldx < D)";
    case CCONV_ERR_DTYPE: return "CCONV_ERR_DTYPE: unknown weight dtype";
    case CCONV_ERR_WORKSPACE: return "CCONV_ERR_WORKSPACE: workspace missing or too small";
    case CCONV_ERR_INDEX: return "CCONV_ERR_INDEX: state_indices invalid";
    case CCONV_ERR_CUDA: return "CCONV_ERR_CUDA: a CUDA call failed";
    case CCONV_ERR_DEVICE: return "CCONV_ERR_DEVICE: a kernel gave up a bounded wait";
    default: return "unknown cconv status";
  }
}

CCONV_API int cconv_describe_begin(void) {
  cconv::t_records.clear();
  cconv::t_recording = true;
  return CCONV_OK;
}

CCONV_API int cconv_describe_end(cconv_kernel_desc* out, int max, int* count) {
  using namespace cconv;
  t_recording = false;
  if (!count || (max > 0 && !out)) return CCONV_ERR_NULL;
  *count = static_cast<int>(t_records.size());
  int rc = CCONV_OK;
  for (int i = 0; i < max && i < static_cast<int>(t_records.size()); ++i) {
    const LaunchRecord& r = t_records[i];
    cconv_kernel_desc& d = out[i];
    memset(&d, 0, sizeof(d));
    cudaFuncAttributes fa{};
    if (report_cuda("cudaFuncGetAttributes", cudaFuncGetAttributes(&fa, r.func)) != cudaSuccess) {
      rc = CCONV_ERR_CUDA;
      continue;
    }
    const int threads = static_cast<int>(r.block.x * r.block.y * r.block.z);
    int per_sm = 0;
    if (report_cuda("cudaOccupancyMaxActiveBlocksPerMultiprocessor",
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, r.func, threads,
                                                                  r.smem)) != cudaSuccess)
      rc = CCONV_ERR_CUDA;
    const char* mangled = nullptr;
    if (cudaFuncGetName(&mangled, r.func) == cudaSuccess && mangled) {
      int st = 0;
      char* dem = abi::__cxa_demangle(mangled, nullptr, nullptr, &st);
      copy_name(d.name, sizeof(d.name), st == 0 && dem ? dem : mangled);
      free(dem);
    }
    d.registers = fa.numRegs;
    d.local_bytes = static_cast<int>(fa.localSizeBytes);
    d.static_shared_bytes = static_cast<int>(fa.sharedSizeBytes);
    d.dynamic_shared_bytes = static_cast<int>(r.smem);
    d.threads = threads;
    d.ctas_per_sm = per_sm;
    d.ctas = static_cast<int64_t>(r.grid.x) * r.grid.y * r.grid.z;
  }
  t_records.clear();
  return rc;
}

CCONV_API int cconv_device_fault(int32_t* fault) {
  if (!fault) return CCONV_ERR_NULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return CCONV_ERR_CUDA;
  unsigned a = 0, b = 0;
  int rc = cconv::read_clear_fault_fwd(&a);
  if (rc != CCONV_OK) return rc;
  rc = cconv::read_clear_fault_bwd(&b);
  if (rc != CCONV_OK) return rc;
  *fault = static_cast<int32_t>(a | b);
  return CCONV_OK;
}

}  // extern "C"
