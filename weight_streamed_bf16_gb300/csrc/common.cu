// common.cu -- error reporting, the device error record, tensor-map
// encoding and device queries shared by the kernels and the runtime.
#include <atomic>
#include <cstdio>
#include <mutex>
#include <string>
#include <cudaTypedefs.h>
#include "internal.h"

namespace psi {

// Kernel-side error record (see DevError).  A module-scope device variable:
// it is part of the library's loaded image, not a device allocation.
__device__ DevError g_dev_error;

namespace {
thread_local std::string t_last_error;

constexpr int kMaxDevices = 64;
DevError* g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_status = cudaSuccess;

int g_sms[kMaxDevices] = {};
}  // namespace

psi_status set_error(psi_status s, const std::string& msg) {
  t_last_error = msg;
  return s;
}

psi_status cuda_error(cudaError_t e, const char* what) {
  return set_error(PSI_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                                     cudaGetErrorString(e) + ")");
}

const char* last_error_cstr() { return t_last_error.c_str(); }

psi_status check_flags(uint32_t flags, uint32_t allowed, const char* what) {
  const uint32_t bad = flags & ~allowed;
  if (!bad) return PSI_OK;
  char buf[160];
  snprintf(buf, sizeof buf, "%s: flag bits 0x%x are not honoured by this entry point", what,
           static_cast<unsigned>(bad));
  return set_error(PSI_ERR_UNSUPPORTED, buf);
}

DevError* dev_error_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<DevError*>(p);
  }
  return g_err_ptr[dev];
}

cudaError_t dev_error_take(DevError* out) {
  DevError zero = {0, 0, 0, 0};
  cudaError_t e = cudaMemcpyFromSymbol(out, g_dev_error, sizeof(DevError));
  if (e != cudaSuccess) return e;
  if (out->code != 0) e = cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(DevError));
  return e;
}

// kernels launched by the library in this process (all entry points)
static std::atomic<uint64_t> g_kernel_launches{0};
void count_launch() { g_kernel_launches.fetch_add(1, std::memory_order_relaxed); }

int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  if (g_sms[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return g_sms[dev];
}

psi_status ensure_smem_attr(std::atomic<uint64_t>* done, const void* fn, int bytes,
                            const char* what) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, what);
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(PSI_ERR_UNSUPPORTED, std::string(what) + ": device index above 63");
  const uint64_t bit = 1ull << dev;
  if (done->load(std::memory_order_acquire) & bit) return PSI_OK;
  // setting the attribute twice (two threads racing here) is harmless
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return cuda_error(e, what);
  done->fetch_or(bit, std::memory_order_release);
  return PSI_OK;
}

static psi_status get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    g_encode_status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                       cudaEnableDefault, &q);
    if (g_encode_status == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) {
    return set_error(PSI_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  }
  return PSI_OK;
}

psi_status make_tmap_2d_ex(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                           uint64_t ld, uint32_t box_rows, uint32_t box_cols, int elem_bytes,
                           int swizzle_bytes) {
  psi_status st = get_encoder();
  if (st != PSI_OK) return st;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || ((ld * elem_bytes) & 15))
    return set_error(PSI_ERR_INVALID_ARG, "tensor map: base or row stride not 16-byte aligned");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled(2d) failed: %d (rows %llu cols %llu)",
             static_cast<int>(r), static_cast<unsigned long long>(rows),
             static_cast<unsigned long long>(cols));
    return set_error(PSI_ERR_CUDA, buf);
  }
  return PSI_OK;
}

psi_status make_tmap_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                        uint64_t ld, uint32_t box_rows, uint32_t box_cols) {
  return make_tmap_2d_ex(m, base, rows, cols, ld, box_rows, box_cols, 2, 128);
}

}  // namespace psi

extern "C" uint64_t psi_kernel_launches(void) {
  return psi::g_kernel_launches.load(std::memory_order_relaxed);
}
