// noalloc.cu -- a paged-FFN entry point that allocates nothing.
//
// Some callers cannot call cudaMalloc at all: code that runs inside another
// framework's memory pool or a fixed memory budget handed out at start-up,
// plug-ins that get device pointers but no allocator, and processes whose
// device memory is carved up before this library is loaded.  For them
// psi_ffn_resident_noalloc runs the FFN with its two workspaces (the BF16
// hidden slices of one group and the FP32 accumulator) in a fixed array
// that is part of this library's device image, so the only memory it
// touches is the caller's inputs and outputs and that array.
#include <mutex>
#include <string>
#include "internal.h"

// The workspace array: every GPU that loads the library holds these bytes
// until the process exits.  All calls share it.
constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_ffn_scratch[kNoAllocScratchBytes];

namespace psi {
namespace {

constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of g_ffn_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
psi_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "ffn_resident_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDev)
    return set_error(PSI_ERR_UNSUPPORTED, "ffn_resident_noalloc: device index out of range");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_ffn_scratch);
    if (e != cudaSuccess) return cuda_error(e, "ffn_resident_noalloc: cudaGetSymbolAddress");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PSI_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace psi

using namespace psi;

extern "C" psi_status psi_ffn_resident_noalloc(const void* X, int64_t N, const psi_ffn_weight* W,
                                               const void* av, const void* bv,
                                               const void* residual, void* Y, void* stream,
                                               uint32_t flags) {
  psi_status fs = check_flags(flags, kFlagsFfnNoAlloc, "ffn_resident_noalloc");
  if (fs != PSI_OK) return fs;
  if (!X || !W || !W->dev_resident || !av || !bv || !Y)
    return set_error(PSI_ERR_INVALID_ARG, "ffn_resident_noalloc: null argument");
  const int64_t d = W->d, h = W->h, r = W->r, sl = W->slice;
  if (N < 0 || d <= 0 || h <= 0 || r <= 0 || sl <= 0 || h % sl)
    return set_error(PSI_ERR_INVALID_ARG,
                     "ffn_resident_noalloc: bad shape (h must be a multiple of slice)");
  if (d % 8 || r % 8 || sl % 16)
    return set_error(PSI_ERR_INVALID_ARG,
                     "ffn_resident_noalloc: d, r must be multiples of 8, slice of 16");
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!al16(X) || !al16(Y) || !al16(av) || !al16(bv) || !al16(W->dev_resident) ||
      (residual && !al16(residual)))
    return set_error(PSI_ERR_INVALID_ARG, "ffn_resident_noalloc: pointers must be 16-byte aligned");
  if (N > 0x7FFFFFFF || d > 0x7FFFFFFF || h > 0x7FFFFFFF || r > 0x7FFFFFFF)
    return set_error(PSI_ERR_UNSUPPORTED, "ffn_resident_noalloc: dimension above 2^31");
  if (N == 0) return PSI_OK;
  // the slice grouping of psi_ffn_paged (the same function), so both sum the
  // down projections in the same order and give the same bytes
  const int64_t S = h / sl;
  const int64_t G = ffn_group(S, sl);
  const size_t hid_bytes = round256(static_cast<size_t>(N) * G * sl * 2);
  const size_t acc_bytes = static_cast<size_t>(N) * r * 4;
  if (hid_bytes + acc_bytes > kNoAllocScratchBytes)
    return set_error(PSI_ERR_CAPACITY,
                     "ffn_resident_noalloc: needs " + std::to_string(hid_bytes + acc_bytes) +
                         " bytes of workspace (N*G*slice*2 rounded up to 256, plus N*r*4), "
                         "the fixed array holds " +
                         std::to_string(kNoAllocScratchBytes));
  void* base = nullptr;
  psi_status st = scratch_address(&base);
  if (st != PSI_OK) return st;
  DevError* err = dev_error_ptr();
  if (!err) return set_error(PSI_ERR_CUDA, "ffn_resident_noalloc: kernel error record not reachable");
  uint16_t* Hg = static_cast<uint16_t*>(base);
  float* acc = reinterpret_cast<float*>(static_cast<char*>(base) + hid_bytes);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const char* src = static_cast<const char*>(W->dev_resident);
  const size_t pb = psi_ffn_page_bytes(d, r, sl);
  const uint16_t* a16 = static_cast<const uint16_t*>(av);
  const int32_t bias_after = (flags & PSI_BIAS_AFTER_BF16) ? 1 : 0;
  for (int64_t J0 = 0; J0 < S; J0 += G) {
    const int64_t gs = (S - J0) < G ? (S - J0) : G;
    // one up-projection launch per slice (psi_ffn_paged merges a group's two
    // slices into one launch when slice % 256 == 0); the per-element
    // arithmetic of the epilogue is the same either way
    for (int64_t u = 0; u < gs; ++u) {
      const int64_t J = J0 + u;
      GemmArgs up{};
      up.M = static_cast<int32_t>(N);
      up.N = static_cast<int32_t>(sl);
      up.K = static_cast<int32_t>(d);
      up.epi = EPI_GELU;
      up.pregelu = (flags & PSI_BOUNDARY_PREGELU_BF16) ? 1 : 0;
      up.bias_after_bf16 = bias_after;
      up.bias = a16 + J * sl;
      up.out = Hg + u * sl;
      up.ldo = G * sl;
      up.err = err;
      up.timeout_ns = kWaitLimitNs;
      st = launch_page_gemm(X, d, src + static_cast<size_t>(J) * pb, d, up, cs);
      if (st != PSI_OK) return st;
    }
    // the accumulator is written by the first group before it is read, so
    // the array needs no clearing between calls
    GemmArgs dn{};
    dn.M = static_cast<int32_t>(N);
    dn.N = static_cast<int32_t>(r);
    dn.K = static_cast<int32_t>(gs * sl);
    dn.k_split = gs > 1 ? static_cast<int32_t>(sl / 64) : 0;
    dn.accf = acc;
    dn.ldacc = r;
    dn.err = err;
    dn.timeout_ns = kWaitLimitNs;
    dn.bias_after_bf16 = bias_after;
    const bool first = J0 == 0, last = J0 + gs >= S;
    if (last) {
      dn.epi = first ? EPI_LINEAR : EPI_ACC_FINAL;
      dn.bias = static_cast<const uint16_t*>(bv);
      dn.resid = static_cast<const uint16_t*>(residual);
      dn.out = static_cast<uint16_t*>(Y);
      dn.ldo = r;
    } else {
      dn.epi = first ? EPI_ACC_STORE : EPI_ACC_ADD;
    }
    const size_t voff = static_cast<size_t>(sl) * d * 2;
    const char* p0 = src + static_cast<size_t>(J0) * pb + voff;
    const char* p1 = gs > 1 ? src + static_cast<size_t>(J0 + 1) * pb + voff : nullptr;
    st = launch_page_gemm(Hg, G * sl, p0, sl, dn, cs, p1);
    if (st != PSI_OK) return st;
  }
  return PSI_OK;
}
