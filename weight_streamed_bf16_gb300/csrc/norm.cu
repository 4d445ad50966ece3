// norm.cu -- full-row RMS normalisation (PSI section II-B): every width
// tile of a row is scaled by the one denominator sqrt(s/d + eps) formed
// from the global sum of squares s.  HBM-bound: one read of X and one BF16
// write of Y; gamma stays in L1/L2.
//
// One warp per row.  The row lives in registers (NV 16-byte vectors per
// lane, lane-strided so each warp load instruction covers 512 contiguous
// bytes); each lane's partial sum over its vectors and a butterfly over the
// lanes give s, i.e. the sum is taken over width partitions (one per lane)
// and combined once, in a fixed order.
#include "internal.h"
#include "ptx.cuh"

namespace psi {
namespace {

constexpr int kNormWarps = 8;

template <int NV>
__global__ void __launch_bounds__(kNormWarps * 32)
    rmsnorm_kernel(const uint16_t* __restrict__ X, int64_t ldx, int N, int d,
                   const uint16_t* __restrict__ gamma, float eps, uint16_t* __restrict__ Y,
                   int64_t ldy) {
  // rows up to 4096 wide stay in registers between the two passes; wider
  // rows are read twice (the second read hits L2)
  constexpr bool kKeep = NV <= 16;
  const int lane = threadIdx.x & 31;
  const int nv = d >> 3;  // 16-byte vectors per row
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  for (int row = blockIdx.x * kNormWarps + (threadIdx.x >> 5); row < N;
       row += gridDim.x * kNormWarps) {
    const uint4* x4 = reinterpret_cast<const uint4*>(X + static_cast<int64_t>(row) * ldx);
    uint4 v[kKeep ? NV : 1];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = i * 32 + lane;
      uint4 x = make_uint4(0, 0, 0, 0);
      if (idx < nv) x = kKeep ? __ldcs(x4 + idx) : __ldg(x4 + idx);
      if constexpr (kKeep) v[i] = x;
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float a = bf16_lo(w[t]), b = bf16_hi(w[t]);
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float r = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
    uint4* y4 = reinterpret_cast<uint4*>(Y + static_cast<int64_t>(row) * ldy);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = i * 32 + lane;
      if (idx < nv) {
        uint4 x;
        if constexpr (kKeep) x = v[i];
        else x = __ldcs(x4 + idx);
        const uint4 g = __ldg(g4 + idx);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
        uint32_t o[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          o[t] = pack_bf16x2(bf16_lo(gw[t]) * (bf16_lo(w[t]) * r),
                             bf16_hi(gw[t]) * (bf16_hi(w[t]) * r));
        __stcs(y4 + idx, make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
  }
}

template <int NV>
psi_status launch_nv(const uint16_t* X, int64_t ldx, int N, int d, const uint16_t* gamma,
                     float eps, uint16_t* Y, int64_t ldy, cudaStream_t s) {
  const int blocks_needed = (N + kNormWarps - 1) / kNormWarps;
  const int grid = std::min(blocks_needed, num_sms() * 8);
  rmsnorm_kernel<NV><<<grid, kNormWarps * 32, 0, s>>>(X, ldx, N, d, gamma, eps, Y, ldy);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "rmsnorm launch");
  return PSI_OK;
}

}  // namespace

psi_status launch_rmsnorm(const void* X, int64_t ldx, int64_t N, int64_t d, const void* gamma,
                          float eps, void* Y, int64_t ldy, cudaStream_t stream) {
  const auto* x = static_cast<const uint16_t*>(X);
  const auto* g = static_cast<const uint16_t*>(gamma);
  auto* y = static_cast<uint16_t*>(Y);
  const int n = static_cast<int>(N), dd = static_cast<int>(d);
  const int per_lane = (static_cast<int>(d / 8) + 31) / 32;  // vectors per lane
  if (per_lane <= 1) return launch_nv<1>(x, ldx, n, dd, g, eps, y, ldy, stream);
  if (per_lane <= 2) return launch_nv<2>(x, ldx, n, dd, g, eps, y, ldy, stream);
  if (per_lane <= 4) return launch_nv<4>(x, ldx, n, dd, g, eps, y, ldy, stream);
  if (per_lane <= 8) return launch_nv<8>(x, ldx, n, dd, g, eps, y, ldy, stream);
  if (per_lane <= 16) return launch_nv<16>(x, ldx, n, dd, g, eps, y, ldy, stream);
  return launch_nv<32>(x, ldx, n, dd, g, eps, y, ldy, stream);
}

}  // namespace psi
