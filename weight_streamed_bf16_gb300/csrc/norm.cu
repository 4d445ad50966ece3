// norm.cu -- full-row RMS normalisation (PSI section II-B): every width
// tile of a row is scaled by the one denominator sqrt(s/d + eps) formed
// from the global sum of squares s.
//
// HBM-bound: one read of X and one BF16 write of Y.  Rows of up to 4096
// elements: 12 to 16 warps per SM (chosen per launch from the row count)
// each normalise whole rows from registers (16 vectors of 16 bytes per
// lane), so that many rows are in flight per SM; gamma is staged in shared
// memory once per CTA.  Wider rows: a persistent CTA per SM
// stages whole rows in shared memory with untiled bulk copies (one producer
// thread keeps a ring of up to 24 rows in flight), consumer warps normalise
// a row in place, and a bulk store writes it back.  (The bulk-copy form is
// slower for the narrower rows: its producer issues one 8 KB copy about
// every 0.27 us per SM.)
//
// Sum of squares: each lane adds the squares of its lane-strided 8-element
// vectors (the width partitions), then a butterfly over the 32 lanes
// combines them: one fixed order, one denominator per row.
#include <algorithm>
#include <utility>
#include "internal.h"
#include "ptx.cuh"

namespace psi {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kNormThreads = 32 * (1 + kConsumerWarps);
constexpr int kStageBudget = 200 * 1024;  // shared bytes for gamma and the row ring
constexpr int kMaxStages = 24;

__device__ __forceinline__ void norm_error(DevError* e, int role, int i0, int i1) {
  if (atomicCAS(&e->code, 0, 1) == 0) {
    e->where = KID_NORM * 16 + role;
    e->info0 = i0;
    e->info1 = i1;
  }
}

struct NormArgs {
  const uint16_t* X;
  int64_t ldx;
  uint16_t* Y;
  int64_t ldy;
  const uint16_t* gamma;
  int N;
  int d;
  int stages;
  float eps;
  DevError* err;
  uint64_t timeout_ns;
};

__global__ void __launch_bounds__(kNormThreads, 1) rmsnorm_kernel(NormArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], gbar;
  __shared__ int abort_flag;
  __shared__ int n_issued;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rb = static_cast<uint32_t>(a.d) * 2;          // row bytes
  const uint32_t stage_bytes = (rb + 127) & ~127u;
  uint8_t* sg = smem;                                          // gamma
  uint8_t* ring = smem + stage_bytes;
  const int S = a.stages;
  const int nrows = a.N > static_cast<int>(blockIdx.x)
                        ? (a.N - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1
                        : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&gbar, 1);
    abort_flag = 0;
    n_issued = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------- producer --
    if (lane == 0) {
      mbar_arrive_expect_tx(&gbar, rb);
      bulk_load(sg, a.gamma, rb, &gbar);
      for (int k = 0; k < nrows; ++k) {
        const int s = k % S;
        if (k >= S && !mbar_wait(&empty[s], ((k / S) - 1) & 1, &abort_flag, a.timeout_ns)) {
          norm_error(a.err, 0, k, s);
          abort_flag = 1;
          break;
        }
        const int row = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
        mbar_arrive_expect_tx(&full[s], rb);
        bulk_load(ring + static_cast<size_t>(s) * stage_bytes,
                  a.X + static_cast<int64_t>(row) * a.ldx, rb, &full[s]);
        n_issued = k + 1;
      }
    }
  } else {
    // ------------------------------------------------------ consumers --
    const int c = warp - 1;
    const int nv = a.d >> 3;  // 16-byte vectors per row
    const float inv_d = 1.0f / static_cast<float>(a.d);
    bool ok = mbar_wait(&gbar, 0, &abort_flag, a.timeout_ns);
    if (!ok && lane == 0) norm_error(a.err, 1, -1, c);
    const uint4* g4 = reinterpret_cast<const uint4*>(sg);
    int prev_s = -1;
    for (int k = c; ok && k < nrows; k += kConsumerWarps) {
      const int s = k % S;
      if (!mbar_wait(&full[s], (k / S) & 1, &abort_flag, a.timeout_ns)) {
        if (lane == 0) norm_error(a.err, 2, k, s);
        abort_flag = 1;
        break;
      }
      uint4* r4 = reinterpret_cast<uint4*>(ring + static_cast<size_t>(s) * stage_bytes);
      float ss = 0.f;
#pragma unroll 4
      for (int idx = lane; idx < nv; idx += 32) {
        const uint4 x = r4[idx];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float lo = bf16_lo(w[t]), hi = bf16_hi(w[t]);
          ss = fmaf(lo, lo, ss);
          ss = fmaf(hi, hi, ss);
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float r = 1.0f / sqrtf(ss * inv_d + a.eps);
#pragma unroll 4
      for (int idx = lane; idx < nv; idx += 32) {
        const uint4 x = r4[idx];
        const uint4 g = g4[idx];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
        uint32_t o[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          o[t] = pack_bf16x2(bf16_lo(gw[t]) * (bf16_lo(w[t]) * r),
                             bf16_hi(gw[t]) * (bf16_hi(w[t]) * r));
        r4[idx] = make_uint4(o[0], o[1], o[2], o[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int row = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
        bulk_store(a.Y + static_cast<int64_t>(row) * a.ldy, r4, rb);
        bulk_commit();
        // the previous row's store has read its stage: hand that stage back
        if (prev_s >= 0) {
          bulk_wait_read<1>();
          mbar_arrive(&empty[prev_s]);
        }
      }
      prev_s = s;
      __syncwarp();
    }
    if (lane == 0) bulk_wait<0>();  // this warp's stores are complete
  }
  __syncthreads();
  // every load the producer issued has landed before the CTA's shared
  // memory is released (normally the consumers already waited for them)
  if (threadIdx.x == 0) {
    const int issued = n_issued;
    for (int s = 0; s < S && s < issued; ++s) {
      const int last_k = s + ((issued - 1 - s) / S) * S;
      int none = 0;
      if (!mbar_wait(&full[s], (last_k / S) & 1, &none, a.timeout_ns))
        norm_error(a.err, 3, last_k, s);
    }
  }
}


// Rows of up to 4096 elements, whole rows per warp from registers; W warps
// per CTA, one CTA per SM (the launch picks W so that the rows fill the
// warps' last round as fully as possible).
template <int W>
__global__ void __launch_bounds__(32 * W, 1) rmsnorm_reg_kernel(NormArgs a) {
  constexpr int kRegWarps = W;
  __shared__ __align__(16) uint4 g4s[512];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = a.d >> 3;
  for (int i = threadIdx.x; i < nv; i += blockDim.x)
    g4s[i] = reinterpret_cast<const uint4*>(a.gamma)[i];
  __syncthreads();
  const float inv_d = 1.0f / static_cast<float>(a.d);
  const int nw = gridDim.x * kRegWarps;
  for (int row = blockIdx.x * kRegWarps + warp; row < a.N; row += nw) {
    const uint4* x4 = reinterpret_cast<const uint4*>(a.X + static_cast<int64_t>(row) * a.ldx);
    uint4* y4 = reinterpret_cast<uint4*>(a.Y + static_cast<int64_t>(row) * a.ldy);
    uint4 xr[16];
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      const int idx = lane + 32 * v;
      xr[v] = idx < nv ? __ldcs(x4 + idx) : make_uint4(0, 0, 0, 0);
    }
    float ss = 0.f;
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      const uint32_t w[4] = {xr[v].x, xr[v].y, xr[v].z, xr[v].w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float lo = bf16_lo(w[t]), hi = bf16_hi(w[t]);
        ss = fmaf(lo, lo, ss);
        ss = fmaf(hi, hi, ss);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float r = 1.0f / sqrtf(ss * inv_d + a.eps);
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      const int idx = lane + 32 * v;
      if (idx < nv) {
        const uint4 g = g4s[idx];
        const uint32_t w[4] = {xr[v].x, xr[v].y, xr[v].z, xr[v].w};
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
        uint32_t o[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          o[t] = pack_bf16x2(bf16_lo(gw[t]) * (bf16_lo(w[t]) * r),
                             bf16_hi(gw[t]) * (bf16_hi(w[t]) * r));
        y4[idx] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

constexpr int kMinRegWarps = 12;
constexpr int kMaxRegWarps = 16;
using RegKernel = void (*)(NormArgs);
template <int... Ws>
const RegKernel* reg_kernel_table(std::integer_sequence<int, Ws...>) {
  static const RegKernel table[] = {&rmsnorm_reg_kernel<kMinRegWarps + Ws>...};
  return table;
}
const RegKernel* reg_kernels() {
  return reg_kernel_table(std::make_integer_sequence<int, kMaxRegWarps - kMinRegWarps + 1>{});
}

}  // namespace

psi_status launch_rmsnorm(const void* X, int64_t ldx, int64_t N, int64_t d, const void* gamma,
                          float eps, void* Y, int64_t ldy, cudaStream_t stream) {
  NormArgs a{};
  a.X = static_cast<const uint16_t*>(X);
  a.ldx = ldx;
  a.Y = static_cast<uint16_t*>(Y);
  a.ldy = ldy;
  a.gamma = static_cast<const uint16_t*>(gamma);
  a.N = static_cast<int>(N);
  a.d = static_cast<int>(d);
  a.eps = eps;
  a.err = dev_error_ptr();
  if (!a.err) return set_error(PSI_ERR_CUDA, "rmsnorm: kernel error record not reachable");
  a.timeout_ns = kWaitLimitNs;
  const int stage_bytes = static_cast<int>((d * 2 + 127) / 128 * 128);
  a.stages = std::min(kMaxStages, (kStageBudget - stage_bytes) / stage_bytes);
  if (a.stages <= kConsumerWarps)
    return set_error(PSI_ERR_UNSUPPORTED, "rmsnorm: row too wide for the shared-memory ring");
  const int smem = stage_bytes * (1 + a.stages);
  static std::atomic<uint64_t> attr_done{0};
  psi_status st = ensure_smem_attr(&attr_done, reinterpret_cast<const void*>(rmsnorm_kernel),
                                   kStageBudget, "rmsnorm: shared-memory attribute");
  if (st != PSI_OK) return st;
  const int grid = static_cast<int>(std::min<int64_t>(N, num_sms()));
  if (d <= 4096) {
    // warps per CTA: each warp takes whole rows in rounds of sms * W rows;
    // choose W in [kMinRegWarps, kMaxRegWarps] with the fewest idle warp
    // slots in the last round (ties: fewer warps)
    const int64_t sms = num_sms();
    int best_w = kMinRegWarps;
    int64_t best_idle = -1;
    for (int w = kMinRegWarps; w <= kMaxRegWarps; ++w) {
      const int64_t slots = sms * w;
      const int64_t idle = (N + slots - 1) / slots * slots - N;
      if (best_idle < 0 || idle < best_idle) {
        best_idle = idle;
        best_w = w;
      }
    }
    const int g2 = static_cast<int>(std::min<int64_t>((N + best_w - 1) / best_w, sms));
    reg_kernels()[best_w - kMinRegWarps]<<<g2, 32 * best_w, 0, stream>>>(a);
  } else {
    rmsnorm_kernel<<<grid, kNormThreads, smem, stream>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "rmsnorm launch");
  count_launch();
  return PSI_OK;
}

}  // namespace psi
