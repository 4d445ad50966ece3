// gemm_epilogue.cuh -- device helpers shared by the page GEMM kernels: the
// fused epilogue (bias, GELU, FP32 accumulator, residual, BF16 cast) and the
// staging of results for TMA tensor stores.
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace psi {
namespace {

constexpr int BM = 128;   // accumulator rows per CTA (TMEM lanes)
constexpr int BK = 64;    // one 128-byte swizzle row of BF16
constexpr int kEpiWarps = 8;

__device__ __forceinline__ void record_error(DevError* e, int code, int where, int i0, int i1) {
  if (atomicCAS(&e->code, 0, code) == 0) {
    e->where = where;
    e->info0 = i0;
    e->info1 = i1;
  }
}

__device__ __forceinline__ float gelu_tanh(float x) {
  // tanh form of GELU: x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
  const float k0 = 0.7978845608028654f;
  const float k1 = 0.044715f;
  const float u = k0 * fmaf(k1 * x * x, x, x);
  return 0.5f * x * (1.0f + tanhf(u));
}

__device__ __forceinline__ float round_bf16_f(float x) {
  return bf16_lo(pack_bf16x2(x, 0.f));
}

__device__ __forceinline__ bool epi_reads_acc(int epi) {
  return epi == EPI_ACC_ADD || epi == EPI_ACC_FINAL;
}
__device__ __forceinline__ bool epi_writes_f32(int epi) {
  return epi == EPI_ACC_STORE || epi == EPI_ACC_ADD;
}

// The 32 FP32 accumulator values of one row chunk (full chunks only).
__device__ __forceinline__ void load_acc32(const GemmArgs& a, int row, int col0,
                                           float4 (&q)[8]) {
  const float4* p4 =
      reinterpret_cast<const float4*>(a.accf + static_cast<int64_t>(row) * a.ldacc + col0);
#pragma unroll
  for (int j = 0; j < 8; ++j) q[j] = p4[j];
}

// Fused epilogue of 32 consecutive columns of one row.  v[] holds the FP32
// MMA results; col0 is the first column, ncol <= 32 of them exist, row_ok
// says whether the row exists (inputs of missing rows/columns are not read;
// their outputs are clipped by the tensor store).  wq[] holds the FP32
// workspace values of a full chunk, loaded ahead.  The results go to the
// warp's staging buffer `stg` (row = lane) in the layout of the tensor
// store (BF16 rows of 64 B with 64-byte swizzle); FP32 results are left in
// v[] for the caller.
__device__ __forceinline__ void epilogue_row32(const GemmArgs& a, int row, bool row_ok,
                                               int col0, int ncol, float (&v)[32],
                                               const float4 (&wq)[8], uint8_t* stg, int lane) {
  const bool full = (ncol == 32) && row_ok;
  if (epi_writes_f32(a.epi)) {
    if (a.epi == EPI_ACC_ADD) {
      if (full) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[4 * j] = wq[j].x + v[4 * j];
          v[4 * j + 1] = wq[j].y + v[4 * j + 1];
          v[4 * j + 2] = wq[j].z + v[4 * j + 2];
          v[4 * j + 3] = wq[j].w + v[4 * j + 3];
        }
      } else if (row_ok) {
        const float* p = a.accf + static_cast<int64_t>(row) * a.ldacc + col0;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < ncol) v[j] = p[j] + v[j];
      }
    }
    return;  // FP32 results stay in v; the caller stages them per 16 columns
  }
  // BF16 outputs: bias (+ FP32 accumulator) (+ GELU) (+ residual)
  float bia[32];
  if (col0 + 32 <= a.N) {
    const uint4* b4 = reinterpret_cast<const uint4*>(a.bias + col0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 q = __ldg(b4 + j);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        bia[8 * j + 2 * t] = bf16_lo(w[t]);
        bia[8 * j + 2 * t + 1] = bf16_hi(w[t]);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      bia[j] = j < ncol ? __uint_as_float(static_cast<uint32_t>(a.bias[col0 + j]) << 16) : 0.f;
  }
  if (a.epi == EPI_ACC_FINAL) {
    if (full) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[4 * j] = wq[j].x + v[4 * j];
        v[4 * j + 1] = wq[j].y + v[4 * j + 1];
        v[4 * j + 2] = wq[j].z + v[4 * j + 2];
        v[4 * j + 3] = wq[j].w + v[4 * j + 3];
      }
    } else if (row_ok) {
      const float* p = a.accf + static_cast<int64_t>(row) * a.ldacc + col0;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < ncol) v[j] = p[j] + v[j];
    }
  }
  if (a.bias_after_bf16) {  // the baseline variant: product rounded before the bias
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = round_bf16_f(v[j]);
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = v[j] + bia[j];
  if (a.epi == EPI_GELU) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float t = v[j];
      if (a.pregelu) t = round_bf16_f(t);
      v[j] = gelu_tanh(t);
    }
  }
  if (a.resid && row_ok) {
    const uint16_t* res = a.resid + static_cast<int64_t>(row) * a.ldo + col0;
    if (ncol == 32) {
      const uint4* r4 = reinterpret_cast<const uint4*>(res);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 q = r4[j];
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          v[8 * j + 2 * t] += bf16_lo(w[t]);
          v[8 * j + 2 * t + 1] += bf16_hi(w[t]);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < ncol) v[j] += __uint_as_float(static_cast<uint32_t>(res[j]) << 16);
    }
  }
  uint8_t* rowp = stg + lane * 64;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(rowp + ((c ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(pack_bf16x2(v[8 * c + 0], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                   pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
}

// The chunks of one tile owned by one epilogue warp: TMEM columns of its
// column half, fused epilogue, staged tensor stores.  `nxt` holds the FP32
// workspace values of the first chunk when `pre` (loaded by the caller
// before it waited for the accumulator).
template <int BN>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& args, const CUtensorMap* tmOut,
                                              uint32_t tbase, int m0, int n0, int q, int row,
                                              bool row_ok, int lane, bool pre, bool f32,
                                              uint8_t* stg_base, int& nstore, float4 (&nxt)[8]) {
  constexpr int CH = BN / 64;  // 32-column chunks per half
#pragma unroll 1
  for (int c = 0; c < CH; ++c) {
    float4 cur[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
    const int col0 = n0 + c * 32;
    if (pre && c + 1 < CH && row_ok && col0 + 64 <= args.N)
      load_acc32(args, row, col0 + 32, nxt);
    __syncwarp();
    uint32_t r[32];
    tmem_ld_32x32b_x32(tbase + c * 32, r);
    tmem_wait_ld();
    if (col0 < args.N && m0 + q * 32 < args.M) {  // warp-uniform
      // The warp's 4 KiB holds two 2 KiB buffers used alternately: a BF16
      // chunk (32 rows x 64 B) or an FP32 half chunk (32 rows x 16
      // columns x 4 B) per buffer, so one tensor store drains while the
      // next buffer is written.
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
      const int ncol = min(32, args.N - col0);
      const int nparts = f32 ? 2 : 1;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        if (part >= nparts) break;
        uint8_t* stg = stg_base + (nstore & 1) * 2048;
        if (lane == 0) bulk_wait_read<1>();  // this buffer's last store has read it
        __syncwarp();
        if (!f32) {
          epilogue_row32(args, row, row_ok, col0, ncol, v, cur, stg, lane);
        } else {
          if (part == 0) epilogue_row32(args, row, row_ok, col0, ncol, v, cur, stg, lane);
          uint8_t* rowp = stg + lane * 64;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int b = 16 * part + 4 * k4;
            *reinterpret_cast<float4*>(rowp + ((k4 ^ ((lane >> 1) & 3)) << 4)) =
                make_float4(v[b], v[b + 1], v[b + 2], v[b + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (col0 + 16 * part < args.N)
            tma_store_2d(tmOut, stg, col0 + 16 * part, m0 + q * 32);
          bulk_commit();
        }
        ++nstore;
      }
    }
  }
}

}  // namespace
}  // namespace psi
