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
  // tanh form of GELU: x/2 (1 + tanh(u)), u = sqrt(2/pi) (x + 0.044715 x^3).
  // (1 + tanh u) / 2 is the logistic function of 2u, so the same value is
  // x / (1 + e^{-2u}), with e^{-2u} = 2^{-2u log2(e)} from ex2 (relative
  // error about 2^-22) and the approximate quotient (2 ulp).  Unlike
  // 1 + tanh(u), which cancels for negative u, this keeps about 2^-21
  // relative accuracy for every x; where e^{-2u} exceeds 2^126 (x below
  // about -9.7) the quotient is 0, against a true magnitude below 2^-126 |x|.
  const float k0 = 0.7978845608028654f;
  const float k1 = 0.044715f;
  const float u = k0 * fmaf(k1 * x * x, x, x);
  return __fdividef(x, 1.0f + ex2_approx(-2.8853900817779268f * u));
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

// The BF16 bias of 32 consecutive columns (0 past column ncol).
__device__ __forceinline__ void load_bias32(const GemmArgs& a, int col0, int ncol,
                                            float (&bia)[32]) {
  if (ncol == 32) {
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
}

// One row of 32 BF16 results into the staging layout of the tensor store
// (rows of 64 B, 64-byte swizzle; row = lane).
__device__ __forceinline__ void stage_bf16_32(const float (&v)[32], uint8_t* stg, int lane) {
  uint8_t* rowp = stg + lane * 64;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(rowp + ((c ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(pack_bf16x2(v[8 * c + 0], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                   pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
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
  load_bias32(a, col0, ncol, bia);
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
  stage_bf16_32(v, stg, lane);
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

// The BF16 bias of 16 consecutive columns (0 past column ncol).
__device__ __forceinline__ void load_bias16(const GemmArgs& a, int col0, int ncol,
                                            float (&bia)[16]) {
  if (ncol >= 16) {
    const uint4* b4 = reinterpret_cast<const uint4*>(a.bias + col0);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
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
    for (int j = 0; j < 16; ++j)
      bia[j] = j < ncol ? __uint_as_float(static_cast<uint32_t>(a.bias[col0 + j]) << 16) : 0.f;
  }
}

// Stage one row of 32 packed BF16 results (16 words) and store the warp's
// chunk with the tensor map; the warp's two 2 KiB staging buffers alternate
// so a store drains while the next chunk is written.
__device__ __forceinline__ void store_chunk_packed(const CUtensorMap* tmOut,
                                                   const uint32_t (&p)[16], uint8_t* stg_base,
                                                   int& nstore, int col0, int row0, int lane) {
  uint8_t* stg = stg_base + (nstore & 1) * 2048;
  if (lane == 0) bulk_wait_read<1>();  // this buffer's last store has read it
  __syncwarp();
  uint8_t* rowp = stg + lane * 64;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(rowp + ((c ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmOut, stg, col0, row0);
    bulk_commit();
  }
  ++nstore;
}

// The linear epilogue with split RoPE on the leading args.rope_cols columns
// (the query and key heads): each head of dh = args.rope_dh columns pairs
// column j with j + dh/2 and writes B(c a - s b), B(s a + c b) from the
// FP32 values a, b (bias included) and the FP32 table entries c, s of this
// row (token) and index j.  Columns from rope_cols on get the plain linear
// result B(t + bias).  The warp's column half (BN/2 columns) holds whole
// heads; a 32-column chunk and its partner dh/2 columns on are handled
// together, 16 columns at a time, and kept as packed BF16 until stored.
template <int BN>
__device__ __forceinline__ void epilogue_tile_rope(const GemmArgs& args, const CUtensorMap* tmOut,
                                                   uint32_t tbase, int m0, int n0, int q, int row,
                                                   bool row_ok, int lane, uint8_t* stg_base,
                                                   int& nstore) {
  const int dh = args.rope_dh;
  const int hh = dh >> 1;  // pair offset: 32 or 64 columns
  const int row0 = m0 + q * 32;
  if (row0 >= args.M) return;
  const float* crow = args.rope_cos + static_cast<int64_t>(row_ok ? row : 0) * args.rope_ld;
  const float* srow = args.rope_sin + static_cast<int64_t>(row_ok ? row : 0) * args.rope_ld;
#pragma unroll 1
  for (int c0 = 0; c0 < BN / 2; c0 += 32) {
    const int in_head = c0 % dh;
    if (in_head >= hh) continue;  // second halves go with their first halves
    const int colA = n0 + c0, colB = colA + hh;
    if (colA >= args.N) break;
    const int ncolA = min(32, args.N - colA);
    const int ncolB = max(0, min(32, args.N - colB));
    const bool rot = colA < args.rope_cols;  // a query or key head (warp-uniform)
    uint32_t pa[16], pb[16];
#pragma unroll
    for (int hq = 0; hq < 2; ++hq) {
      __syncwarp();
      uint32_t ra[16], rb[16];
      tmem_ld_32x32b_x16(tbase + c0 + 16 * hq, ra);
      tmem_ld_32x32b_x16(tbase + c0 + hh + 16 * hq, rb);
      tmem_wait_ld();
      float va[16], vb[16], bia[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        va[j] = __uint_as_float(ra[j]);
        vb[j] = __uint_as_float(rb[j]);
      }
      if (args.bias_after_bf16) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          va[j] = round_bf16_f(va[j]);
          vb[j] = round_bf16_f(vb[j]);
        }
      }
      load_bias16(args, colA + 16 * hq, ncolA - 16 * hq, bia);
#pragma unroll
      for (int j = 0; j < 16; ++j) va[j] += bia[j];
      load_bias16(args, colB + 16 * hq, ncolB - 16 * hq, bia);
#pragma unroll
      for (int j = 0; j < 16; ++j) vb[j] += bia[j];
      if (rot) {
        if (args.rope_after_bf16) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            va[j] = round_bf16_f(va[j]);
            vb[j] = round_bf16_f(vb[j]);
          }
        }
        const int jt = in_head + 16 * hq;  // table index of the first pair
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          float4 c4 = make_float4(1.f, 1.f, 1.f, 1.f), s4 = make_float4(0.f, 0.f, 0.f, 0.f);
          if (row_ok) {
            c4 = __ldg(reinterpret_cast<const float4*>(crow + jt) + j4);
            s4 = __ldg(reinterpret_cast<const float4*>(srow + jt) + j4);
          }
          const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
          const float ss[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float a = va[4 * j4 + t], b = vb[4 * j4 + t];
            va[4 * j4 + t] = fmaf(cc[t], a, -ss[t] * b);
            vb[4 * j4 + t] = fmaf(ss[t], a, cc[t] * b);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        pa[8 * hq + j] = pack_bf16x2(va[2 * j], va[2 * j + 1]);
        pb[8 * hq + j] = pack_bf16x2(vb[2 * j], vb[2 * j + 1]);
      }
    }
    store_chunk_packed(tmOut, pa, stg_base, nstore, colA, row0, lane);
    if (ncolB > 0) store_chunk_packed(tmOut, pb, stg_base, nstore, colB, row0, lane);
  }
}

}  // namespace
}  // namespace psi
