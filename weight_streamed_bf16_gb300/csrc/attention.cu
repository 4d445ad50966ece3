// attention.cu -- partitioned attention with FP32 online softmax on tcgen05.
//
// Paper: Precision-Preserving Subtensor Inference, section II-B Eqs.(3)-(4)
// (online-softmax invariant over disjoint key tiles: m' = max(m, max s_j),
// eta = e^{m-m'}, l' = eta*l + sum e^{s_j-m'}, z' = eta*z + sum e^{s_j-m'}
// v_j, output z/l) and section III-A (FP32 online accumulation in place of
// BF16 numerator exponential weights).
//
// One CTA per (head, 256 queries) = two 128-query tiles that share every K
// and V tile.  Key tiles of 128:
//   warp 0      TMA producer: Q (both tiles) once, then K_j and V_j into
//               2-stage rings
//   warp 1      TMEM owner and MMA issuer, ping-ponging the two query tiles:
//                 S_t = Q_t K_j^T          (M=128, N=128 keys, K=128) into
//                                          the S/P columns of tile t
//                 O_t += P_t,hi V_j + P_t,lo V_j   (P read from tensor memory,
//                                          V read MN-major from shared memory)
//   warps 2..5  softmax of tile 0, warps 6..9 softmax of tile 1, one query
//               row per thread: scores scaled to log2 units in FP32, running
//               max m and sum l in FP32, weights p = 2^(s - m) in FP32 split
//               into p_hi = B(p) and p_lo = B(p - p_hi) (the tensor-core
//               operand then carries p to within 2^-17 relative) and written
//               over the row's S columns (two passes over tensor memory:
//               row extremum, then exponentials); O rescaled by eta in
//               tensor memory when the max moves; O / l written as BF16.
// While one softmax warpgroup works on its tile, the tensor core runs the
// other tile's MMAs.
#include "internal.h"
#include "ptx.cuh"

namespace psi {
namespace {

constexpr int BQ = 128;      // queries per tile
constexpr int NT = 2;        // query tiles per CTA
constexpr int BKEY = 128;    // keys per tile
constexpr int DH = 128;
constexpr int kThreads = 64 + NT * 128;
constexpr int TILE64 = 128 * 128;  // one [128 rows x 64 cols] BF16 swizzled block, bytes

constexpr int OFF_Q = 0;                              // NT tiles x 2 column blocks
constexpr int OFF_K = OFF_Q + NT * 2 * TILE64;        // 2 stages x 2 column blocks
constexpr int OFF_V = OFF_K + 2 * 2 * TILE64;
constexpr int OFF_BAR = OFF_V + 2 * 2 * TILE64;       // 192 KiB
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;

// tensor memory: tile t uses columns [256 t, 256 t + 128) for S and P over
// it (for keys 32c..32c+31: p_hi pairs in columns 32c..32c+15, p_lo pairs in
// 32c+16..32c+31) and [256 t + 128, 256 t + 256) for O
constexpr uint32_t TM_COLS = 512;
__device__ __forceinline__ uint32_t tm_s(int t) { return 256u * t; }
__device__ __forceinline__ uint32_t tm_o(int t) { return 256u * t + 128u; }

struct __align__(8) ABars {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[NT], p_full[NT], pv_done[NT];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Coordinates of (head, token) in a 2-D tensor map: x = col + h*hx,
// y = token + h*hy.
struct View {
  int32_t hx;
  int32_t hy;
};

__device__ __forceinline__ void record_error(DevError* e, int code, int where, int i0, int i1) {
  if (atomicCAS(&e->code, 0, code) == 0) {
    e->where = where;
    e->info0 = i0;
    e->info1 = i1;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const View vq, const View vk,
                const View vv, const AttnArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  ABars* bars = reinterpret_cast<ABars*>(smem + OFF_BAR);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q_blocks = (args.Nq + NT * BQ - 1) / (NT * BQ);
  const int head = blockIdx.x / q_blocks;
  const int q0 = (blockIdx.x % q_blocks) * (NT * BQ);
  const int nb = (args.Nk + BKEY - 1) / BKEY;
  volatile int* abort_flag = &bars->abort_flag;
  constexpr int kWhere = KID_ATTN * 16;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int t = 0; t < NT; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 128);
      mbar_init(&bars->pv_done[t], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      uint32_t k_armed = 0, v_armed = 0;  // per-stage parity of the last arming
      int k_cnt[2] = {0, 0}, v_cnt[2] = {0, 0};
      mbar_arrive_expect_tx(&bars->q_full, NT * 2 * TILE64);
      for (int t = 0; t < NT; ++t)
        for (int cb = 0; cb < 2; ++cb)
          tma_load_2d(smem + OFF_Q + (t * 2 + cb) * TILE64, &tmQ, &bars->q_full,
                      head * vq.hx + cb * 64, head * vq.hy + q0 + t * BQ);
      for (int j = 0; j < nb; ++j) {
        const int s = j & 1;
        const uint32_t par = ((j >> 1) & 1) ^ 1;
        const int key0 = j * BKEY;
        if (!mbar_wait(&bars->k_empty[s], par, abort_flag, args.timeout_ns)) {
          record_error(args.err, 1, kWhere + 0, j, 0);
          bars->abort_flag = 1;
          break;
        }
        uint8_t* kd = smem + OFF_K + s * 2 * TILE64;
        mbar_arrive_expect_tx(&bars->k_full[s], 2 * TILE64);
        tma_load_2d(kd, &tmK, &bars->k_full[s], head * vk.hx, head * vk.hy + key0);
        tma_load_2d(kd + TILE64, &tmK, &bars->k_full[s], head * vk.hx + 64, head * vk.hy + key0);
        k_armed = (k_armed & ~(1u << s)) | (static_cast<uint32_t>(k_cnt[s] & 1) << s);
        ++k_cnt[s];
        if (!mbar_wait(&bars->v_empty[s], par, abort_flag, args.timeout_ns)) {
          record_error(args.err, 1, kWhere + 0, j, 1);
          bars->abort_flag = 1;
          break;
        }
        uint8_t* vd = smem + OFF_V + s * 2 * TILE64;
        mbar_arrive_expect_tx(&bars->v_full[s], 2 * TILE64);
        tma_load_2d(vd, &tmV, &bars->v_full[s], head * vv.hx, head * vv.hy + key0);
        tma_load_2d(vd + TILE64, &tmV, &bars->v_full[s], head * vv.hx + 64, head * vv.hy + key0);
        v_armed = (v_armed & ~(1u << s)) | (static_cast<uint32_t>(v_cnt[s] & 1) << s);
        ++v_cnt[s];
      }
      // drain this thread's copies before the CTA exits
      int dummy = 0;
      if (!mbar_wait(&bars->q_full, 0, &dummy, args.timeout_ns))
        record_error(args.err, 1, kWhere + 4, -1, 0);
      for (int s = 0; s < 2; ++s) {
        if (k_cnt[s] && !mbar_wait(&bars->k_full[s], (k_armed >> s) & 1, &dummy, args.timeout_ns))
          record_error(args.err, 1, kWhere + 4, s, 1);
        if (v_cnt[s] && !mbar_wait(&bars->v_full[s], (v_armed >> s) & 1, &dummy, args.timeout_ns))
          record_error(args.err, 1, kWhere + 4, s, 2);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, 128, 0, 1);  // V is MN-major
      bool ok = true, issued = false;
      auto fail = [&](int j, int what) {
        record_error(args.err, 1, kWhere + 1, j, what);
        bars->abort_flag = 1;
        ok = false;
      };
      // S_t = Q_t K_j^T into tile t's S/P columns
      auto issue_s = [&](int j, int t) {
        const int s = j & 1;
        if (t == 0) {
          if (!mbar_wait(&bars->k_full[s], (j >> 1) & 1, abort_flag, args.timeout_ns)) {
            fail(j, 0);
            return;
          }
          tc_fence_after();
        }
        const uint32_t sK = smem_u32(smem + OFF_K + s * 2 * TILE64);
        const uint32_t sQ = smem_u32(smem + OFF_Q + t * 2 * TILE64);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t off = (kk >> 2) * TILE64 + (kk & 3) * 32;
          mma_bf16_ss(tmem + tm_s(t), sdesc_sw128(sQ + off, 16, 1024),
                      sdesc_sw128(sK + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[t]);
        if (t == NT - 1) mma_commit(&bars->k_empty[s]);  // both tiles have read K_j
        issued = true;
      };
      if (!mbar_wait(&bars->q_full, 0, abort_flag, args.timeout_ns)) fail(-1, 2);
      for (int t = 0; t < NT && ok; ++t) issue_s(0, t);
      for (int j = 0; j < nb && ok; ++j) {
        const int s = j & 1;
        if (!mbar_wait(&bars->v_full[s], (j >> 1) & 1, abort_flag, args.timeout_ns)) {
          fail(j, 4);
          break;
        }
        const uint32_t sV = smem_u32(smem + OFF_V + s * 2 * TILE64);
        for (int t = 0; t < NT && ok; ++t) {
          if (!mbar_wait(&bars->p_full[t], j & 1, abort_flag, args.timeout_ns)) {
            fail(j, 3);
            break;
          }
          tc_fence_after();
          // O_t += P_hi V_j + P_lo V_j: P from tensor memory, keys 16kk..16kk+15
          // at columns 32(kk/2) + 8(kk%2) (hi) and 16 further (lo); V rows
          // 16kk.. of both 64-wide dh blocks (LBO apart)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int kk = 0; kk < BKEY / 16; ++kk) {
              const uint32_t pcol = 32 * (kk >> 1) + 8 * (kk & 1) + 16 * half;
              mma_bf16_ts(tmem + tm_o(t), tmem + tm_s(t) + pcol,
                          sdesc_sw128(sV + kk * 2048, TILE64, 1024), idesc_o,
                          (j | half | kk) != 0 ? 1u : 0u);
            }
          }
          mma_commit(&bars->pv_done[t]);
          // tile t's next scores overwrite its P: issued after its PV MMAs,
          // which the tensor core executes first
          if (j + 1 < nb) issue_s(j + 1, t);
        }
        if (!ok) break;
        mma_commit(&bars->v_empty[s]);
      }
      if (issued) {
        mma_commit(&bars->drain);
        int dummy = 0;
        if (!mbar_wait(&bars->drain, 0, &dummy, args.timeout_ns))
          record_error(args.err, 1, kWhere + 5, 0, 0);
      }
    }
  } else {
    // ---------------------------------------------------------- softmax --
    const int t = (warp - 2) >> 2;   // query tile of this warpgroup
    const int q = warp & 3;          // TMEM lane quarter
    const int row = q * 32 + lane;   // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t tS = tmem + tm_s(t) + lane_off;
    const uint32_t tO = tmem + tm_o(t) + lane_off;
    float m2 = -INFINITY;  // running max, log2 units
    float l = 0.f;         // running sum of weights
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      if (!mbar_wait(&bars->s_full[t], j & 1, abort_flag, args.timeout_ns)) {
        if (lane == 0) record_error(args.err, 1, kWhere + 2, j, t * 4 + q);
        bars->abort_flag = 1;
        ok = false;
        break;
      }
      tc_fence_after();
      // pass 1: row extremum of the raw scores (max, or min for a negative
      // scale); all four chunks are loaded before one wait
      const float c = args.scale_log2;  // scale * log2(e)
      const int kvalid = args.Nk - j * BKEY;  // keys of this tile that exist
      float ext = c >= 0.f ? -INFINITY : INFINITY;
      {
        uint32_t ra[32], rb[32], rc[32], rd[32];
        tmem_ld_32x32b_x32(tS + 0, ra);
        tmem_ld_32x32b_x32(tS + 32, rb);
        tmem_ld_32x32b_x32(tS + 64, rc);
        tmem_ld_32x32b_x32(tS + 96, rd);
        tmem_wait_ld();
        auto scan = [&](const uint32_t (&r)[32], int base) {
          if (kvalid >= BKEY) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              ext = c >= 0.f ? fmaxf(ext, __uint_as_float(r[i])) : fminf(ext, __uint_as_float(r[i]));
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (base + i < kvalid)
                ext = c >= 0.f ? fmaxf(ext, __uint_as_float(r[i]))
                               : fminf(ext, __uint_as_float(r[i]));
          }
        };
        scan(ra, 0);
        scan(rb, 32);
        scan(rc, 64);
        scan(rd, 96);
      }
      const float m_new = fmaxf(m2, ext * c);
      const float eta = ex2_approx(m2 - m_new);  // 0 on the first tile
      // pass 2: p = 2^(s*c - m) with one FFMA; the chunk of 32 keys is
      // written back over its own 32 columns as 16 columns of p_hi pairs and
      // 16 of p_lo pairs (keys 2i, 2i+1 share a column).  The next chunk's
      // load is in flight while this chunk is processed.
      float rs = 0.f;
      auto expo = [&](const uint32_t (&r)[32], int cc) {
        float p[32];
        if (kvalid >= BKEY) {
#pragma unroll
          for (int i = 0; i < 32; ++i) p[i] = ex2_approx(fmaf(__uint_as_float(r[i]), c, -m_new));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            p[i] = cc * 32 + i < kvalid ? ex2_approx(fmaf(__uint_as_float(r[i]), c, -m_new)) : 0.f;
        }
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          rs += p[2 * i] + p[2 * i + 1];
          hi[i] = pack_bf16x2(p[2 * i], p[2 * i + 1]);
          lo[i] = pack_bf16x2(p[2 * i] - bf16_lo(hi[i]), p[2 * i + 1] - bf16_hi(hi[i]));
        }
        tmem_st_32x32b_x16(tS + cc * 32, hi);
        tmem_st_32x32b_x16(tS + cc * 32 + 16, lo);
      };
      {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(tS + 0, r0);
        tmem_wait_ld();
        tmem_ld_32x32b_x32(tS + 32, r1);
        expo(r0, 0);
        tmem_wait_ld();
        tmem_ld_32x32b_x32(tS + 64, r0);
        expo(r1, 1);
        tmem_wait_ld();
        tmem_ld_32x32b_x32(tS + 96, r1);
        expo(r0, 2);
        tmem_wait_ld();
        expo(r1, 3);
      }
      l = eta * l + rs;
      m2 = m_new;
      if (j > 0) {
        // the previous PV of this tile has finished: O is stable
        if (!mbar_wait(&bars->pv_done[t], (j - 1) & 1, abort_flag, args.timeout_ns)) {
          if (lane == 0) record_error(args.err, 1, kWhere + 3, j, t * 4 + q);
          bars->abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, eta != 1.0f)) {
#pragma unroll 1
          for (int cc = 0; cc < DH / 32; cc += 2) {
            uint32_t ra[32], rb[32];
            tmem_ld_32x32b_x32(tO + cc * 32, ra);
            tmem_ld_32x32b_x32(tO + cc * 32 + 32, rb);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              ra[i] = __float_as_uint(__uint_as_float(ra[i]) * eta);
              rb[i] = __float_as_uint(__uint_as_float(rb[i]) * eta);
            }
            tmem_st_32x32b_x32(tO + cc * 32, ra);
            tmem_st_32x32b_x32(tO + cc * 32 + 32, rb);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[t]);
    }
    if (ok && nb > 0) {
      if (!mbar_wait(&bars->pv_done[t], (nb - 1) & 1, abort_flag, args.timeout_ns)) {
        if (lane == 0) record_error(args.err, 1, kWhere + 3, nb, t * 4 + q);
        bars->abort_flag = 1;
      } else {
        tc_fence_after();
        const int tok = q0 + t * BQ + row;
        uint16_t* orow =
            args.O + head * args.o_ld_head + static_cast<int64_t>(tok) * args.o_ld_token;
#pragma unroll 1
        for (int c = 0; c < DH / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tO + c * 32, r);
          tmem_wait_ld();
          if (tok < args.Nq) {
            uint4* o4 = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float v[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) v[i] = __fdiv_rn(__uint_as_float(r[8 * u + i]), l);
              o4[u] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                 pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// Choose the 2-D tensor map of a psi_heads view: head-major rows (ld_head a
// multiple of ld_token) or heads interleaved along the row.
psi_status make_view(const psi_heads* h, int heads, int64_t tokens, CUtensorMap* m, View* v) {
  if (!h || !h->ptr) return set_error(PSI_ERR_INVALID_ARG, "attention: null tensor");
  if (h->ld_token < DH) return set_error(PSI_ERR_INVALID_ARG, "attention: ld_token < dh");
  if (h->ld_head >= h->ld_token && h->ld_head % h->ld_token == 0) {
    const int64_t hy = h->ld_head / h->ld_token;
    if (hy < tokens && heads > 1)
      return set_error(PSI_ERR_INVALID_ARG, "attention: heads overlap (ld_head too small)");
    v->hx = 0;
    v->hy = static_cast<int32_t>(hy);
    return make_tmap_2d(m, h->ptr, (heads - 1) * hy + tokens, DH, h->ld_token, 128, 64);
  }
  if (h->ld_head >= DH && (heads - 1) * h->ld_head + DH <= h->ld_token && h->ld_head % 8 == 0) {
    v->hx = static_cast<int32_t>(h->ld_head);
    v->hy = 0;
    return make_tmap_2d(m, h->ptr, tokens, (heads - 1) * h->ld_head + DH, h->ld_token, 128, 64);
  }
  return set_error(PSI_ERR_UNSUPPORTED, "attention: head layout is neither head-major nor "
                                        "interleaved within a row");
}

}  // namespace

psi_status launch_attention(const psi_heads* Q, const psi_heads* K, const psi_heads* V,
                            const AttnArgs& a, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  View vq, vk, vv;
  psi_status st = make_view(Q, a.heads, a.Nq, &mq, &vq);
  if (st != PSI_OK) return st;
  if ((st = make_view(K, a.heads, a.Nk, &mk, &vk)) != PSI_OK) return st;
  if ((st = make_view(V, a.heads, a.Nk, &mv, &vv)) != PSI_OK) return st;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(attn)");
    attr_set = true;
  }
  const int q_blocks = (a.Nq + NT * BQ - 1) / (NT * BQ);
  const long long grid = static_cast<long long>(q_blocks) * a.heads;
  if (grid <= 0) return PSI_OK;
  if (grid > 0x7FFFFFFFLL) return set_error(PSI_ERR_UNSUPPORTED, "attention: grid too large");
  attn_kernel<<<static_cast<unsigned>(grid), kThreads, SMEM_BYTES, stream>>>(mq, mk, mv, vq, vk,
                                                                             vv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "attention launch");
  return PSI_OK;
}

}  // namespace psi
