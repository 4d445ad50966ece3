// page_gemm.cu -- the page GEMM: D = X * P^T for one weight page, on the
// 5th-generation tensor cores (tcgen05.mma kind::f16, BF16 in, FP32
// accumulator in tensor memory), operands staged by TMA, with the bias /
// GELU / FP32-accumulate / BF16-cast epilogues fused.
//
// Paper: Precision-Preserving Subtensor Inference, section II-B Eq.(2) (each
// output entry receives its complete dot product; output bias added once),
// section III-A (bias added in FP32 before the single BF16 write) and
// section III-B (hidden slice computed once, written as BF16, reused by the
// down projection; ordered down-projection accumulation).
//
// Structure (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0      TMA producer: X tile [128 x 64] and page tile [BN x 64] per
//               stage into a STAGES-deep shared-memory ring (128B swizzle);
//               the K range may span two pages (grouped FFN down slices)
//   warp 1      TMEM allocation and the MMA issuer: 4 MMAs of K = 16 per
//               stage into one of two TMEM accumulators (2 x BN columns)
//   warps 2..9  epilogue, two warps per TMEM lane quarter (one per column
//               half): tcgen05.ld of the accumulator rows, fused epilogue,
//               global stores, FP32 accumulator loads issued ahead of use;
//               frees the accumulator so the next tile's MMAs overlap this
//               tile's epilogue
// Every wait is bounded; on expiry the kernel records an error, drains its
// own copies and MMAs, frees TMEM and returns.
#include "gemm_epilogue.cuh"

namespace psi {
namespace {

constexpr int kThreads = 320;  // producer, MMA, 8 epilogue warps

template <int BN>
struct Cfg {
  static constexpr int STAGES = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BAR_OFFSET = STAGES * STAGE_BYTES;
  // one 4 KiB store-staging buffer per epilogue warp after the barriers
  static constexpr int STG_OFFSET = BAR_OFFSET + 1024;
  static constexpr int STG_BYTES = 4096;
  static constexpr int SMEM_BYTES = STG_OFFSET + 8 * STG_BYTES + 1024;  // + align slack
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct __align__(8) Bars {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    page_gemm_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmP,
                     const __grid_constant__ CUtensorMap tmP2,
                     const __grid_constant__ CUtensorMap tmOut, const GemmArgs args) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                              // STAGES x [128 x 64] bf16
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;     // STAGES x [BN x 64] bf16
  Bars* bars = reinterpret_cast<Bars*>(smem + C::BAR_OFFSET);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tiles = (args.M + BM - 1) / BM;
  const int n_tiles = (args.N + BN - 1) / BN;
  const int tiles = m_tiles * n_tiles;
  const int kblocks = (args.K + BK - 1) / BK;
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->tfull[a], 1);
      mbar_init(&bars->tempty[a], kEpiWarps);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmP);
    if (args.k_split || args.n_split) tma_prefetch_desc(&tmP2);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;  // bit s: stage s has been armed at least once
      uint32_t last_parity = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok && !args.debug_stall; t += gridDim.x) {
        const int m0 = (t % m_tiles) * BM;
        const int n0 = (t / m_tiles) * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1, abort_flag, args.timeout_ns)) {
            record_error(args.err, 1, KID_GEMM * 16 + 0, t, kb);
            bars->abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->full[stage], C::STAGE_BYTES);
          tma_load_2d(sA + stage * C::A_BYTES, &tmX, &bars->full[stage], kb * BK, m0);
          if (args.n_split > 0 && n0 >= args.n_split)
            tma_load_2d(sB + stage * C::B_BYTES, &tmP2, &bars->full[stage], kb * BK,
                        n0 - args.n_split);
          else if (args.k_split == 0 || kb < args.k_split)
            tma_load_2d(sB + stage * C::B_BYTES, &tmP, &bars->full[stage], kb * BK, n0);
          else
            tma_load_2d(sB + stage * C::B_BYTES, &tmP2, &bars->full[stage],
                        (kb - args.k_split) * BK, n0);
          armed |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // drain: every armed stage's last load has landed before exit
      for (int s = 0; s < C::STAGES; ++s) {
        if (armed & (1u << s)) {
          int dummy = 0;
          if (!mbar_wait(&bars->full[s], (last_parity >> s) & 1, &dummy, args.timeout_ns))
            record_error(args.err, 1, KID_GEMM * 16 + 4, s, 0);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, 0);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued = false;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1, abort_flag, args.timeout_ns)) {
          record_error(args.err, 1, KID_GEMM * 16 + 1, t, -1);
          bars->abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&bars->full[stage], phase, abort_flag, args.timeout_ns)) {
            record_error(args.err, 1, KID_GEMM * 16 + 1, t, kb);
            bars->abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b_base + kk * 32, 16, 1024);
            mma_bf16_ss(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          issued = true;
          mma_commit(&bars->empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&bars->tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (issued) {  // all MMAs complete before TMEM is released
        mma_commit(&bars->drain);
        int dummy = 0;
        if (!mbar_wait(&bars->drain, 0, &dummy, args.timeout_ns))
          record_error(args.err, 1, KID_GEMM * 16 + 5, 0, 0);
      }
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;       // column half of the tile
    const bool pre = epi_reads_acc(args.epi);
    const bool f32 = epi_writes_f32(args.epi);
    // staging: 4 KiB per warp; FP32 chunks use all of it, BF16 chunks
    // alternate between its two halves so a store can drain while the next
    // chunk is written
    uint8_t* stg_base = smem + C::STG_OFFSET + (warp - 2) * C::STG_BYTES;
    int nstore = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
      const int m0 = (t % m_tiles) * BM;
      const int n0 = (t / m_tiles) * BN + half * (BN / 2);
      const int row = m0 + q * 32 + lane;
      const bool row_ok = row < args.M;
      // the FP32 workspace does not depend on this tile's MMAs: start its
      // loads before waiting for the accumulator
      float4 nxt[8];
      if (pre && row_ok && n0 + 32 <= args.N) load_acc32(args, row, n0, nxt);
      if (!mbar_wait(&bars->tfull[acc], acc_phase, abort_flag, args.timeout_ns)) {
        if (lane == 0) record_error(args.err, 1, KID_GEMM * 16 + 2, t, q);
        bars->abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem + static_cast<uint32_t>(acc * BN + half * (BN / 2)) +
                             (static_cast<uint32_t>(q * 32) << 16);
      if constexpr (BN == 256) {
        if (args.rope_dh)
          epilogue_tile_rope<BN>(args, &tmOut, tbase, m0, n0, q, row, row_ok, lane, stg_base,
                                 nstore);
        else
          epilogue_tile<BN>(args, &tmOut, tbase, m0, n0, q, row, row_ok, lane, pre, f32,
                            stg_base, nstore, nxt);
      } else {
        epilogue_tile<BN>(args, &tmOut, tbase, m0, n0, q, row, row_ok, lane, pre, f32, stg_base,
                          nstore, nxt);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (lane == 0) bulk_wait<0>();  // this warp's stores are complete
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int BN>
psi_status launch_bn(const CUtensorMap& tx, const CUtensorMap& tp, const CUtensorMap& tp2,
                     const CUtensorMap& to, const GemmArgs& a, cudaStream_t s) {
  using C = Cfg<BN>;
  static std::atomic<uint64_t> attr_done{0};
  psi_status st = ensure_smem_attr(&attr_done, reinterpret_cast<const void*>(page_gemm_kernel<BN>),
                                   C::SMEM_BYTES, "cudaFuncSetAttribute(page_gemm)");
  if (st != PSI_OK) return st;
  const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
  const int grid = tiles < num_sms() ? tiles : num_sms();
  page_gemm_kernel<BN><<<grid, kThreads, C::SMEM_BYTES, s>>>(tx, tp, tp2, to, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "page_gemm launch");
  count_launch();
  return PSI_OK;
}

}  // namespace

int gemm_bn_for(int64_t N) { return N > 128 ? 256 : (N > 64 ? 128 : 64); }

// page_gemm_pair.cu
psi_status launch_page_gemm_pair(const CUtensorMap& tx, const CUtensorMap& tp,
                                 const CUtensorMap& tp2, const CUtensorMap& to, const GemmArgs& a,
                                 cudaStream_t s);

psi_status launch_page_gemm(const void* X, int64_t ldx, const void* P, int64_t ldp,
                            const GemmArgs& a, cudaStream_t stream, const void* P2) {
  if (a.M <= 0 || a.N <= 0 || a.K <= 0) return PSI_OK;
  // tiles of 256 x 256 on CTA pairs where the shape fills them, else one CTA
  // per 128 x BN tile; the choice depends on the shape only
  const bool pair = gemm_use_pair(a.M, a.N);
  // split RoPE needs whole heads in each epilogue warp's column half
  const int bn = pair ? 128 : (a.rope_dh ? 256 : gemm_bn_for(a.N));  // page rows per CTA and box
  if (a.rope_dh) {
    if ((a.rope_dh != 64 && a.rope_dh != 128) || a.epi != EPI_LINEAR || a.resid ||
        a.k_split > 0 || a.rope_cols % a.rope_dh || a.rope_ld % 4 ||
        (reinterpret_cast<uintptr_t>(a.rope_cos) & 15) ||
        (reinterpret_cast<uintptr_t>(a.rope_sin) & 15))
      return set_error(PSI_ERR_INVALID_ARG, "page_gemm: bad RoPE arguments");
  }
  CUtensorMap tx, tp, tp2;
  psi_status st = make_tmap_2d(&tx, X, a.M, a.K, ldx, BM, BK);
  if (st != PSI_OK) return st;
  if (a.k_split > 0 && a.n_split > 0)
    return set_error(PSI_ERR_INVALID_ARG, "page_gemm: K and N split together");
  if (a.k_split > 0) {
    const int64_t k1 = static_cast<int64_t>(a.k_split) * BK;
    if (!P2 || k1 >= a.K) return set_error(PSI_ERR_INVALID_ARG, "page_gemm: bad K split");
    st = make_tmap_2d(&tp, P, a.N, k1, ldp, bn, BK);
    if (st != PSI_OK) return st;
    st = make_tmap_2d(&tp2, P2, a.N, a.K - k1, ldp, bn, BK);
  } else if (a.n_split > 0) {
    if (!P2 || a.n_split >= a.N || a.n_split % (pair ? 256 : bn))
      return set_error(PSI_ERR_INVALID_ARG, "page_gemm: bad N split");
    st = make_tmap_2d(&tp, P, a.n_split, a.K, ldp, bn, BK);
    if (st != PSI_OK) return st;
    st = make_tmap_2d(&tp2, P2, a.N - a.n_split, a.K, ldp, bn, BK);
  } else {
    st = make_tmap_2d(&tp, P, a.N, a.K, ldp, bn, BK);
    tp2 = tp;
  }
  if (st != PSI_OK) return st;
  // the output tensor the epilogue stores into, in 32 x 32 boxes
  CUtensorMap to;
  if (a.epi == EPI_ACC_STORE || a.epi == EPI_ACC_ADD)
    st = make_tmap_2d_ex(&to, a.accf, a.M, a.N, a.ldacc, 32, 16, 4, 64);
  else
    st = make_tmap_2d_ex(&to, a.out, a.M, a.N, a.ldo, 32, 32, 2, 64);
  if (st != PSI_OK) return st;
  if (pair) return launch_page_gemm_pair(tx, tp, tp2, to, a, stream);
  switch (bn) {
    case 256: return launch_bn<256>(tx, tp, tp2, to, a, stream);
    case 128: return launch_bn<128>(tx, tp, tp2, to, a, stream);
    default: return launch_bn<64>(tx, tp, tp2, to, a, stream);
  }
}

}  // namespace psi
