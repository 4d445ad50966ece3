// page_gemm_pair.cu -- the page GEMM on a CTA pair: D = X * P^T in 256 x 256
// tiles, each tile computed by two CTAs of a cluster with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16, BF16 in, FP32
// accumulator in tensor memory).
//
// Paper: Precision-Preserving Subtensor Inference, section II-B Eq.(2) (each
// output entry receives its complete dot product), section III-A (bias in
// FP32 before the single BF16 write), section III-B (hidden slices reused by
// the down projection, ordered accumulation).  Same arithmetic and epilogues
// as page_gemm.cu; only the tiling of the tensor-core work differs.
//
// Why a pair: with one CTA per 128 x 256 tile, every 64-deep k-block moves
// 48 KiB into shared memory (TMA) and 48 KiB out of it (MMA operand reads)
// in 512 tensor cycles, more than the shared-memory bandwidth.  In a pair,
// each CTA holds 128 rows of X and 128 of the 256 page rows; the tensor cores
// share the page rows across the pair, so each CTA moves 32 KiB in and 32 KiB
// out per k-block for the same MMA time.
//
// Roles in each CTA (320 threads):
//   warp 0      TMA producer: this CTA's X rows [128 x 128] and page rows
//               [128 x 128] per stage (two 64-wide swizzled blocks of each;
//               3-stage ring), completion signalled on the even CTA's stage
//               barrier.  Stages 128 deep rather than six of 64 halve the
//               barrier round trips per MMA (8 pair MMAs per stage): the
//               resident QKV projection runs 9 % faster with the same bytes
//               in flight.
//   warp 1      TMEM allocation for the pair (both CTAs); in the even CTA the
//               MMA issuer, whose commits arrive on both CTAs' barriers
//   warps 2..9  epilogue over this CTA's 128 accumulator rows (shared with
//               the one-CTA kernel), then an arrive on the even CTA's
//               accumulator-empty barrier
// Every mbarrier wait is bounded; the two cluster barriers (after set-up and
// before tensor memory is freed) are reached by both CTAs on every path.
#include "gemm_epilogue.cuh"

namespace psi {
namespace {

constexpr int kThreadsP = 320;
constexpr int PSTAGES = 3;
constexpr int KD = 2 * BK;                    // k depth of a stage: two swizzled blocks
constexpr int PA_BLOCK = BM * BK * 2;         // one [128 x 64] block of X rows
constexpr int PB_BLOCK = 128 * BK * 2;        // one [128 x 64] block of page rows
constexpr int PA_BYTES = 2 * PA_BLOCK;        // this CTA's X rows
constexpr int PB_BYTES = 2 * PB_BLOCK;        // this CTA's half of the page rows
constexpr int PSTAGE_BYTES = PA_BYTES + PB_BYTES;
constexpr int PTILE_N = 256;                  // output columns per pair tile
constexpr int PTMEM_COLS = 2 * PTILE_N;       // double-buffered accumulator
constexpr int PBAR_OFFSET = PSTAGES * PSTAGE_BYTES;
constexpr int PSTG_OFFSET = PBAR_OFFSET + 1024;
constexpr int PSTG_BYTES = 4096;
constexpr int PSMEM_BYTES = PSTG_OFFSET + kEpiWarps * PSTG_BYTES + 1024;
static_assert(PSMEM_BYTES <= 232448, "shared memory");

struct __align__(8) PBars {
  uint64_t full[PSTAGES];
  uint64_t empty[PSTAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(kThreadsP, 1)
    page_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmX,
                          const __grid_constant__ CUtensorMap tmP,
                          const __grid_constant__ CUtensorMap tmP2,
                          const __grid_constant__ CUtensorMap tmOut, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + PSTAGES * PA_BYTES;
  PBars* bars = reinterpret_cast<PBars*>(smem + PBAR_OFFSET);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: the even CTA, which issues the MMAs
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int m_pairs = (args.M + 2 * BM - 1) / (2 * BM);
  const int n_tiles = (args.N + PTILE_N - 1) / PTILE_N;
  const int tiles = m_pairs * n_tiles;
  const int kblocks = (args.K + KD - 1) / KD;  // stages of KD; K tails read zeros
  volatile int* abort_flag = &bars->abort_flag;
  constexpr int kWhere = KID_GEMM * 16 + 8;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PSTAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->tfull[a], 1);
      mbar_init(&bars->tempty[a], 2 * kEpiWarps);  // both CTAs' epilogue warps
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
    tmem_alloc_pair(&bars->tmem_base, PTMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // both CTAs' barriers exist before either CTA signals the other's
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, last_parity = 0;
      bool ok = true;
      for (int t = pair; t < tiles && ok && !args.debug_stall; t += npairs) {
        const int m0 = (t % m_pairs) * 2 * BM + static_cast<int>(rank) * BM;
        const int n0 = (t / m_pairs) * PTILE_N + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1, abort_flag, args.timeout_ns)) {
            record_error(args.err, 1, kWhere + 0, t, kb);
            bars->abort_flag = 1;
            ok = false;
            break;
          }
          const uint32_t full_leader = mapa_shared(smem_u32(&bars->full[stage]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&bars->full[stage], 2 * PSTAGE_BYTES);
          for (int h = 0; h < 2; ++h) {  // the stage's two 64-deep blocks
            const int k64 = 2 * kb + h;
            tma_load_2d_pair(sA + stage * PA_BYTES + h * PA_BLOCK, &tmX, full_leader, k64 * BK,
                             m0);
            uint8_t* dB = sB + stage * PB_BYTES + h * PB_BLOCK;
            if (args.n_split > 0 && n0 >= args.n_split)
              tma_load_2d_pair(dB, &tmP2, full_leader, k64 * BK, n0 - args.n_split);
            else if (args.k_split == 0 || k64 < args.k_split)
              tma_load_2d_pair(dB, &tmP, full_leader, k64 * BK, n0);
            else
              tma_load_2d_pair(dB, &tmP2, full_leader, (k64 - args.k_split) * BK, n0);
          }
          armed |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == PSTAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // drain: a stage's loads have landed once the MMAs that read it have
      // completed, which the (multicast) empty barrier reports
      for (int s = 0; s < PSTAGES; ++s) {
        if (armed & (1u << s)) {
          int dummy = 0;
          if (!mbar_wait(&bars->empty[s], (last_parity >> s) & 1, &dummy, args.timeout_ns))
            record_error(args.err, 1, kWhere + 4, s, 0);
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------- MMA issuer (even CTA) --
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, PTILE_N, 0, 0);
      // Shared-memory descriptors formed once: the start-address field holds
      // address / 16 and every operand lies below 256 KB, so the descriptor
      // of base + off is the base's descriptor + off / 16.
      const uint64_t da0 = sdesc_sw128(smem_u32(sA), 16, 1024);
      const uint64_t db0 = sdesc_sw128(smem_u32(sB), 16, 1024);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int t = pair; t < tiles && ok; t += npairs) {
        if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1, abort_flag, args.timeout_ns)) {
          record_error(args.err, 1, kWhere + 1, t, -1);
          bars->abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * PTILE_N;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&bars->full[stage], phase, abort_flag, args.timeout_ns)) {
            record_error(args.err, 1, kWhere + 1, t, kb);
            bars->abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = da0 + static_cast<uint64_t>((stage * PA_BYTES) >> 4);
          const uint64_t db = db0 + static_cast<uint64_t>((stage * PB_BYTES) >> 4);
          static_assert(PA_BLOCK == PB_BLOCK, "one offset serves both operands");
#pragma unroll
          for (int kk = 0; kk < KD / 16; ++kk) {
            // k 16kk..: block kk / 4, 32 bytes per 16 k within its 128-byte rows
            const uint64_t off = static_cast<uint64_t>((kk >> 2) * (PA_BLOCK >> 4) + 2 * (kk & 3));
            mma_bf16_ss_pair(d_tmem, da + off, db + off, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          issued = true;
          mma_commit_pair(&bars->empty[stage], 0x3);  // both CTAs' stage is free
          if (++stage == PSTAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair(&bars->tfull[acc], 0x3);  // both CTAs' accumulator rows are ready
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (issued) {  // all MMAs complete before the pair frees tensor memory
        mma_commit_pair(&bars->drain, 0x1);
        int dummy = 0;
        if (!mbar_wait(&bars->drain, 0, &dummy, args.timeout_ns))
          record_error(args.err, 1, kWhere + 5, 0, 0);
      }
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const bool pre = epi_reads_acc(args.epi);
    const bool f32 = epi_writes_f32(args.epi);
    uint8_t* stg_base = smem + PSTG_OFFSET + (warp - 2) * PSTG_BYTES;
    int nstore = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < tiles; t += npairs) {
      const int m0 = (t % m_pairs) * 2 * BM + static_cast<int>(rank) * BM;
      const int n0 = (t / m_pairs) * PTILE_N + half * (PTILE_N / 2);
      const int row = m0 + q * 32 + lane;
      const bool row_ok = row < args.M;
      float4 nxt[8];
      if (pre && row_ok && n0 + 32 <= args.N) load_acc32(args, row, n0, nxt);
      if (!mbar_wait(&bars->tfull[acc], acc_phase, abort_flag, args.timeout_ns)) {
        if (lane == 0) record_error(args.err, 1, kWhere + 2, t, q);
        bars->abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem + static_cast<uint32_t>(acc * PTILE_N + half * (PTILE_N / 2)) +
                             (static_cast<uint32_t>(q * 32) << 16);
      if (args.rope_dh)
        epilogue_tile_rope<PTILE_N>(args, &tmOut, tbase, m0, n0, q, row, row_ok, lane, stg_base,
                                    nstore);
      else
        epilogue_tile<PTILE_N>(args, &tmOut, tbase, m0, n0, q, row, row_ok, lane, pre, f32,
                               stg_base, nstore, nxt);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&bars->tempty[acc]), 0));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (lane == 0) bulk_wait<0>();  // this warp's stores are complete
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA frees tensor memory or exits while the pair still works
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, PTMEM_COLS);
  }
}

}  // namespace

bool gemm_use_pair(int64_t M, int64_t N) { return M >= 256 && N >= 256; }

psi_status launch_page_gemm_pair(const CUtensorMap& tx, const CUtensorMap& tp,
                                 const CUtensorMap& tp2, const CUtensorMap& to, const GemmArgs& a,
                                 cudaStream_t s) {
  static std::atomic<uint64_t> attr_done{0};
  psi_status st = ensure_smem_attr(&attr_done, reinterpret_cast<const void*>(page_gemm_pair_kernel),
                                   PSMEM_BYTES, "cudaFuncSetAttribute(page_gemm_pair)");
  if (st != PSI_OK) return st;
  const int tiles = ((a.M + 2 * BM - 1) / (2 * BM)) * ((a.N + PTILE_N - 1) / PTILE_N);
  const int max_pairs = num_sms() / 2;
  const int pairs = tiles < max_pairs ? tiles : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kThreadsP, 1, 1);
  cfg.dynamicSmemBytes = PSMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, page_gemm_pair_kernel, tx, tp, tp2, to, a);
  if (e != cudaSuccess) return cuda_error(e, "page_gemm_pair launch");
  count_launch();
  return PSI_OK;
}

}  // namespace psi
