// attention.cu -- partitioned attention with FP32 online softmax on tcgen05.
//
// Paper: Precision-Preserving Subtensor Inference, section II-B Eqs.(3)-(4)
// (online-softmax invariant over disjoint key tiles: m' = max(m, max s_j),
// eta = e^{m-m'}, l' = eta*l + sum e^{s_j-m'}, z' = eta*z + sum e^{s_j-m'}
// v_j, output z/l) and section III-A (FP32 online accumulation in place of
// BF16 numerator exponential weights).
//
// Keys are visited in blocks of key_block = 128 or 256 (one online update per
// block), read as 128-key K/V sub-tiles.  A CTA holds NT query tiles of 128
// (NT = 2 for 128-key blocks, 1 for 256-key blocks):
//   warp 0      TMA producer: Q once, then per block its K sub-tiles and its
//               V sub-tiles into rings (V of block j and K of block j + 1
//               complete one barrier per sub-tile, so the MMA issuer waits
//               once per sub-tile for its copies; with 256-key blocks the K
//               ring has 3 stages so that this pairing never delays V)
//   warp 1      TMEM owner and MMA issuer:
//                 S_t = Q_t K^T            (M=128, N=128 per sub-tile, K=128)
//                                          into the S/P columns of tile t
//                 O_t += P_t,hi V + P_t,lo V   (P read from tensor memory,
//                                          V read MN-major from shared memory)
//               with two tiles it ping-pongs them: tile t's next S is issued
//               right after its PV, while the other tile is in softmax
//   warps 2..   softmax, 4 warps per query tile, one query row per thread:
//               two passes over tensor memory (row extremum, then
//               p = 2^(s*scale*log2e - m) by one FFMA and ex2), reference
//               point m (the running max, moved when it grows by more than
//               2^8) and sum l in FP32, p split into p_hi = B(p) and
//               p_lo = B(p - p_hi) (the tensor-core operand carries p to
//               within 2^-17 relative) and written over the row's S
//               columns; O rescaled by eta in tensor memory when the max
//               moves; O / l written as BF16 at the end.
//
// Tail split: with one CTA per SM, the last wave of (head, query tile)
// units is usually partial.  Given a workspace, the launch keeps whole
// units for every full wave and cuts each unit of the last wave into
// contiguous ranges of key blocks, one CTA per range.  Such a CTA stores its
// unnormalised state (z, m, l) in FP32; merge_kernel then combines the
// ranges of a unit by the same update as Eq.(4) (M = max m_r,
// l = sum 2^(m_r - M) l_r, z = sum 2^(m_r - M) z_r) and writes B(z / l).
#include <algorithm>
#include "internal.h"
#include "ptx.cuh"

namespace psi {
namespace {

constexpr int BQ = 128;      // queries per tile
constexpr int SUB = 128;     // keys per K/V sub-tile (one S = QK^T MMA of N = 128)
constexpr int DH = 128;
constexpr int TILE64 = 128 * 128;  // one [128 rows x 64 cols] BF16 swizzled block, bytes

// Kernel shape for key blocks of KSUB sub-tiles (key_block = 128 * KSUB):
// NT query tiles per CTA (two when the block is 128 keys, so the softmax
// warpgroups ping-pong; one when it is 256 keys, whose S needs 256 TMEM
// columns).  Tensor memory per tile: S and P over it (128 * KSUB columns;
// for keys 32c..32c+31 of the block: p_hi pairs in columns 32c..32c+15, p_lo
// pairs in 32c+16..32c+31), then O (128 columns).
template <int KSUB>
struct AShape {
  static constexpr int NT = KSUB == 1 ? 2 : 1;
  static constexpr int KB = SUB * KSUB;
  // softmax warps per TMEM lane quarter (key ranges): 2 with two tiles, 4
  // with one, which halves each warp's share of a 256-key block
  static constexpr int SPLIT = KSUB == 1 ? 2 : 4;
  static constexpr int kThreads = 64 + NT * 128 * SPLIT;
  static constexpr int OFF_Q = 0;                          // NT tiles x 2 column blocks
  // K ring stages (x 2 column blocks): 3 with 256-key blocks, so that K of
  // block j + 1 can share a copy barrier with V of block j without waiting
  // for the scores that read the stage before it
  static constexpr int KSTAGES = KSUB == 1 ? 2 : 3;
  static constexpr int OFF_K = OFF_Q + NT * 2 * TILE64;
  static constexpr int OFF_V = OFF_K + KSTAGES * 2 * TILE64;
  static constexpr int OFF_BAR = OFF_V + 2 * 2 * TILE64;
  // row-extremum and row-sum exchange between the key ranges of a row:
  // [2 parities][NT tiles][SPLIT ranges][128 rows] floats
  static constexpr int OFF_X = OFF_BAR + 256;
  static constexpr int X_BYTES = 2 * NT * SPLIT * 128 * 4;
  static constexpr int SMEM_BYTES = OFF_X + X_BYTES + 1024;
  static constexpr uint32_t TILE_COLS = KB + 128;
  static constexpr uint32_t TM_COLS = 512;
  static_assert(NT * TILE_COLS <= TM_COLS, "tensor memory");
  __device__ static uint32_t tm_s(int t) { return TILE_COLS * t; }
  __device__ static uint32_t tm_o(int t) { return TILE_COLS * t + KB; }
};
// 256-key blocks keep sub-tile 0's P in the columns after O
static_assert(AShape<2>::TILE_COLS + SUB <= AShape<2>::TM_COLS, "tensor memory");

// Workspace slot of one tail-split CTA: z [NT*128 rows x 128] then (m, l)
// per row, FP32.
template <int NT>
struct PartSlot {
  static constexpr int ROWS = NT * BQ;
  static constexpr size_t FLOATS = static_cast<size_t>(ROWS) * (DH + 2);
};

struct __align__(8) ABars {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[3];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t xbar[2][4];  // per tile and lane quarter: the row's key ranges met
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

// Publish a row value to the other warps of the row (same rows, other key
// ranges) and gather the row's SPLIT values in range order (out[h] = v):
// every warp writes its slot, arrives on the row group's mbarrier and waits
// (bounded) for the phase, then reads the other slots.  All warps of the row
// then combine the same values in the same order.  Returns false on timeout.
template <int SPLIT>
__device__ __forceinline__ bool exchange(float* slots, int h, float v, uint64_t* bar,
                                         uint32_t parity, float (&out)[SPLIT],
                                         volatile int* abort, uint64_t limit_ns) {
  slots[h * 128] = v;
  mbar_arrive(bar);
  if (!mbar_wait(bar, parity, abort, limit_ns)) return false;
  if constexpr (SPLIT == 2) {
    const float w = slots[(h ^ 1) * 128];
    out[0] = h == 0 ? v : w;
    out[1] = h == 0 ? w : v;
  } else {
#pragma unroll
    for (int i = 0; i < SPLIT; ++i) out[i] = slots[i * 128];
  }
  return true;
}

// The softmax role of one warp (both attention kernels).  SPLIT warps share
// each TMEM lane quarter of a tile: warp h owns the keys
// [h*KB/SPLIT, (h+1)*KB/SPLIT) of every block (and O columns
// [h*DH/SPLIT, ...)); the warps of a row exchange the row extremum once per
// block and the row sum once at the end.
template <int KSUB, int NT, int SPLIT, class Bars>
__device__ __forceinline__ void softmax_role(Bars* bars, uint8_t* smem, int off_x, uint32_t tmem,
                                             uint32_t tile_cols, int warp, int lane,
                                             const AttnArgs& args, int nb, int jb0, int slot,
                                             int head, int q0, volatile int* abort_flag) {
  constexpr int KB = SUB * KSUB;
  constexpr int kWhere = KID_ATTN * 16;
  const int e = warp - 2;
  const int t = e / (4 * SPLIT);           // query tile
  const int h = (e % (4 * SPLIT)) / 4;     // key range
  const int q = warp & 3;                  // TMEM lane quarter
  const int row = q * 32 + lane;           // query row within the tile
  const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
  const uint32_t tS = tmem + (tile_cols * static_cast<uint32_t>(t)) + lane_off;
  const uint32_t tO = tmem + (tile_cols * static_cast<uint32_t>(t) + KB) + lane_off;
  constexpr int NCH = KB / 32 / SPLIT;     // 32-key chunks of this range per block
  static_assert(NCH == 2, "each softmax warp owns 64 keys of a block");
  const int ch0 = h * NCH;                 // first chunk of this range
  float* xbase = reinterpret_cast<float*>(smem + off_x);
  uint64_t* xb = &bars->xbar[t][q];
  auto xslots = [&](int par) { return xbase + ((par * NT + t) * SPLIT) * 128 + row; };
  float m2 = -INFINITY;  // running max, log2 units
  float l = 0.f;         // running sum of this range's weights
  bool ok = true;
  for (int j = 0; j < nb; ++j) {
    if (!mbar_wait(&bars->s_full[t], j & 1, abort_flag, args.timeout_ns)) {
      if (lane == 0) record_error(args.err, 1, kWhere + 2, j, t * 8 + h * 4 + q);
      bars->abort_flag = 1;
      ok = false;
      break;
    }
    tc_fence_after();
    // S(j) of the last tile is issued after both tiles' S(j) and that tile's
    // PV(j - 1), so once it is complete K(j) and V(j - 1) are free: one
    // thread of the last tile hands both stages back to the producer (the
    // MMA issuer then commits two barriers fewer per block)
    if (t == NT - 1 && e % (4 * SPLIT) == 0 && lane == 0) {
      mbar_arrive(&bars->k_empty[j & 1]);
      if (j > 0) mbar_arrive(&bars->v_empty[(j - 1) & 1]);
    }
    // pass 1: row extremum of this range's raw scores (max, or min for a
    // negative scale), then the other ranges' through shared memory
    const float c = args.scale_log2;  // scale * log2(e)
    const int kvalid = args.Nk - (jb0 + j) * KB;  // keys of this block that exist
    float ext = c >= 0.f ? -INFINITY : INFINITY;
    auto scan = [&](const uint32_t (&r)[32], int base) {
      if (kvalid >= KB) {
        if (c >= 0.f) {
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            ext = max3f(ext, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            ext = min3f(ext, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (base + i < kvalid)
            ext = c >= 0.f ? fmaxf(ext, __uint_as_float(r[i])) : fminf(ext, __uint_as_float(r[i]));
      }
    };
    // the range's two chunks stay in registers for pass 2
    uint32_t ra[32], rb[32];
    tmem_ld_32x32b_x32(tS + ch0 * 32, ra);
    tmem_ld_32x32b_x32(tS + (ch0 + 1) * 32, rb);
    tmem_wait_ld();
    scan(ra, ch0 * 32);
    scan(rb, (ch0 + 1) * 32);
    float others[SPLIT];
    if (!exchange<SPLIT>(xslots(j & 1), h, ext, xb, j & 1, others, abort_flag,
                         args.timeout_ns)) {
      if (lane == 0) record_error(args.err, 1, kWhere + 6, j, t * 8 + h * 4 + q);
      bars->abort_flag = 1;
      ok = false;
      break;
    }
#pragma unroll
    for (int i = 0; i < SPLIT; ++i)
      ext = c >= 0.f ? fmaxf(ext, others[i]) : fminf(ext, others[i]);
    // reference point of the exponents: moved only when the running max
    // exceeds it by more than 2^8 (the weights then stay below 2^8 and O is
    // rescaled rarely); z and l are scaled alike, so z / l is unchanged.
    // The BF16-weights variant keeps the exact running max: its rounded
    // weights depend on the reference point.
    const float mx = fmaxf(m2, ext * c);
    const float m_new = mx > m2 + (args.bf16_weights ? 0.f : 8.f) ? mx : m2;
    const float eta = ex2_approx(m2 - m_new);  // 0 on the first block, 1 if unmoved
    // pass 2: p = 2^(s*c - m) with one FFMA; each chunk of 32 keys is
    // written back over its own 32 columns as 16 columns of p_hi pairs and
    // 16 of p_lo pairs (keys 2i, 2i+1 share a column).
    float rs = 0.f;
    auto expo = [&](const uint32_t (&r)[32], int cc) {
      float p[32];
      uint32_t hl[32];  // the chunk's 32 columns: 16 of p_hi pairs, then 16 of p_lo
      if (kvalid >= KB) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          p[i] = ex2_approx(fmaf(__uint_as_float(r[i]), c, -m_new));
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          p[i] = cc * 32 + i < kvalid ? ex2_approx(fmaf(__uint_as_float(r[i]), c, -m_new))
                                      : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        rs += p[2 * i] + p[2 * i + 1];
        hl[i] = pack_bf16x2(p[2 * i], p[2 * i + 1]);
        hl[16 + i] = pack_bf16x2(p[2 * i] - bf16_lo(hl[i]), p[2 * i + 1] - bf16_hi(hl[i]));
      }
      tmem_st_32x32b_x32(tS + cc * 32, hl);  // one store for both halves
    };
    expo(ra, ch0);
    expo(rb, ch0 + 1);
    l = eta * l + rs;
    m2 = m_new;
    // O is stable: this tile's PV(j - 1) was issued before its S(j), whose
    // completion (the S-ready barrier above) covers every earlier MMA
    if (j > 0) {
      if (__any_sync(0xffffffffu, eta != 1.0f)) {
        // this range's O columns
        constexpr int OCH = DH / 32 / SPLIT;
        if constexpr (OCH == 1) {
          uint32_t ra[32];
          tmem_ld_32x32b_x32(tO + h * 32, ra);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ra[i] = __float_as_uint(__uint_as_float(ra[i]) * eta);
          tmem_st_32x32b_x32(tO + h * 32, ra);
        } else {
#pragma unroll 1
          for (int cc = h * OCH; cc < (h + 1) * OCH; cc += 2) {
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
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bars->p_full[t]);
  }
  if (ok && nb > 0) {
    float ls[SPLIT];
    // the tile's last PV product (the only one with a completion barrier)
    if (!mbar_wait(&bars->pv_done[t], 0, abort_flag, args.timeout_ns)) {
      if (lane == 0) record_error(args.err, 1, kWhere + 3, nb, t * 8 + h * 4 + q);
      bars->abort_flag = 1;
    } else if (!exchange<SPLIT>(xslots(nb & 1), h, l, xb, nb & 1, ls, abort_flag,
                                args.timeout_ns)) {
      if (lane == 0) record_error(args.err, 1, kWhere + 6, nb, t * 8 + h * 4 + q);
      bars->abort_flag = 1;
    } else {
      // the ranges' sums, added in range order in every warp of the row
      float lt = ls[0];
#pragma unroll
      for (int i = 1; i < SPLIT; ++i) lt += ls[i];
      tc_fence_after();
      const int tok = q0 + t * BQ + row;
      if (slot >= 0) {
        // a key range of a split unit: unnormalised z, and (m, l), FP32
        float* zs = args.part + static_cast<size_t>(slot) * PartSlot<NT>::FLOATS;
        float* zr = zs + static_cast<size_t>(t * BQ + row) * DH;
        constexpr int OCH = DH / 32 / SPLIT;
#pragma unroll 1
        for (int cc = h * OCH; cc < (h + 1) * OCH; ++cc) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tO + cc * 32, r);
          tmem_wait_ld();
          float4* z4 = reinterpret_cast<float4*>(zr + cc * 32);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            z4[u] = make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3]));
        }
        if (h == 0) {
          float* ml = zs + static_cast<size_t>(PartSlot<NT>::ROWS) * DH + 2 * (t * BQ + row);
          ml[0] = m2;
          ml[1] = lt;
        }
      } else {
      uint16_t* orow =
          args.O + head * args.o_ld_head + static_cast<int64_t>(tok) * args.o_ld_token;
      constexpr int OCH = DH / 32 / SPLIT;
#pragma unroll 1
      for (int cc = h * OCH; cc < (h + 1) * OCH; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tO + cc * 32, r);
        tmem_wait_ld();
        if (tok < args.Nq) {
          uint4* o4 = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __fdiv_rn(__uint_as_float(r[8 * u + i]), lt);
            o4[u] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                               pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
          }
        }
      }
      }
    }
  }
}

// The softmax role of one warp for 256-key blocks (one query tile, two
// 128-key sub-tiles per block, four warps per TMEM lane quarter): warp h
// owns chunk h of each sub-tile (keys 32h.. and 128 + 32h..) and O columns
// [32h, 32h + 32).  Each sub-tile has its own S-ready and P-ready barrier,
// and sub-tile 0's weights (in the columns after O) are published first, so
// its PV product (and the next block's scores for it) run on the tensor
// core while sub-tile 1's weights are formed.  The extremum and row-sum
// exchanges are those of the 128-key role.
template <int NT, int SPLIT, class Bars>
__device__ __forceinline__ void softmax_role_sub(Bars* bars, uint8_t* smem, int off_x, uint32_t tmem,
                                             uint32_t tile_cols, int warp, int lane,
                                             const AttnArgs& args, int nb, int jb0, int slot,
                                             int head, int q0, volatile int* abort_flag) {
  constexpr int KB = 2 * SUB;
  constexpr int kWhere = KID_ATTN * 16;
  const int e = warp - 2;
  constexpr int t = 0;                     // the query tile
  const int h = e / 4;                     // key range
  const int q = warp & 3;                  // TMEM lane quarter
  const int row = q * 32 + lane;           // query row within the tile
  const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
  const uint32_t tS = tmem + (tile_cols * static_cast<uint32_t>(t)) + lane_off;
  const uint32_t tO = tmem + (tile_cols * static_cast<uint32_t>(t) + KB) + lane_off;
  static_assert(NT == 1 && SPLIT == 4, "one tile, four warps per lane quarter");
  const int c0 = h, c1 = 4 + h;            // this warp's chunks of a block
  float* xbase = reinterpret_cast<float*>(smem + off_x);
  uint64_t* xb = &bars->xbar[t][q];
  auto xslots = [&](int par) { return xbase + ((par * NT + t) * SPLIT) * 128 + row; };
  float m2 = -INFINITY;  // running max, log2 units
  float l = 0.f;         // running sum of this range's weights
  bool ok = true;
  // P of sub-tile 0 goes to the 128 columns after O, so that S of sub-tile
  // 0 stays readable until the block's reference point is known
  const uint32_t tP0 = tmem + tile_cols + lane_off;
  const float c = args.scale_log2;  // scale * log2(e)
  for (int j = 0; j < nb; ++j) {
    if (!mbar_wait(&bars->s_full[0], j & 1, abort_flag, args.timeout_ns)) {
      if (lane == 0) record_error(args.err, 1, kWhere + 2, j, h * 4 + q);
      bars->abort_flag = 1;
      ok = false;
      break;
    }
    tc_fence_after();
    const int kvalid = args.Nk - (jb0 + j) * KB;  // keys of this block that exist
    // S(j, u) is issued after PV(j - 1, u), so once it is complete K(j, u)
    // and V(j - 1, u) are free: one thread hands both stages back to the
    // producer (here for sub-tile 0, below for sub-tile 1), and the MMA
    // issuer commits no barrier for them
    const bool relay = e == 0 && lane == 0;
    if (relay) {
      mbar_arrive(&bars->k_empty[(2 * j) % 3]);
      if (j > 0) mbar_arrive(&bars->v_empty[0]);
    }
    // pass 1: row extremum of this range's raw scores (max, or min for a
    // negative scale), then the other ranges' through shared memory
    float ext = c >= 0.f ? -INFINITY : INFINITY;
    auto scan = [&](const uint32_t (&r)[32], int base) {
      if (kvalid >= KB) {
        if (c >= 0.f) {
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            ext = max3f(ext, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            ext = min3f(ext, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (base + i < kvalid)
            ext = c >= 0.f ? fmaxf(ext, __uint_as_float(r[i])) : fminf(ext, __uint_as_float(r[i]));
      }
    };
    // pass 2: p = 2^(s*c - m) with one FFMA; each chunk of 32 keys goes to
    // 32 columns at `dst` as 16 columns of p_hi pairs and 16 of p_lo pairs
    // (keys 2i, 2i+1 share a column); `rs` gets the chunk's sum
    auto expo = [&](const uint32_t (&r)[32], int cc, uint32_t dst, float m, float& rs) {
      float p[32];
      uint32_t hi[16], lo[16];
      if (kvalid >= KB) {
#pragma unroll
        for (int i = 0; i < 32; ++i) p[i] = ex2_approx(fmaf(__uint_as_float(r[i]), c, -m));
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          p[i] = cc * 32 + i < kvalid ? ex2_approx(fmaf(__uint_as_float(r[i]), c, -m)) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        rs += p[2 * i] + p[2 * i + 1];
        hi[i] = pack_bf16x2(p[2 * i], p[2 * i + 1]);
        lo[i] = pack_bf16x2(p[2 * i] - bf16_lo(hi[i]), p[2 * i + 1] - bf16_hi(hi[i]));
      }
      tmem_st_32x32b_x16(dst, hi);
      tmem_st_32x32b_x16(dst + 16, lo);
    };
    // Sub-tile 0 is scanned while sub-tile 1's scores are computed.  With
    // the lagging reference point (below) the reference rarely moves after
    // the first block, so sub-tile 0's weights are formed against the
    // current one meanwhile and the row exchange only confirms them; where
    // it moves a row of the warp, the warp forms them again from S.
    const bool speculate = j > 0 && !args.bf16_weights;
    float rs0 = 0.f, rs1 = 0.f;
    {
      uint32_t ra[32];
      tmem_ld_32x32b_x32(tS + c0 * 32, ra);
      tmem_wait_ld();
      scan(ra, c0 * 32);
      if (speculate) expo(ra, c0, tP0 + c0 * 32, m2, rs0);
    }
    if (!mbar_wait(&bars->s_full[1], j & 1, abort_flag, args.timeout_ns)) {
      if (lane == 0) record_error(args.err, 1, kWhere + 2, j, 64 + h * 4 + q);
      bars->abort_flag = 1;
      ok = false;
      break;
    }
    tc_fence_after();
    if (relay) {
      if (kvalid > SUB) mbar_arrive(&bars->k_empty[(2 * j + 1) % 3]);  // K(j, 1) exists
      if (j > 0) mbar_arrive(&bars->v_empty[1]);
    }
    uint32_t rb[32];
    tmem_ld_32x32b_x32(tS + c1 * 32, rb);
    tmem_wait_ld();
    scan(rb, c1 * 32);
    float others[SPLIT];
    if (!exchange<SPLIT>(xslots(j & 1), h, ext, xb, j & 1, others, abort_flag,
                         args.timeout_ns)) {
      if (lane == 0) record_error(args.err, 1, kWhere + 6, j, h * 4 + q);
      bars->abort_flag = 1;
      ok = false;
      break;
    }
#pragma unroll
    for (int i = 0; i < SPLIT; ++i)
      ext = c >= 0.f ? fmaxf(ext, others[i]) : fminf(ext, others[i]);
    // reference point of the exponents: moved only when the running max
    // exceeds it by more than 2^8 (the weights then stay below 2^8 and O is
    // rescaled rarely); z and l are scaled alike, so z / l is unchanged.
    // The BF16-weights variant keeps the exact running max: its rounded
    // weights depend on the reference point.
    const float mx = fmaxf(m2, ext * c);
    const float m_new = mx > m2 + (args.bf16_weights ? 0.f : 8.f) ? mx : m2;
    const float eta = ex2_approx(m2 - m_new);  // 0 on the first block, 1 if unmoved
    if (!speculate || __any_sync(0xffffffffu, m_new != m2)) {
      if (speculate) tmem_wait_st();  // the first stores land before they are replaced
      uint32_t ra[32];
      tmem_ld_32x32b_x32(tS + c0 * 32, ra);
      tmem_wait_ld();
      rs0 = 0.f;
      expo(ra, c0, tP0 + c0 * 32, m_new, rs0);
    }
    // O is stable: PV(j - 1, 1) was issued before S(j, 1), whose completion
    // (the S-ready barrier above) covers every earlier MMA
    if (j > 0) {
      if (__any_sync(0xffffffffu, eta != 1.0f)) {  // this range's O columns
        uint32_t r[32];
        tmem_ld_32x32b_x32(tO + h * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * eta);
        tmem_st_32x32b_x32(tO + h * 32, r);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bars->p_full[0]);  // sub-tile 0's weights (and the rescaled O)
    expo(rb, c1, tS + c1 * 32, m_new, rs1);  // over sub-tile 1's S
    l = eta * l + (rs0 + rs1);
    m2 = m_new;
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bars->p_full[1]);
  }
  if (ok && nb > 0) {
    float ls[SPLIT];
    // the last PV product (the only one with a completion barrier)
    if (!mbar_wait(&bars->pv_done[t], 0, abort_flag, args.timeout_ns)) {
      if (lane == 0) record_error(args.err, 1, kWhere + 3, nb, t * 8 + h * 4 + q);
      bars->abort_flag = 1;
    } else if (!exchange<SPLIT>(xslots(nb & 1), h, l, xb, nb & 1, ls, abort_flag,
                                args.timeout_ns)) {
      if (lane == 0) record_error(args.err, 1, kWhere + 6, nb, t * 8 + h * 4 + q);
      bars->abort_flag = 1;
    } else {
      // the ranges' sums, added in range order in every warp of the row
      float lt = ls[0];
#pragma unroll
      for (int i = 1; i < SPLIT; ++i) lt += ls[i];
      tc_fence_after();
      const int tok = q0 + t * BQ + row;
      if (slot >= 0) {
        // a key range of a split unit: unnormalised z, and (m, l), FP32
        float* zs = args.part + static_cast<size_t>(slot) * PartSlot<NT>::FLOATS;
        float* zr = zs + static_cast<size_t>(t * BQ + row) * DH;
        constexpr int OCH = DH / 32 / SPLIT;
#pragma unroll 1
        for (int cc = h * OCH; cc < (h + 1) * OCH; ++cc) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tO + cc * 32, r);
          tmem_wait_ld();
          float4* z4 = reinterpret_cast<float4*>(zr + cc * 32);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            z4[u] = make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3]));
        }
        if (h == 0) {
          float* ml = zs + static_cast<size_t>(PartSlot<NT>::ROWS) * DH + 2 * (t * BQ + row);
          ml[0] = m2;
          ml[1] = lt;
        }
      } else {
      uint16_t* orow =
          args.O + head * args.o_ld_head + static_cast<int64_t>(tok) * args.o_ld_token;
      constexpr int OCH = DH / 32 / SPLIT;
#pragma unroll 1
      for (int cc = h * OCH; cc < (h + 1) * OCH; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tO + cc * 32, r);
        tmem_wait_ld();
        if (tok < args.Nq) {
          uint4* o4 = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __fdiv_rn(__uint_as_float(r[8 * u + i]), lt);
            o4[u] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                               pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
          }
        }
      }
      }
    }
  }
}

template <int KSUB>
__global__ void __launch_bounds__(AShape<KSUB>::kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const View vq, const View vk,
                const View vv, const AttnArgs args) {
  using A = AShape<KSUB>;
  constexpr int NT = A::NT;
  constexpr int KB = A::KB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  ABars* bars = reinterpret_cast<ABars*>(smem + A::OFF_BAR);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q_blocks = (args.Nq + NT * BQ - 1) / (NT * BQ);
  const int nsub = (args.Nk + SUB - 1) / SUB;  // K/V sub-tiles
  const int nb_all = (args.Nk + KB - 1) / KB;  // online-softmax key blocks
  // this CTA's unit and key-block range [jb0, jb0 + nb)
  int unit = blockIdx.x, jb0 = 0, nb = nb_all, slot = -1;
  if (args.pieces > 0 && static_cast<int>(blockIdx.x) >= args.units_full) {
    slot = blockIdx.x - args.units_full;
    unit = args.units_full + slot / args.pieces;
    const int piece = slot % args.pieces;
    jb0 = piece * nb_all / args.pieces;
    nb = (piece + 1) * nb_all / args.pieces - jb0;
  }
  const int head = unit / q_blocks;
  const int q0 = (unit % q_blocks) * (NT * BQ);
  const int js0 = jb0 * KSUB;                  // first sub-tile of the range
  volatile int* abort_flag = &bars->abort_flag;
  constexpr int kWhere = KID_ATTN * 16;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      if (s == 0 && A::KSTAGES == 3) mbar_init(&bars->k_empty[2], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    if constexpr (KSUB == 2) {  // one tile: S-ready and P-ready per sub-tile
      mbar_init(&bars->s_full[1], 1);
      mbar_init(&bars->p_full[1], 128 * A::SPLIT);
    }
    for (int t = 0; t < NT; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 128 * A::SPLIT);
      mbar_init(&bars->pv_done[t], 1);
      for (int qq = 0; qq < 4; ++qq) mbar_init(&bars->xbar[t][qq], 32 * A::SPLIT);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, A::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    // Q once; then per key block its K sub-tiles, then its V sub-tiles
    // (sub-tile js lives in ring stage js & 1)
    if (lane == 0) {
      uint32_t k_armed = 0, v_armed = 0;  // per-stage parity of the last arming
      int k_cnt[2] = {0, 0}, v_cnt[2] = {0, 0};
      mbar_arrive_expect_tx(&bars->q_full, NT * 2 * TILE64);
      for (int t = 0; t < NT; ++t)
        for (int cb = 0; cb < 2; ++cb)
          tma_load_2d(smem + A::OFF_Q + (t * 2 + cb) * TILE64, &tmQ, &bars->q_full,
                      head * vq.hx + cb * 64, head * vq.hy + q0 + t * BQ);
      bool ok = true;
      // sub-tile js of the range (128 keys) into ring stage `stage` at `off`
      auto load_kv = [&](const CUtensorMap* m, const View& vw, int off, int stage, int js,
                         uint64_t* full) {
        uint8_t* dst = smem + off + stage * 2 * TILE64;
        const int key0 = (js0 + js) * SUB;
        tma_load_2d(dst, m, full, head * vw.hx, head * vw.hy + key0);
        tma_load_2d(dst + TILE64, m, full, head * vw.hx + 64, head * vw.hy + key0);
      };
      if constexpr (KSUB == 1) {
        // K(0) on k_full[0]; then per block j, V(j) and K(j+1) together on
        // v_full[j & 1], so the MMA issuer waits once per block for both
        if (nb > 0) {
          mbar_arrive_expect_tx(&bars->k_full[0], 2 * TILE64);
          load_kv(&tmK, vk, A::OFF_K, 0, 0, &bars->k_full[0]);
          k_cnt[0] = 1;
        }
        for (int j = 0; j < nb && ok; ++j) {
          const int sv = j & 1, sk = (j + 1) & 1;
          const bool knext = j + 1 < nb;
          if (!mbar_wait(&bars->v_empty[sv], ((j >> 1) & 1) ^ 1, abort_flag, args.timeout_ns) ||
              (knext && !mbar_wait(&bars->k_empty[sk], (((j + 1) >> 1) & 1) ^ 1, abort_flag,
                                   args.timeout_ns))) {
            record_error(args.err, 1, kWhere + 0, j, 2);
            bars->abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->v_full[sv], (knext ? 4 : 2) * TILE64);
          load_kv(&tmV, vv, A::OFF_V, sv, j, &bars->v_full[sv]);
          if (knext) load_kv(&tmK, vk, A::OFF_K, sk, j + 1, &bars->v_full[sv]);
          v_armed = (v_armed & ~(1u << sv)) | (static_cast<uint32_t>(v_cnt[sv] & 1) << sv);
          ++v_cnt[sv];
        }
      } else {
        // 256-key blocks: K of block 0's sub-tiles on k_full[u]; then, per
        // sub-tile u of block j, V(j, u) and K(j + 1, u) together on
        // v_full[u].  K sub-tile js lives in stage js % 3, V sub-tile js in
        // stage js & 1 (= u).
        for (int u = 0; u < KSUB; ++u) {
          if (js0 + u >= nsub) break;
          mbar_arrive_expect_tx(&bars->k_full[u], 2 * TILE64);
          load_kv(&tmK, vk, A::OFF_K, u, u, &bars->k_full[u]);
          k_cnt[u] = 1;
        }
        for (int j = 0; j < nb && ok; ++j) {
          for (int u = 0; u < KSUB && ok; ++u) {
            const int js = j * KSUB + u;
            if (js0 + js >= nsub) break;
            const int kn = js + KSUB, sk = kn % 3;
            const bool knext = j + 1 < nb && js0 + kn < nsub;
            if (!mbar_wait(&bars->v_empty[u], (j & 1) ^ 1, abort_flag, args.timeout_ns) ||
                (knext && !mbar_wait(&bars->k_empty[sk], ((kn / 3) & 1) ^ 1, abort_flag,
                                     args.timeout_ns))) {
              record_error(args.err, 1, kWhere + 0, js, 2);
              bars->abort_flag = 1;
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars->v_full[u], (knext ? 4 : 2) * TILE64);
            load_kv(&tmV, vv, A::OFF_V, u, js, &bars->v_full[u]);
            if (knext) load_kv(&tmK, vk, A::OFF_K, sk, kn, &bars->v_full[u]);
            v_armed = (v_armed & ~(1u << u)) | (static_cast<uint32_t>(v_cnt[u] & 1) << u);
            ++v_cnt[u];
          }
        }
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
      // Shared-memory descriptors are formed once: the start-address field
      // holds address / 16 in its low 14 bits, and every operand lies below
      // 256 KB, so the descriptor of base + off is the base's descriptor +
      // off / 16.  The tensor core queues about one instruction, so the
      // issue loops keep only that addition between MMAs.
      const uint64_t dq0 = sdesc_sw128(smem_u32(smem + A::OFF_Q), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(smem + A::OFF_K), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(smem + A::OFF_V), TILE64, 1024);
      // S_t = Q_t K^T for the sub-tiles of key block j, into tile t's S columns
      auto issue_s = [&](int j, int t) {
        const uint64_t dq = dq0 + static_cast<uint64_t>((t * 2 * TILE64) >> 4);
        for (int u = 0; u < KSUB; ++u) {
          const int js = j * KSUB + u;
          if (js0 + js >= nsub) break;
          const int s = js & 1;
          // with one 128-key sub-tile per block, K(j) for j > 0 arrived with
          // V(j - 1), whose barrier the PV MMAs of block j - 1 waited for
          if (t == 0 && (KSUB != 1 || j == 0)) {
            if (!mbar_wait(&bars->k_full[s], (js >> 1) & 1, abort_flag, args.timeout_ns)) {
              fail(js, 0);
              return;
            }
            tc_fence_after();
          }
          const uint64_t dk = dk0 + static_cast<uint64_t>((s * 2 * TILE64) >> 4);
          const uint32_t d_tm = tmem + A::tm_s(t) + SUB * u;
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * TILE64 + (kk & 3) * 32) >> 4;
            mma_bf16_ss(d_tm, dq + off, dk + off, idesc_s, kk > 0 ? 1u : 0u);
          }
          issued = true;  // K(j) is handed back by the softmax role (S-ready)
        }
        mma_commit(&bars->s_full[t]);
      };
      if (!mbar_wait(&bars->q_full, 0, abort_flag, args.timeout_ns)) fail(-1, 2);
      if constexpr (KSUB == 2) {
        // one tile; per sub-tile u of block j: wait for its weights, O +=
        // P_hi V + P_lo V over it, then the next block's scores for u (they
        // overwrite its P after the PV MMAs, which the tensor core executes
        // first)
        auto issue_sub = [&](int j, int u) {
          const int js = j * KSUB + u;
          if (js0 + js < nsub) {
            // K of block j > 0 arrived with V of block j - 1, whose barrier
            // the PV MMAs of that sub-tile waited for
            const int s = js % 3;
            if (j == 0) {
              if (!mbar_wait(&bars->k_full[u], 0, abort_flag, args.timeout_ns)) {
                fail(js, 0);
                return;
              }
              tc_fence_after();
            }
            const uint64_t dk = dk0 + static_cast<uint64_t>((s * 2 * TILE64) >> 4);
            const uint32_t d_tm = tmem + A::tm_s(0) + SUB * u;
#pragma unroll
            for (int kk = 0; kk < DH / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * TILE64 + (kk & 3) * 32) >> 4;
              mma_bf16_ss(d_tm, dq0 + off, dk + off, idesc_s, kk > 0 ? 1u : 0u);
            }
            issued = true;  // K(j, u) is handed back by the softmax role
          }
          mma_commit(&bars->s_full[u]);  // also when the sub-tile is past the keys
        };
        for (int u = 0; u < KSUB && ok; ++u) issue_sub(0, u);
        for (int j = 0; j < nb && ok; ++j) {
          for (int u = 0; u < KSUB && ok; ++u) {
            if (!mbar_wait(&bars->p_full[u], j & 1, abort_flag, args.timeout_ns)) {
              fail(j, 3);
              break;
            }
            tc_fence_after();
            const int js = j * KSUB + u;
            if (js0 + js < nsub) {
              const int s = js & 1;
              if (!mbar_wait(&bars->v_full[s], (js >> 1) & 1, abort_flag, args.timeout_ns)) {
                fail(js, 4);
                break;
              }
              tc_fence_after();
              const uint64_t dv = dv0 + static_cast<uint64_t>((s * 2 * TILE64) >> 4);
              const int halves = args.bf16_weights ? 1 : 2;  // p_hi (and p_lo)
              // sub-tile 0's P is in the columns after O, sub-tile 1's over its S
              const uint32_t pbase = tmem + (u == 0 ? A::TILE_COLS : SUB);
              const uint32_t o_tm = tmem + A::tm_o(0);
              const uint32_t first = (j | u) != 0 ? 1u : 0u;
              // both halves unrolled: one straight run of MMAs for the issuer
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                if (half == halves) break;
#pragma unroll
                for (int kk = 0; kk < SUB / 16; ++kk) {
                  const uint32_t pcol = 32 * (kk >> 1) + 8 * (kk & 1) + 16 * half;
                  mma_bf16_ts(o_tm, pbase + pcol, dv + ((kk * 2048) >> 4), idesc_o,
                              (half | kk) != 0 ? 1u : first);
                }
              }
            }
            // V(j, u) is handed back by the softmax role once S(j + 1, u) is
            // complete, which also tells it that this PV is; only the last
            // block's PV gets a barrier of its own
            if (u == KSUB - 1 && j == nb - 1) mma_commit(&bars->pv_done[0]);
            if (j + 1 < nb) issue_sub(j + 1, u);
          }
        }
      } else {
        // two tiles of 128-key blocks (one sub-tile per block, every block of
        // the range exists).  Per block and tile: wait for P, the PV run,
        // then the tile's next scores, with every operand address formed
        // before the waits, so the issuer runs no bookkeeping between MMA
        // runs while the softmax warps keep its SM sub-partition busy.
        static_assert(KSUB == 1, "the two-tile kernel takes 128-key blocks");
        for (int t = 0; t < NT && ok; ++t) issue_s(0, t);
        const int halves = args.bf16_weights ? 1 : 2;  // p_hi (and p_lo)
        for (int j = 0; j < nb && ok; ++j) {
          const uint64_t dv = dv0 + static_cast<uint64_t>(((j & 1) * 2 * TILE64) >> 4);
          const uint64_t dkn = dk0 + static_cast<uint64_t>((((j + 1) & 1) * 2 * TILE64) >> 4);
          const bool next = j + 1 < nb;
          const uint32_t first = j != 0 ? 1u : 0u;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (!mbar_wait(&bars->p_full[t], j & 1, abort_flag, args.timeout_ns)) {
              fail(j, 3);
              break;
            }
            tc_fence_after();
            if (t == 0) {
              // V(j), and K(j + 1) with it
              if (!mbar_wait(&bars->v_full[j & 1], (j >> 1) & 1, abort_flag, args.timeout_ns)) {
                fail(j, 4);
                break;
              }
              tc_fence_after();
            }
            // O_t += P_hi V + P_lo V: P from tensor memory (keys 16kk.. at
            // column 32(kk/2) + 8(kk%2), lo 16 further), V rows 16kk.. of
            // both 64-wide dh blocks; both halves as one unrolled run
            const uint32_t pbase = tmem + A::tm_s(t);
            const uint32_t o_tm = tmem + A::tm_o(t);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              if (half == halves) break;
#pragma unroll
              for (int kk = 0; kk < SUB / 16; ++kk) {
                const uint32_t pcol = 32 * (kk >> 1) + 8 * (kk & 1) + 16 * half;
                mma_bf16_ts(o_tm, pbase + pcol, dv + ((kk * 2048) >> 4), idesc_o,
                            (half | kk) != 0 ? 1u : first);
              }
            }
            if (!next) {
              // the softmax learns that PV(j) is complete from S(j + 1)'s
              // barrier; only the last block's PV gets a barrier of its own
              mma_commit(&bars->pv_done[t]);
              continue;
            }
            // tile t's next scores overwrite its P: the tensor core runs them
            // after its PV MMAs.  K(j + 1) and V(j) are handed back to the
            // producer by the softmax role when it sees these scores.
            const uint64_t dq = dq0 + static_cast<uint64_t>((t * 2 * TILE64) >> 4);
            const uint32_t d_tm = tmem + A::tm_s(t);
#pragma unroll
            for (int kk = 0; kk < DH / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * TILE64 + (kk & 3) * 32) >> 4;
              mma_bf16_ss(d_tm, dq + off, dkn + off, idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bars->s_full[t]);
          }
        }
      }
      if (issued) {
        mma_commit(&bars->drain);
        int dummy = 0;
        if (!mbar_wait(&bars->drain, 0, &dummy, args.timeout_ns))
          record_error(args.err, 1, kWhere + 5, 0, 0);
      }
    }
  } else {
    if constexpr (KSUB == 2)
      softmax_role_sub<NT, A::SPLIT>(bars, smem, A::OFF_X, tmem, A::TILE_COLS, warp, lane, args,
                                     nb, jb0, slot, head, q0, abort_flag);
    else
      softmax_role<KSUB, NT, A::SPLIT>(bars, smem, A::OFF_X, tmem, A::TILE_COLS, warp, lane,
                                       args, nb, jb0, slot, head, q0, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, A::TM_COLS);
  }
}

// Combine the key ranges of each split unit: one warp per query row, four
// output columns per lane; ranges in their order, FP32.
template <int NT>
__global__ void __launch_bounds__(256) merge_kernel(const AttnArgs a, int q_blocks,
                                                    int n_tail) {
  constexpr int ROWS = PartSlot<NT>::ROWS;
  const int wg = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int u = wg / ROWS, row = wg % ROWS;
  if (u >= n_tail) return;
  const int unit = a.units_full + u;
  const int head = unit / q_blocks;
  const int tok = (unit % q_blocks) * ROWS + row;
  if (tok >= a.Nq) return;
  const float* base = a.part + static_cast<size_t>(u) * a.pieces * PartSlot<NT>::FLOATS;
  // the ranges' (m, l) are read one per lane (32 ranges at a time); the
  // maximum, the weights and the sum are formed across the warp in a fixed
  // order; every lane then accumulates its four columns of z
  float M = -INFINITY;
  for (int r0 = 0; r0 < a.pieces; r0 += 32) {
    const int r = r0 + lane;
    if (r < a.pieces) M = fmaxf(M, base[r * PartSlot<NT>::FLOATS + ROWS * DH + 2 * row]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float l = 0.f, z[4] = {0.f, 0.f, 0.f, 0.f};
  for (int r0 = 0; r0 < a.pieces; r0 += 32) {
    const int r = r0 + lane;
    float w = 0.f, wl = 0.f;
    if (r < a.pieces) {
      const float* ml = base + r * PartSlot<NT>::FLOATS + ROWS * DH + 2 * row;
      w = exp2f(ml[0] - M);
      wl = w * ml[1];
    }
    const int n = min(32, a.pieces - r0);
#pragma unroll 8
    for (int k = 0; k < n; ++k) {
      const float wk = __shfl_sync(0xffffffffu, w, k);
      l += __shfl_sync(0xffffffffu, wl, k);
      const float4 zv = *reinterpret_cast<const float4*>(
          base + (r0 + k) * PartSlot<NT>::FLOATS + row * DH + 4 * lane);
      z[0] = fmaf(wk, zv.x, z[0]);
      z[1] = fmaf(wk, zv.y, z[1]);
      z[2] = fmaf(wk, zv.z, z[2]);
      z[3] = fmaf(wk, zv.w, z[3]);
    }
  }
  uint16_t* orow = a.O + head * a.o_ld_head + static_cast<int64_t>(tok) * a.o_ld_token;
  *reinterpret_cast<uint2*>(orow + 4 * lane) =
      make_uint2(pack_bf16x2(__fdiv_rn(z[0], l), __fdiv_rn(z[1], l)),
                 pack_bf16x2(__fdiv_rn(z[2], l), __fdiv_rn(z[3], l)));
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

template <int KSUB>
psi_status launch_k(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                    const View& vq, const View& vk, const View& vv, const AttnArgs& a,
                    cudaStream_t stream) {
  using A = AShape<KSUB>;
  static std::atomic<uint64_t> attr_done{0};
  psi_status st = ensure_smem_attr(&attr_done, reinterpret_cast<const void*>(attn_kernel<KSUB>),
                                   A::SMEM_BYTES, "cudaFuncSetAttribute(attn)");
  if (st != PSI_OK) return st;
  const int q_blocks = (a.Nq + A::NT * BQ - 1) / (A::NT * BQ);
  const long long units = static_cast<long long>(q_blocks) * a.heads;
  if (units <= 0) return PSI_OK;
  if (units > 0x3FFFFFFFLL) return set_error(PSI_ERR_UNSUPPORTED, "attention: grid too large");
  // one CTA per SM: split the units of a partial last wave into key ranges
  AttnArgs g = a;
  g.units_full = static_cast<int32_t>(units);
  g.pieces = 0;
  int n_tail = 0;
  const int sms = num_sms();
  const int nb = (a.Nk + A::KB - 1) / A::KB;
  if (a.part && !a.bf16_weights && units > sms && units % sms) {
    const int tail = static_cast<int>(units % sms);
    const int pieces = std::min(nb, sms / tail);
    if (pieces >= 2) {
      n_tail = tail;
      g.units_full = static_cast<int32_t>(units - tail);
      g.pieces = pieces;
    }
  }
  const long long grid = g.units_full + static_cast<long long>(n_tail) * g.pieces;
  attn_kernel<KSUB><<<static_cast<unsigned>(grid), A::kThreads, A::SMEM_BYTES, stream>>>(
      mq, mk, mv, vq, vk, vv, g);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "attention launch");
  count_launch();
  if (n_tail) {
    const int warps = n_tail * PartSlot<A::NT>::ROWS;
    merge_kernel<A::NT><<<(warps + 7) / 8, 256, 0, stream>>>(g, q_blocks, n_tail);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "attention merge launch");
    count_launch();
  }
  return PSI_OK;
}

}  // namespace

size_t attention_workspace_bytes(int key_block) {
  const size_t per = key_block == 128 ? PartSlot<AShape<1>::NT>::FLOATS
                                      : PartSlot<AShape<2>::NT>::FLOATS;
  return per * sizeof(float) * static_cast<size_t>(num_sms());
}

psi_status launch_attention(const psi_heads* Q, const psi_heads* K, const psi_heads* V,
                            const AttnArgs& a, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  View vq, vk, vv;
  psi_status st = make_view(Q, a.heads, a.Nq, &mq, &vq);
  if (st != PSI_OK) return st;
  if ((st = make_view(K, a.heads, a.Nk, &mk, &vk)) != PSI_OK) return st;
  if ((st = make_view(V, a.heads, a.Nk, &mv, &vv)) != PSI_OK) return st;
  if (a.key_block == 128) return launch_k<1>(mq, mk, mv, vq, vk, vv, a, stream);
  if (a.key_block == 256) return launch_k<2>(mq, mk, mv, vq, vk, vv, a, stream);
  return set_error(PSI_ERR_UNSUPPORTED, "attention: key_block must be 128 or 256");
}

}  // namespace psi
