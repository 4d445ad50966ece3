// internal.h -- declarations shared by the translation units of libpsi.
#pragma once
#include <atomic>
#include <cstdint>
#include <cstddef>
#include <string>
#include <cuda_runtime.h>
#include <cuda.h>
#include "../../include/psi.h"

namespace psi {

// Error record written by kernels (first error wins); lives in device
// memory of the library module (a __device__ variable, not an allocation).
struct DevError {
  int code;   // 0 = none; 1 = bounded wait expired; 2 = bad range
  int where;  // kernel id * 16 + role
  int info0;
  int info1;
};

enum KernelId : int { KID_GEMM = 1, KID_ATTN = 2, KID_NORM = 3 };

// Returns the device address of the error record on the current device.
DevError* dev_error_ptr();
// Copies the record to the host and clears it (synchronous, current device).
cudaError_t dev_error_take(DevError* out);

// thread-local last-error message
psi_status set_error(psi_status s, const std::string& msg);
psi_status cuda_error(cudaError_t e, const char* what);

// The flags each entry point honours; any other bit is refused with
// PSI_ERR_UNSUPPORTED before anything is enqueued.
constexpr uint32_t kFlagsPageStream = PSI_SYNC_COPY;
constexpr uint32_t kFlagsLinear = PSI_RESIDENT | PSI_SYNC_COPY | PSI_BIAS_AFTER_BF16;
constexpr uint32_t kFlagsLinearRope = kFlagsLinear | PSI_ROPE_AFTER_BF16;
constexpr uint32_t kFlagsFfn =
    PSI_RESIDENT | PSI_SYNC_COPY | PSI_BOUNDARY_PREGELU_BF16 | PSI_BIAS_AFTER_BF16;
constexpr uint32_t kFlagsFfnNoAlloc = PSI_RESIDENT | PSI_BOUNDARY_PREGELU_BF16 | PSI_BIAS_AFTER_BF16;
constexpr uint32_t kFlagsAttn = PSI_ATTN_BF16_WEIGHTS;
psi_status check_flags(uint32_t flags, uint32_t allowed, const char* what);

// Hidden slices per FFN down-projection pass (psi_ffn_paged): two slices
// share one FP32 accumulator read-modify-write when there are at least two
// and the slice is a whole number of 64-deep k-blocks, else one.  Fixed by
// the shape, never by the arena, so every FFN entry point sums in the same
// order.
constexpr int64_t kFfnGroupMax = 2;
inline int64_t ffn_group(int64_t S, int64_t sl) { return (S >= 2 && sl % 64 == 0) ? 2 : 1; }

// Tensor maps (driver entry point obtained through the runtime).
// 2-D BF16 tensor [rows x cols] with row stride ld (elements), box
// {box_cols, box_rows}, 128-byte swizzle.
psi_status make_tmap_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                        uint64_t ld, uint32_t box_rows, uint32_t box_cols);
// The same for a BF16 (elem_bytes 2) or FP32 (4) tensor with a 128-, 64-byte
// or no swizzle (swizzle_bytes 128, 64, 0).
psi_status make_tmap_2d_ex(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                           uint64_t ld, uint32_t box_rows, uint32_t box_cols, int elem_bytes,
                           int swizzle_bytes);
int num_sms();
// Count one kernel launch (psi_kernel_launches).
void count_launch();
// Raise `fn`'s dynamic shared-memory limit to `bytes` on the current device,
// once per device (the attribute belongs to the device context, so a
// process that drives several GPUs sets it on each).  `done` is the call
// site's per-device record (bit d: device d done); safe to call from
// several host threads.
psi_status ensure_smem_attr(std::atomic<uint64_t>* done, const void* fn, int bytes,
                            const char* what);

// ------------------------------------------------------------ page GEMM --
enum Epilogue : int {
  EPI_LINEAR = 0,     // out = B(acc + bias [+ resid])
  EPI_GELU = 1,       // out = B(phi(acc + bias)), optional pre-GELU rounding
  EPI_ACC_STORE = 2,  // accf = acc
  EPI_ACC_ADD = 3,    // accf += acc
  EPI_ACC_FINAL = 4   // out = B(accf + acc + bias [+ resid])
};

struct GemmArgs {
  int32_t M;  // output rows (tokens)
  int32_t N;  // output columns (page rows)
  int32_t K;
  int32_t epi;
  int32_t pregelu;
  int32_t debug_stall;  // test hook: the producer issues no loads, so the
                        // consumers' bounded waits expire (see timeout_ns)
  int32_t k_split;      // k-blocks (of 64) read from the first page; the rest
                        // come from the second page (0: one page)
  int32_t n_split;      // output columns served by the first page; columns from
                        // n_split on come from the second page (0: one page)
  int32_t bias_after_bf16;  // round the FP32 product to BF16 before adding bias
  int32_t rope_dh;          // split RoPE head width (64 or 128); 0: no RoPE
  int32_t rope_cols;        // leading output columns rotated (whole heads)
  int32_t rope_after_bf16;  // round to BF16 before the rotation
  const float* rope_cos;    // [M x rope_ld] FP32 table, row = token, index j < dh/2
  const float* rope_sin;
  int64_t rope_ld;
  const uint16_t* bias;   // [N]
  const uint16_t* resid;  // [M x ldo] or null
  uint16_t* out;          // [M x ldo]
  float* accf;            // [M x ldacc]
  int64_t ldo;
  int64_t ldacc;
  DevError* err;
  uint64_t timeout_ns;
};

// D[M x N] = X[M x K] * P[N x K]^T with the chosen epilogue, on `stream`.
// X and P are BF16 row-major with row strides ldx and ldp (elements).  With
// args.k_split > 0 the K range is split over two pages: columns
// [0, 64*k_split) of P come from P, the rest from P2 (same row stride); with
// args.n_split > 0 the output columns are: rows [0, n_split) of P, then the
// rows of P2 (n_split a multiple of the tile width).
psi_status launch_page_gemm(const void* X, int64_t ldx, const void* P, int64_t ldp,
                            const GemmArgs& args, cudaStream_t stream,
                            const void* P2 = nullptr);
// Whether an M x N page GEMM runs on CTA pairs (256 x 256 tiles); the choice
// depends on the shape only.
bool gemm_use_pair(int64_t M, int64_t N);

// ------------------------------------------------------------ attention --
struct AttnArgs {
  int32_t heads;
  int32_t Nq;
  int32_t Nk;
  int32_t key_block;
  float scale_log2;  // scale * log2(e)
  int32_t bf16_weights;  // numerator with B(p) only (no p_lo correction)
  uint16_t* O;
  int64_t o_ld_token;
  int64_t o_ld_head;
  // tail split: CTAs [0, units_full) take whole (head, query tile) units;
  // the remaining units are cut into `pieces` contiguous key-block ranges,
  // one CTA each, whose unnormalised partial results go to `part` and are
  // combined by the merge kernel (pieces = 0: no split)
  int32_t units_full;
  int32_t pieces;
  float* part;
  DevError* err;
  uint64_t timeout_ns;
};

// Bytes of the tail-split workspace for key_block (128 or 256) on this device.
size_t attention_workspace_bytes(int key_block);

psi_status launch_rmsnorm(const void* X, int64_t ldx, int64_t N, int64_t d, const void* gamma,
                          float eps, void* Y, int64_t ldy, cudaStream_t stream);
psi_status launch_attention(const psi_heads* Q, const psi_heads* K, const psi_heads* V,
                            const AttnArgs& args, cudaStream_t stream);

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per in-kernel wait

}  // namespace psi
