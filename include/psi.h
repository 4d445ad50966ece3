/*
 * psi.h -- C ABI of the paged BF16 operator library (libpsi).
 *
 * Precision-Preserving Subtensor Inference (PSI, arXiv 2611.08023):
 *  - section II-A: a fixed device arena of reusable weight pages; every
 *    library device buffer comes from caller memory (the library itself never
 *    allocates device memory); each page has at most one unreleased slice
 *    request; reuse follows the copy and consumer dependencies; operators
 *    declare their BF16 write boundaries.
 *  - section II-D: page lifecycle free -> filling (H2D copy) -> ready ->
 *    consuming -> free, enforced by stream order and cross-stream events;
 *    release records an event after all uses are enqueued and the next copy
 *    into the page waits for it.
 *  - section II-B Eq.(2): hidden-partitioned FFN, Eqs.(3)-(4): online-softmax
 *    attention over disjoint key tiles.
 *  - section III-A: bias added in FP32 before the only BF16 write; FP32
 *    attention weights.
 *
 * Conventions (all entry points):
 *  - BF16 tensors are row-major arrays of uint16 bit patterns; "dev" pointers
 *    are device addresses, "host" pointers are pinned host addresses.
 *  - Calls enqueue work on the given CUDA streams and return; results are
 *    valid once the stream has finished.  Asynchronous failures (a CUDA error
 *    or an error recorded by a kernel) are returned by psi_sync or
 *    psi_stream_wait.
 *  - The caller owns every buffer.  The library creates only CUDA events, one
 *    auxiliary stream per arena and host-side tensor-map descriptors.
 *  - Errors: a psi_status is returned; psi_last_error() gives a message for
 *    the last failing call of the calling thread.  An argument error enqueues
 *    nothing.
 *  - One arena is used by one host thread at a time.
 */
#ifndef PSI_H
#define PSI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PSI_OK = 0,
  PSI_ERR_INVALID_ARG = 1,  /* null pointer, bad shape, stride or alignment */
  PSI_ERR_CAPACITY = 2,     /* a page or workspace is too small for its tile */
  PSI_ERR_PAGE_BUSY = 3,    /* a second request on an unreleased page */
  PSI_ERR_CUDA = 4,         /* a CUDA runtime or driver call failed */
  PSI_ERR_TIMEOUT = 5,      /* a host wait passed its deadline */
  PSI_ERR_UNSUPPORTED = 6,  /* a shape or flag this build does not handle */
  PSI_ERR_DEVICE = 7        /* a kernel recorded an error (bounded wait expired) */
} psi_status;

/* flags (bitwise or).  Each entry point lists the flags it honours; a call
 * given any other bit fails with PSI_ERR_UNSUPPORTED and enqueues nothing. */
#define PSI_RESIDENT              0x1u /* weights read from dev_resident: no copies */
#define PSI_SYNC_COPY             0x2u /* H2D page copies on the compute stream */
#define PSI_BOUNDARY_PREGELU_BF16 0x4u /* FFN: extra BF16 write of the biased
                                          pre-activation before GELU, the rounding
                                          order of the paper's native prototype
                                          (section III-A) */
#define PSI_BIAS_AFTER_BF16       0x8u /* the paper's baseline variant (section
                                          III-A): the FP32 matrix product is
                                          rounded to BF16 before the bias (and
                                          residual) is added, in every epilogue
                                          that adds a bias */
#define PSI_ATTN_BF16_WEIGHTS     0x10u /* attention: the numerator uses the
                                          exponential weights rounded to BF16
                                          (p_hi only), the baseline variant of
                                          section III-A; the denominator keeps
                                          the FP32 weights */
#define PSI_ROPE_AFTER_BF16       0x20u /* psi_linear_rope_paged: the projection
                                          is rounded to BF16 before the rotation
                                          and rounded again after it (an extra
                                          materialisation, the baseline
                                          variant's RoPE order) */

typedef struct psi_arena psi_arena;

/* A page handed out by psi_page_stream: slot index, request sequence number,
 * device address of the slot and the bytes copied into it. */
typedef struct {
  int32_t slot;
  uint64_t seq;
  void* dev;
  size_t bytes;
} psi_page;

/* Weight of a paged linear layer, W [rows x cols] BF16 row-major (rows =
 * output features, cols = input features, the U layout of Eq.(2)).  Page p
 * holds output rows [p*page_rows, min(rows, (p+1)*page_rows)), which are
 * contiguous in W, so `host` is W itself.  `dev_resident` is a device copy of
 * the same bytes, read instead of streaming when PSI_RESIDENT is given. */
typedef struct {
  const void* host;
  const void* dev_resident;
  int64_t rows;
  int64_t cols;
  int64_t page_rows;
} psi_linear_weight;

/* Weight of a paged FFN (Eq.(2)): U [h x d], V [r x h].  The hidden
 * dimension is cut into slices J of `slice` channels; page J holds U_J
 * ([slice x d], contiguous in U) followed by V_:,J ([r x slice], gathered).
 * `host` is the packed image written by psi_ffn_pack (h/slice pages of
 * psi_ffn_page_bytes each); `dev_resident` is a device copy of that image. */
typedef struct {
  const void* host;
  const void* dev_resident;
  int64_t d;
  int64_t h;
  int64_t r;
  int64_t slice;
} psi_ffn_weight;

/* A BF16 tensor with a head dimension: element (head, token, c) is at
 * ptr[head*ld_head + token*ld_token + c] (strides in elements, c contiguous). */
typedef struct {
  void* ptr;
  int64_t ld_token;
  int64_t ld_head;
} psi_heads;

/* Split RoPE table (section II-B): token n's head pair j (j < dh/2) is
 * rotated by c = cos[n*ld + j], s = sin[n*ld + j] (device FP32; 16-byte
 * aligned, ld % 4 == 0, ld >= dh/2).  The rotation covers the leading `cols`
 * output columns (whole heads of dh = 64 or 128 columns: the query and key
 * heads of a fused QKV projection); later columns pass through. */
typedef struct {
  const float* cos;
  const float* sin;
  int64_t ld;
  int64_t cols;
  int32_t dh;
  int32_t pad_;
} psi_rope;

typedef struct {
  uint64_t pages_streamed;   /* H2D page requests */
  uint64_t h2d_bytes;        /* bytes copied into pages */
  uint64_t resident_pages;   /* pages read from dev_resident */
  uint64_t kernels_launched; /* kernels this arena enqueued */
  uint64_t timed_gemms;      /* page-GEMM launches bracketed by events */
  double gemm_ms;            /* their summed device time */
  double gemm_flops;         /* their summed algorithmic FLOPs (2*M*N*K) */
  uint64_t timed_copies;     /* H2D copies bracketed by events */
  double copy_ms;            /* their summed device time */
  double copy_bytes;
  double gemm_busy_ms;       /* length of the union of the timed page-GEMM
                                intervals (launches on the two streams may
                                overlap, so this can be below gemm_ms) */
  double copy_busy_ms;       /* the same for the timed copies */
} psi_stats;

/* One record of the page timeline (psi_arena_trace_begin/get). */
enum { PSI_TRACE_COPY = 0, PSI_TRACE_GEMM = 1 };
typedef struct {
  int32_t kind;     /* PSI_TRACE_COPY: H2D copy of a page; PSI_TRACE_GEMM: page GEMM */
  int32_t slot;     /* arena slot of the page; -1: a resident page or no arena page */
  int32_t stream;   /* 0 compute stream, 1 the arena's auxiliary stream, 2 copy stream */
  int32_t pad_;
  uint64_t seq;     /* copy: the page request's sequence number; GEMM: launch number */
  double start_ms;  /* from the origin event of psi_arena_trace_begin */
  double end_ms;
  double work;      /* copy: bytes; GEMM: algorithmic FLOPs 2*M*N*K */
} psi_trace_record;

/* ---------------------------------------------------------------- misc -- */
const char* psi_version(void);
const char* psi_status_string(psi_status s);
/* Message of the last failing call on this thread ("" if none). */
const char* psi_last_error(void);

/* ------------------------------------------------------- page plans ----- */
/* Output rows per page of a linear weight [rows x cols] for pages of
 * page_bytes: the largest multiple of 256 (or, below 256 rows, of 16) whose
 * rows fit, capped at `rows`.  PSI_ERR_CAPACITY if not even 16 rows fit
 * (the "weight tile exceeds page" outcome of the capacity study, Table V).
 * The plan depends on the page size only, never on the arena size. */
psi_status psi_plan_linear(int64_t rows, int64_t cols, size_t page_bytes,
                           int64_t* page_rows);

/* Output-column partition for sharding an operator over `parts` devices
 * (the column-partition invariant of section II-B: every output entry still
 * receives its complete dot product from one device, so the gathered
 * columns equal the unpartitioned result bit for bit).  Part `part` of
 * `parts` gets the contiguous columns [*c0, *c1) of [0, cols): boundaries
 * are multiples of `align` (the last part ends at cols), and the parts'
 * widths differ by at most `align`, earlier parts taking the larger ones.
 * A part may be empty (c0 == c1) when cols < parts * align.
 * PSI_ERR_INVALID_ARG for cols < 0, align < 1, parts < 1 or part outside
 * [0, parts).  Host arithmetic only, no CUDA call. */
psi_status psi_plan_columns(int64_t cols, int64_t align, int32_t parts, int32_t part,
                            int64_t* c0, int64_t* c1);

/* Bytes of one FFN page: slice*d*2 + r*slice*2. */
size_t psi_ffn_page_bytes(int64_t d, int64_t r, int64_t slice);

/* Pack U [h x d] and V [r x h] (host BF16) into the page image `dst` (host,
 * h/slice pages of psi_ffn_page_bytes).  h must be a multiple of slice.
 * Runs on host threads; no CUDA call. */
psi_status psi_ffn_pack(const void* U, const void* V, int64_t d, int64_t h,
                        int64_t r, int64_t slice, void* dst);

/* Workspace of psi_ffn_paged: hidden_bytes = 2*2*N*slice*2 (two groups of
 * two BF16 hidden slices, so the next group's up projections never
 * overwrite the group the down projection is reading), acc_bytes = N*r*4
 * (FP32 accumulator). */
psi_status psi_ffn_workspace(int64_t N, int64_t r, int64_t slice,
                             size_t* hidden_bytes, size_t* acc_bytes);

/* ------------------------------------------------------------- arena ---- */
/* Create an arena over caller device memory [dev_base, dev_base+dev_bytes):
 * floor(dev_bytes / page_bytes) page slots (at least 1).  dev_base must be
 * 1024-byte aligned and page_bytes a multiple of 1024.  compute_stream and
 * copy_stream are cudaStream_t handles (they may be equal; NULL is the
 * legacy default stream).  The arena owns events and one auxiliary stream:
 * an operator forks it from the compute stream when it starts, runs some of
 * its page GEMMs on it, and joins it back into the compute stream before it
 * returns, so each operator's work is complete when the compute stream
 * reaches the point after the call. */
psi_status psi_arena_create(void* dev_base, size_t dev_bytes, size_t page_bytes,
                            void* compute_stream, void* copy_stream,
                            psi_arena** out);
/* Waits for the arena's streams, then frees its events. */
psi_status psi_arena_destroy(psi_arena* arena);
int32_t psi_arena_slots(const psi_arena* arena);

/* Request the next slot of the ring and enqueue the H2D copy of
 * host_src[0..bytes) into it.  The copy stream first waits for the slot's
 * last release (its previous consumers); the compute stream then waits for
 * the copy.  With PSI_SYNC_COPY the copy is enqueued on the compute stream
 * instead.  PSI_ERR_PAGE_BUSY if that slot still has an unreleased request,
 * PSI_ERR_CAPACITY if bytes > page_bytes.  Flags: PSI_SYNC_COPY. */
psi_status psi_page_stream(psi_arena* arena, const void* host_src, size_t bytes,
                           uint32_t flags, psi_page* out);
/* End a request: records the slot's consumed event on the compute stream
 * after every use enqueued so far.  PSI_ERR_INVALID_ARG for a stale page. */
psi_status psi_page_release(psi_arena* arena, psi_page page);

/* Poll the arena's streams until both are idle or timeout_ms passes
 * (PSI_ERR_TIMEOUT; timeout_ms < 0 waits without limit), then report any
 * asynchronous CUDA error or kernel-recorded error (PSI_ERR_DEVICE, which
 * is cleared by the report). */
psi_status psi_sync(psi_arena* arena, int64_t timeout_ms);
/* The same for one stream, without an arena. */
psi_status psi_stream_wait(void* stream, int64_t timeout_ms);

psi_status psi_arena_stats(const psi_arena* arena, psi_stats* out);
/* Kernels the library has launched in this process, over every entry point
 * and device (a monotonic count). */
uint64_t psi_kernel_launches(void);
psi_status psi_arena_reset_stats(psi_arena* arena);
/* enable != 0: bracket every page GEMM (compute stream) and every H2D copy
 * (copy stream) with CUDA events; psi_arena_stats sums them (it waits for
 * the events).  Off by default. */
psi_status psi_arena_set_timing(psi_arena* arena, int32_t enable);
/* Page timeline (the lifecycle of section II-D made visible): turn timing on
 * and keep one psi_trace_record per timed page copy and page GEMM, at most
 * `capacity` of them (later ones are dropped), with times measured from an
 * event recorded now on the compute stream.  Drops the records of an
 * earlier trace.  PSI_ERR_INVALID_ARG for a null arena or capacity 0. */
psi_status psi_arena_trace_begin(psi_arena* arena, size_t capacity);
/* Wait for the events of the records taken so far (a host wait) and copy
 * min(capacity, held) of them, ordered by start time, to `out` (host
 * memory, may be null when capacity is 0); *count = records held.  The
 * timing sums of psi_arena_stats include the same launches.
 * PSI_ERR_INVALID_ARG without an active trace or for null arena/count. */
psi_status psi_arena_trace_get(psi_arena* arena, psi_trace_record* out, size_t capacity,
                               size_t* count);
/* Test hook: the next psi_page_stream call on this arena fails with
 * PSI_ERR_CUDA before enqueuing anything (host-side fault injection). */
psi_status psi_arena_fail_next_copy(psi_arena* arena);
/* Test hook: the next page GEMM this process launches gets a producer that
 * issues no copies and in-kernel waits bounded by timeout_ns, so its
 * consumers' waits expire; the kernel records the error, frees its tensor
 * memory and returns (no fault, no hang).  The following psi_sync reports
 * PSI_ERR_DEVICE and the context stays usable.  timeout_ns in (0, 1e10]. */
psi_status psi_debug_stall_next_gemm(uint64_t timeout_ns);

/* ---------------------------------------------------------- operators --- */
/* Paged linear, section IV-B ("projection tiles ... output columns per
 * group"): for each page p, Y[:, rows_p] = B(X W_p^T + b_p [+ R[:, rows_p]]),
 * FP32 accumulation over all of K, bias (and residual) added in FP32 before
 * the single BF16 write.
 *   X    dev [N x K] BF16, row stride K; 16-byte aligned, K % 8 == 0
 *   W    weight descriptor; W->cols == K
 *   bias dev [W->rows] BF16 (required)
 *   residual  dev [N x W->rows] BF16 with row stride ldy, or NULL
 *   Y    dev [N x W->rows] BF16 with row stride ldy (ldy >= rows, ldy % 8 == 0)
 * Weights stream through the arena page by page (or are read in place with
 * PSI_RESIDENT); page GEMMs alternate between the compute stream and the
 * arena's auxiliary stream (disjoint output columns), so one launch's tail
 * overlaps the next launch's start.  With four or more slots, streamed pages
 * of 256-aligned row counts that run on CTA pairs go two to a launch after
 * the first page (which runs alone: its slot is the ring's oldest) whenever
 * the ring slot after the next one is also free; resident pages on CTA pairs
 * run as one launch.  The per-element arithmetic is the
 * same in every mode, so resident and streamed results are bitwise equal.
 * Flags: PSI_RESIDENT, PSI_SYNC_COPY, PSI_BIAS_AFTER_BF16. */
psi_status psi_linear_paged(psi_arena* arena, const void* X, int64_t N, int64_t K,
                            const psi_linear_weight* W, const void* bias,
                            const void* residual, void* Y, int64_t ldy,
                            uint32_t flags);

/* Paged linear with split RoPE in the epilogue (section II-B): as
 * psi_linear_paged without residual, and in each head among the leading
 * rope->cols output columns the pair (a, b) = (t_j, t_{j+dh/2}) of the FP32
 * values t = X W^T + b is written as B(c a - s b), B(s a + c b) with the
 * table entries of the row's token: one BF16 write, the rotation applied to
 * the exact pre-rotation pair.  W->page_rows must be a multiple of rope->dh
 * (or cover W in one page).  Flags: PSI_RESIDENT, PSI_SYNC_COPY,
 * PSI_BIAS_AFTER_BF16, PSI_ROPE_AFTER_BF16. */
psi_status psi_linear_rope_paged(psi_arena* arena, const void* X, int64_t N, int64_t K,
                                 const psi_linear_weight* W, const void* bias,
                                 const psi_rope* rope, void* Y, int64_t ldy,
                                 uint32_t flags);

/* Full-row RMS normalisation, section II-B:
 *   Y[n, i] = B(gamma_i * X[n, i] / sqrt(s_n/d + eps)),  s_n = sum_i X[n, i]^2
 * with s_n summed in FP32 over the whole row (partial sums over width tiles
 * combined once, in a fixed order) and one denominator for every tile.
 *   X [N x d] row stride ldx, Y [N x d] row stride ldy, gamma [d]: device
 *   BF16, 16-byte aligned, d, ldx, ldy multiples of 8, 1 <= d <= 8192.
 *   eps >= 0 (finite).  Y must not overlap X.
 * Enqueued on `stream` (cudaStream_t). */
psi_status psi_rmsnorm(const void* X, int64_t ldx, int64_t N, int64_t d, const void* gamma,
                       float eps, void* Y, int64_t ldy, void* stream);

/* Paged FFN, Eq.(2) with the reuse schedule of section III-B.  Hidden
 * slices are taken in order in groups of G (G = 2 when there are at least
 * two slices and slice % 64 == 0, else 1; fixed by the shape): for each
 * slice J of a group, page J is streamed and
 *   H_J  = B(phi(X U_J^T + a_J))            (BF16 write; phi = tanh-GELU;
 *                                            with PSI_BOUNDARY_PREGELU_BF16
 *                                            the pre-activation is rounded too)
 * then one down projection covers the group:
 *   Acc  = Acc + sum_{J in group} H_J V_:,J^T   (FP32, the first group stores)
 * and the last group writes Y = B(Acc + its partial + b [+ residual]).
 * A streamed FFN needs an arena of at least G slots (PSI_ERR_CAPACITY).
 *   X [N x d], residual and Y [N x r] (row stride r), a [h], b [r]: dev BF16
 *   hidden_ws, acc_ws: dev workspace of psi_ffn_workspace sizes (16-byte
 *   aligned); the full [N x h] hidden tensor is never formed.
 * Flags: PSI_RESIDENT, PSI_SYNC_COPY, PSI_BOUNDARY_PREGELU_BF16,
 * PSI_BIAS_AFTER_BF16. */
psi_status psi_ffn_paged(psi_arena* arena, const void* X, int64_t N,
                         const psi_ffn_weight* W, const void* a, const void* b,
                         void* hidden_ws, void* acc_ws, const void* residual,
                         void* Y, uint32_t flags);

/* psi_ffn_paged with Y and the residual at row stride ldy (elements; ldy >=
 * W->r, a multiple of 8), so an FFN over a range of output columns (the
 * rows [c0, c1) of V, packed into their own page image) can write straight
 * into those columns of a wider activation, e.g. Y = y + c0 with ldy = the
 * full width.  The accumulator workspace stays [N x r].  Same flags;
 * psi_ffn_paged is this call with ldy = W->r. */
psi_status psi_ffn_paged_strided(psi_arena* arena, const void* X, int64_t N,
                                 const psi_ffn_weight* W, const void* a, const void* b,
                                 void* hidden_ws, void* acc_ws, const void* residual,
                                 void* Y, int64_t ldy, uint32_t flags);

/* Partitioned attention, Eqs.(3)-(4): for every head and query row,
 * s_j = scale * q.k_j in FP32; keys are visited in blocks of key_block and
 * combined by the online-softmax update in FP32 (m, l, z); O = B(z / l).
 * Unmasked, noncausal, no dropout; Nk >= 1.
 *   Q [heads x Nq x dh], K, V [heads x Nk x dh], O [heads x Nq x dh]: dev
 *   BF16 views (psi_heads strides, 16-byte aligned rows).  dh == 128.
 *   key_block: 128 or 256 keys per online-softmax update (the kernel reads
 *   K and V in 128-key sub-tiles; with 256 a CTA holds one 128-query tile,
 *   with 128 two).
 * Enqueued on `stream` (cudaStream_t).  No arena: inputs are resident.
 * Flags: PSI_ATTN_BF16_WEIGHTS. */
psi_status psi_attn_partitioned(const psi_heads* Q, const psi_heads* K,
                                const psi_heads* V, const psi_heads* O,
                                int32_t heads, int64_t Nq, int64_t Nk, int32_t dh,
                                float scale, int32_t key_block, void* stream,
                                uint32_t flags);
/* The same with a device workspace (16-byte aligned, at least
 * psi_attn_workspace_size bytes) for the tail split: the kernel runs one
 * CTA per SM and (head, query tile) units; when the last wave of units is
 * partial, each of its units is cut into ranges of whole key blocks, one
 * CTA per range, and a second kernel combines the ranges' FP32 states
 * (m, l, z) by the update of Eq.(4) before the one BF16 write.  Only the
 * rounding of those units changes.  No split with PSI_ATTN_BF16_WEIGHTS
 * (its rounded weights follow the kernel's running maximum).
 * workspace NULL: no split (psi_attn_partitioned). */
psi_status psi_attn_partitioned_ws(const psi_heads* Q, const psi_heads* K,
                                   const psi_heads* V, const psi_heads* O,
                                   int32_t heads, int64_t Nq, int64_t Nk, int32_t dh,
                                   float scale, int32_t key_block, void* workspace,
                                   size_t workspace_bytes, void* stream, uint32_t flags);
/* Workspace bytes psi_attn_partitioned_ws needs on the current device. */
psi_status psi_attn_workspace_size(int32_t key_block, size_t* bytes);

/* ------------------------------------------------------ state journal --- */
/* Indexed host BF16 journal, section II-D (with the asynchronous pinned-host
 * transport of section III-B): inactive state tensors are kept in a pinned
 * host region, indexed by (block, branch, role), so that only the live state
 * occupies device memory (the S_live term of Eq.(1)).
 *
 * The host region is cut into equal slots; an entry takes one slot.  The
 * journal owns two copy streams (D2H and H2D, so both directions run at
 * once) and orders every copy against the arena's compute stream:
 *   - commit:  the D2H copy waits for the producer (the compute stream's
 *              position at the call); the entry becomes valid when the copy
 *              completes;
 *   - reload:  the H2D copy waits for the entry to be valid, for the
 *              consumers of the destination (the compute stream's position at
 *              the call) and for every journal copy still reading the
 *              destination; the compute stream waits for it only at
 *              psi_journal_acquire, so a reload can run ahead of the work
 *              enqueued before the acquire;
 *   - a slot is rewritten only after its last reload has read it.
 * The steady state needs no host-blocking wait.  Copies are byte-preserving:
 * a reloaded tensor is bitwise the committed one.  One journal per arena,
 * used by one host thread at a time. */
typedef struct psi_journal psi_journal;

typedef struct {
  int32_t block;
  int32_t branch;
  int32_t role;
} psi_key;

typedef struct {
  uint64_t commits;          /* D2H copies enqueued */
  uint64_t reloads;          /* H2D copies enqueued */
  uint64_t d2h_bytes;
  uint64_t h2d_bytes;
  uint64_t host_waits;       /* host-blocking waits (psi_journal_host_view) */
  uint64_t hazard_waits;     /* cross-stream waits added for device-range hazards */
  int32_t slots_in_use;
  int32_t slots_total;
} psi_journal_stats;

/* host_base: pinned host memory (cudaHostAlloc/cudaHostRegister; pageable
 * memory is refused with PSI_ERR_INVALID_ARG), 16-byte aligned, host_bytes
 * >= slot_bytes; slot_bytes: a multiple of 256, the largest entry. */
psi_status psi_journal_create(psi_arena* arena, void* host_base, size_t host_bytes,
                              size_t slot_bytes, psi_journal** out);
/* Waits (without limit) for the journal's copies, then frees its streams and
 * events. */
psi_status psi_journal_destroy(psi_journal* j);

/* Journal `bytes` of device memory at dev_src under `key` (replacing an
 * earlier entry of that key).  PSI_ERR_CAPACITY if bytes > slot_bytes or no
 * slot is free.  dev_src must not be written until the copy has read it:
 * call psi_journal_fence on the range first (the journal's own reloads
 * already wait for it). */
psi_status psi_journal_commit(psi_journal* j, psi_key key, const void* dev_src, size_t bytes);
/* Copy the entry of `key` into dev_dst (bytes must equal the committed
 * size; PSI_ERR_INVALID_ARG for an unknown key or another size). */
psi_status psi_journal_reload(psi_journal* j, psi_key key, void* dev_dst, size_t bytes);
/* The compute stream waits for the latest reload of `key`
 * (PSI_ERR_INVALID_ARG if there is none since the last acquire or commit). */
psi_status psi_journal_acquire(psi_journal* j, psi_key key);
/* The compute stream waits for every journal copy that reads or writes
 * [dev_ptr, dev_ptr + bytes) (none: no wait). */
psi_status psi_journal_fence(psi_journal* j, const void* dev_ptr, size_t bytes);
/* Free the entry's slot (its last reload still completes first). */
psi_status psi_journal_drop(psi_journal* j, psi_key key);
/* Host view of a committed entry: waits for its D2H copy (bounded by
 * timeout_ms; PSI_ERR_TIMEOUT) and returns the host address and size. */
psi_status psi_journal_host_view(psi_journal* j, psi_key key, int64_t timeout_ms,
                                 const void** host_ptr, size_t* bytes);
psi_status psi_journal_get_stats(const psi_journal* j, psi_journal_stats* out);
/* Test hook: the next commit or reload fails with PSI_ERR_CUDA before it
 * enqueues anything (host-side fault injection). */
psi_status psi_journal_fail_next_copy(psi_journal* j);

/* ------------------------------------------------- no-allocation FFN --- */
/* The paper has no counterpart of this entry point; it serves callers that
 * cannot allocate device memory (code running inside another framework's
 * memory pool or a fixed budget handed out at start-up, plug-ins given
 * device pointers but no allocator).  It computes what psi_ffn_paged
 * computes with PSI_RESIDENT: the same slice grouping G, the same FP32
 * accumulation order and the same per-element epilogue arithmetic, so the
 * same bytes (the up projections of a group are launched one slice at a
 * time rather than merged).  It runs on `stream` (cudaStream_t), with
 * weights read in place from W->dev_resident (the packed page image,
 * W->host is not used) and no arena.
 *   X [N x d], residual (or NULL) and Y [N x r] (row stride r), a [h],
 *   b [r]: device BF16, 16-byte aligned.
 *   flags: PSI_BOUNDARY_PREGELU_BF16, PSI_BIAS_AFTER_BF16 (as for
 *   psi_ffn_paged); PSI_RESIDENT is accepted and implied; any other bit
 *   gives PSI_ERR_UNSUPPORTED.
 * Workspace: the hidden slices of one group (N*G*slice*2 bytes, rounded up
 * to 256, with G as for psi_ffn_paged) and the FP32 accumulator (N*r*4
 * bytes) live in one fixed 16 MiB device array inside the library, held on
 * every GPU that loads it until the process exits.  Larger problems fail
 * with PSI_ERR_CAPACITY before anything is enqueued.  The call makes no cudaMalloc or cudaFree and
 * calls no allocating library routine.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call shares the array: calls whose work overlaps on the GPU (other
 * streams, other host threads) race on it and must be serialised by the
 * caller.  The accumulator is written before it is read, so no clearing
 * is needed between calls. */
psi_status psi_ffn_resident_noalloc(const void* X, int64_t N, const psi_ffn_weight* W,
                                    const void* a, const void* b, const void* residual,
                                    void* Y, void* stream, uint32_t flags);

#ifdef __cplusplus
}
#endif

#endif /* PSI_H */
