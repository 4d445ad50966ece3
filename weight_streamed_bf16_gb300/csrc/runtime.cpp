// runtime.cpp -- the fixed arena of weight pages, the page ring with its
// copy/consumer events, and the paged operators (C ABI of include/psi.h).
//
// Paper: Precision-Preserving Subtensor Inference, section II-A (managed
// working set M <= S_live + W + 2P + eps; the four arena rules), section
// II-D (page lifecycle free -> filling -> ready -> consuming; release
// records an event after all uses, the next copy waits on it), section III-B
// (weight prefetch into alternating pages; FFN reuse schedule).
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <string>
#include <thread>
#include <utility>
#include <vector>
#include "internal.h"

namespace psi {
const char* last_error_cstr();
int gemm_bn_for(int64_t N);
}  // namespace psi

using namespace psi;

namespace {

enum SlotState : int { SLOT_FREE = 0, SLOT_REQUESTED = 1 };

struct TimedLaunch {
  cudaEvent_t start;
  cudaEvent_t stop;
  double work;  // FLOPs for a GEMM, bytes for a copy
  int32_t kind = PSI_TRACE_GEMM;
  int32_t slot = -1;    // arena slot of the page, -1 if none
  int32_t stream = 0;   // 0 compute, 1 auxiliary, 2 copy
  uint64_t seq = 0;     // page request or launch number
};

}  // namespace

struct psi_arena {
  int device = 0;
  char* base = nullptr;
  size_t bytes = 0;
  size_t page_bytes = 0;
  int nslots = 0;
  cudaStream_t compute = nullptr;
  cudaStream_t copy = nullptr;
  // second consumer stream owned by the arena: consecutive page GEMMs run on
  // alternating streams so one kernel's tail overlaps the next one's start
  cudaStream_t aux = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  cudaEvent_t ev_up[2] = {nullptr, nullptr}, ev_down[2] = {nullptr, nullptr};
  std::vector<cudaEvent_t> ready;      // copy into the slot complete
  std::vector<cudaEvent_t> consumed;   // last consumer of the slot complete
  std::vector<uint8_t> has_consumed;   // consumed[s] has been recorded
  std::vector<int> state;              // host shadow of the request state
  std::vector<uint64_t> slot_seq;      // sequence number of the open request
  int next = 0;
  uint64_t seq = 0;
  psi_stats stats{};
  bool timing = false;
  bool fail_next_copy = false;
  std::vector<TimedLaunch> gemm_t, copy_t;
  std::vector<cudaEvent_t> pool;
  uint64_t gemm_seq = 0;  // page-GEMM launches while timing
  // page timeline: records of the timed launches since psi_arena_trace_begin
  bool tracing = false;
  size_t trace_cap = 0;
  cudaEvent_t trace_origin = nullptr;
  std::vector<psi_trace_record> trace;
};

namespace psi {
// the arena's compute stream and device, for the journal (journal.cpp)
cudaStream_t arena_compute_stream(psi_arena* a) { return a->compute; }
int arena_device(psi_arena* a) { return a->device; }
}  // namespace psi

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

cudaEvent_t pool_get(psi_arena* a) {
  if (!a->pool.empty()) {
    cudaEvent_t e = a->pool.back();
    a->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

psi_status timed_begin(psi_arena* a, cudaStream_t s, TimedLaunch* t) {
  t->start = pool_get(a);
  t->stop = pool_get(a);
  if (!t->start || !t->stop) return set_error(PSI_ERR_CUDA, "cudaEventCreate failed");
  cudaError_t e = cudaEventRecord(t->start, s);
  return e == cudaSuccess ? PSI_OK : cuda_error(e, "cudaEventRecord");
}

psi_status timed_end(psi_arena* a, cudaStream_t s, TimedLaunch t, std::vector<TimedLaunch>* v) {
  cudaError_t e = cudaEventRecord(t.stop, s);
  if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord");
  v->push_back(t);
  (void)a;
  return PSI_OK;
}

uint64_t g_stall_next_ns = 0;  // test hook, see psi_debug_stall_next_gemm

// Launch one page GEMM on the arena's compute stream (timed if enabled).
psi_status arena_gemm(psi_arena* a, cudaStream_t sm, const void* X, int64_t ldx, const void* P,
                      int64_t ldp, const GemmArgs& g0, const void* P2 = nullptr) {
  GemmArgs g = g0;
  if (g_stall_next_ns) {
    g.debug_stall = 1;
    g.timeout_ns = g_stall_next_ns;
    g_stall_next_ns = 0;
  }
  TimedLaunch t{};
  psi_status st;
  if (a->timing && (st = timed_begin(a, sm, &t)) != PSI_OK) return st;
  st = launch_page_gemm(X, ldx, P, ldp, g, sm, P2);
  if (st != PSI_OK) return st;
  a->stats.kernels_launched++;
  if (a->timing) {
    t.work = 2.0 * g.M * static_cast<double>(g.N) * g.K;
    t.kind = PSI_TRACE_GEMM;
    t.stream = sm == a->aux ? 1 : 0;
    const char* pc = static_cast<const char*>(P);
    t.slot = (pc >= a->base && pc < a->base + a->bytes)
                 ? static_cast<int32_t>((pc - a->base) / static_cast<ptrdiff_t>(a->page_bytes))
                 : -1;
    t.seq = ++a->gemm_seq;
    return timed_end(a, sm, t, &a->gemm_t);
  }
  return PSI_OK;
}

psi_status wait_stream(cudaStream_t s, std::chrono::steady_clock::time_point deadline,
                       bool bounded) {
  while (true) {
    cudaError_t e = cudaStreamQuery(s);
    if (e == cudaSuccess) return PSI_OK;
    if (e != cudaErrorNotReady) return cuda_error(e, "stream");
    if (bounded && std::chrono::steady_clock::now() > deadline)
      return set_error(PSI_ERR_TIMEOUT, "stream did not finish before the deadline");
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

psi_status report_device_errors() {
  DevError d{};
  cudaError_t e = dev_error_take(&d);
  if (e != cudaSuccess) return cuda_error(e, "reading the kernel error record");
  if (d.code != 0) {
    char buf[200];
    snprintf(buf, sizeof buf,
             "kernel error %d (%s) in kernel %d role %d, info %d %d", d.code,
             d.code == 1 ? "bounded wait expired" : "range", d.where / 16, d.where % 16, d.info0,
             d.info1);
    return set_error(PSI_ERR_DEVICE, buf);
  }
  return PSI_OK;
}

}  // namespace

extern "C" {

const char* psi_version(void) { return "psi-gb300 0.1 (sm_103a, tcgen05)"; }

const char* psi_status_string(psi_status s) {
  switch (s) {
    case PSI_OK: return "PSI_OK";
    case PSI_ERR_INVALID_ARG: return "PSI_ERR_INVALID_ARG";
    case PSI_ERR_CAPACITY: return "PSI_ERR_CAPACITY";
    case PSI_ERR_PAGE_BUSY: return "PSI_ERR_PAGE_BUSY";
    case PSI_ERR_CUDA: return "PSI_ERR_CUDA";
    case PSI_ERR_TIMEOUT: return "PSI_ERR_TIMEOUT";
    case PSI_ERR_UNSUPPORTED: return "PSI_ERR_UNSUPPORTED";
    case PSI_ERR_DEVICE: return "PSI_ERR_DEVICE";
  }
  return "PSI_ERR_UNKNOWN";
}

const char* psi_last_error(void) { return last_error_cstr(); }

psi_status psi_plan_linear(int64_t rows, int64_t cols, size_t page_bytes, int64_t* page_rows) {
  if (!page_rows || rows <= 0 || cols <= 0)
    return set_error(PSI_ERR_INVALID_ARG, "plan_linear: bad arguments");
  const int64_t fit = static_cast<int64_t>(page_bytes / (static_cast<size_t>(cols) * 2));
  if (fit >= rows) {
    *page_rows = rows;
    return PSI_OK;
  }
  int64_t pr = fit >= 256 ? (fit / 256) * 256 : (fit / 16) * 16;
  if (pr < 16)
    return set_error(PSI_ERR_CAPACITY, "plan_linear: weight tile exceeds page (16 rows do not fit)");
  *page_rows = pr;
  return PSI_OK;
}

psi_status psi_plan_columns(int64_t cols, int64_t align, int32_t parts, int32_t part,
                            int64_t* c0, int64_t* c1) {
  if (!c0 || !c1 || cols < 0 || align < 1 || parts < 1 || part < 0 || part >= parts)
    return set_error(PSI_ERR_INVALID_ARG, "plan_columns: bad arguments");
  // units of `align` columns (the last unit may be short), dealt out as
  // evenly as possible, the remainder to the first parts
  const int64_t units = (cols + align - 1) / align;
  const int64_t base = units / parts, extra = units % parts;
  const int64_t u0 = part * base + std::min<int64_t>(part, extra);
  const int64_t u1 = u0 + base + (part < extra ? 1 : 0);
  *c0 = std::min(u0 * align, cols);
  *c1 = std::min(u1 * align, cols);
  return PSI_OK;
}

size_t psi_ffn_page_bytes(int64_t d, int64_t r, int64_t slice) {
  if (d <= 0 || r <= 0 || slice <= 0) return 0;
  return static_cast<size_t>(slice) * static_cast<size_t>(d) * 2 +
         static_cast<size_t>(r) * static_cast<size_t>(slice) * 2;
}

psi_status psi_ffn_pack(const void* U, const void* V, int64_t d, int64_t h, int64_t r,
                        int64_t slice, void* dst) {
  if (!U || !V || !dst || d <= 0 || h <= 0 || r <= 0 || slice <= 0 || h % slice)
    return set_error(PSI_ERR_INVALID_ARG, "ffn_pack: bad arguments (h must be a multiple of slice)");
  const int64_t S = h / slice;
  const size_t pb = psi_ffn_page_bytes(d, r, slice);
  const uint16_t* u = static_cast<const uint16_t*>(U);
  const uint16_t* v = static_cast<const uint16_t*>(V);
  char* out = static_cast<char*>(dst);
  auto pack_one = [&](int64_t J) {
    char* page = out + J * pb;
    std::memcpy(page, u + J * slice * d, static_cast<size_t>(slice * d) * 2);
    uint16_t* vj = reinterpret_cast<uint16_t*>(page + static_cast<size_t>(slice * d) * 2);
    for (int64_t o = 0; o < r; ++o)
      std::memcpy(vj + o * slice, v + o * h + J * slice, static_cast<size_t>(slice) * 2);
  };
  unsigned nt = std::max(1u, std::min<unsigned>(std::thread::hardware_concurrency(), 32u));
  nt = static_cast<unsigned>(std::min<int64_t>(nt, S));
  std::vector<std::thread> th;
  for (unsigned t = 0; t < nt; ++t)
    th.emplace_back([&, t] {
      for (int64_t J = t; J < S; J += nt) pack_one(J);
    });
  for (auto& x : th) x.join();
  return PSI_OK;
}

psi_status psi_ffn_workspace(int64_t N, int64_t r, int64_t slice, size_t* hidden_bytes,
                             size_t* acc_bytes) {
  if (N < 0 || r <= 0 || slice <= 0 || !hidden_bytes || !acc_bytes)
    return set_error(PSI_ERR_INVALID_ARG, "ffn_workspace: bad arguments");
  *hidden_bytes = 2 * static_cast<size_t>(kFfnGroupMax) * static_cast<size_t>(N) *
                  static_cast<size_t>(slice) * 2;
  *acc_bytes = static_cast<size_t>(N) * static_cast<size_t>(r) * 4;
  return PSI_OK;
}

psi_status psi_arena_create(void* dev_base, size_t dev_bytes, size_t page_bytes,
                            void* compute_stream, void* copy_stream, psi_arena** out) {
  if (!out) return set_error(PSI_ERR_INVALID_ARG, "arena_create: out is null");
  *out = nullptr;
  if (!dev_base || page_bytes == 0 || (page_bytes % 1024) ||
      (reinterpret_cast<uintptr_t>(dev_base) % 1024))
    return set_error(PSI_ERR_INVALID_ARG,
                     "arena_create: base must be 1024-byte aligned, page_bytes a multiple of 1024");
  if (dev_bytes < page_bytes)
    return set_error(PSI_ERR_CAPACITY, "arena_create: arena smaller than one page");
  psi_arena* a = new psi_arena();
  cudaGetDevice(&a->device);
  a->base = static_cast<char*>(dev_base);
  a->bytes = dev_bytes;
  a->page_bytes = page_bytes;
  a->nslots = static_cast<int>(dev_bytes / page_bytes);
  a->compute = static_cast<cudaStream_t>(compute_stream);
  a->copy = static_cast<cudaStream_t>(copy_stream);
  a->ready.resize(a->nslots);
  a->consumed.resize(a->nslots);
  a->has_consumed.assign(a->nslots, 0);
  a->state.assign(a->nslots, SLOT_FREE);
  a->slot_seq.assign(a->nslots, 0);
  for (int s = 0; s < a->nslots; ++s) {
    cudaError_t e1 = cudaEventCreateWithFlags(&a->ready[s], cudaEventDisableTiming);
    cudaError_t e2 = cudaEventCreateWithFlags(&a->consumed[s], cudaEventDisableTiming);
    if (e1 != cudaSuccess || e2 != cudaSuccess) {
      psi_arena_destroy(a);
      return cuda_error(e1 != cudaSuccess ? e1 : e2, "arena_create: cudaEventCreate");
    }
  }
  {
    cudaError_t e = cudaStreamCreateWithFlags(&a->aux, cudaStreamNonBlocking);
    cudaEvent_t* evs[] = {&a->ev_fork, &a->ev_join, &a->ev_up[0], &a->ev_up[1], &a->ev_down[0],
                          &a->ev_down[1]};
    for (auto* ev : evs)
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      psi_arena_destroy(a);
      return cuda_error(e, "arena_create: auxiliary stream or events");
    }
  }
  if (!dev_error_ptr()) {
    psi_arena_destroy(a);
    return set_error(PSI_ERR_CUDA, "arena_create: kernel error record not reachable");
  }
  *out = a;
  return PSI_OK;
}

psi_status psi_arena_destroy(psi_arena* a) {
  if (!a) return PSI_OK;
  cudaStreamSynchronize(a->compute);
  if (a->copy != a->compute) cudaStreamSynchronize(a->copy);
  if (a->aux) {
    cudaStreamSynchronize(a->aux);
    cudaStreamDestroy(a->aux);
  }
  for (cudaEvent_t e : {a->ev_fork, a->ev_join, a->ev_up[0], a->ev_up[1], a->ev_down[0],
                        a->ev_down[1]})
    if (e) cudaEventDestroy(e);
  for (auto e : a->ready)
    if (e) cudaEventDestroy(e);
  for (auto e : a->consumed)
    if (e) cudaEventDestroy(e);
  for (auto& t : a->gemm_t) {
    cudaEventDestroy(t.start);
    cudaEventDestroy(t.stop);
  }
  for (auto& t : a->copy_t) {
    cudaEventDestroy(t.start);
    cudaEventDestroy(t.stop);
  }
  for (auto e : a->pool) cudaEventDestroy(e);
  if (a->trace_origin) cudaEventDestroy(a->trace_origin);
  delete a;
  return PSI_OK;
}

int32_t psi_arena_slots(const psi_arena* a) { return a ? a->nslots : 0; }

}  // extern "C"

namespace {
// Request the next slot for a consumer on stream `cs` (see psi_page_stream).
psi_status page_stream_to(psi_arena* a, const void* host_src, size_t bytes, uint32_t flags,
                          cudaStream_t cs, psi_page* out) {
  if (!a || !host_src || !out) return set_error(PSI_ERR_INVALID_ARG, "page_stream: null argument");
  if (bytes > a->page_bytes)
    return set_error(PSI_ERR_CAPACITY, "page_stream: slice larger than the page");
  const int s = a->next;
  if (a->state[s] != SLOT_FREE)
    return set_error(PSI_ERR_PAGE_BUSY, "page_stream: slot " + std::to_string(s) +
                                            " still has an unreleased request");
  if (a->fail_next_copy) {
    a->fail_next_copy = false;
    return set_error(PSI_ERR_CUDA, "page_stream: injected copy failure (test hook)");
  }
  void* dst = a->base + static_cast<size_t>(s) * a->page_bytes;
  cudaError_t e;
  const bool sync_copy = (flags & PSI_SYNC_COPY) || a->copy == a->compute;
  TimedLaunch t{};
  psi_status st;
  if (sync_copy) {
    // the copy runs on the consumer's stream, after the slot's last consumer
    if (a->has_consumed[s]) {
      e = cudaStreamWaitEvent(cs, a->consumed[s], 0);
      if (e != cudaSuccess) return cuda_error(e, "page_stream: wait consumed");
    }
    if (a->timing && (st = timed_begin(a, cs, &t)) != PSI_OK) return st;
    e = cudaMemcpyAsync(dst, host_src, bytes, cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) return cuda_error(e, "page_stream: cudaMemcpyAsync");
  } else {
    if (a->has_consumed[s]) {
      e = cudaStreamWaitEvent(a->copy, a->consumed[s], 0);  // previous consumers done
      if (e != cudaSuccess) return cuda_error(e, "page_stream: wait consumed");
    }
    if (a->timing && (st = timed_begin(a, a->copy, &t)) != PSI_OK) return st;
    e = cudaMemcpyAsync(dst, host_src, bytes, cudaMemcpyHostToDevice, a->copy);
    if (e != cudaSuccess) return cuda_error(e, "page_stream: cudaMemcpyAsync");
    e = cudaEventRecord(a->ready[s], a->copy);
    if (e != cudaSuccess) return cuda_error(e, "page_stream: record ready");
    e = cudaStreamWaitEvent(cs, a->ready[s], 0);  // consumers wait for the copy
    if (e != cudaSuccess) return cuda_error(e, "page_stream: wait ready");
  }
  if (a->timing) {
    t.work = static_cast<double>(bytes);
    t.kind = PSI_TRACE_COPY;
    t.slot = s;
    t.stream = sync_copy ? (cs == a->aux ? 1 : 0) : 2;
    t.seq = a->seq + 1;  // the number this request gets below
    if ((st = timed_end(a, sync_copy ? cs : a->copy, t, &a->copy_t)) != PSI_OK) return st;
  }
  a->state[s] = SLOT_REQUESTED;
  a->slot_seq[s] = ++a->seq;
  a->next = (s + 1) % a->nslots;
  a->stats.pages_streamed++;
  a->stats.h2d_bytes += bytes;
  out->slot = s;
  out->seq = a->slot_seq[s];
  out->dev = dst;
  out->bytes = bytes;
  return PSI_OK;
}

// End a request whose last consumer was enqueued on stream `cs`.
psi_status page_release_on(psi_arena* a, psi_page p, cudaStream_t cs) {
  if (!a || p.slot < 0 || p.slot >= a->nslots)
    return set_error(PSI_ERR_INVALID_ARG, "page_release: bad page");
  if (a->state[p.slot] != SLOT_REQUESTED || a->slot_seq[p.slot] != p.seq)
    return set_error(PSI_ERR_INVALID_ARG, "page_release: stale or already released page");
  cudaError_t e = cudaEventRecord(a->consumed[p.slot], cs);
  if (e != cudaSuccess) return cuda_error(e, "page_release: record consumed");
  a->has_consumed[p.slot] = 1;
  a->state[p.slot] = SLOT_FREE;
  return PSI_OK;
}

// aux (or compute) waits for everything enqueued so far on `from`.
psi_status stream_after(cudaEvent_t ev, cudaStream_t from, cudaStream_t to) {
  cudaError_t e = cudaEventRecord(ev, from);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(to, ev, 0);
  return e == cudaSuccess ? PSI_OK : cuda_error(e, "fork/join event");
}
}  // namespace

extern "C" {

psi_status psi_page_stream(psi_arena* a, const void* host_src, size_t bytes, uint32_t flags,
                           psi_page* out) {
  psi_status fs = check_flags(flags, kFlagsPageStream, "page_stream");
  if (fs != PSI_OK) return fs;
  if (!a) return set_error(PSI_ERR_INVALID_ARG, "page_stream: null arena");
  return page_stream_to(a, host_src, bytes, flags, a->compute, out);
}

psi_status psi_page_release(psi_arena* a, psi_page p) {
  if (!a) return set_error(PSI_ERR_INVALID_ARG, "page_release: null arena");
  return page_release_on(a, p, a->compute);
}

psi_status psi_sync(psi_arena* a, int64_t timeout_ms) {
  if (!a) return set_error(PSI_ERR_INVALID_ARG, "sync: null arena");
  const bool bounded = timeout_ms >= 0;
  const auto dl = std::chrono::steady_clock::now() + std::chrono::milliseconds(bounded ? timeout_ms : 0);
  psi_status st = wait_stream(a->compute, dl, bounded);
  if (st != PSI_OK) return st;
  if (a->copy != a->compute && (st = wait_stream(a->copy, dl, bounded)) != PSI_OK) return st;
  if ((st = wait_stream(a->aux, dl, bounded)) != PSI_OK) return st;
  return report_device_errors();
}

psi_status psi_stream_wait(void* stream, int64_t timeout_ms) {
  const bool bounded = timeout_ms >= 0;
  const auto dl = std::chrono::steady_clock::now() + std::chrono::milliseconds(bounded ? timeout_ms : 0);
  psi_status st = wait_stream(static_cast<cudaStream_t>(stream), dl, bounded);
  if (st != PSI_OK) return st;
  return report_device_errors();
}

psi_status psi_arena_stats(const psi_arena* ca, psi_stats* out) {
  if (!ca || !out) return set_error(PSI_ERR_INVALID_ARG, "arena_stats: null argument");
  psi_arena* a = const_cast<psi_arena*>(ca);
  // sums of the launch durations, and the union of the launch intervals
  // (timestamps relative to the first event of the batch)
  auto fold = [&](std::vector<TimedLaunch>& v, uint64_t* n, double* ms, double* work,
                  double* busy) -> psi_status {
    std::vector<std::pair<double, double>> iv;
    for (auto& t : v) {
      cudaError_t e = cudaEventSynchronize(t.stop);
      if (e != cudaSuccess) return cuda_error(e, "arena_stats: event");
      float f = 0.f, t0 = 0.f;
      e = cudaEventElapsedTime(&f, t.start, t.stop);
      if (e == cudaSuccess) e = cudaEventElapsedTime(&t0, v.front().start, t.start);
      if (e != cudaSuccess) return cuda_error(e, "arena_stats: elapsed");
      *n += 1;
      *ms += f;
      *work += t.work;
      iv.emplace_back(t0, t0 + f);
      if (a->tracing && a->trace.size() < a->trace_cap) {
        float ts = 0.f, te = 0.f;
        e = cudaEventElapsedTime(&ts, a->trace_origin, t.start);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&te, a->trace_origin, t.stop);
        if (e != cudaSuccess) return cuda_error(e, "arena trace: elapsed");
        psi_trace_record r{};
        r.kind = t.kind;
        r.slot = t.slot;
        r.stream = t.stream;
        r.seq = t.seq;
        r.start_ms = ts;
        r.end_ms = te;
        r.work = t.work;
        a->trace.push_back(r);
      }
    }
    std::sort(iv.begin(), iv.end());
    double end = -1e300;
    for (auto& x : iv) {
      if (x.first >= end) {
        *busy += x.second - x.first;
        end = x.second;
      } else if (x.second > end) {
        *busy += x.second - end;
        end = x.second;
      }
    }
    for (auto& t : v) {
      a->pool.push_back(t.start);
      a->pool.push_back(t.stop);
    }
    v.clear();
    return PSI_OK;
  };
  psi_status st = fold(a->gemm_t, &a->stats.timed_gemms, &a->stats.gemm_ms,
                       &a->stats.gemm_flops, &a->stats.gemm_busy_ms);
  if (st != PSI_OK) return st;
  st = fold(a->copy_t, &a->stats.timed_copies, &a->stats.copy_ms, &a->stats.copy_bytes,
            &a->stats.copy_busy_ms);
  if (st != PSI_OK) return st;
  *out = a->stats;
  return PSI_OK;
}

psi_status psi_arena_reset_stats(psi_arena* a) {
  if (!a) return set_error(PSI_ERR_INVALID_ARG, "arena_reset_stats: null arena");
  psi_stats tmp;
  psi_status st = psi_arena_stats(a, &tmp);  // folds and recycles pending events
  a->stats = psi_stats{};
  return st;
}

psi_status psi_arena_set_timing(psi_arena* a, int32_t enable) {
  if (!a) return set_error(PSI_ERR_INVALID_ARG, "arena_set_timing: null arena");
  a->timing = enable != 0;
  return PSI_OK;
}

psi_status psi_arena_trace_begin(psi_arena* a, size_t capacity) {
  if (!a || capacity == 0)
    return set_error(PSI_ERR_INVALID_ARG, "arena_trace_begin: null arena or capacity 0");
  psi_stats tmp;
  a->tracing = false;
  psi_status st = psi_arena_stats(a, &tmp);  // launches before the origin stay out
  if (st != PSI_OK) return st;
  cudaError_t e = cudaSuccess;
  if (!a->trace_origin) e = cudaEventCreate(&a->trace_origin);
  if (e == cudaSuccess) e = cudaEventRecord(a->trace_origin, a->compute);
  if (e != cudaSuccess) return cuda_error(e, "arena_trace_begin: origin event");
  a->trace.clear();
  a->trace.reserve(std::min<size_t>(capacity, 1 << 16));
  a->trace_cap = capacity;
  a->tracing = true;
  a->timing = true;
  return PSI_OK;
}

psi_status psi_arena_trace_get(psi_arena* a, psi_trace_record* out, size_t capacity,
                               size_t* count) {
  if (!a || !count || (capacity > 0 && !out))
    return set_error(PSI_ERR_INVALID_ARG, "arena_trace_get: null argument");
  if (!a->tracing) return set_error(PSI_ERR_INVALID_ARG, "arena_trace_get: no trace begun");
  psi_stats tmp;
  psi_status st = psi_arena_stats(a, &tmp);  // waits for and folds the pending launches
  if (st != PSI_OK) return st;
  std::stable_sort(a->trace.begin(), a->trace.end(),
                   [](const psi_trace_record& x, const psi_trace_record& y) {
                     return x.start_ms < y.start_ms;
                   });
  const size_t n = std::min(capacity, a->trace.size());
  for (size_t i = 0; i < n; ++i) out[i] = a->trace[i];
  *count = a->trace.size();
  return PSI_OK;
}

psi_status psi_debug_stall_next_gemm(uint64_t timeout_ns) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull)
    return set_error(PSI_ERR_INVALID_ARG, "debug_stall_next_gemm: timeout must be in (0, 10 s]");
  g_stall_next_ns = timeout_ns;
  return PSI_OK;
}

psi_status psi_arena_fail_next_copy(psi_arena* a) {
  if (!a) return set_error(PSI_ERR_INVALID_ARG, "arena_fail_next_copy: null arena");
  a->fail_next_copy = true;
  return PSI_OK;
}

// --------------------------------------------------------------------------
static psi_status linear_paged(psi_arena* a, const void* X, int64_t N, int64_t K,
                               const psi_linear_weight* W, const void* bias,
                               const void* residual, void* Y, int64_t ldy, uint32_t flags,
                               const psi_rope* rope) {
  {
    psi_status fs = rope ? check_flags(flags, kFlagsLinearRope, "linear_rope_paged")
                         : check_flags(flags, kFlagsLinear, "linear_paged");
    if (fs != PSI_OK) return fs;
  }
  if (!a || !X || !W || !bias || !Y)
    return set_error(PSI_ERR_INVALID_ARG, "linear_paged: null argument");
  if (N < 0 || K <= 0 || W->cols != K || W->rows <= 0 || W->page_rows <= 0)
    return set_error(PSI_ERR_INVALID_ARG, "linear_paged: bad shape (W->cols must equal K)");
  if (K % 8 || ldy < W->rows || ldy % 8)
    return set_error(PSI_ERR_INVALID_ARG, "linear_paged: K and ldy must be multiples of 8, ldy >= rows");
  if (W->page_rows < W->rows && W->page_rows % 16)
    return set_error(PSI_ERR_INVALID_ARG, "linear_paged: page_rows must be a multiple of 16");
  if (!aligned16(X) || !aligned16(Y) || !aligned16(bias) || (residual && !aligned16(residual)))
    return set_error(PSI_ERR_INVALID_ARG, "linear_paged: pointers must be 16-byte aligned");
  if (N > 0x7FFFFFFF || K > 0x7FFFFFFF || W->rows > 0x7FFFFFFF)
    return set_error(PSI_ERR_UNSUPPORTED, "linear_paged: dimension above 2^31");
  const bool resident = flags & PSI_RESIDENT;
  const char* src = static_cast<const char*>(resident ? W->dev_resident : W->host);
  if (!src)
    return set_error(PSI_ERR_INVALID_ARG, resident ? "linear_paged: dev_resident is null"
                                                   : "linear_paged: host is null");
  const size_t max_page = static_cast<size_t>(std::min(W->page_rows, W->rows)) * K * 2;
  if (!resident && max_page > a->page_bytes)
    return set_error(PSI_ERR_CAPACITY, "linear_paged: weight tile exceeds page");
  if (rope) {
    if (rope->dh != 64 && rope->dh != 128)
      return set_error(PSI_ERR_UNSUPPORTED, "linear_rope_paged: dh must be 64 or 128");
    if (!rope->cos || !rope->sin || !aligned16(rope->cos) || !aligned16(rope->sin) ||
        rope->ld % 4 || rope->ld < rope->dh / 2)
      return set_error(PSI_ERR_INVALID_ARG,
                       "linear_rope_paged: tables must be 16-byte aligned, ld % 4 == 0, ld >= dh/2");
    if (rope->cols < 0 || rope->cols % rope->dh || rope->cols > W->rows)
      return set_error(PSI_ERR_INVALID_ARG,
                       "linear_rope_paged: cols must be whole heads within the output");
    if (W->page_rows < W->rows && W->page_rows % rope->dh)
      return set_error(PSI_ERR_INVALID_ARG,
                       "linear_rope_paged: page_rows must be a multiple of dh");
  }
  int64_t npages = (W->rows + W->page_rows - 1) / W->page_rows;
  DevError* err = dev_error_ptr();
  // Resident weights need no page ring: when every page would run on CTA
  // pairs with page boundaries on 256-row tile boundaries, one launch covers
  // all pages with exactly the per-page launches' tiles (the same kernel and
  // per-element arithmetic, so the result is bit for bit the same), and the
  // ramp, last-tile epilogue and launch gap are paid once per operator.
  const int64_t last_rows = W->rows - (npages - 1) * W->page_rows;
  const bool one_launch = resident && npages > 1 && W->page_rows % 256 == 0 &&
                          gemm_use_pair(N, W->page_rows) && gemm_use_pair(N, last_rows);
  int64_t page_rows = W->page_rows;
  if (one_launch) {
    a->stats.resident_pages += npages - 1;  // pages covered, counted as before
    page_rows = W->rows;
    npages = 1;
  }
  // After the first page, streamed pages go two to a launch when both run
  // on CTA pairs and their boundary falls on a 256-row tile boundary: the
  // launch reads its output columns from two tensor maps (one per page),
  // with the tiles and per-element arithmetic of the two single-page
  // launches, so the bytes are the same; the pair has 2 x 192 tiles of
  // 256 x 256 on a 6144-token batch instead of two launches of 192, each
  // with its own ramp and tail.  The first page runs alone because its slot
  // is the ring's oldest, the one a copy stream blocked on a full ring waits
  // for (in the streamed block, pairs from the first page measured 2.535 ms
  // per step, one page per launch 2.521, pairs after the first 2.503).  The
  // ring must hold the next pair while one computes (four slots or more).
  const bool merge2 = !resident && a->nslots >= 4 && W->page_rows % 256 == 0;
  // launches alternate between the compute and the auxiliary stream (outputs
  // are disjoint column blocks); aux first catches up with the compute stream
  psi_status fst = stream_after(a->ev_fork, a->compute, a->aux);
  if (fst != PSI_OK) return fst;
  for (int64_t p = 0, launch = 0; p < npages; ++launch) {
    cudaStream_t cs = (launch & 1) ? a->aux : a->compute;
    const int64_t r0 = p * page_rows;
    const int64_t rows_p = std::min(page_rows, W->rows - r0);
    int64_t rows_q = 0;  // rows of the second page of the launch (0: none)
    if (merge2 && p > 0 && p + 1 < npages && a->state[(a->next + 1) % a->nslots] == SLOT_FREE) {
      rows_q = std::min(page_rows, W->rows - r0 - page_rows);
      if (!gemm_use_pair(N, rows_p) || !gemm_use_pair(N, rows_q)) rows_q = 0;
    }
    const size_t off = static_cast<size_t>(r0) * K * 2;
    const size_t nbytes = static_cast<size_t>(rows_p) * K * 2;
    psi_page pg{}, pg2{};
    const void* dev;
    const void* dev2 = nullptr;
    if (resident) {
      dev = src + off;
      a->stats.resident_pages++;
    } else {
      psi_status st = page_stream_to(a, src + off, nbytes, flags, cs, &pg);
      if (st != PSI_OK) return st;
      dev = pg.dev;
      if (rows_q) {
        st = page_stream_to(a, src + off + nbytes, static_cast<size_t>(rows_q) * K * 2, flags,
                            cs, &pg2);
        if (st != PSI_OK) return st;
        dev2 = pg2.dev;
      }
    }
    GemmArgs g{};
    g.M = static_cast<int32_t>(N);
    g.N = static_cast<int32_t>(rows_p + rows_q);
    g.n_split = rows_q ? static_cast<int32_t>(rows_p) : 0;
    g.K = static_cast<int32_t>(K);
    g.epi = EPI_LINEAR;
    g.bias_after_bf16 = (flags & PSI_BIAS_AFTER_BF16) ? 1 : 0;
    g.bias = static_cast<const uint16_t*>(bias) + r0;
    g.resid = residual ? static_cast<const uint16_t*>(residual) + r0 : nullptr;
    g.out = static_cast<uint16_t*>(Y) + r0;
    g.ldo = ldy;
    if (rope && rope->cols > r0) {
      g.rope_dh = rope->dh;
      g.rope_cols = static_cast<int32_t>(std::min(rope->cols - r0, rows_p + rows_q));
      g.rope_after_bf16 = (flags & PSI_ROPE_AFTER_BF16) ? 1 : 0;
      g.rope_cos = rope->cos;
      g.rope_sin = rope->sin;
      g.rope_ld = rope->ld;
    }
    g.err = err;
    g.timeout_ns = kWaitLimitNs;
    psi_status st = arena_gemm(a, cs, X, K, dev, K, g, dev2);
    if (st != PSI_OK) return st;
    if (!resident && (st = page_release_on(a, pg, cs)) != PSI_OK) return st;
    if (rows_q && (st = page_release_on(a, pg2, cs)) != PSI_OK) return st;
    p += rows_q ? 2 : 1;
  }
  return stream_after(a->ev_join, a->aux, a->compute);
}

psi_status psi_linear_paged(psi_arena* a, const void* X, int64_t N, int64_t K,
                            const psi_linear_weight* W, const void* bias, const void* residual,
                            void* Y, int64_t ldy, uint32_t flags) {
  return linear_paged(a, X, N, K, W, bias, residual, Y, ldy, flags, nullptr);
}

psi_status psi_linear_rope_paged(psi_arena* a, const void* X, int64_t N, int64_t K,
                                 const psi_linear_weight* W, const void* bias,
                                 const psi_rope* rope, void* Y, int64_t ldy, uint32_t flags) {
  if (!rope) return set_error(PSI_ERR_INVALID_ARG, "linear_rope_paged: null rope table");
  return linear_paged(a, X, N, K, W, bias, nullptr, Y, ldy, flags, rope);
}

psi_status psi_rmsnorm(const void* X, int64_t ldx, int64_t N, int64_t d, const void* gamma,
                       float eps, void* Y, int64_t ldy, void* stream) {
  if (!X || !gamma || !Y) return set_error(PSI_ERR_INVALID_ARG, "rmsnorm: null argument");
  if (N < 0 || d < 1 || d % 8 || ldx < d || ldy < d || ldx % 8 || ldy % 8)
    return set_error(PSI_ERR_INVALID_ARG,
                     "rmsnorm: need d, ldx, ldy multiples of 8 with ldx, ldy >= d");
  if (d > 8192) return set_error(PSI_ERR_UNSUPPORTED, "rmsnorm: this build handles d <= 8192");
  if (!(eps >= 0.0f) || !std::isfinite(eps))
    return set_error(PSI_ERR_INVALID_ARG, "rmsnorm: eps must be finite and >= 0");
  if (!aligned16(X) || !aligned16(Y) || !aligned16(gamma))
    return set_error(PSI_ERR_INVALID_ARG, "rmsnorm: pointers must be 16-byte aligned");
  {
    const auto x0 = reinterpret_cast<uintptr_t>(X), y0 = reinterpret_cast<uintptr_t>(Y);
    const uintptr_t xb = static_cast<uintptr_t>(((N - 1) * ldx + d) * 2);
    const uintptr_t yb = static_cast<uintptr_t>(((N > 0 ? N - 1 : 0) * ldy + d) * 2);
    if (N > 0 && x0 < y0 + yb && y0 < x0 + xb)
      return set_error(PSI_ERR_INVALID_ARG, "rmsnorm: Y must not overlap X");
  }
  if (N > 0x7FFFFFFF) return set_error(PSI_ERR_UNSUPPORTED, "rmsnorm: row count above 2^31");
  if (N == 0) return PSI_OK;
  return launch_rmsnorm(X, ldx, N, d, gamma, eps, Y, ldy, static_cast<cudaStream_t>(stream));
}

psi_status psi_ffn_paged(psi_arena* a, const void* X, int64_t N, const psi_ffn_weight* W,
                         const void* av, const void* bv, void* hidden_ws, void* acc_ws,
                         const void* residual, void* Y, uint32_t flags) {
  return psi_ffn_paged_strided(a, X, N, W, av, bv, hidden_ws, acc_ws, residual, Y,
                               W ? W->r : 0, flags);
}

psi_status psi_ffn_paged_strided(psi_arena* a, const void* X, int64_t N, const psi_ffn_weight* W,
                                 const void* av, const void* bv, void* hidden_ws, void* acc_ws,
                                 const void* residual, void* Y, int64_t ldy, uint32_t flags) {
  psi_status fs = check_flags(flags, kFlagsFfn, "ffn_paged");
  if (fs != PSI_OK) return fs;
  if (!a || !X || !W || !av || !bv || !hidden_ws || !acc_ws || !Y)
    return set_error(PSI_ERR_INVALID_ARG, "ffn_paged: null argument");
  const int64_t d = W->d, h = W->h, r = W->r, sl = W->slice;
  if (N < 0 || d <= 0 || h <= 0 || r <= 0 || sl <= 0 || h % sl)
    return set_error(PSI_ERR_INVALID_ARG, "ffn_paged: bad shape (h must be a multiple of slice)");
  if (d % 8 || r % 8 || sl % 16)
    return set_error(PSI_ERR_INVALID_ARG, "ffn_paged: d, r must be multiples of 8, slice of 16");
  if (ldy < r || ldy % 8)
    return set_error(PSI_ERR_INVALID_ARG, "ffn_paged: ldy must be >= r and a multiple of 8");
  if (!aligned16(X) || !aligned16(Y) || !aligned16(av) || !aligned16(bv) ||
      !aligned16(hidden_ws) || !aligned16(acc_ws) || (residual && !aligned16(residual)))
    return set_error(PSI_ERR_INVALID_ARG, "ffn_paged: pointers must be 16-byte aligned");
  if (N > 0x7FFFFFFF || d > 0x7FFFFFFF || h > 0x7FFFFFFF || r > 0x7FFFFFFF)
    return set_error(PSI_ERR_UNSUPPORTED, "ffn_paged: dimension above 2^31");
  const bool resident = flags & PSI_RESIDENT;
  const char* src = static_cast<const char*>(resident ? W->dev_resident : W->host);
  if (!src)
    return set_error(PSI_ERR_INVALID_ARG, resident ? "ffn_paged: dev_resident is null"
                                                   : "ffn_paged: host is null");
  const size_t pb = psi_ffn_page_bytes(d, r, sl);
  if (!resident && pb > a->page_bytes)
    return set_error(PSI_ERR_CAPACITY, "ffn_paged: FFN weight tile exceeds page");
  const int64_t S = h / sl;
  const int64_t G = ffn_group(S, sl);
  if (!resident && G > a->nslots)
    return set_error(PSI_ERR_CAPACITY, "ffn_paged: a slice group needs " + std::to_string(G) +
                                           " page slots, the arena has " +
                                           std::to_string(a->nslots));
  DevError* err = dev_error_ptr();
  const uint16_t* a16 = static_cast<const uint16_t*>(av);
  uint16_t* hid = static_cast<uint16_t*>(hidden_ws);
  // up projections run on the auxiliary stream, one group ahead of the down
  // projections on the compute stream; hidden buffer g&1 is rewritten only
  // after the down projection of group g-2 has read it
  psi_status fst = stream_after(a->ev_fork, a->compute, a->aux);
  if (fst != PSI_OK) return fst;
  for (int64_t J0 = 0, g = 0; J0 < S; J0 += G, ++g) {
    const int64_t gs = std::min(G, S - J0);
    uint16_t* Hg = hid + static_cast<size_t>(g & 1) * N * G * sl;
    // Streamed, the second group's up projection also waits for the first
    // group's down projection: when the FFN starts, the copy stream is
    // usually blocked on a full ring (the FFN pages queued while attention
    // ran), and the first group, running alone, frees its slots sooner
    // (block step 2.58 -> 2.53 ms; the order of the FP32 accumulation is
    // unchanged)
    if (g >= 2 || (!resident && g == 1)) {
      const int64_t gw = g >= 2 ? g - 2 : 0;
      cudaError_t e = cudaStreamWaitEvent(a->aux, a->ev_down[gw & 1], 0);
      if (e != cudaSuccess) return cuda_error(e, "ffn_paged: wait down projection");
    }
    psi_page pg[kFfnGroupMax]{};
    const char* dev[kFfnGroupMax];
    for (int64_t u = 0; u < gs; ++u) {
      const int64_t J = J0 + u;
      if (resident) {
        dev[u] = src + static_cast<size_t>(J) * pb;
        a->stats.resident_pages++;
      } else {
        psi_status st =
            page_stream_to(a, src + static_cast<size_t>(J) * pb, pb, flags, a->aux, &pg[u]);
        if (st != PSI_OK) return st;
        dev[u] = static_cast<const char*>(pg[u].dev);
      }
    }
    // up projection of the group: H_J = B(phi(X U_J^T + a_J)) for each slice J,
    // one launch over both pages when the slice is a whole number of tiles
    const bool merged = gs > 1 && sl % 256 == 0;
    for (int64_t u = 0; u < gs; u += merged ? gs : 1) {
      const int64_t J = J0 + u;
      GemmArgs up{};
      up.M = static_cast<int32_t>(N);
      up.N = static_cast<int32_t>(merged ? gs * sl : sl);
      up.K = static_cast<int32_t>(d);
      up.n_split = merged ? static_cast<int32_t>(sl) : 0;
      up.epi = EPI_GELU;
      up.pregelu = (flags & PSI_BOUNDARY_PREGELU_BF16) ? 1 : 0;
      up.bias_after_bf16 = (flags & PSI_BIAS_AFTER_BF16) ? 1 : 0;
      up.bias = a16 + J * sl;
      up.out = Hg + u * sl;
      up.ldo = G * sl;
      up.err = err;
      up.timeout_ns = kWaitLimitNs;
      psi_status st = arena_gemm(a, a->aux, X, d, dev[u], d, up, merged ? dev[u + 1] : nullptr);
      if (st != PSI_OK) return st;
    }
    {
      psi_status st = stream_after(a->ev_up[g & 1], a->aux, a->compute);
      if (st != PSI_OK) return st;
    }
    // down projection of the group: Acc (+)= [H_J0 .. H_J0+gs-1] [V_:,J0 .. ]^T,
    // ordered FP32 accumulation over groups; output bias once, at the end
    GemmArgs dn{};
    dn.M = static_cast<int32_t>(N);
    dn.N = static_cast<int32_t>(r);
    dn.K = static_cast<int32_t>(gs * sl);
    dn.k_split = gs > 1 ? static_cast<int32_t>(sl / 64) : 0;
    dn.accf = static_cast<float*>(acc_ws);
    dn.ldacc = r;
    dn.err = err;
    dn.timeout_ns = kWaitLimitNs;
    dn.bias_after_bf16 = (flags & PSI_BIAS_AFTER_BF16) ? 1 : 0;
    const bool first = J0 == 0, last = J0 + gs >= S;
    if (last) {
      dn.epi = first ? EPI_LINEAR : EPI_ACC_FINAL;
      dn.bias = static_cast<const uint16_t*>(bv);
      dn.resid = static_cast<const uint16_t*>(residual);
      dn.out = static_cast<uint16_t*>(Y);
      dn.ldo = ldy;
    } else {
      dn.epi = first ? EPI_ACC_STORE : EPI_ACC_ADD;
    }
    const size_t voff = static_cast<size_t>(sl) * d * 2;
    psi_status st = arena_gemm(a, a->compute, Hg, G * sl, dev[0] + voff, sl, dn,
                               gs > 1 ? dev[1] + voff : nullptr);
    if (st != PSI_OK) return st;
    cudaError_t e = cudaEventRecord(a->ev_down[g & 1], a->compute);
    if (e != cudaSuccess) return cuda_error(e, "ffn_paged: record down projection");
    if (!resident)
      for (int64_t u = 0; u < gs; ++u)
        if ((st = page_release_on(a, pg[u], a->compute)) != PSI_OK) return st;
  }
  return stream_after(a->ev_join, a->aux, a->compute);
}

psi_status psi_attn_workspace_size(int32_t key_block, size_t* bytes) {
  if (!bytes) return set_error(PSI_ERR_INVALID_ARG, "attn_workspace_size: null");
  if (key_block != 128 && key_block != 256)
    return set_error(PSI_ERR_UNSUPPORTED, "attn: key_block must be 128 or 256");
  *bytes = attention_workspace_bytes(key_block);
  return PSI_OK;
}

psi_status psi_attn_partitioned(const psi_heads* Q, const psi_heads* K, const psi_heads* V,
                                const psi_heads* O, int32_t heads, int64_t Nq, int64_t Nk,
                                int32_t dh, float scale, int32_t key_block, void* stream,
                                uint32_t flags) {
  return psi_attn_partitioned_ws(Q, K, V, O, heads, Nq, Nk, dh, scale, key_block, nullptr, 0,
                                 stream, flags);
}

psi_status psi_attn_partitioned_ws(const psi_heads* Q, const psi_heads* K, const psi_heads* V,
                                   const psi_heads* O, int32_t heads, int64_t Nq, int64_t Nk,
                                   int32_t dh, float scale, int32_t key_block, void* workspace,
                                   size_t workspace_bytes, void* stream, uint32_t flags) {
  psi_status fs = check_flags(flags, kFlagsAttn, "attn");
  if (fs != PSI_OK) return fs;
  if (!Q || !K || !V || !O || !O->ptr)
    return set_error(PSI_ERR_INVALID_ARG, "attn: null argument");
  if (heads <= 0 || Nq < 0 || Nk < 1)
    return set_error(PSI_ERR_INVALID_ARG, "attn: need heads >= 1, Nq >= 0 and at least one key");
  if (dh != 128) return set_error(PSI_ERR_UNSUPPORTED, "attn: this build handles dh = 128");
  if (key_block != 128 && key_block != 256)
    return set_error(PSI_ERR_UNSUPPORTED, "attn: key_block must be 128 or 256");
  if (!std::isfinite(scale)) return set_error(PSI_ERR_INVALID_ARG, "attn: scale not finite");
  if (!aligned16(O->ptr) || O->ld_token % 8 || O->ld_head % 8 || O->ld_token < dh)
    return set_error(PSI_ERR_INVALID_ARG, "attn: O rows must be 16-byte aligned");
  if (Nq > 0x7FFFFFFF || Nk > 0x7FFFFFFF)
    return set_error(PSI_ERR_UNSUPPORTED, "attn: token count above 2^31");
  if (Nq == 0) return PSI_OK;
  AttnArgs g{};
  g.heads = heads;
  g.Nq = static_cast<int32_t>(Nq);
  g.Nk = static_cast<int32_t>(Nk);
  g.key_block = key_block;
  g.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  g.bf16_weights = (flags & PSI_ATTN_BF16_WEIGHTS) ? 1 : 0;
  g.O = static_cast<uint16_t*>(O->ptr);
  g.o_ld_token = O->ld_token;
  g.o_ld_head = O->ld_head;
  if (workspace) {
    if (!aligned16(workspace) || workspace_bytes < attention_workspace_bytes(key_block))
      return set_error(PSI_ERR_INVALID_ARG,
                       "attn: workspace must be 16-byte aligned and psi_attn_workspace_size bytes");
    g.part = static_cast<float*>(workspace);
  }
  g.err = dev_error_ptr();
  if (!g.err) return set_error(PSI_ERR_CUDA, "attn: kernel error record not reachable");
  g.timeout_ns = kWaitLimitNs;
  return launch_attention(Q, K, V, g, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
