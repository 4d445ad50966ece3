// journal.cpp -- the indexed host BF16 journal (C ABI of include/psi.h).
//
// Paper: Precision-Preserving Subtensor Inference, section II-D (inactive
// state is kept in a host journal indexed by block, branch and tensor role;
// the D2H copy waits for the producer, the host commit waits for the D2H
// copy, a reload keeps the consumer dependencies) and section III-B (the
// journal transport runs asynchronously through pinned host memory, so
// state copies overlap compute).
//
// Host side only: the pinned region is cut into equal slots, a key maps to
// a slot, and every copy is ordered by CUDA events against the arena's
// compute stream and the journal's two copy streams.  Device-range hazards
// of the journal's own copies (a reload into memory that a commit is still
// reading, a commit of memory a reload is still writing) are tracked here,
// so callers only fence before their own kernels write committed memory.
#include <algorithm>
#include <chrono>
#include <map>
#include <string>
#include <thread>
#include <tuple>
#include <vector>
#include "internal.h"

namespace psi {
cudaStream_t arena_compute_stream(psi_arena* a);
int arena_device(psi_arena* a);
}  // namespace psi

using namespace psi;

namespace {

struct Slot {
  size_t off = 0;
  size_t bytes = 0;           // committed size (0: free)
  cudaEvent_t written = nullptr;  // last D2H into the slot complete
  cudaEvent_t read = nullptr;     // last H2D out of the slot complete
  bool has_written = false;
  bool has_read = false;
  bool reload_pending = false;    // a reload not yet acquired
};

// A journal copy still in flight on a device range.
struct Pending {
  uintptr_t lo, hi;
  cudaEvent_t done;
  bool device_write;  // H2D (writes the range) or D2H (reads it)
};

using Key = std::tuple<int32_t, int32_t, int32_t>;

}  // namespace

struct psi_journal {
  psi_arena* arena = nullptr;
  int device = 0;
  char* host = nullptr;
  size_t host_bytes = 0;
  size_t slot_bytes = 0;
  std::vector<Slot> slots;
  std::vector<int> free_slots;
  std::map<Key, int> index;
  cudaStream_t d2h = nullptr, h2d = nullptr;
  cudaEvent_t point = nullptr;  // scratch: a position of the compute stream
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> pool;
  psi_journal_stats stats{};
  bool fail_next = false;
};

namespace {

psi_status mk_event(cudaEvent_t* e) {
  cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
  return r == cudaSuccess ? PSI_OK : cuda_error(r, "cudaEventCreate");
}

cudaEvent_t pool_take(psi_journal* j) {
  if (!j->pool.empty()) {
    cudaEvent_t e = j->pool.back();
    j->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  return mk_event(&e) == PSI_OK ? e : nullptr;
}

// Retire finished copies from the hazard list.
void prune(psi_journal* j) {
  size_t k = 0;
  for (size_t i = 0; i < j->pending.size(); ++i) {
    if (cudaEventQuery(j->pending[i].done) == cudaSuccess) {
      j->pool.push_back(j->pending[i].done);
    } else {
      j->pending[k++] = j->pending[i];
    }
  }
  j->pending.resize(k);
  (void)cudaGetLastError();  // a not-ready query leaves no sticky error
}

// `s` waits for every pending journal copy overlapping [lo, hi) whose kind
// matches (device writes, device reads, or both).
psi_status wait_hazards(psi_journal* j, cudaStream_t s, uintptr_t lo, uintptr_t hi,
                        bool writes, bool reads) {
  for (const Pending& p : j->pending) {
    if (p.hi <= lo || hi <= p.lo) continue;
    if ((p.device_write && !writes) || (!p.device_write && !reads)) continue;
    cudaError_t e = cudaStreamWaitEvent(s, p.done, 0);
    if (e != cudaSuccess) return cuda_error(e, "cudaStreamWaitEvent");
    j->stats.hazard_waits++;
  }
  return PSI_OK;
}

psi_status track(psi_journal* j, cudaStream_t s, const void* p, size_t bytes, bool write) {
  cudaEvent_t e = pool_take(j);
  if (!e) return set_error(PSI_ERR_CUDA, "journal: cudaEventCreate failed");
  cudaError_t r = cudaEventRecord(e, s);
  if (r != cudaSuccess) {
    j->pool.push_back(e);
    return cuda_error(r, "cudaEventRecord");
  }
  const auto lo = reinterpret_cast<uintptr_t>(p);
  j->pending.push_back({lo, lo + bytes, e, write});
  return PSI_OK;
}

// `s` waits for the compute stream's current position.
psi_status after_compute(psi_journal* j, cudaStream_t s) {
  cudaError_t e = cudaEventRecord(j->point, arena_compute_stream(j->arena));
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, j->point, 0);
  return e == cudaSuccess ? PSI_OK : cuda_error(e, "journal: compute-stream dependency");
}

bool key_ok(const psi_key& k) { return k.block >= 0 && k.branch >= 0 && k.role >= 0; }

psi_status find(psi_journal* j, const psi_key& k, const char* what, int* slot) {
  if (!key_ok(k)) return set_error(PSI_ERR_INVALID_ARG, std::string(what) + ": negative key");
  auto it = j->index.find(Key{k.block, k.branch, k.role});
  if (it == j->index.end())
    return set_error(PSI_ERR_INVALID_ARG,
                     std::string(what) + ": no entry for key (" + std::to_string(k.block) +
                         ", " + std::to_string(k.branch) + ", " + std::to_string(k.role) + ")");
  *slot = it->second;
  return PSI_OK;
}

void destroy_all(psi_journal* j) {
  for (Slot& s : j->slots) {
    if (s.written) cudaEventDestroy(s.written);
    if (s.read) cudaEventDestroy(s.read);
  }
  for (Pending& p : j->pending) cudaEventDestroy(p.done);
  for (cudaEvent_t e : j->pool) cudaEventDestroy(e);
  if (j->point) cudaEventDestroy(j->point);
  if (j->d2h) cudaStreamDestroy(j->d2h);
  if (j->h2d) cudaStreamDestroy(j->h2d);
}

}  // namespace

extern "C" {

psi_status psi_journal_create(psi_arena* arena, void* host_base, size_t host_bytes,
                              size_t slot_bytes, psi_journal** out) {
  if (!arena || !host_base || !out) return set_error(PSI_ERR_INVALID_ARG, "journal: null argument");
  *out = nullptr;
  if (slot_bytes == 0 || slot_bytes % 256 || host_bytes < slot_bytes)
    return set_error(PSI_ERR_INVALID_ARG,
                     "journal: slot_bytes must be a positive multiple of 256 and fit host_bytes");
  if (reinterpret_cast<uintptr_t>(host_base) & 15)
    return set_error(PSI_ERR_INVALID_ARG, "journal: host region must be 16-byte aligned");
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, host_base);
  if (e != cudaSuccess || attr.type != cudaMemoryTypeHost) {
    (void)cudaGetLastError();
    return set_error(PSI_ERR_INVALID_ARG, "journal: host region is not pinned host memory");
  }
  const size_t n = host_bytes / slot_bytes;
  if (n > 0x7FFFFFFF) return set_error(PSI_ERR_UNSUPPORTED, "journal: too many slots");
  auto* j = new psi_journal();
  j->arena = arena;
  j->device = arena_device(arena);
  j->host = static_cast<char*>(host_base);
  j->host_bytes = host_bytes;
  j->slot_bytes = slot_bytes;
  j->slots.resize(n);
  psi_status st = PSI_OK;
  for (size_t i = 0; i < n && st == PSI_OK; ++i) {
    j->slots[i].off = i * slot_bytes;
    st = mk_event(&j->slots[i].written);
    if (st == PSI_OK) st = mk_event(&j->slots[i].read);
  }
  for (size_t i = n; i-- > 0;) j->free_slots.push_back(static_cast<int>(i));
  if (st == PSI_OK) st = mk_event(&j->point);
  if (st == PSI_OK) {
    e = cudaStreamCreateWithFlags(&j->d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&j->h2d, cudaStreamNonBlocking);
    if (e != cudaSuccess) st = cuda_error(e, "journal: cudaStreamCreate");
  }
  if (st != PSI_OK) {
    destroy_all(j);
    delete j;
    return st;
  }
  j->stats.slots_total = static_cast<int32_t>(n);
  *out = j;
  return PSI_OK;
}

psi_status psi_journal_destroy(psi_journal* j) {
  if (!j) return set_error(PSI_ERR_INVALID_ARG, "journal: null");
  cudaError_t e1 = cudaStreamSynchronize(j->d2h);
  cudaError_t e2 = cudaStreamSynchronize(j->h2d);
  destroy_all(j);
  delete j;
  if (e1 != cudaSuccess) return cuda_error(e1, "journal: D2H stream");
  if (e2 != cudaSuccess) return cuda_error(e2, "journal: H2D stream");
  return PSI_OK;
}

psi_status psi_journal_commit(psi_journal* j, psi_key key, const void* dev_src, size_t bytes) {
  if (!j || !dev_src) return set_error(PSI_ERR_INVALID_ARG, "journal_commit: null argument");
  if (!key_ok(key)) return set_error(PSI_ERR_INVALID_ARG, "journal_commit: negative key");
  if (bytes == 0) return set_error(PSI_ERR_INVALID_ARG, "journal_commit: empty tensor");
  if (bytes > j->slot_bytes)
    return set_error(PSI_ERR_CAPACITY, "journal_commit: " + std::to_string(bytes) +
                                           " bytes exceed the slot size " +
                                           std::to_string(j->slot_bytes));
  const Key k{key.block, key.branch, key.role};
  auto it = j->index.find(k);
  int slot;
  if (it != j->index.end()) {
    slot = it->second;
  } else {
    if (j->free_slots.empty())
      return set_error(PSI_ERR_CAPACITY, "journal_commit: every slot holds an entry");
    slot = j->free_slots.back();
  }
  if (j->fail_next) {
    j->fail_next = false;
    return set_error(PSI_ERR_CUDA, "journal_commit: injected copy failure");
  }
  prune(j);
  Slot& s = j->slots[slot];
  // producer, then the slot's last reader, then any reload still writing
  // the source range
  psi_status st = after_compute(j, j->d2h);
  if (st != PSI_OK) return st;
  cudaError_t e = cudaSuccess;
  if (s.has_read) e = cudaStreamWaitEvent(j->d2h, s.read, 0);
  if (e != cudaSuccess) return cuda_error(e, "cudaStreamWaitEvent");
  const auto lo = reinterpret_cast<uintptr_t>(dev_src);
  if ((st = wait_hazards(j, j->d2h, lo, lo + bytes, true, false)) != PSI_OK) return st;
  e = cudaMemcpyAsync(j->host + s.off, dev_src, bytes, cudaMemcpyDeviceToHost, j->d2h);
  if (e != cudaSuccess) return cuda_error(e, "journal_commit: cudaMemcpyAsync");
  e = cudaEventRecord(s.written, j->d2h);
  if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord");
  if ((st = track(j, j->d2h, dev_src, bytes, false)) != PSI_OK) return st;
  if (it == j->index.end()) {
    j->free_slots.pop_back();
    j->index.emplace(k, slot);
    j->stats.slots_in_use++;
  }
  s.bytes = bytes;
  s.has_written = true;
  s.reload_pending = false;
  j->stats.commits++;
  j->stats.d2h_bytes += bytes;
  return PSI_OK;
}

psi_status psi_journal_reload(psi_journal* j, psi_key key, void* dev_dst, size_t bytes) {
  if (!j || !dev_dst) return set_error(PSI_ERR_INVALID_ARG, "journal_reload: null argument");
  int slot;
  psi_status st = find(j, key, "journal_reload", &slot);
  if (st != PSI_OK) return st;
  Slot& s = j->slots[slot];
  if (bytes != s.bytes)
    return set_error(PSI_ERR_INVALID_ARG, "journal_reload: size differs from the entry (" +
                                              std::to_string(s.bytes) + " bytes)");
  if (j->fail_next) {
    j->fail_next = false;
    return set_error(PSI_ERR_CUDA, "journal_reload: injected copy failure");
  }
  prune(j);
  // consumers of the destination, the entry's D2H copy, journal reads of
  // the destination range
  if ((st = after_compute(j, j->h2d)) != PSI_OK) return st;
  cudaError_t e = cudaStreamWaitEvent(j->h2d, s.written, 0);
  if (e != cudaSuccess) return cuda_error(e, "cudaStreamWaitEvent");
  const auto lo = reinterpret_cast<uintptr_t>(dev_dst);
  if ((st = wait_hazards(j, j->h2d, lo, lo + bytes, false, true)) != PSI_OK) return st;
  e = cudaMemcpyAsync(dev_dst, j->host + s.off, bytes, cudaMemcpyHostToDevice, j->h2d);
  if (e != cudaSuccess) return cuda_error(e, "journal_reload: cudaMemcpyAsync");
  e = cudaEventRecord(s.read, j->h2d);
  if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord");
  if ((st = track(j, j->h2d, dev_dst, bytes, true)) != PSI_OK) return st;
  s.has_read = true;
  s.reload_pending = true;
  j->stats.reloads++;
  j->stats.h2d_bytes += bytes;
  return PSI_OK;
}

psi_status psi_journal_acquire(psi_journal* j, psi_key key) {
  if (!j) return set_error(PSI_ERR_INVALID_ARG, "journal_acquire: null");
  int slot;
  psi_status st = find(j, key, "journal_acquire", &slot);
  if (st != PSI_OK) return st;
  Slot& s = j->slots[slot];
  if (!s.reload_pending)
    return set_error(PSI_ERR_INVALID_ARG, "journal_acquire: no reload of this entry to wait for");
  cudaError_t e = cudaStreamWaitEvent(arena_compute_stream(j->arena), s.read, 0);
  if (e != cudaSuccess) return cuda_error(e, "cudaStreamWaitEvent");
  s.reload_pending = false;
  return PSI_OK;
}

psi_status psi_journal_fence(psi_journal* j, const void* dev_ptr, size_t bytes) {
  if (!j || !dev_ptr) return set_error(PSI_ERR_INVALID_ARG, "journal_fence: null argument");
  prune(j);
  const auto lo = reinterpret_cast<uintptr_t>(dev_ptr);
  return wait_hazards(j, arena_compute_stream(j->arena), lo, lo + bytes, true, true);
}

psi_status psi_journal_drop(psi_journal* j, psi_key key) {
  if (!j) return set_error(PSI_ERR_INVALID_ARG, "journal_drop: null");
  int slot;
  psi_status st = find(j, key, "journal_drop", &slot);
  if (st != PSI_OK) return st;
  j->index.erase(Key{key.block, key.branch, key.role});
  Slot& s = j->slots[slot];
  s.bytes = 0;
  s.reload_pending = false;
  j->free_slots.push_back(slot);  // its next commit waits for s.read
  j->stats.slots_in_use--;
  return PSI_OK;
}

psi_status psi_journal_host_view(psi_journal* j, psi_key key, int64_t timeout_ms,
                                 const void** host_ptr, size_t* bytes) {
  if (!j || !host_ptr || !bytes) return set_error(PSI_ERR_INVALID_ARG, "journal_host_view: null");
  int slot;
  psi_status st = find(j, key, "journal_host_view", &slot);
  if (st != PSI_OK) return st;
  const Slot& s = j->slots[slot];
  j->stats.host_waits++;
  const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms);
  while (true) {
    cudaError_t e = cudaEventQuery(s.written);
    if (e == cudaSuccess) break;
    if (e != cudaErrorNotReady) return cuda_error(e, "journal_host_view");
    if (timeout_ms >= 0 && std::chrono::steady_clock::now() > deadline)
      return set_error(PSI_ERR_TIMEOUT, "journal_host_view: D2H copy not finished in time");
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  *host_ptr = j->host + s.off;
  *bytes = s.bytes;
  return PSI_OK;
}

psi_status psi_journal_get_stats(const psi_journal* j, psi_journal_stats* out) {
  if (!j || !out) return set_error(PSI_ERR_INVALID_ARG, "journal_get_stats: null");
  *out = j->stats;
  return PSI_OK;
}

psi_status psi_journal_fail_next_copy(psi_journal* j) {
  if (!j) return set_error(PSI_ERR_INVALID_ARG, "journal_fail_next_copy: null");
  j->fail_next = true;
  return PSI_OK;
}

}  // extern "C"
