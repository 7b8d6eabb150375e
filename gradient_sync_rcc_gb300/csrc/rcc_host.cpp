// rcc_host.cpp -- librcc host layer: session registry, argument validation,
// launch planning and the gradient-sync step driver.  Implements include/rcc.h.
//
// Every call validates on the host before it launches anything, in this order:
//   1. the argument arrays themselves (NULL array -> INVALID_ARGUMENT)
//   2. the session handle (dead or unknown -> MISSING_REGISTRATION)
//   3. per-rank counts (SHAPE_MISMATCH), ops (INCONSISTENT_OP),
//      roots (INCONSISTENT_ROOT), broadcast senders (BROADCAST_SENDERS)
//   4. a count of 0 returns RCC_OK here (valid no-op)
//   5. per-rank buffers (NULL -> MISSING_REGISTRATION: that rank did not
//      take part)
//   6. overlaps and other malformed arguments (INVALID_ARGUMENT)
//   7. the current CUDA device against the session's (INVALID_ARGUMENT)
// [ruCCL README §3 "Registration and call contract", §4 "Errors and
// lifecycle"; Monarch "Struct Communicator": each call returns a status.]
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "rcc.h"
#include "rcc_internal.h"

namespace {

using rcc::MultiPtrArgs;

// ---- errors and counters ---------------------------------------------------

thread_local std::string t_err;
std::atomic<uint64_t> g_launches{0};

rcc_status fail(rcc_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return st;
}

rcc_status cuda_fail(cudaError_t e, const char* what) {
  cudaGetLastError();  // clear a sticky launch error so later calls can run
  return fail(RCC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int wait_limit_ms() {
  const char* v = std::getenv("RCC_WAIT_LIMIT_MS");
  if (v && *v) {
    int ms = std::atoi(v);
    if (ms > 0) return ms;
  }
  return 120000;
}

// Wait for an event with a time limit: poll, yield, then back off with short
// sleeps.  Never blocks forever.
rcc_status wait_event(cudaEvent_t ev, const char* what) {
  const auto t0 = std::chrono::steady_clock::now();
  const int limit = wait_limit_ms();
  for (long spins = 0;; ++spins) {
    cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return RCC_OK;
    if (e != cudaErrorNotReady) return cuda_fail(e, what);
    const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                        std::chrono::steady_clock::now() - t0)
                        .count();
    if (ms > limit)
      return fail(RCC_ERR_TIMEOUT, "%s: GPU work did not complete within %d ms", what, limit);
    if (spins < 2000)
      std::this_thread::yield();
    else
      std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

// ---- sessions ----------------------------------------------------------------

constexpr size_t kCombineRegionBytes = 49200;   // 4096 level-1 rows + 4 level-2 rows, 12 B each
constexpr uint64_t kMaxStatsRows = 4096ull * 1024ull;
constexpr uint32_t kDefaultElemsPerRow = 8192;
constexpr uint64_t kFanIn = 1024;

struct Scratch {
  void* rows = nullptr;
  size_t rows_cap = 0;
  void* combine = nullptr;          // the reused reduction region, kCombineRegionBytes
  uint32_t* report_dev = nullptr;   // 12-byte report (16 allocated)
  uint32_t* report_host = nullptr;  // pinned readback slot
  void* desc_dev = nullptr;         // tensor table + grad table + state table
  size_t desc_cap = 0;
  void* desc_host = nullptr;        // pinned staging for the tables
  size_t desc_host_cap = 0;
  std::vector<unsigned char> last_desc;  // bytes most recently uploaded
  cudaEvent_t report_ev = nullptr;
  cudaEvent_t done_ev = nullptr;    // end of the previous call's work
  bool done_recorded = false;
  uint64_t desc_gen = 0;            // bumped at every descriptor upload
  // device decision
  rcc::GsDecision* decision_dev = nullptr;
  rcc::AdamWScalars* scalars_dev = nullptr;
  rcc::AdamWScalars* scalars_host = nullptr;  // pinned staging
  // captured update launches: a fork/join graph of kBranches parallel chains
  static constexpr int kBranches = 8;
  cudaStream_t capture_stream = nullptr;
  cudaStream_t branch[kBranches] = {};
  cudaEvent_t fork_ev = nullptr;
  cudaEvent_t join_ev[kBranches] = {};
  cudaGraphExec_t graph_exec = nullptr;
  uint64_t graph_gen = 0;           // desc_gen the graph was captured for
  size_t graph_P = 0;
};

// Per-rank arrival: one collective at a time collects each rank's arguments;
// the last arrival validates and launches, the others wait for its result.
struct Arrival {
  int kind;  // 0 all_reduce, 1 reduce, 2 broadcast, 3 reduce_scatter, 4 all_gather
  const void* send;
  void* recv;
  size_t count;
  int op;
  int root;
  cudaStream_t stream;
};

struct Pending {
  uint64_t seq = 0;            // number of the collective being collected
  int arrived = 0;
  bool launching = false;      // all ranks in; the last one is launching
  std::vector<char> has;       // per rank: arrived for `seq`
  std::vector<Arrival> args;
  // outcome of the most recently completed collective (seq - 1)
  rcc_status last_status = RCC_OK;
  std::string last_msg;
  bool last_launched = false;
};

struct Session {
  int device;
  int R;
  rcc_dtype dtype;
  std::atomic<unsigned> flags;
  std::mutex mu;  // serialises scratch use and teardown
  Scratch sc;
  std::mutex pmu;  // guards pend and dead
  std::condition_variable pcv;
  Pending pend;
  bool dead = false;  // finished or reset: waiters give up
  std::vector<cudaEvent_t> arr_ev;  // one per rank: the rank's stream at arrival
  cudaEvent_t rank_done_ev = nullptr;  // after the per-rank collective's kernel
  Session(int d, int r, rcc_dtype t, unsigned f) : device(d), R(r), dtype(t), flags(f) {
    pend.has.assign(r, 0);
    pend.args.resize(r);
  }
  ~Session() {
    for (cudaEvent_t e : arr_ev)
      if (e) cudaEventDestroy(e);
    if (rank_done_ev) cudaEventDestroy(rank_done_ev);
  }
};

// Orders a per-rank collective against every rank's stream: the kernel waits
// for the work each rank had queued at arrival, and records rank_done_ev.
struct ArrivalSync {
  Session* s;
  const cudaStream_t* streams;  // [R]
  bool launched = false;
};

void free_scratch(Scratch& s) {
  if (s.rows) cudaFree(s.rows);
  if (s.combine) cudaFree(s.combine);
  if (s.report_dev) cudaFree(s.report_dev);
  if (s.report_host) cudaFreeHost(s.report_host);
  if (s.desc_dev) cudaFree(s.desc_dev);
  if (s.desc_host) cudaFreeHost(s.desc_host);
  if (s.report_ev) cudaEventDestroy(s.report_ev);
  if (s.done_ev) cudaEventDestroy(s.done_ev);
  if (s.decision_dev) cudaFree(s.decision_dev);
  if (s.scalars_dev) cudaFree(s.scalars_dev);
  if (s.scalars_host) cudaFreeHost(s.scalars_host);
  if (s.graph_exec) cudaGraphExecDestroy(s.graph_exec);
  if (s.capture_stream) cudaStreamDestroy(s.capture_stream);
  for (int k = 0; k < Scratch::kBranches; ++k) {
    if (s.branch[k]) cudaStreamDestroy(s.branch[k]);
    if (s.join_ev[k]) cudaEventDestroy(s.join_ev[k]);
  }
  if (s.fork_ev) cudaEventDestroy(s.fork_ev);
  s = Scratch{};
}

constexpr int kSlots = 255;
struct Slot {
  std::shared_ptr<Session> s;
  uint32_t gen = 0;
};
std::mutex g_reg_mu;
Slot g_slots[kSlots];

rcc_comm encode(int slot, uint32_t gen) {
  return reinterpret_cast<rcc_comm>(
      static_cast<uintptr_t>((static_cast<uint64_t>(gen) << 8) | static_cast<uint64_t>(slot + 1)));
}

std::shared_ptr<Session> lookup(rcc_comm h, int* slot_out = nullptr) {
  const uint64_t v = static_cast<uint64_t>(reinterpret_cast<uintptr_t>(h));
  if (v == 0) return nullptr;
  const int slot = static_cast<int>(v & 0xFF) - 1;
  const uint32_t gen = static_cast<uint32_t>(v >> 8);
  if (slot < 0 || slot >= kSlots) return nullptr;
  std::lock_guard<std::mutex> lock(g_reg_mu);
  if (!g_slots[slot].s || g_slots[slot].gen != gen) return nullptr;
  if (slot_out) *slot_out = slot;
  return g_slots[slot].s;
}

// Remove a session from the registry; returns it (nullptr if already gone).
std::shared_ptr<Session> unregister(rcc_comm h) {
  int slot = -1;
  auto s = lookup(h, &slot);
  if (!s) return nullptr;
  std::lock_guard<std::mutex> lock(g_reg_mu);
  if (g_slots[slot].s != s) return nullptr;
  g_slots[slot].s.reset();
  return s;
}

rcc_status missing_session() {
  return fail(RCC_ERR_MISSING_REGISTRATION,
              "session handle is not registered (never registered, finished or reset)");
}

// ---- validation helpers ----------------------------------------------------

size_t elem_bytes(rcc_dtype t) { return t == RCC_F32 ? 4 : 2; }
bool valid_op(int op) { return op >= RCC_SUM && op <= RCC_MIN; }

bool overlap(const void* a, size_t an, const void* b, size_t bn) {
  if (an == 0 || bn == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bn && y < x + an;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte ranges that must not overlap one another; returns the indices of an
// overlapping pair, or {-1, -1}.  Sorting keeps this O(n log n) for the R*R
// outputs of the list all_gather.
struct Span {
  uintptr_t lo, hi;
  int id;
};
std::pair<int, int> first_overlap(std::vector<Span> v) {
  std::sort(v.begin(), v.end(), [](const Span& x, const Span& y) { return x.lo < y.lo; });
  uintptr_t reach = 0;
  int reach_id = -1;
  for (const Span& sp : v) {
    if (sp.hi == sp.lo) continue;
    if (reach_id >= 0 && sp.lo < reach) return {reach_id, sp.id};
    if (sp.hi > reach) {
      reach = sp.hi;
      reach_id = sp.id;
    }
  }
  return {-1, -1};
}

// Byte ranges, each written or only read; returns true if a written range
// overlaps any other range (read-only ranges may overlap each other).
struct RwSpan {
  uintptr_t lo, hi;
  bool written;
};
bool written_overlap(std::vector<RwSpan> v) {
  std::sort(v.begin(), v.end(), [](const RwSpan& x, const RwSpan& y) { return x.lo < y.lo; });
  uintptr_t reach_w = 0, reach_any = 0;
  for (const RwSpan& sp : v) {
    if (sp.hi == sp.lo) continue;
    if (sp.lo < reach_w) return true;                 // inside an earlier written range
    if (sp.written && sp.lo < reach_any) return true;  // a written range inside any earlier one
    if (sp.written && sp.hi > reach_w) reach_w = sp.hi;
    if (sp.hi > reach_any) reach_any = sp.hi;
  }
  return false;
}

rcc_status check_counts(const size_t* counts, int R, size_t* n) {
  for (int r = 1; r < R; ++r)
    if (counts[r] != counts[0])
      return fail(RCC_ERR_SHAPE_MISMATCH, "rank %d has %zu elements, rank 0 has %zu", r,
                  counts[r], counts[0]);
  *n = counts[0];
  return RCC_OK;
}

rcc_status check_ops(const rcc_op* ops, int R) {
  for (int r = 0; r < R; ++r) {
    if (!valid_op(ops[r]))
      return fail(RCC_ERR_INCONSISTENT_OP, "rank %d passes op %d, not an rcc_op", r, (int)ops[r]);
    if (ops[r] != ops[0])
      return fail(RCC_ERR_INCONSISTENT_OP, "rank %d passes op %d, rank 0 passes %d", r,
                  (int)ops[r], (int)ops[0]);
  }
  return RCC_OK;
}

rcc_status check_device(int dev) {
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (cur != dev)
    return fail(RCC_ERR_INVALID_ARGUMENT, "current CUDA device %d is not the session's device %d",
                cur, dev);
  return RCC_OK;
}

rcc::Red red_of(rcc_op op) {
  switch (op) {
    case RCC_MAX: return rcc::kRedMax;
    case RCC_MIN: return rcc::kRedMin;
    default: return rcc::kRedSum;
  }
}

rcc_status launch(const Session& s, rcc::Red red, int nseg, const MultiPtrArgs& a,
                  rcc_stream_t stream, ArrivalSync* sync = nullptr) {
  const bool fast = (s.flags.load() & RCC_DETERMINISTIC) == 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (sync) {
    Session& ms = *sync->s;
    if (ms.arr_ev.empty()) ms.arr_ev.assign(ms.R, nullptr);
    for (int r = 0; r < ms.R; ++r) {
      cudaError_t e = cudaSuccess;
      if (!ms.arr_ev[r]) e = cudaEventCreateWithFlags(&ms.arr_ev[r], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventRecord(ms.arr_ev[r], sync->streams[r]);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ms.arr_ev[r], 0);
      if (e != cudaSuccess) return cuda_fail(e, "arrival ordering");
    }
    if (!ms.rank_done_ev) {
      cudaError_t e = cudaEventCreateWithFlags(&ms.rank_done_ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
    }
  }
  cudaError_t e = s.dtype == RCC_F32 ? rcc::launch_multi_ptr_f32(red, fast, nseg, a, st)
                                     : rcc::launch_multi_ptr_bf16(red, fast, nseg, a, st);
  if (e != cudaSuccess) return cuda_fail(e, "collective kernel launch");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (sync) {
    e = cudaEventRecord(sync->s->rank_done_ev, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    sync->launched = true;
  }
  return RCC_OK;
}

// The widest vector (32 or 16 bytes, else 0) that every base address and
// every per-segment offset is a multiple of.
int vec_ok(const MultiPtrArgs& a, int nsrc_ptrs, int ndst_ptrs, size_t seg_bytes_src,
           size_t seg_bytes_dst) {
  uintptr_t bits = seg_bytes_src | seg_bytes_dst;
  for (int i = 0; i < nsrc_ptrs; ++i) bits |= reinterpret_cast<uintptr_t>(a.src[i]);
  for (int i = 0; i < ndst_ptrs; ++i) bits |= reinterpret_cast<uintptr_t>(a.dst[i]);
  if ((bits & 31u) == 0) return 32;
  if ((bits & 15u) == 0) return 16;
  return 0;
}

}  // namespace

// The session is gone: every rank waiting in a per-rank collective returns
// RCC_ERR_MISSING_REGISTRATION.
static void wake_waiters(Session& s) {
  {
    std::lock_guard<std::mutex> lock(s.pmu);
    s.dead = true;
  }
  s.pcv.notify_all();
}

namespace rcc {
rcc_status set_error(rcc_status st, const char* msg) { return fail(st, "%s", msg); }
void add_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace rcc

// ============================================================================
extern "C" {

const char* rcc_last_error_message(void) { return t_err.c_str(); }

const char* rcc_status_string(rcc_status st) {
  switch (st) {
    case RCC_OK: return "RCC_OK";
    case RCC_ERR_DUPLICATE_REGISTRATION: return "RCC_ERR_DUPLICATE_REGISTRATION";
    case RCC_ERR_MISSING_REGISTRATION: return "RCC_ERR_MISSING_REGISTRATION";
    case RCC_ERR_SHAPE_MISMATCH: return "RCC_ERR_SHAPE_MISMATCH";
    case RCC_ERR_INCONSISTENT_OP: return "RCC_ERR_INCONSISTENT_OP";
    case RCC_ERR_INCONSISTENT_ROOT: return "RCC_ERR_INCONSISTENT_ROOT";
    case RCC_ERR_BROADCAST_SENDERS: return "RCC_ERR_BROADCAST_SENDERS";
    case RCC_ERR_INVALID_ARGUMENT: return "RCC_ERR_INVALID_ARGUMENT";
    case RCC_ERR_TIMEOUT: return "RCC_ERR_TIMEOUT";
    case RCC_ERR_CUDA: return "RCC_ERR_CUDA";
  }
  return "unknown rcc_status";
}

uint64_t rcc_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

// ---- lifecycle ---------------------------------------------------------------

rcc_status rcc_register(int device, int num_ranks, rcc_dtype dtype, unsigned flags,
                        rcc_comm* out) {
  t_err.clear();
  if (!out) return fail(RCC_ERR_INVALID_ARGUMENT, "out is NULL");
  *out = nullptr;
  if (device < 0) return fail(RCC_ERR_INVALID_ARGUMENT, "device %d < 0", device);
  if (num_ranks < 1 || num_ranks > RCC_MAX_RANKS)
    return fail(RCC_ERR_INVALID_ARGUMENT, "num_ranks %d outside [1, %d]", num_ranks,
                RCC_MAX_RANKS);
  if (dtype != RCC_F32 && dtype != RCC_BF16)
    return fail(RCC_ERR_INVALID_ARGUMENT, "dtype %d is not an rcc_dtype", (int)dtype);
  if (flags & ~RCC_DETERMINISTIC)
    return fail(RCC_ERR_INVALID_ARGUMENT, "unknown flag bits 0x%x", flags & ~RCC_DETERMINISTIC);
  std::lock_guard<std::mutex> lock(g_reg_mu);
  int free_slot = -1;
  for (int i = 0; i < kSlots; ++i) {
    if (g_slots[i].s) {
      if (g_slots[i].s->device == device)
        return fail(RCC_ERR_DUPLICATE_REGISTRATION,
                    "device %d already has a live session (finish or reset it first)", device);
    } else if (free_slot < 0) {
      free_slot = i;
    }
  }
  if (free_slot < 0) return fail(RCC_ERR_INVALID_ARGUMENT, "too many live sessions");
  Slot& sl = g_slots[free_slot];
  sl.gen = (sl.gen + 1) & 0x00FFFFFFu;
  if (sl.gen == 0) sl.gen = 1;
  sl.s = std::make_shared<Session>(device, num_ranks, dtype, flags);
  *out = encode(free_slot, sl.gen);
  return RCC_OK;
}

rcc_status rcc_set_flags(rcc_comm comm, unsigned flags) {
  t_err.clear();
  auto s = lookup(comm);
  if (!s) return missing_session();
  if (flags & ~RCC_DETERMINISTIC)
    return fail(RCC_ERR_INVALID_ARGUMENT, "unknown flag bits 0x%x", flags & ~RCC_DETERMINISTIC);
  s->flags.store(flags);
  return RCC_OK;
}

rcc_status rcc_finish(rcc_comm comm, rcc_stream_t stream) {
  t_err.clear();
  auto s = lookup(comm);
  if (!s) return missing_session();
  {
    std::lock_guard<std::mutex> lock(s->mu);
    rcc_status st = check_device(s->device);
    if (st != RCC_OK) return st;
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
    e = cudaEventRecord(ev, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
      cudaEventDestroy(ev);
      return cuda_fail(e, "cudaEventRecord");
    }
    st = wait_event(ev, "rcc_finish");
    cudaEventDestroy(ev);
    if (st != RCC_OK) return st;  // the session stays live: retry or reset
    free_scratch(s->sc);
  }
  unregister(comm);
  wake_waiters(*s);
  // a bulk-copy CTA that gave up waiting leaves its flag raised
  uint32_t f32 = 0, bf16 = 0;
  if (rcc::bulk_copy_timeouts_f32(&f32) == cudaSuccess &&
      rcc::bulk_copy_timeouts_bf16(&bf16) == cudaSuccess && (f32 | bf16))
    return fail(RCC_ERR_TIMEOUT, "a bulk-copy wait gave up: some copy output is incomplete");
  return RCC_OK;
}

rcc_status rcc_reset(rcc_comm comm) {
  t_err.clear();
  auto s = unregister(comm);
  if (!s) return missing_session();
  wake_waiters(*s);  // a half-arrived per-rank collective is discarded
  std::lock_guard<std::mutex> lock(s->mu);
  free_scratch(s->sc);
  return RCC_OK;
}

// ---- collectives ---------------------------------------------------------------

static rcc_status all_reduce_impl(rcc_comm comm, const void* const* send, void* const* recv,
                          const size_t* counts, const rcc_op* ops, rcc_stream_t stream,
    ArrivalSync* sync) {
  t_err.clear();
  if (!send || !recv || !counts || !ops)
    return fail(RCC_ERR_INVALID_ARGUMENT, "send, recv, counts and ops arrays are required");
  auto s = lookup(comm);
  if (!s) return missing_session();
  const int R = s->R;
  size_t n;
  rcc_status st = check_counts(counts, R, &n);
  if (st != RCC_OK) return st;
  if ((st = check_ops(ops, R)) != RCC_OK) return st;
  if (n == 0) return RCC_OK;
  for (int r = 0; r < R; ++r)
    if (!send[r] || !recv[r])
      return fail(RCC_ERR_MISSING_REGISTRATION, "rank %d supplies no %s buffer", r,
                  send[r] ? "recv" : "send");
  const size_t bytes = n * elem_bytes(s->dtype);
  for (int r = 0; r < R; ++r)
    for (int q = 0; q < R; ++q) {
      if (q != r && overlap(recv[r], bytes, recv[q], bytes))
        return fail(RCC_ERR_INVALID_ARGUMENT, "recv buffers of ranks %d and %d overlap", r, q);
      if (overlap(recv[r], bytes, send[q], bytes) && !(q == r && recv[r] == send[r]))
        return fail(RCC_ERR_INVALID_ARGUMENT,
                    "recv of rank %d overlaps send of rank %d (only recv[r] == send[r] may alias)",
                    r, q);
    }
  if ((st = check_device(s->device)) != RCC_OK) return st;
  MultiPtrArgs a{};
  for (int r = 0; r < R; ++r) {
    a.src[r] = send[r];
    a.dst[r] = recv[r];
  }
  a.n = n;
  a.nsrc = a.ndst = R;
  a.mean_div = ops[0] == RCC_MEAN ? R : 0;
  a.vec_ok = vec_ok(a, R, R, 0, 0);
  return launch(*s, red_of(ops[0]), 1, a, stream, sync);
}

rcc_status rcc_all_reduce(rcc_comm comm, const void* const* send, void* const* recv,
                          const size_t* counts, const rcc_op* ops, rcc_stream_t stream) {
  return all_reduce_impl(comm, send, recv, counts, ops, stream, nullptr);
}

static rcc_status reduce_impl(rcc_comm comm, const void* const* send, void* const* recv,
                      const size_t* counts, const rcc_op* ops, const int* roots,
                      rcc_stream_t stream,
    ArrivalSync* sync) {
  t_err.clear();
  if (!send || !recv || !counts || !ops || !roots)
    return fail(RCC_ERR_INVALID_ARGUMENT, "send, recv, counts, ops and roots arrays are required");
  auto s = lookup(comm);
  if (!s) return missing_session();
  const int R = s->R;
  size_t n;
  rcc_status st = check_counts(counts, R, &n);
  if (st != RCC_OK) return st;
  if ((st = check_ops(ops, R)) != RCC_OK) return st;
  for (int r = 0; r < R; ++r) {
    if (roots[r] < 0 || roots[r] >= R)
      return fail(RCC_ERR_INCONSISTENT_ROOT, "rank %d names root %d outside [0, %d)", r, roots[r],
                  R);
    if (roots[r] != roots[0])
      return fail(RCC_ERR_INCONSISTENT_ROOT, "rank %d names root %d, rank 0 names %d", r, roots[r],
                  roots[0]);
  }
  if (n == 0) return RCC_OK;
  const int root = roots[0];
  for (int r = 0; r < R; ++r)
    if (!send[r]) return fail(RCC_ERR_MISSING_REGISTRATION, "rank %d supplies no send buffer", r);
  if (!recv[root])
    return fail(RCC_ERR_MISSING_REGISTRATION, "root rank %d supplies no recv buffer", root);
  const size_t bytes = n * elem_bytes(s->dtype);
  for (int q = 0; q < R; ++q)
    if (overlap(recv[root], bytes, send[q], bytes) && !(q == root && recv[root] == send[root]))
      return fail(RCC_ERR_INVALID_ARGUMENT, "root recv overlaps send of rank %d", q);
  if ((st = check_device(s->device)) != RCC_OK) return st;
  MultiPtrArgs a{};
  for (int r = 0; r < R; ++r) a.src[r] = send[r];
  a.dst[0] = recv[root];
  a.n = n;
  a.nsrc = R;
  a.ndst = 1;
  a.mean_div = ops[0] == RCC_MEAN ? R : 0;
  a.vec_ok = vec_ok(a, R, 1, 0, 0);
  return launch(*s, red_of(ops[0]), 1, a, stream, sync);
}

rcc_status rcc_reduce(rcc_comm comm, const void* const* send, void* const* recv,
                      const size_t* counts, const rcc_op* ops, const int* roots,
                      rcc_stream_t stream) {
  return reduce_impl(comm, send, recv, counts, ops, roots, stream, nullptr);
}

static rcc_status broadcast_impl(rcc_comm comm, const void* const* send, void* const* recv,
                         const size_t* counts, rcc_stream_t stream,
    ArrivalSync* sync) {
  t_err.clear();
  if (!send || !recv || !counts)
    return fail(RCC_ERR_INVALID_ARGUMENT, "send, recv and counts arrays are required");
  auto s = lookup(comm);
  if (!s) return missing_session();
  const int R = s->R;
  size_t n;
  rcc_status st = check_counts(counts, R, &n);
  if (st != RCC_OK) return st;
  int senders = 0, root = -1;
  for (int r = 0; r < R; ++r)
    if (send[r]) {
      ++senders;
      root = r;
    }
  if (senders != 1)
    return fail(RCC_ERR_BROADCAST_SENDERS, "broadcast needs exactly one sender, got %d", senders);
  if (n == 0) return RCC_OK;
  for (int r = 0; r < R; ++r)
    if (r != root && !recv[r])
      return fail(RCC_ERR_MISSING_REGISTRATION, "receiving rank %d supplies no recv buffer", r);
  const size_t bytes = n * elem_bytes(s->dtype);
  MultiPtrArgs a{};
  int nd = 0;
  for (int r = 0; r < R; ++r) {
    if (!recv[r] || recv[r] == send[root]) continue;
    if (overlap(recv[r], bytes, send[root], bytes))
      return fail(RCC_ERR_INVALID_ARGUMENT, "recv of rank %d overlaps the root's send buffer", r);
    for (int q = 0; q < r; ++q)
      if (recv[q] && recv[q] != send[root] && overlap(recv[r], bytes, recv[q], bytes))
        return fail(RCC_ERR_INVALID_ARGUMENT, "recv buffers of ranks %d and %d overlap", q, r);
    a.dst[nd++] = recv[r];
  }
  if (nd == 0) return RCC_OK;  // only the root, in place
  if ((st = check_device(s->device)) != RCC_OK) return st;
  a.src[0] = send[root];
  a.n = n;
  a.nsrc = 1;
  a.ndst = nd;
  a.vec_ok = vec_ok(a, 1, nd, 0, 0);
  return launch(*s, rcc::kRedCopy, 1, a, stream, sync);
}

rcc_status rcc_broadcast(rcc_comm comm, const void* const* send, void* const* recv,
                         const size_t* counts, rcc_stream_t stream) {
  return broadcast_impl(comm, send, recv, counts, stream, nullptr);
}

static rcc_status reduce_scatter_impl(rcc_comm comm, const void* const* send, void* const* recv,
                              const size_t* in_counts, const rcc_op* ops, rcc_stream_t stream,
    ArrivalSync* sync) {
  t_err.clear();
  if (!send || !recv || !in_counts || !ops)
    return fail(RCC_ERR_INVALID_ARGUMENT, "send, recv, in_counts and ops arrays are required");
  auto s = lookup(comm);
  if (!s) return missing_session();
  const int R = s->R;
  size_t N;
  rcc_status st = check_counts(in_counts, R, &N);
  if (st != RCC_OK) return st;
  if (N % (size_t)R != 0)
    return fail(RCC_ERR_SHAPE_MISMATCH, "input count %zu is not a multiple of %d ranks", N, R);
  if ((st = check_ops(ops, R)) != RCC_OK) return st;
  if (N == 0) return RCC_OK;
  for (int r = 0; r < R; ++r)
    if (!send[r] || !recv[r])
      return fail(RCC_ERR_MISSING_REGISTRATION, "rank %d supplies no %s buffer", r,
                  send[r] ? "recv" : "send");
  const size_t es = elem_bytes(s->dtype), n = N / (size_t)R;
  for (int r = 0; r < R; ++r)
    for (int q = 0; q < R; ++q) {
      if (q != r && overlap(recv[r], n * es, recv[q], n * es))
        return fail(RCC_ERR_INVALID_ARGUMENT, "recv buffers of ranks %d and %d overlap", r, q);
      if (overlap(recv[r], n * es, send[q], N * es))
        return fail(RCC_ERR_INVALID_ARGUMENT, "recv of rank %d overlaps send of rank %d", r, q);
    }
  if ((st = check_device(s->device)) != RCC_OK) return st;
  MultiPtrArgs a{};
  for (int r = 0; r < R; ++r) {
    a.src[r] = send[r];
    a.dst[r] = recv[r];
  }
  a.n = n;
  a.nsrc = R;
  a.ndst = 1;
  a.src_seg_stride = n;
  a.dst_per_seg = 1;
  a.mean_div = ops[0] == RCC_MEAN ? R : 0;
  a.vec_ok = vec_ok(a, R, R, n * es, 0);
  return launch(*s, red_of(ops[0]), R, a, stream, sync);
}

rcc_status rcc_reduce_scatter(rcc_comm comm, const void* const* send, void* const* recv,
                              const size_t* in_counts, const rcc_op* ops, rcc_stream_t stream) {
  return reduce_scatter_impl(comm, send, recv, in_counts, ops, stream, nullptr);
}

static rcc_status all_gather_impl(rcc_comm comm, const void* const* send, void* const* recv,
                          const size_t* in_counts, rcc_stream_t stream,
    ArrivalSync* sync) {
  t_err.clear();
  if (!send || !recv || !in_counts)
    return fail(RCC_ERR_INVALID_ARGUMENT, "send, recv and in_counts arrays are required");
  auto s = lookup(comm);
  if (!s) return missing_session();
  const int R = s->R;
  size_t n;
  rcc_status st = check_counts(in_counts, R, &n);
  if (st != RCC_OK) return st;
  if (n == 0) return RCC_OK;
  for (int r = 0; r < R; ++r)
    if (!send[r] || !recv[r])
      return fail(RCC_ERR_MISSING_REGISTRATION, "rank %d supplies no %s buffer", r,
                  send[r] ? "recv" : "send");
  const size_t es = elem_bytes(s->dtype), N = n * (size_t)R;
  for (int r = 0; r < R; ++r)
    for (int q = 0; q < R; ++q) {
      if (q != r && overlap(recv[r], N * es, recv[q], N * es))
        return fail(RCC_ERR_INVALID_ARGUMENT, "recv buffers of ranks %d and %d overlap", r, q);
      // in place: rank q's input may be its own slot q of its own output
      const bool own_slot =
          q == r && send[q] == static_cast<const char*>(recv[r]) + (size_t)q * n * es;
      if (overlap(recv[r], N * es, send[q], n * es) && !own_slot)
        return fail(RCC_ERR_INVALID_ARGUMENT, "recv of rank %d overlaps send of rank %d", r, q);
    }
  if ((st = check_device(s->device)) != RCC_OK) return st;
  MultiPtrArgs a{};
  for (int r = 0; r < R; ++r) {
    a.src[r] = send[r];
    a.dst[r] = recv[r];
  }
  a.n = n;
  a.nsrc = 1;
  a.ndst = R;
  a.src_per_seg = 1;
  a.dst_seg_stride = n;
  a.vec_ok = vec_ok(a, R, R, 0, n * es);
  return launch(*s, rcc::kRedCopy, R, a, stream, sync);
}

rcc_status rcc_all_gather(rcc_comm comm, const void* const* send, void* const* recv,
                          const size_t* in_counts, rcc_stream_t stream) {
  return all_gather_impl(comm, send, recv, in_counts, stream, nullptr);
}

// ---- all_to_all_single and the list all_gather ---------------------------------

rcc_status rcc_all_to_all_single(rcc_comm comm, const void* const* send, void* const* recv,
                                 const size_t* in_counts, rcc_stream_t stream) {
  t_err.clear();
  if (!send || !recv || !in_counts)
    return fail(RCC_ERR_INVALID_ARGUMENT, "send, recv and in_counts arrays are required");
  auto s = lookup(comm);
  if (!s) return missing_session();
  const int R = s->R;
  size_t N;
  rcc_status st = check_counts(in_counts, R, &N);
  if (st != RCC_OK) return st;
  if (N % (size_t)R != 0)
    return fail(RCC_ERR_SHAPE_MISMATCH, "count %zu is not a multiple of %d ranks", N, R);
  if (N == 0) return RCC_OK;
  for (int r = 0; r < R; ++r)
    if (!send[r] || !recv[r])
      return fail(RCC_ERR_MISSING_REGISTRATION, "rank %d supplies no %s buffer", r,
                  send[r] ? "recv" : "send");
  const size_t es = elem_bytes(s->dtype), n = N / (size_t)R;
  std::vector<Span> spans;
  for (int r = 0; r < R; ++r) {
    const uintptr_t o = reinterpret_cast<uintptr_t>(recv[r]);
    spans.push_back({o, o + N * es, r});
  }
  auto ov = first_overlap(spans);
  if (ov.first >= 0)
    return fail(RCC_ERR_INVALID_ARGUMENT, "recv buffers of ranks %d and %d overlap", ov.first,
                ov.second);
  for (int r = 0; r < R; ++r)
    for (int q = 0; q < R; ++q)
      if (overlap(recv[r], N * es, send[q], N * es))
        return fail(RCC_ERR_INVALID_ARGUMENT, "recv of rank %d overlaps send of rank %d", r, q);
  if ((st = check_device(s->device)) != RCC_OK) return st;
  MultiPtrArgs a{};
  for (int r = 0; r < R; ++r) {
    a.src[r] = send[r];
    a.dst[r] = recv[r];
  }
  a.n = n;
  a.nsrc = 1;
  a.ndst = 1;
  a.a2a_ranks = R;
  a.vec_ok = vec_ok(a, R, R, n * es, 0);
  return launch(*s, rcc::kRedCopy, R * R, a, stream);
}

rcc_status rcc_all_gather_list(rcc_comm comm, const void* const* send, void* const* recv,
                               const size_t* in_counts, rcc_stream_t stream) {
  t_err.clear();
  if (!send || !recv || !in_counts)
    return fail(RCC_ERR_INVALID_ARGUMENT, "send, recv and in_counts arrays are required");
  auto s = lookup(comm);
  if (!s) return missing_session();
  const int R = s->R;
  size_t n;
  rcc_status st = check_counts(in_counts, R, &n);
  if (st != RCC_OK) return st;
  if (n == 0) return RCC_OK;
  for (int q = 0; q < R; ++q)
    if (!send[q]) return fail(RCC_ERR_MISSING_REGISTRATION, "rank %d supplies no send buffer", q);
  for (int i = 0; i < R * R; ++i)
    if (!recv[i])
      return fail(RCC_ERR_MISSING_REGISTRATION, "rank %d supplies no output for rank %d's tensor",
                  i / R, i % R);
  const size_t es = elem_bytes(s->dtype), bytes = n * es;
  // outputs disjoint from each other and from every input; rank r's own
  // entry may be its input (in place: nothing to copy)
  auto in_place = [&](int i) { return i / R == i % R && recv[i] == send[i % R]; };
  std::vector<Span> spans;
  for (int i = 0; i < R * R; ++i) {
    if (in_place(i)) continue;
    const uintptr_t o = reinterpret_cast<uintptr_t>(recv[i]);
    spans.push_back({o, o + bytes, i});
  }
  auto ov = first_overlap(spans);
  if (ov.first >= 0)
    return fail(RCC_ERR_INVALID_ARGUMENT, "outputs %d and %d of the list overlap", ov.first,
                ov.second);
  for (int i = 0; i < R * R; ++i)
    for (int q = 0; q < R && !in_place(i); ++q)
      if (overlap(recv[i], bytes, send[q], bytes))
        return fail(RCC_ERR_INVALID_ARGUMENT, "output %d of the list overlaps send of rank %d", i,
                    q);
  if ((st = check_device(s->device)) != RCC_OK) return st;
  // one copy pass per source rank: send[q] -> recv[r*R + q] for every r
  for (int q = 0; q < R; ++q) {
    MultiPtrArgs a{};
    a.src[0] = send[q];
    int nd = 0;
    for (int r = 0; r < R; ++r)
      if (!(r == q && recv[r * R + q] == send[q])) a.dst[nd++] = recv[r * R + q];
    if (nd == 0) continue;
    a.n = n;
    a.nsrc = 1;
    a.ndst = nd;
    a.vec_ok = vec_ok(a, 1, nd, 0, 0);
    if ((st = launch(*s, rcc::kRedCopy, 1, a, stream)) != RCC_OK) return st;
  }
  return RCC_OK;
}

// ---- per-rank arrival ------------------------------------------------------------

}  // extern "C"

namespace {

// Every rank's arguments are in: check they describe one collective and run
// it through the group implementation, ordered against every rank's stream.
rcc_status launch_arrived(rcc_comm comm, const Session& s, const std::vector<Arrival>& args,
                          ArrivalSync* sync, cudaStream_t launch_stream) {
  const int R = s.R;
  for (int r = 1; r < R; ++r)
    if (args[r].kind != args[0].kind)
      return fail(RCC_ERR_INCONSISTENT_OP, "rank %d called a different collective than rank 0", r);
  std::vector<const void*> send(R);
  std::vector<void*> recv(R);
  std::vector<size_t> counts(R);
  std::vector<rcc_op> ops(R);
  std::vector<int> roots(R);
  std::vector<cudaStream_t> streams(R);
  for (int r = 0; r < R; ++r) {
    send[r] = args[r].send;
    recv[r] = args[r].recv;
    counts[r] = args[r].count;
    ops[r] = static_cast<rcc_op>(args[r].op);
    roots[r] = args[r].root;
    streams[r] = args[r].stream;
  }
  sync->streams = streams.data();
  rcc_stream_t st = reinterpret_cast<rcc_stream_t>(launch_stream);
  switch (args[0].kind) {
    case 0: return all_reduce_impl(comm, send.data(), recv.data(), counts.data(), ops.data(), st, sync);
    case 1:
      return reduce_impl(comm, send.data(), recv.data(), counts.data(), ops.data(), roots.data(), st,
                         sync);
    case 2: return broadcast_impl(comm, send.data(), recv.data(), counts.data(), st, sync);
    case 3:
      return reduce_scatter_impl(comm, send.data(), recv.data(), counts.data(), ops.data(), st, sync);
    default: return all_gather_impl(comm, send.data(), recv.data(), counts.data(), st, sync);
  }
}

void complete(Pending& pd) {
  ++pd.seq;
  pd.arrived = 0;
  pd.launching = false;
  std::fill(pd.has.begin(), pd.has.end(), 0);
}

// One rank's arrival: record its arguments; the last rank launches for all,
// the others wait (bounded) for that outcome and order their stream after it.
rcc_status rank_arrive(rcc_comm comm, int rank, const Arrival& a) {
  t_err.clear();
  auto s = lookup(comm);
  if (!s) return missing_session();
  if (rank < 0 || rank >= s->R)
    return fail(RCC_ERR_INVALID_ARGUMENT, "rank %d outside [0, %d)", rank, s->R);
  std::unique_lock<std::mutex> lk(s->pmu);
  if (s->dead) return missing_session();
  Pending& pd = s->pend;
  if (pd.has[rank])
    return fail(RCC_ERR_INVALID_ARGUMENT, "rank %d arrived twice for one collective", rank);
  pd.has[rank] = 1;
  pd.args[rank] = a;
  ++pd.arrived;
  const uint64_t my_seq = pd.seq;
  if (pd.arrived < s->R) {
    const auto deadline =
        std::chrono::steady_clock::now() + std::chrono::milliseconds(wait_limit_ms());
    while (pd.seq == my_seq && !s->dead) {
      if (pd.launching) {
        s->pcv.wait(lk);  // all ranks are in: the outcome is moments away
        continue;
      }
      if (s->pcv.wait_until(lk, deadline) == std::cv_status::timeout && pd.seq == my_seq &&
          !s->dead && !pd.launching) {
        // give up: the collective is discarded for every rank waiting on it
        pd.last_status = RCC_ERR_TIMEOUT;
        pd.last_msg = "not every rank arrived within the wait limit; collective discarded";
        pd.last_launched = false;
        complete(pd);
        lk.unlock();
        s->pcv.notify_all();
        return fail(RCC_ERR_TIMEOUT, "%s", "not every rank arrived within the wait limit; "
                                           "collective discarded");
      }
    }
    if (pd.seq == my_seq) return missing_session();  // finished or reset meanwhile
    const rcc_status st = pd.last_status;
    const std::string msg = pd.last_msg;
    const bool launched = pd.last_launched;
    cudaEvent_t done = s->rank_done_ev;
    lk.unlock();
    if (st != RCC_OK) {
      t_err = msg;
      return st;
    }
    if (launched) {
      cudaError_t e = cudaStreamWaitEvent(a.stream, done, 0);
      if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
    }
    return RCC_OK;
  }
  pd.launching = true;
  const std::vector<Arrival> args = pd.args;
  lk.unlock();
  ArrivalSync sync{s.get(), nullptr};
  const rcc_status st = launch_arrived(comm, *s, args, &sync, a.stream);
  const std::string msg = t_err;
  lk.lock();
  pd.last_status = st;
  pd.last_msg = msg;
  pd.last_launched = sync.launched;
  complete(pd);
  lk.unlock();
  s->pcv.notify_all();
  return st;
}

}  // namespace

extern "C" {

rcc_status rcc_all_reduce_rank(rcc_comm comm, int rank, const void* send, void* recv,
                               size_t count, rcc_op op, rcc_stream_t stream) {
  return rank_arrive(comm, rank,
                     Arrival{0, send, recv, count, (int)op, 0, reinterpret_cast<cudaStream_t>(stream)});
}

rcc_status rcc_reduce_rank(rcc_comm comm, int rank, const void* send, void* recv, size_t count,
                           rcc_op op, int root, rcc_stream_t stream) {
  return rank_arrive(comm, rank, Arrival{1, send, recv, count, (int)op, root,
                                         reinterpret_cast<cudaStream_t>(stream)});
}

rcc_status rcc_broadcast_rank(rcc_comm comm, int rank, const void* send, void* recv,
                              size_t count, rcc_stream_t stream) {
  return rank_arrive(comm, rank,
                     Arrival{2, send, recv, count, 0, 0, reinterpret_cast<cudaStream_t>(stream)});
}

rcc_status rcc_reduce_scatter_rank(rcc_comm comm, int rank, const void* send, void* recv,
                                   size_t in_count, rcc_op op, rcc_stream_t stream) {
  return rank_arrive(comm, rank, Arrival{3, send, recv, in_count, (int)op, 0,
                                         reinterpret_cast<cudaStream_t>(stream)});
}

rcc_status rcc_all_gather_rank(rcc_comm comm, int rank, const void* send, void* recv,
                               size_t in_count, rcc_stream_t stream) {
  return rank_arrive(comm, rank,
                     Arrival{4, send, recv, in_count, 0, 0, reinterpret_cast<cudaStream_t>(stream)});
}

// ---- gradient sync + fused AdamW ------------------------------------------------

}  // extern "C"

namespace {

template <typename T>
rcc_status ensure_dev(T** p, size_t* cap, size_t need, const char* what) {
  if (*p && *cap >= need) return RCC_OK;
  if (*p) cudaFree(*p);
  *p = nullptr;
  *cap = 0;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), need);
  if (e != cudaSuccess) return cuda_fail(e, what);
  *cap = need;
  return RCC_OK;
}

rcc_status ensure_fixed_scratch(Scratch& sc) {
  cudaError_t e;
  if (!sc.combine) {
    e = cudaMalloc(&sc.combine, kCombineRegionBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(combine region)");
  }
  if (!sc.report_dev) {
    e = cudaMalloc(reinterpret_cast<void**>(&sc.report_dev), 16);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(report)");
  }
  if (!sc.report_host) {
    e = cudaMallocHost(reinterpret_cast<void**>(&sc.report_host), 16);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocHost(report)");
  }
  if (!sc.report_ev) {
    e = cudaEventCreateWithFlags(&sc.report_ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
  }
  if (!sc.done_ev) {
    e = cudaEventCreateWithFlags(&sc.done_ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
  }
  return RCC_OK;
}

rcc_status ensure_decision_scratch(Scratch& sc) {
  cudaError_t e;
  if (!sc.decision_dev) {
    e = cudaMalloc(reinterpret_cast<void**>(&sc.decision_dev), sizeof(rcc::GsDecision));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(decision)");
  }
  if (!sc.scalars_dev) {
    e = cudaMalloc(reinterpret_cast<void**>(&sc.scalars_dev), sizeof(rcc::AdamWScalars));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(scalars)");
  }
  if (!sc.scalars_host) {
    e = cudaMallocHost(reinterpret_cast<void**>(&sc.scalars_host), sizeof(rcc::AdamWScalars));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocHost(scalars)");
  }
  return RCC_OK;
}

// Host copy of the device decision kernel: the same IEEE double arithmetic.
void host_decision(double sum_sq, uint32_t nonfinite, double max_grad_norm, double* norm,
                   bool* skip, float* coef) {
  *norm = std::sqrt(sum_sq);
  *skip = nonfinite > 0 || !std::isfinite(*norm);
  *coef = 1.0f;
  if (!*skip && max_grad_norm > 0.0 && *norm > max_grad_norm)
    *coef = (float)(max_grad_norm / *norm);
}

rcc::AdamWScalars step_scalars(const rcc_adamw_cfg* cfg, int64_t t) {
  rcc::AdamWScalars s{};
  const double bc1 = 1.0 - std::pow(cfg->beta1, (double)t);
  const double bc2 = 1.0 - std::pow(cfg->beta2, (double)t);
  s.step_size = (float)(cfg->lr / bc1);
  s.inv_bc2_sqrt = (float)(1.0 / std::sqrt(bc2));
  s.decay = (float)(1.0 - cfg->lr * cfg->weight_decay);
  s.beta1 = (float)cfg->beta1;
  s.one_minus_beta1 = (float)(1.0 - cfg->beta1);
  s.beta2 = (float)cfg->beta2;
  s.one_minus_beta2 = (float)(1.0 - cfg->beta2);
  s.eps = (float)cfg->eps;
  return s;
}

bool finite_pos(double x) { return std::isfinite(x) && x > 0.0; }

}  // namespace

extern "C" {

rcc_status rcc_grad_sync_adamw(rcc_comm comm, const rcc_param_set* params, int num_params,
                               const rcc_adamw_cfg* cfg, rcc_optim_state* state,
                               rcc_step_report* report, rcc_stream_t stream) {
  t_err.clear();
  if (!params || !cfg || !state || num_params < 1)
    return fail(RCC_ERR_INVALID_ARGUMENT, "params, cfg, state and num_params >= 1 are required");
  auto s = lookup(comm);
  if (!s) return missing_session();
  const int R = s->R;
  // shapes must match across ranks [ruCCL §6]
  for (int p = 0; p < num_params; ++p) {
    const rcc_param_set& ps = params[p];
    if (ps.rank_numel)
      for (int r = 0; r < R; ++r)
        if (ps.rank_numel[r] != ps.numel)
          return fail(RCC_ERR_SHAPE_MISMATCH, "tensor %d: rank %d has %zu elements, expected %zu",
                      p, r, ps.rank_numel[r], ps.numel);
  }
  const int rep = cfg->replicas;
  for (int p = 0; p < num_params; ++p) {
    const rcc_param_set& ps = params[p];
    if (!ps.grads)
      return fail(RCC_ERR_MISSING_REGISTRATION, "tensor %d has no grads array", p);
    for (int r = 0; r < R; ++r)
      if (!ps.grads[r])
        return fail(RCC_ERR_MISSING_REGISTRATION, "tensor %d: rank %d supplies no gradient", p, r);
  }
  if (s->dtype != RCC_F32)
    return fail(RCC_ERR_INVALID_ARGUMENT, "gradient sync needs an RCC_F32 session");
  if (rep != 1 && rep != R)
    return fail(RCC_ERR_INVALID_ARGUMENT, "replicas %d must be 1 or %d", rep, R);
  if (cfg->flags & ~(RCC_ADAMW_DEVICE_DECISION | RCC_ADAMW_GRAPH | RCC_ADAMW_MULTI_TENSOR))
    return fail(RCC_ERR_INVALID_ARGUMENT, "unknown cfg->flags bits 0x%x", cfg->flags);
  if ((cfg->flags & RCC_ADAMW_GRAPH) && (cfg->flags & RCC_ADAMW_MULTI_TENSOR))
    return fail(RCC_ERR_INVALID_ARGUMENT, "RCC_ADAMW_GRAPH and RCC_ADAMW_MULTI_TENSOR exclude "
                                          "each other (the multi-tensor update is one launch)");
  if (!finite_pos(cfg->lr) && cfg->lr != 0.0)
    return fail(RCC_ERR_INVALID_ARGUMENT, "lr must be finite and >= 0");
  if (!(cfg->beta1 >= 0.0 && cfg->beta1 < 1.0 && cfg->beta2 >= 0.0 && cfg->beta2 < 1.0))
    return fail(RCC_ERR_INVALID_ARGUMENT, "betas must lie in [0, 1)");
  if (!finite_pos(cfg->eps)) return fail(RCC_ERR_INVALID_ARGUMENT, "eps must be finite and > 0");
  if (!std::isfinite(cfg->weight_decay) || !std::isfinite(cfg->max_grad_norm))
    return fail(RCC_ERR_INVALID_ARGUMENT, "weight_decay and max_grad_norm must be finite");
  const uint32_t epr = cfg->elems_per_row ? cfg->elems_per_row : kDefaultElemsPerRow;
  if (epr % 4 != 0 || epr > (1u << 24))
    return fail(RCC_ERR_INVALID_ARGUMENT, "elems_per_row %u must be a multiple of 4 in [4, 2^24]",
                epr);
  if (!finite_pos(state->scale))
    return fail(RCC_ERR_INVALID_ARGUMENT, "loss scale must be finite and > 0");
  if (state->growth_interval < 1 || !finite_pos(state->growth_factor) ||
      !finite_pos(state->backoff_factor) || state->step < 0)
    return fail(RCC_ERR_INVALID_ARGUMENT, "malformed optimizer/scaler state");
  uint64_t total_rows = 0;
  for (int p = 0; p < num_params; ++p) {
    const rcc_param_set& ps = params[p];
    if (ps.numel == 0) return fail(RCC_ERR_INVALID_ARGUMENT, "tensor %d has 0 elements", p);
    if (!ps.params || !ps.exp_avg || !ps.exp_avg_sq)
      return fail(RCC_ERR_INVALID_ARGUMENT, "tensor %d lacks params/exp_avg/exp_avg_sq arrays", p);
    for (int k = 0; k < rep; ++k)
      if (!ps.params[k] || !ps.exp_avg[k] || !ps.exp_avg_sq[k])
        return fail(RCC_ERR_INVALID_ARGUMENT, "tensor %d: replica %d state pointer is NULL", p, k);
    total_rows += (ps.numel + epr - 1) / epr;
  }
  if (total_rows > kMaxStatsRows)
    return fail(RCC_ERR_INVALID_ARGUMENT,
                "%llu statistics rows exceed %llu (two fan-in-1024 levels); raise elems_per_row",
                (unsigned long long)total_rows, (unsigned long long)kMaxStatsRows);
  rcc_status st = check_device(s->device);
  if (st != RCC_OK) return st;

  std::lock_guard<std::mutex> lock(s->mu);
  Scratch& sc = s->sc;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if ((st = ensure_fixed_scratch(sc)) != RCC_OK) return st;
  if ((st = ensure_dev(&sc.rows, &sc.rows_cap, (size_t)total_rows * 12, "cudaMalloc(rows)")) !=
      RCC_OK)
    return st;

  // descriptor tables: tensors | grad pointers | state pointers
  const size_t P = (size_t)num_params;
  const size_t off_grads = P * sizeof(rcc::GsTensor);
  const size_t off_state = off_grads + P * R * sizeof(void*);
  const size_t desc_bytes = off_state + P * 3 * rep * sizeof(void*);
  const bool dev_grew = !sc.desc_dev || sc.desc_cap < desc_bytes;
  if ((st = ensure_dev(&sc.desc_dev, &sc.desc_cap, desc_bytes, "cudaMalloc(descriptors)")) !=
      RCC_OK)
    return st;
  if (!sc.desc_host || sc.desc_host_cap < desc_bytes) {
    if (sc.desc_host) cudaFreeHost(sc.desc_host);
    sc.desc_host = nullptr;
    cudaError_t e = cudaMallocHost(&sc.desc_host, desc_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocHost(descriptors)");
    sc.desc_host_cap = desc_bytes;
  }
  std::vector<unsigned char> desc(desc_bytes);
  auto* tens = reinterpret_cast<rcc::GsTensor*>(desc.data());
  auto* gtab = reinterpret_cast<const float**>(desc.data() + off_grads);
  auto* stab = reinterpret_cast<float**>(desc.data() + off_state);
  std::vector<int> upd_vec(P);
  uint64_t row = 0;
  for (size_t p = 0; p < P; ++p) {
    const rcc_param_set& ps = params[p];
    bool gv = ps.mean_grad == nullptr || aligned16(ps.mean_grad);
    for (int r = 0; r < R; ++r) {
      gtab[p * R + r] = ps.grads[r];
      gv = gv && aligned16(ps.grads[r]);
    }
    bool uv = gv;
    for (int k = 0; k < rep; ++k) {
      stab[p * 3 * rep + k] = ps.params[k];
      stab[p * 3 * rep + rep + k] = ps.exp_avg[k];
      stab[p * 3 * rep + 2 * rep + k] = ps.exp_avg_sq[k];
      uv = uv && aligned16(ps.params[k]) && aligned16(ps.exp_avg[k]) && aligned16(ps.exp_avg_sq[k]);
    }
    upd_vec[p] = uv ? 1 : 0;
    rcc::GsTensor t{};
    t.numel = ps.numel;
    t.row_begin = row;
    t.mean_grad = ps.mean_grad;
    t.grad_slot = (uint32_t)(p * R);
    t.vec_ok = (gv ? 1u : 0u) | (uv ? 2u : 0u);
    tens[p] = t;
    row += (ps.numel + epr - 1) / epr;
  }
  // the previous call's update kernels may still read the tables
  cudaError_t e;
  if (sc.done_recorded) {
    e = cudaStreamWaitEvent(cs, sc.done_ev, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
  }
  if (sc.last_desc != desc) {
    // new tensors: the state and mean-gradient buffers (written) may not
    // overlap each other or any gradient (gradients are only read)
    std::vector<RwSpan> spans;
    spans.reserve(P * (R + 3 * rep + 1));
    for (size_t p = 0; p < P; ++p) {
      const rcc_param_set& ps = params[p];
      const size_t bytes = ps.numel * sizeof(float);
      auto add = [&](const void* ptr, bool w) {
        const uintptr_t o = reinterpret_cast<uintptr_t>(ptr);
        spans.push_back({o, o + bytes, w});
      };
      for (int r = 0; r < R; ++r) add(ps.grads[r], false);
      for (int k = 0; k < rep; ++k) {
        add(ps.params[k], true);
        add(ps.exp_avg[k], true);
        add(ps.exp_avg_sq[k], true);
      }
      if (ps.mean_grad) add(ps.mean_grad, true);
    }
    if (written_overlap(std::move(spans)))
      return fail(RCC_ERR_INVALID_ARGUMENT,
                  "a parameter, moment or mean-gradient buffer overlaps another buffer");
  }
  if (dev_grew || sc.last_desc != desc) {
    std::memcpy(sc.desc_host, desc.data(), desc_bytes);
    e = cudaMemcpyAsync(sc.desc_dev, sc.desc_host, desc_bytes, cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) return cuda_fail(e, "descriptor upload");
    sc.last_desc.swap(desc);
    ++sc.desc_gen;
  }
  const bool on_device = (cfg->flags & (RCC_ADAMW_DEVICE_DECISION | RCC_ADAMW_GRAPH)) != 0;
  const int64_t t_next = state->step + 1;
  if (on_device) {
    // the scalars of step t+1; used only if the device decides not to skip
    if ((st = ensure_decision_scratch(sc)) != RCC_OK) return st;
    *sc.scalars_host = step_scalars(cfg, t_next);
    sc.scalars_host->inv_scale = (float)(1.0 / state->scale);
    e = cudaMemcpyAsync(sc.scalars_dev, sc.scalars_host, sizeof(rcc::AdamWScalars),
                        cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) return cuda_fail(e, "scalar upload");
  }
  const char* dbase = static_cast<const char*>(sc.desc_dev);
  const float inv_scale = (float)(1.0 / state->scale);

  // statistics pass + hierarchy
  rcc::GsStatsArgs ga{};
  ga.tensors = reinterpret_cast<const rcc::GsTensor*>(dbase);
  ga.grads = reinterpret_cast<const float* const*>(dbase + off_grads);
  ga.rows = static_cast<uint32_t*>(sc.rows);
  ga.total_rows = total_rows;
  ga.num_tensors = (uint32_t)P;
  ga.elems_per_row = epr;
  ga.R = R;
  ga.inv_scale = inv_scale;
  if ((e = rcc::launch_gs_stats(ga, cs)) != cudaSuccess) return cuda_fail(e, "statistics kernel");
  g_launches.fetch_add(1, std::memory_order_relaxed);

  const uint32_t* src = static_cast<const uint32_t*>(sc.rows);
  uint64_t rows = total_rows;
  int levels = 0;
  uint64_t region_bytes = 0;
  if (cfg->hierarchical_stats) {
    uint32_t* region = static_cast<uint32_t*>(sc.combine);
    while (rows > kFanIn) {
      // level 1 writes rows [0, 4096) of the region, level 2 rows [4096, 4100)
      uint32_t* out = region + (levels == 0 ? 0 : 4096 * 3);
      const uint64_t out_rows = (rows + kFanIn - 1) / kFanIn;
      if ((e = rcc::launch_gs_combine(src, rows, out, cs)) != cudaSuccess)
        return cuda_fail(e, "combine kernel");
      g_launches.fetch_add(1, std::memory_order_relaxed);
      region_bytes = (levels == 0 ? 0 : 4096 * 12) + out_rows * 12;
      src = out;
      rows = out_rows;
      ++levels;
    }
  }
  if ((e = rcc::launch_gs_report(src, rows, sc.report_dev, cs)) != cudaSuccess)
    return cuda_fail(e, "report kernel");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if ((e = cudaMemcpyAsync(sc.report_host, sc.report_dev, 12, cudaMemcpyDeviceToHost, cs)) !=
      cudaSuccess)
    return cuda_fail(e, "report readback");
  if ((e = cudaEventRecord(sc.report_ev, cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");

  // One update kernel per tensor, spread over parallel chains forked from
  // (and joined back into) `origin`: largest tensors first onto the least
  // loaded chain.  The tensors are disjoint (checked above), so their kernels
  // may run concurrently and the many small ones no longer queue one behind
  // another.
  rcc::GsUpdateArgs ua{};
  ua.R = R;
  ua.replicas = rep;
  ua.inv_scale = inv_scale;
  auto enqueue_one = [&](size_t p, cudaStream_t where) -> cudaError_t {
    ua.state = reinterpret_cast<float* const*>(dbase + off_state) + p * 3 * rep;
    ua.mean_grad = params[p].mean_grad;
    ua.grads = reinterpret_cast<const float* const*>(dbase + off_grads) + p * R;
    ua.numel = params[p].numel;
    ua.vec_ok = upd_vec[p];
    return rcc::launch_gs_update(ua, where);
  };
  auto enqueue_branched = [&](cudaStream_t origin) -> cudaError_t {
    cudaError_t le;
    if (!sc.fork_ev && (le = cudaEventCreateWithFlags(&sc.fork_ev, cudaEventDisableTiming)))
      return le;
    for (int k = 0; k < Scratch::kBranches; ++k) {
      if (!sc.branch[k] &&
          (le = cudaStreamCreateWithFlags(&sc.branch[k], cudaStreamNonBlocking)) != cudaSuccess)
        return le;
      if (!sc.join_ev[k] &&
          (le = cudaEventCreateWithFlags(&sc.join_ev[k], cudaEventDisableTiming)) != cudaSuccess)
        return le;
    }
    if ((le = cudaEventRecord(sc.fork_ev, origin)) != cudaSuccess) return le;
    for (int k = 0; k < Scratch::kBranches; ++k)
      if ((le = cudaStreamWaitEvent(sc.branch[k], sc.fork_ev, 0)) != cudaSuccess) return le;
    std::vector<size_t> order(P);
    for (size_t p = 0; p < P; ++p) order[p] = p;
    std::stable_sort(order.begin(), order.end(),
                     [&](size_t x, size_t y) { return params[x].numel > params[y].numel; });
    uint64_t load[Scratch::kBranches] = {};
    for (size_t p : order) {
      int k = 0;
      for (int j = 1; j < Scratch::kBranches; ++j)
        if (load[j] < load[k]) k = j;
      load[k] += params[p].numel;
      if ((le = enqueue_one(p, sc.branch[k])) != cudaSuccess) return le;
    }
    for (int k = 0; k < Scratch::kBranches; ++k) {
      if ((le = cudaEventRecord(sc.join_ev[k], sc.branch[k])) != cudaSuccess) return le;
      if ((le = cudaStreamWaitEvent(origin, sc.join_ev[k], 0)) != cudaSuccess) return le;
    }
    return cudaSuccess;
  };

  const bool multi = (cfg->flags & RCC_ADAMW_MULTI_TENSOR) != 0;
  auto enqueue_multi = [&](cudaStream_t where) -> cudaError_t {
    rcc::GsMultiUpdateArgs ma{};
    ma.tensors = reinterpret_cast<const rcc::GsTensor*>(dbase);
    ma.grads = reinterpret_cast<const float* const*>(dbase + off_grads);
    ma.state = reinterpret_cast<float* const*>(dbase + off_state);
    ma.total_rows = total_rows;
    ma.num_tensors = (uint32_t)P;
    ma.elems_per_row = epr;
    ma.R = R;
    ma.replicas = rep;
    ma.inv_scale = ua.inv_scale;
    ma.clip_coef = ua.clip_coef;
    ma.s = ua.s;
    ma.decision = ua.decision;
    ma.dev_scalars = ua.dev_scalars;
    return rcc::launch_gs_update_multi(ma, where);
  };
  const uint64_t launches_per_update = multi ? 1 : P;

  uint64_t device_updates = 0;
  if (on_device) {
    // decide on the GPU and enqueue the updates behind it, before waiting
    if ((e = rcc::launch_gs_decide(sc.report_dev, cfg->max_grad_norm, sc.decision_dev, cs)) !=
        cudaSuccess)
      return cuda_fail(e, "decision kernel");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    ua.clip_coef = 1.0f;
    ua.decision = sc.decision_dev;
    ua.dev_scalars = sc.scalars_dev;
    if (cfg->flags & RCC_ADAMW_GRAPH) {
      if (!sc.graph_exec || sc.graph_gen != sc.desc_gen || sc.graph_P != P) {
        // capture the P update launches once for these tables
        if (sc.graph_exec) cudaGraphExecDestroy(sc.graph_exec);
        sc.graph_exec = nullptr;
        if (!sc.capture_stream &&
            (e = cudaStreamCreateWithFlags(&sc.capture_stream, cudaStreamNonBlocking)) != cudaSuccess)
          return cuda_fail(e, "cudaStreamCreate");
        if ((e = cudaStreamBeginCapture(sc.capture_stream, cudaStreamCaptureModeThreadLocal)) !=
            cudaSuccess)
          return cuda_fail(e, "cudaStreamBeginCapture");
        cudaError_t le = enqueue_branched(sc.capture_stream);
        cudaGraph_t graph = nullptr;
        e = cudaStreamEndCapture(sc.capture_stream, &graph);
        if (le != cudaSuccess) {
          if (graph) cudaGraphDestroy(graph);
          return cuda_fail(le, "update capture");
        }
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture");
        e = cudaGraphInstantiate(&sc.graph_exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGraphInstantiate");
        sc.graph_gen = sc.desc_gen;
        sc.graph_P = P;
      }
      if ((e = cudaGraphLaunch(sc.graph_exec, cs)) != cudaSuccess)
        return cuda_fail(e, "cudaGraphLaunch");
    } else {
      if ((e = multi ? enqueue_multi(cs) : enqueue_branched(cs)) != cudaSuccess)
        return cuda_fail(e, "update kernel");
    }
    device_updates = launches_per_update;
    g_launches.fetch_add(launches_per_update, std::memory_order_relaxed);
  }
  if ((st = wait_event(sc.report_ev, "12-byte report readback")) != RCC_OK) return st;

  // the decision [RUDA docs, native PyTorch section]: skip on non-finite,
  // clip after unscale when the global norm exceeds max_grad_norm
  uint64_t bits = ((uint64_t)sc.report_host[1] << 32) | sc.report_host[0];
  double sum_sq;
  std::memcpy(&sum_sq, &bits, 8);
  const uint32_t nonfinite = sc.report_host[2];
  double norm;
  bool skip;
  float coef;
  host_decision(sum_sq, nonfinite, cfg->max_grad_norm, &norm, &skip, &coef);

  rcc_step_report rep_out{};
  rep_out.sum_sq = sum_sq;
  rep_out.grad_norm = norm;
  rep_out.scale_used = state->scale;
  rep_out.nonfinite = nonfinite;
  rep_out.skipped = skip ? 1 : 0;
  rep_out.clip_coef = skip ? 1.0f : coef;
  rep_out.combine_launches = levels;
  rep_out.stats_rows = total_rows;
  rep_out.combine_region_bytes = region_bytes;

  rep_out.update_launches = device_updates;
  if (skip) {
    state->scale *= state->backoff_factor;
    state->growth_tracker = 0;
  } else if (on_device) {
    state->step = t_next;
    state->growth_tracker += 1;
    if (state->growth_tracker >= state->growth_interval) {
      state->scale *= state->growth_factor;
      state->growth_tracker = 0;
    }
  } else {
    const int64_t t = t_next;
    ua.s = step_scalars(cfg, t);
    ua.clip_coef = coef;
    if ((e = multi ? enqueue_multi(cs) : enqueue_branched(cs)) != cudaSuccess)
      return cuda_fail(e, "update kernel");
    g_launches.fetch_add(launches_per_update, std::memory_order_relaxed);
    rep_out.update_launches = launches_per_update;
    state->step = t;
    state->growth_tracker += 1;
    if (state->growth_tracker >= state->growth_interval) {
      state->scale *= state->growth_factor;
      state->growth_tracker = 0;
    }
  }
  if ((e = cudaEventRecord(sc.done_ev, cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  sc.done_recorded = true;
  if (report) *report = rep_out;
  return RCC_OK;
}

}  // extern "C"
