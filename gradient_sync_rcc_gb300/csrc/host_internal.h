// host_internal.h -- state and helpers shared by the host layer's translation
// units (rcc_host.cpp: sessions and collectives; rcc_rank.cpp: per-rank
// arrival; rcc_gradsync_host.cpp: the gradient-sync driver).  Not public.
#pragma once

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

namespace rcc {
namespace host {

using rcc::MultiPtrArgs;

// ---- errors and counters ---------------------------------------------------

inline thread_local std::string t_err;
inline std::atomic<uint64_t> g_launches{0};

inline rcc_status fail(rcc_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return st;
}

inline rcc_status cuda_fail(cudaError_t e, const char* what) {
  cudaGetLastError();  // clear a sticky launch error so later calls can run
  return fail(RCC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

inline int wait_limit_ms() {
  const char* v = std::getenv("RCC_WAIT_LIMIT_MS");
  if (v && *v) {
    int ms = std::atoi(v);
    if (ms > 0) return ms;
  }
  return 120000;
}

// The default grad-sync flow replays its per-tensor update launches from a
// captured graph once the same tensors come back (RCC_AUTO_GRAPH=0: never).
inline bool auto_graph_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("RCC_AUTO_GRAPH");
    return !(v && v[0] == '0');
  }();
  return on;
}

// Parallel chains of the per-tensor update launches: RCC_CHAINS (1..32),
// default 16 (measured best with 24; 8 and 32 were slower).
inline int chain_count() {
  static const int n = [] {
    const char* v = std::getenv("RCC_CHAINS");
    const int k = v ? std::atoi(v) : 16;
    return k < 1 ? 1 : (k > 32 ? 32 : k);
  }();
  return n;
}

// Wait for an event with a time limit; never blocks forever.  Polls with
// yields for the first 20 ms (a grad-sync readback waits for a statistics pass
// of up to a few ms and sits on the step's critical path), then sleeps 50 us
// between polls up to the limit.
inline rcc_status wait_event(cudaEvent_t ev, const char* what) {
  const auto t0 = std::chrono::steady_clock::now();
  const int limit = wait_limit_ms();
  for (;;) {
    cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return RCC_OK;
    if (e != cudaErrorNotReady) return cuda_fail(e, what);
    const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                        std::chrono::steady_clock::now() - t0)
                        .count();
    if (ms > limit)
      return fail(RCC_ERR_TIMEOUT, "%s: GPU work did not complete within %d ms", what, limit);
    if (ms < 20)
      std::this_thread::yield();
    else
      std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

// Wait (bounded, as wait_event) for the 12-byte report: the kernel that writes
// it stores the call's sequence number to `seq_word` in the mapped host slot
// once the report words are visible there.  `ev`, recorded after that kernel,
// is queried between polls so that a failed kernel is reported at once; once
// it has completed the word must hold `seq`.
inline rcc_status wait_report_word(const uint32_t* seq_word, uint32_t seq, cudaEvent_t ev,
                                   const char* what) {
  const auto t0 = std::chrono::steady_clock::now();
  const int limit = wait_limit_ms();
  for (uint32_t polls = 0;; ++polls) {
    if (__atomic_load_n(seq_word, __ATOMIC_ACQUIRE) == seq) return RCC_OK;
    if ((polls & 15u) == 15u) {
      cudaError_t e = cudaEventQuery(ev);
      if (e == cudaSuccess) {
        if (__atomic_load_n(seq_word, __ATOMIC_ACQUIRE) == seq) return RCC_OK;
        return fail(RCC_ERR_CUDA, "%s: the report kernel completed without writing the report",
                    what);
      }
      if (e != cudaErrorNotReady) return cuda_fail(e, what);
    }
    const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                        std::chrono::steady_clock::now() - t0)
                        .count();
    if (ms > limit)
      return fail(RCC_ERR_TIMEOUT, "%s: GPU work did not complete within %d ms", what, limit);
    if (ms >= 20) std::this_thread::sleep_for(std::chrono::microseconds(50));
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
  uint32_t* report_host = nullptr;  // pinned, mapped readback slot: 3 report words + seq
  uint32_t report_seq = 0;          // sequence number of the last call's report
  uint32_t* report_host_dev = nullptr;  // its device alias (the report kernel writes it), or
                                        // null: then a 12-byte D2H copy fills the slot
  void* desc_dev = nullptr;         // tensor table + grad table + state table
  size_t desc_cap = 0;
  void* desc_host = nullptr;        // pinned, mapped staging for the tables
  void* desc_host_dev = nullptr;    // its device alias (null: copied by DMA)
  size_t desc_host_cap = 0;
  std::vector<unsigned char> last_desc;  // bytes most recently uploaded
  cudaEvent_t report_ev = nullptr;
  cudaEvent_t done_ev = nullptr;    // end of the previous call's work
  bool done_recorded = false;
  // a call gave up waiting for its report: its GPU work (which reads the host
  // staging and the tables) may still be pending, up to done_ev
  bool stale = false;
  uint64_t desc_gen = 0;            // bumped at every descriptor upload
  uint64_t same_tables = 0;         // consecutive calls with unchanged tables
  // device decision
  rcc::GsDecision* decision_dev = nullptr;
  rcc::AdamWScalars* scalars_dev = nullptr;
  rcc::AdamWScalars* scalars_host = nullptr;  // pinned, mapped staging
  rcc::AdamWScalars* scalars_host_dev = nullptr;
  rcc::GsDecision* decision_host = nullptr;   // pinned, mapped staging of a host decision
  rcc::GsDecision* decision_host_dev = nullptr;
  // per-tensor update launches on up to kMaxBranches parallel fork/join
  // chains (chain_count() of them), also the shape of the captured graph
  static constexpr int kMaxBranches = 32;
  cudaStream_t capture_stream = nullptr;
  cudaStream_t branch[kMaxBranches] = {};
  cudaEvent_t fork_ev = nullptr;
  cudaEvent_t join_ev[kMaxBranches] = {};
  // RCC_STEP_TIMING: events around the phases of the last grad-sync call
  static constexpr int kTimeEvents = 5;
  cudaEvent_t time_ev[kTimeEvents] = {};
  bool timed = false;               // the last call recorded all of them
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

inline void free_scratch(Scratch& s) {
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
  if (s.decision_host) cudaFreeHost(s.decision_host);
  if (s.graph_exec) cudaGraphExecDestroy(s.graph_exec);
  if (s.capture_stream) cudaStreamDestroy(s.capture_stream);
  for (int k = 0; k < Scratch::kMaxBranches; ++k) {
    if (s.branch[k]) cudaStreamDestroy(s.branch[k]);
    if (s.join_ev[k]) cudaEventDestroy(s.join_ev[k]);
  }
  if (s.fork_ev) cudaEventDestroy(s.fork_ev);
  for (int k = 0; k < Scratch::kTimeEvents; ++k)
    if (s.time_ev[k]) cudaEventDestroy(s.time_ev[k]);
  s = Scratch{};
}

constexpr int kSlots = 255;
struct Slot {
  std::shared_ptr<Session> s;
  uint32_t gen = 0;
};
inline std::mutex g_reg_mu;
inline Slot g_slots[kSlots];

inline rcc_comm encode(int slot, uint32_t gen) {
  return reinterpret_cast<rcc_comm>(
      static_cast<uintptr_t>((static_cast<uint64_t>(gen) << 8) | static_cast<uint64_t>(slot + 1)));
}

inline std::shared_ptr<Session> lookup(rcc_comm h, int* slot_out = nullptr) {
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
inline std::shared_ptr<Session> unregister(rcc_comm h) {
  int slot = -1;
  auto s = lookup(h, &slot);
  if (!s) return nullptr;
  std::lock_guard<std::mutex> lock(g_reg_mu);
  if (g_slots[slot].s != s) return nullptr;
  g_slots[slot].s.reset();
  return s;
}

inline rcc_status missing_session() {
  return fail(RCC_ERR_MISSING_REGISTRATION,
              "session handle is not registered (never registered, finished or reset)");
}

// ---- validation helpers ----------------------------------------------------

inline size_t elem_bytes(rcc_dtype t) { return t == RCC_F32 ? 4 : 2; }
inline bool valid_op(int op) { return op >= RCC_SUM && op <= RCC_MIN; }
constexpr unsigned kSessionFlags = RCC_DETERMINISTIC | RCC_STEP_TIMING;

inline bool overlap(const void* a, size_t an, const void* b, size_t bn) {
  if (an == 0 || bn == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bn && y < x + an;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// Byte ranges that must not overlap one another; returns the indices of an
// overlapping pair, or {-1, -1}.  Sorting keeps this O(n log n) for the R*R
// outputs of the list all_gather.
struct Span {
  uintptr_t lo, hi;
  int id;
};
inline std::pair<int, int> first_overlap(std::vector<Span> v) {
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
inline bool written_overlap(std::vector<RwSpan> v) {
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

inline rcc_status check_counts(const size_t* counts, int R, size_t* n) {
  for (int r = 1; r < R; ++r)
    if (counts[r] != counts[0])
      return fail(RCC_ERR_SHAPE_MISMATCH, "rank %d has %zu elements, rank 0 has %zu", r,
                  counts[r], counts[0]);
  *n = counts[0];
  return RCC_OK;
}

inline rcc_status check_ops(const rcc_op* ops, int R) {
  for (int r = 0; r < R; ++r) {
    if (!valid_op(ops[r]))
      return fail(RCC_ERR_INCONSISTENT_OP, "rank %d passes op %d, not an rcc_op", r, (int)ops[r]);
    if (ops[r] != ops[0])
      return fail(RCC_ERR_INCONSISTENT_OP, "rank %d passes op %d, rank 0 passes %d", r,
                  (int)ops[r], (int)ops[0]);
  }
  return RCC_OK;
}

inline rcc_status check_device(int dev) {
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (cur != dev)
    return fail(RCC_ERR_INVALID_ARGUMENT, "current CUDA device %d is not the session's device %d",
                cur, dev);
  return RCC_OK;
}

inline rcc::Red red_of(rcc_op op) {
  switch (op) {
    case RCC_MAX: return rcc::kRedMax;
    case RCC_MIN: return rcc::kRedMin;
    default: return rcc::kRedSum;
  }
}

// Picks the build object of the pass: the pairwise tree applies to sums over
// 4..8 sources (with fewer the tree is the rank-order fold; a runtime rank
// count folds in rank order).
template <int DT>
inline cudaError_t launch_multi_ptr_t(rcc::Red red, bool fast, int nseg, const MultiPtrArgs& a,
                                      cudaStream_t st) {
  using rcc::mp::launch_part;
  switch (red) {
    case rcc::kRedSum:
      if (fast && !a.src_per_seg && a.nsrc >= 4 && a.nsrc <= 8)
        return launch_part<DT, rcc::kRedSum, true>(nseg, a, st);
      return launch_part<DT, rcc::kRedSum, false>(nseg, a, st);
    case rcc::kRedMax: return launch_part<DT, rcc::kRedMax, false>(nseg, a, st);
    case rcc::kRedMin: return launch_part<DT, rcc::kRedMin, false>(nseg, a, st);
    case rcc::kRedCopy: return launch_part<DT, rcc::kRedCopy, false>(nseg, a, st);
  }
  return cudaErrorInvalidValue;
}

inline cudaError_t launch_multi_ptr(int dt, rcc::Red red, bool fast, int nseg,
                                    const MultiPtrArgs& a, cudaStream_t st) {
  return dt == 0 ? launch_multi_ptr_t<0>(red, fast, nseg, a, st)
                 : launch_multi_ptr_t<1>(red, fast, nseg, a, st);
}

inline rcc_status launch(const Session& s, rcc::Red red, int nseg, const MultiPtrArgs& a,
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
  cudaError_t e = launch_multi_ptr(s.dtype == RCC_F32 ? 0 : 1, red, fast, nseg, a, st);
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
inline int vec_ok(const MultiPtrArgs& a, int nsrc_ptrs, int ndst_ptrs, size_t seg_bytes_src,
           size_t seg_bytes_dst) {
  uintptr_t bits = seg_bytes_src | seg_bytes_dst;
  for (int i = 0; i < nsrc_ptrs; ++i) bits |= reinterpret_cast<uintptr_t>(a.src[i]);
  for (int i = 0; i < ndst_ptrs; ++i) bits |= reinterpret_cast<uintptr_t>(a.dst[i]);
  if ((bits & 31u) == 0) return 32;
  if ((bits & 15u) == 0) return 16;
  return 0;
}

// Sets a.vec_ok and a.stage for segments at offsets that are multiples of
// seg_bytes.  When those offsets break a 16-byte alignment that the base
// addresses have, the staged kernels align `side` within each segment instead
// of falling back to scalar accesses everywhere.
inline void set_layout(MultiPtrArgs& a, int nsrc_ptrs, int ndst_ptrs, size_t seg_bytes,
                       rcc::Stage side) {
  const int full = vec_ok(a, nsrc_ptrs, ndst_ptrs, seg_bytes, 0);
  const int base = vec_ok(a, nsrc_ptrs, ndst_ptrs, 0, 0);
  a.stage = rcc::kStageNone;
  a.vec_ok = full;
  if (full < 16 && base >= 16) {
    a.vec_ok = base;
    a.stage = side;
  }
}

// The session is gone: every rank waiting in a per-rank collective returns
// RCC_ERR_MISSING_REGISTRATION.
inline void wake_waiters(Session& s) {
  {
    std::lock_guard<std::mutex> lock(s.pmu);
    s.dead = true;
  }
  s.pcv.notify_all();
}

// the group collectives' implementations, also run by the per-rank path
rcc_status all_reduce_impl(rcc_comm comm, const void* const* send, void* const* recv,
                           const size_t* counts, const rcc_op* ops, rcc_stream_t stream,
                           ArrivalSync* sync);
rcc_status reduce_impl(rcc_comm comm, const void* const* send, void* const* recv,
                       const size_t* counts, const rcc_op* ops, const int* roots,
                       rcc_stream_t stream, ArrivalSync* sync);
rcc_status broadcast_impl(rcc_comm comm, const void* const* send, void* const* recv,
                          const size_t* counts, rcc_stream_t stream, ArrivalSync* sync);
rcc_status reduce_scatter_impl(rcc_comm comm, const void* const* send, void* const* recv,
                               const size_t* in_counts, const rcc_op* ops, rcc_stream_t stream,
                               ArrivalSync* sync);
rcc_status all_gather_impl(rcc_comm comm, const void* const* send, void* const* recv,
                           const size_t* in_counts, rcc_stream_t stream, ArrivalSync* sync);

}  // namespace host
}  // namespace rcc
