// rcc_host.cpp -- librcc host layer: session registry and lifecycle, argument
// validation and launch planning of the group collectives, diagnostics.  The
// per-rank entry points live in rcc_rank.cpp, the gradient-sync driver in
// rcc_gradsync_host.cpp, shared helpers in host_internal.h.
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
#include "host_internal.h"

using namespace rcc::host;

// services for the entry points defined in the CUDA translation units
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
  rcc::NvtxRange nvtx_range("rcc_register");
  t_err.clear();
  if (!out) return fail(RCC_ERR_INVALID_ARGUMENT, "out is NULL");
  *out = nullptr;
  if (device < 0) return fail(RCC_ERR_INVALID_ARGUMENT, "device %d < 0", device);
  if (num_ranks < 1 || num_ranks > RCC_MAX_RANKS)
    return fail(RCC_ERR_INVALID_ARGUMENT, "num_ranks %d outside [1, %d]", num_ranks,
                RCC_MAX_RANKS);
  if (dtype != RCC_F32 && dtype != RCC_BF16)
    return fail(RCC_ERR_INVALID_ARGUMENT, "dtype %d is not an rcc_dtype", (int)dtype);
  if (flags & ~kSessionFlags)
    return fail(RCC_ERR_INVALID_ARGUMENT, "unknown flag bits 0x%x", flags & ~kSessionFlags);
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
  rcc::NvtxRange nvtx_range("rcc_set_flags");
  t_err.clear();
  auto s = lookup(comm);
  if (!s) return missing_session();
  if (flags & ~kSessionFlags)
    return fail(RCC_ERR_INVALID_ARGUMENT, "unknown flag bits 0x%x", flags & ~kSessionFlags);
  s->flags.store(flags);
  return RCC_OK;
}

rcc_status rcc_finish(rcc_comm comm, rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_finish");
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
  return RCC_OK;
}

rcc_status rcc_reset(rcc_comm comm) {
  rcc::NvtxRange nvtx_range("rcc_reset");
  t_err.clear();
  auto s = unregister(comm);
  if (!s) return missing_session();
  wake_waiters(*s);  // a half-arrived per-rank collective is discarded
  std::lock_guard<std::mutex> lock(s->mu);
  free_scratch(s->sc);
  return RCC_OK;
}

// ---- collectives ---------------------------------------------------------------

}  // extern "C"

namespace rcc {
namespace host {
rcc_status all_reduce_impl(rcc_comm comm, const void* const* send, void* const* recv,
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
}  // namespace host
}  // namespace rcc

extern "C" {

rcc_status rcc_all_reduce(rcc_comm comm, const void* const* send, void* const* recv,
                          const size_t* counts, const rcc_op* ops, rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_all_reduce");
  return all_reduce_impl(comm, send, recv, counts, ops, stream, nullptr);
}

}  // extern "C"

namespace rcc {
namespace host {
rcc_status reduce_impl(rcc_comm comm, const void* const* send, void* const* recv,
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
}  // namespace host
}  // namespace rcc

extern "C" {

rcc_status rcc_reduce(rcc_comm comm, const void* const* send, void* const* recv,
                      const size_t* counts, const rcc_op* ops, const int* roots,
                      rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_reduce");
  return reduce_impl(comm, send, recv, counts, ops, roots, stream, nullptr);
}

}  // extern "C"

namespace rcc {
namespace host {
rcc_status broadcast_impl(rcc_comm comm, const void* const* send, void* const* recv,
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
}  // namespace host
}  // namespace rcc

extern "C" {

rcc_status rcc_broadcast(rcc_comm comm, const void* const* send, void* const* recv,
                         const size_t* counts, rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_broadcast");
  return broadcast_impl(comm, send, recv, counts, stream, nullptr);
}

}  // extern "C"

namespace rcc {
namespace host {
rcc_status reduce_scatter_impl(rcc_comm comm, const void* const* send, void* const* recv,
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
  set_layout(a, R, R, n * es, rcc::kStageSources);
  return launch(*s, red_of(ops[0]), R, a, stream, sync);
}
}  // namespace host
}  // namespace rcc

extern "C" {

rcc_status rcc_reduce_scatter(rcc_comm comm, const void* const* send, void* const* recv,
                              const size_t* in_counts, const rcc_op* ops, rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_reduce_scatter");
  return reduce_scatter_impl(comm, send, recv, in_counts, ops, stream, nullptr);
}

}  // extern "C"

namespace rcc {
namespace host {
rcc_status all_gather_impl(rcc_comm comm, const void* const* send, void* const* recv,
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
  set_layout(a, R, R, n * es, rcc::kStageDestinations);
  return launch(*s, rcc::kRedCopy, R, a, stream, sync);
}
}  // namespace host
}  // namespace rcc

extern "C" {

rcc_status rcc_all_gather(rcc_comm comm, const void* const* send, void* const* recv,
                          const size_t* in_counts, rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_all_gather");
  return all_gather_impl(comm, send, recv, in_counts, stream, nullptr);
}

// ---- all_to_all_single and the list all_gather ---------------------------------

rcc_status rcc_all_to_all_single(rcc_comm comm, const void* const* send, void* const* recv,
                                 const size_t* in_counts, rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_all_to_all_single");
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
  set_layout(a, R, R, n * es, rcc::kStageDestinations);
  return launch(*s, rcc::kRedCopy, R * R, a, stream);
}

rcc_status rcc_all_gather_list(rcc_comm comm, const void* const* send, void* const* recv,
                               const size_t* in_counts, rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_all_gather_list");
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
}  // extern "C"
