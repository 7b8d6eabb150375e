// rcc_rank.cpp -- per-rank arrival: one host thread (and one stream) per
// logical rank calls the *_rank entry points; the last arrival validates the
// set and launches once for everyone.  [ruCCL README introduction and §1:
// the in_process implementation; §3: matching collectives in the same order;
// §4: reset discards in-flight operation state.]
#include "host_internal.h"

using namespace rcc::host;


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
  rcc::NvtxRange nvtx_range("rcc_all_reduce_rank");
  return rank_arrive(comm, rank,
                     Arrival{0, send, recv, count, (int)op, 0, reinterpret_cast<cudaStream_t>(stream)});
}

rcc_status rcc_reduce_rank(rcc_comm comm, int rank, const void* send, void* recv, size_t count,
                           rcc_op op, int root, rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_reduce_rank");
  return rank_arrive(comm, rank, Arrival{1, send, recv, count, (int)op, root,
                                         reinterpret_cast<cudaStream_t>(stream)});
}

rcc_status rcc_broadcast_rank(rcc_comm comm, int rank, const void* send, void* recv,
                              size_t count, rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_broadcast_rank");
  return rank_arrive(comm, rank,
                     Arrival{2, send, recv, count, 0, 0, reinterpret_cast<cudaStream_t>(stream)});
}

rcc_status rcc_reduce_scatter_rank(rcc_comm comm, int rank, const void* send, void* recv,
                                   size_t in_count, rcc_op op, rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_reduce_scatter_rank");
  return rank_arrive(comm, rank, Arrival{3, send, recv, in_count, (int)op, 0,
                                         reinterpret_cast<cudaStream_t>(stream)});
}

rcc_status rcc_all_gather_rank(rcc_comm comm, int rank, const void* send, void* recv,
                               size_t in_count, rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_all_gather_rank");
  return rank_arrive(comm, rank,
                     Arrival{4, send, recv, in_count, 0, 0, reinterpret_cast<cudaStream_t>(stream)});
}


}  // extern "C"
