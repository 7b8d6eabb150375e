// rcc_gradsync_host.cpp -- the gradient-sync + fused AdamW step driver
// (rcc_grad_sync_adamw): validation, descriptor tables, the statistics
// hierarchy, the report readback, the host or device decision, and the
// per-tensor update launches.  [ruCCL README §6; RUDA docs "Training and
// saving state", native PyTorch section.]
#include "host_internal.h"

using namespace rcc::host;


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

// Pinned host staging mapped into the device's address space; *alias is
// null when no device alias can be had (the upload then goes by DMA).
template <typename T>
cudaError_t alloc_mapped(T** host, T** alias, size_t bytes) {
  cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(host), bytes, cudaHostAllocMapped);
  if (e != cudaSuccess) return e;
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, *host, 0) == cudaSuccess)
    *alias = static_cast<T*>(d);
  else
    (void)cudaGetLastError();
  return cudaSuccess;
}

// Host staging -> device memory on `cs`.  A small kernel reads the staging
// through its device alias: a copy-engine transfer would queue behind large
// host<->device copies that the caller may have in flight on other streams
// (a 64 MiB transfer holds a 4 KB table back by about 0.3 ms).
static_assert(sizeof(rcc::AdamWScalars) % 4 == 0 && sizeof(rcc::GsDecision) % 4 == 0,
              "uploads move whole 32-bit words");
static_assert(sizeof(rcc::GsTensor) % 8 == 0, "descriptor tables are whole 64-bit words");

cudaError_t upload(void* dst, const void* host, const void* alias, size_t bytes, cudaStream_t cs) {
  if (alias) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return rcc::launch_host_upload(alias, dst, bytes, cs);
  }
  return cudaMemcpyAsync(dst, host, bytes, cudaMemcpyHostToDevice, cs);
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
    e = cudaHostAlloc(reinterpret_cast<void**>(&sc.report_host), 16, cudaHostAllocMapped);
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc(report)");
    std::memset(sc.report_host, 0, 16);
    sc.report_seq = 0;
    // the report kernel stores the 12 bytes straight into this slot, so no
    // copy is queued between the report and the host's wait
    void* alias = nullptr;
    if (cudaHostGetDevicePointer(&alias, sc.report_host, 0) == cudaSuccess)
      sc.report_host_dev = static_cast<uint32_t*>(alias);
    else
      (void)cudaGetLastError();
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
    e = alloc_mapped(&sc.scalars_host, &sc.scalars_host_dev, sizeof(rcc::AdamWScalars));
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc(scalars)");
  }
  if (!sc.decision_host) {
    e = alloc_mapped(&sc.decision_host, &sc.decision_host_dev, sizeof(rcc::GsDecision));
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc(decision)");
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
  rcc::NvtxRange nvtx_range("rcc_grad_sync_adamw");
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
  if (cfg->flags & ~(RCC_ADAMW_DEVICE_DECISION | RCC_ADAMW_GRAPH | RCC_ADAMW_MULTI_TENSOR |
                     RCC_ADAMW_HOST_GRAPH))
    return fail(RCC_ERR_INVALID_ARGUMENT, "unknown cfg->flags bits 0x%x", cfg->flags);
  if ((cfg->flags & RCC_ADAMW_HOST_GRAPH) && (cfg->flags & ~RCC_ADAMW_HOST_GRAPH))
    return fail(RCC_ERR_INVALID_ARGUMENT, "RCC_ADAMW_HOST_GRAPH takes no other flag (it is the "
                                          "host decision with the captured update launches)");
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
  if (cfg->hierarchical_stats < 0 || cfg->hierarchical_stats > 1)
    return fail(RCC_ERR_INVALID_ARGUMENT, "hierarchical_stats %d must be 0 or 1",
                cfg->hierarchical_stats);
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
  if (sc.stale) {
    // the previous call timed out with work still queued that reads the
    // staging memory and tables rewritten below: let it finish first
    if ((st = wait_event(sc.done_ev, "the previous call's GPU work")) != RCC_OK) return st;
    sc.stale = false;
  }
  if ((st = ensure_fixed_scratch(sc)) != RCC_OK) return st;
  const bool on_device = (cfg->flags & (RCC_ADAMW_DEVICE_DECISION | RCC_ADAMW_GRAPH)) != 0;
  const bool timing = (s->flags.load() & RCC_STEP_TIMING) != 0;
  sc.timed = false;
  if (timing) {
    for (int k = 0; k < Scratch::kTimeEvents; ++k) {
      if (sc.time_ev[k]) continue;
      cudaError_t te = cudaEventCreate(&sc.time_ev[k]);
      if (te != cudaSuccess) return cuda_fail(te, "cudaEventCreate(timing)");
    }
  }
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
    sc.desc_host_dev = nullptr;
    cudaError_t e = alloc_mapped(&sc.desc_host, &sc.desc_host_dev, desc_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc(descriptors)");
    sc.desc_host_cap = desc_bytes;
  }
  std::vector<unsigned char> desc(desc_bytes);
  auto* tens = reinterpret_cast<rcc::GsTensor*>(desc.data());
  auto* gtab = reinterpret_cast<const float**>(desc.data() + off_grads);
  auto* stab = reinterpret_cast<float**>(desc.data() + off_state);
  std::vector<int> upd_vec(P);
  // 32-byte statistics vectors need rows that start on 8 elements
  // (RCC_VEC_BYTES=16 caps every kernel at 16-byte vectors)
  static const bool wide_ok = [] {
    const char* v = std::getenv("RCC_VEC_BYTES");
    return !(v && std::atoi(v) == 16);
  }();
  const bool rows8 = wide_ok && epr % 8 == 0;
  uint64_t row = 0;
  for (size_t p = 0; p < P; ++p) {
    const rcc_param_set& ps = params[p];
    bool gv = ps.mean_grad == nullptr || aligned16(ps.mean_grad);
    bool gv32 = rows8 && (ps.mean_grad == nullptr || aligned32(ps.mean_grad));
    bool grads32 = true;
    for (int r = 0; r < R; ++r) {
      gtab[p * R + r] = ps.grads[r];
      gv = gv && aligned16(ps.grads[r]);
      grads32 = grads32 && aligned32(ps.grads[r]);
    }
    gv32 = gv32 && grads32;
    bool uv = gv;
    // 32-byte update vectors: the gradient the update reads (the mean
    // gradient, else every rank's) and every state pointer 32-byte aligned
    bool uv32 = wide_ok && (ps.mean_grad ? aligned32(ps.mean_grad) : grads32);
    for (int k = 0; k < rep; ++k) {
      stab[p * 3 * rep + k] = ps.params[k];
      stab[p * 3 * rep + rep + k] = ps.exp_avg[k];
      stab[p * 3 * rep + 2 * rep + k] = ps.exp_avg_sq[k];
      uv = uv && aligned16(ps.params[k]) && aligned16(ps.exp_avg[k]) && aligned16(ps.exp_avg_sq[k]);
      uv32 = uv32 && aligned32(ps.params[k]) && aligned32(ps.exp_avg[k]) &&
             aligned32(ps.exp_avg_sq[k]);
    }
    upd_vec[p] = uv32 && uv ? 32 : (uv ? 16 : 0);
    rcc::GsTensor t{};
    t.numel = ps.numel;
    t.row_begin = row;
    t.mean_grad = ps.mean_grad;
    t.grad_slot = (uint32_t)(p * R);
    t.vec_ok = (gv ? 1u : 0u) | (uv ? 2u : 0u) | (gv32 ? 4u : 0u);
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
    e = upload(sc.desc_dev, sc.desc_host, sc.desc_host_dev, desc_bytes, cs);
    if (e != cudaSuccess) return cuda_fail(e, "descriptor upload");
    sc.last_desc.swap(desc);
    ++sc.desc_gen;
    sc.same_tables = 0;
  } else {
    ++sc.same_tables;
  }
  // The default flow becomes the host-graph flow -- the same decision on the
  // host, the same kernels, the P launches replayed from a captured graph --
  // once the same tensors have come three calls in a row, for P >= 32 (below
  // that the host's launches keep pace with the GPU).
  constexpr size_t kAutoGraphMinTensors = 32;
  const bool repeat_tables =
      P >= kAutoGraphMinTensors && sc.same_tables >= 2 && auto_graph_enabled();
  const bool host_graph =
      (cfg->flags & RCC_ADAMW_HOST_GRAPH) != 0 || (cfg->flags == 0 && repeat_tables);
  // likewise the device-decision flow replays its launches as RCC_ADAMW_GRAPH does
  const bool device_graph =
      (cfg->flags & RCC_ADAMW_GRAPH) != 0 ||
      (cfg->flags == RCC_ADAMW_DEVICE_DECISION && repeat_tables);
  const int64_t t_next = state->step + 1;
  if (on_device || host_graph) {
    // the scalars of step t+1, read by the updates from device memory; used
    // only if the step is not skipped
    if ((st = ensure_decision_scratch(sc)) != RCC_OK) return st;
    *sc.scalars_host = step_scalars(cfg, t_next);
    sc.scalars_host->inv_scale = (float)(1.0 / state->scale);
    e = upload(sc.scalars_dev, sc.scalars_host, sc.scalars_host_dev, sizeof(rcc::AdamWScalars),
               cs);
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
  const uint32_t seq = ++sc.report_seq == 0 ? ++sc.report_seq : sc.report_seq;  // never 0
  // RCC_STEP_TIMING: an event at each phase boundary on the call's stream
  auto mark = [&](int k) -> cudaError_t {
    return timing ? cudaEventRecord(sc.time_ev[k], cs) : cudaSuccess;
  };
  if ((e = mark(0)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing)");
  if ((e = rcc::launch_gs_stats(ga, cs)) != cudaSuccess) return cuda_fail(e, "statistics kernel");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if ((e = mark(1)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing)");

  const uint32_t* src = static_cast<const uint32_t*>(sc.rows);
  uint64_t rows = total_rows;
  int levels = 0;
  int combine_kernels = 0;
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
      ++combine_kernels;
      region_bytes = (levels == 0 ? 0 : 4096 * 12) + out_rows * 12;
      src = out;
      rows = out_rows;
      ++levels;
    }
  }
  if ((e = rcc::launch_gs_report(src, rows, sc.report_dev, sc.report_host_dev, seq, cs)) !=
      cudaSuccess)
    return cuda_fail(e, "report kernel");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!sc.report_host_dev &&
      (e = cudaMemcpyAsync(sc.report_host, sc.report_dev, 12, cudaMemcpyDeviceToHost, cs)) !=
          cudaSuccess)
    return cuda_fail(e, "report readback");
  if ((e = cudaEventRecord(sc.report_ev, cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  if ((e = mark(2)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing)");

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
    ua.inl = rep <= rcc::GsUpdateArgs::kInlineReplicas;
    if (ua.inl) {
      for (int k = 0; k < rep; ++k) {
        ua.inl_state[k] = params[p].params[k];
        ua.inl_state[rep + k] = params[p].exp_avg[k];
        ua.inl_state[2 * rep + k] = params[p].exp_avg_sq[k];
      }
    }
    return rcc::launch_gs_update(ua, where);
  };
  auto enqueue_branched = [&](cudaStream_t origin) -> cudaError_t {
    cudaError_t le;
    const int nb = (int)std::min<size_t>(P, (size_t)chain_count());
    if (nb == 1) {  // one chain (one tensor, or RCC_CHAINS=1): no fork/join
      for (size_t p = 0; p < P; ++p)
        if ((le = enqueue_one(p, origin)) != cudaSuccess) return le;
      return cudaSuccess;
    }
    if (!sc.fork_ev && (le = cudaEventCreateWithFlags(&sc.fork_ev, cudaEventDisableTiming)))
      return le;
    for (int k = 0; k < nb; ++k) {
      if (!sc.branch[k] &&
          (le = cudaStreamCreateWithFlags(&sc.branch[k], cudaStreamNonBlocking)) != cudaSuccess)
        return le;
      if (!sc.join_ev[k] &&
          (le = cudaEventCreateWithFlags(&sc.join_ev[k], cudaEventDisableTiming)) != cudaSuccess)
        return le;
    }
    if ((le = cudaEventRecord(sc.fork_ev, origin)) != cudaSuccess) return le;
    for (int k = 0; k < nb; ++k)
      if ((le = cudaStreamWaitEvent(sc.branch[k], sc.fork_ev, 0)) != cudaSuccess) return le;
    // Chains: tensors taken largest first, each onto the least loaded chain,
    // a launch counting as kLaunchCost elements of fixed cost.  Each chain
    // then runs its tensors alternately from its largest and its smallest
    // end, so the small, latency-bound launches of one chain overlap large,
    // bandwidth-bound ones on the others instead of every chain ending on a
    // run of small ones.  Launches are issued round-robin over the chains.
    constexpr uint64_t kLaunchCost = 65536;
    std::vector<size_t> order(P);
    for (size_t p = 0; p < P; ++p) order[p] = p;
    std::stable_sort(order.begin(), order.end(),
                     [&](size_t x, size_t y) { return params[x].numel > params[y].numel; });
    std::vector<size_t> chain[Scratch::kMaxBranches];
    uint64_t load[Scratch::kMaxBranches] = {};
    for (size_t p : order) {
      int k = 0;
      for (int j = 1; j < nb; ++j)
        if (load[j] < load[k]) k = j;
      load[k] += params[p].numel + kLaunchCost;
      chain[k].push_back(p);
    }
    size_t longest = 0;
    for (int k = 0; k < nb; ++k) {
      std::vector<size_t>& c = chain[k];
      std::vector<size_t> alt;
      alt.reserve(c.size());
      for (size_t lo = 0, hi = c.size(); lo < hi;) {
        alt.push_back(c[lo++]);
        if (lo < hi) alt.push_back(c[--hi]);
      }
      c.swap(alt);
      longest = std::max(longest, c.size());
    }
    for (size_t pos = 0; pos < longest; ++pos)
      for (int k = 0; k < nb; ++k)
        if (pos < chain[k].size() && (le = enqueue_one(chain[k][pos], sc.branch[k])) != cudaSuccess)
          return le;
    for (int k = 0; k < nb; ++k) {
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
  // The per-tensor updates captured once into a graph that reads the
  // decision and the scalars from device memory, replayed while the tables
  // stay the same.
  auto replay_graph = [&]() -> rcc_status {
    ua.clip_coef = 1.0f;
    ua.decision = sc.decision_dev;
    ua.dev_scalars = sc.scalars_dev;
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
    return RCC_OK;
  };

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
    if ((e = mark(3)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing)");
    if (device_graph) {
      if ((st = replay_graph()) != RCC_OK) return st;
    } else {
      if ((e = multi ? enqueue_multi(cs) : enqueue_branched(cs)) != cudaSuccess)
        return cuda_fail(e, "update kernel");
    }
    device_updates = launches_per_update;
    g_launches.fetch_add(launches_per_update, std::memory_order_relaxed);
  }
  {
    rcc::NvtxRange wait_range("rcc_grad_sync_adamw: report readback");
    st = sc.report_host_dev
             ? wait_report_word(sc.report_host + 3, seq, sc.report_ev, "12-byte report readback")
             : wait_event(sc.report_ev, "12-byte report readback");
  }
  if (st != RCC_OK) {
    // nothing of this step is applied by the host (default flow: no update
    // was launched); mark the queued work so that the next call waits for it
    if (cudaEventRecord(sc.done_ev, cs) == cudaSuccess) {
      sc.done_recorded = true;
      sc.stale = true;
    }
    return st;
  }

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
  rep_out.combine_launches = combine_kernels;
  rep_out.combine_levels = levels;
  rep_out.stats_rows = total_rows;
  rep_out.combine_region_bytes = region_bytes;

  rep_out.update_launches = device_updates;
  rep_out.report_words[0] = sc.report_host[0];
  rep_out.report_words[1] = sc.report_host[1];
  rep_out.report_words[2] = sc.report_host[2];
  rep_out.updates_before_readback = on_device ? 1 : 0;
  if (!on_device && (e = mark(3)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing)");
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
    if (host_graph) {
      // the host's decision goes to device memory for the replayed graph
      sc.decision_host->skip = 0u;
      sc.decision_host->coef = coef;
      if ((e = upload(sc.decision_dev, sc.decision_host, sc.decision_host_dev,
                      sizeof(rcc::GsDecision), cs)) != cudaSuccess)
        return cuda_fail(e, "decision upload");
      if ((st = replay_graph()) != RCC_OK) return st;
    } else {
      ua.s = step_scalars(cfg, t);
      ua.clip_coef = coef;
      if ((e = multi ? enqueue_multi(cs) : enqueue_branched(cs)) != cudaSuccess)
        return cuda_fail(e, "update kernel");
    }
    g_launches.fetch_add(launches_per_update, std::memory_order_relaxed);
    rep_out.update_launches = launches_per_update;
    state->step = t;
    state->growth_tracker += 1;
    if (state->growth_tracker >= state->growth_interval) {
      state->scale *= state->growth_factor;
      state->growth_tracker = 0;
    }
  }
  if ((e = mark(4)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing)");
  if ((e = cudaEventRecord(sc.done_ev, cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  sc.done_recorded = true;
  sc.timed = timing;
  if (report) *report = rep_out;
  return RCC_OK;
}

rcc_status rcc_last_step_times(rcc_comm comm, float out_ms[4]) {
  rcc::NvtxRange nvtx_range("rcc_last_step_times");
  t_err.clear();
  if (!out_ms) return fail(RCC_ERR_INVALID_ARGUMENT, "out_ms is NULL");
  auto s = lookup(comm);
  if (!s) return missing_session();
  std::lock_guard<std::mutex> lock(s->mu);
  Scratch& sc = s->sc;
  if (!sc.timed)
    return fail(RCC_ERR_INVALID_ARGUMENT,
                "no timed grad-sync call on this session (set RCC_STEP_TIMING first)");
  rcc_status st = check_device(s->device);
  if (st != RCC_OK) return st;
  if ((st = wait_event(sc.time_ev[Scratch::kTimeEvents - 1], "timed grad-sync call")) != RCC_OK)
    return st;
  for (int k = 0; k + 1 < Scratch::kTimeEvents; ++k) {
    float ms = 0.0f;
    cudaError_t e = cudaEventElapsedTime(&ms, sc.time_ev[k], sc.time_ev[k + 1]);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    out_ms[k] = ms;
  }
  return RCC_OK;
}

}  // extern "C"
