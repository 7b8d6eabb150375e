// collectives.cuh -- the multi-pointer pass behind every librcc collective.
//
// Replaces the ring schedule with host-staged transfers that the ruCCL README
// describes (§5 "CUDA example", §6 data path) by a single pass over HBM: all R
// rank buffers live on one GPU, so each output element is produced by one
// thread that loads the element from every source rank (32-byte vectors where
// every address allows, else 16-byte, else scalars; coalesced, no L1 allocation)
// and stores the result to every destination (streaming stores).  Minimum
// traffic, no staging, no exchange.  Launched with programmatic dependent
// launch (launch.cuh).
//
// Arithmetic is fp32 for both element types (bf16 is widened exactly and the
// result is rounded once to nearest-even).  Sums fold ranks in the order
// 0..R-1 (deterministic mode) or in a pairwise tree (fast mode); mean divides
// the sum by R with an IEEE division; max/min keep the lowest rank among
// equals and turn any NaN into the quiet NaN 0x7FC00000.
//
// Included by collectives_part.cu, which the build compiles once per element
// type and reduction (launch_part below), so that the instantiations build in
// parallel.
#pragma once

#include <cuda_bf16.h>

#include <cstdlib>
#include <mutex>
#include <unordered_map>

#include "launch.cuh"
#include "rcc_internal.h"

namespace rcc {
namespace mp {

constexpr uint32_t kCanonicalNaN = 0x7FC00000u;

// ---- memory access -------------------------------------------------------
// A vector of W 32-bit words: W = 4 (16 bytes) or W = 8 (32 bytes, the
// 256-bit global loads/stores sm_100-class GPUs provide).
template <int W>
struct Vec {
  uint32_t w[W];
};

// Source loads without L1 allocation: every input element is read exactly
// once.  They take the coherent path, not the non-coherent (read-only) one,
// which would be valid only while no thread of the kernel writes the data: a
// destination may alias a source (in-place all_reduce, reduce and
// all_gather).  On GB300 the two measured the same (8 ranks x 2^24 fp32 and
// 2^26 bf16, every collective, within 0.5%).  Volatile keeps the loads and
// stores of one thread in program order (an in-place element is read before
// the same thread overwrites it).
template <int W>
__device__ __forceinline__ Vec<W> ld_vec(const void* p) {
  Vec<W> v;
  if constexpr (W == 4) {
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
  } else {
    asm volatile("ld.global.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]),
                   "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
  }
  return v;
}

// Output stores.  RCC_STORE_HINT 1 marks them streaming (evict-first): this
// pass never re-reads what it writes.  0 uses the default write-back policy.
#ifndef RCC_STORE_HINT
#define RCC_STORE_HINT 1
#endif
#if RCC_STORE_HINT
#define RCC_ST "st.global.cs"
#else
#define RCC_ST "st.global"
#endif

template <int W>
__device__ __forceinline__ void st_vec(void* p, const Vec<W>& v) {
  if constexpr (W == 4) {
    asm volatile(RCC_ST ".v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]),
                 "r"(v.w[2]), "r"(v.w[3])
                 : "memory");
  } else {
    asm volatile(RCC_ST ".v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]),
                 "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
                 "r"(v.w[7])
                 : "memory");
  }
}

// Schedule knobs (build-time).  RCC_BLOCKED 1 gives each CTA one contiguous
// range of vectors instead of a grid-stride sweep; RCC_WAVES caps the grid at
// that many waves of resident CTAs (16 measured best on GB300: with one wave
// all CTAs drain together and HBM idles at the end; with many, finishing CTAs
// are replaced at once); RCC_COPY_U overrides the copy pass's vectors per
// thread; RCC_MIN_BLOCKS (> 0) asks for that many resident CTAs per SM.
#ifndef RCC_BLOCKED
#define RCC_BLOCKED 0
#endif
#ifndef RCC_WAVES
#define RCC_WAVES 16
#endif
#ifndef RCC_COPY_U
#define RCC_COPY_U 4
#endif
#ifndef RCC_MIN_BLOCKS
#define RCC_MIN_BLOCKS 0
#endif
#if RCC_MIN_BLOCKS > 0
#define RCC_BOUNDS __launch_bounds__(kThreads, RCC_MIN_BLOCKS)
#else
#define RCC_BOUNDS __launch_bounds__(kThreads)
#endif

// ---- element types ---------------------------------------------------------

// fp32 -> bf16 bits, round to nearest even (hardware cvt); a NaN keeps its
// sign and high payload bits and is made quiet, the same rule for every op.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  if (lo != lo) r = (r & 0xFFFF0000u) | ((__float_as_uint(lo) >> 16) | 0x40u);
  if (hi != hi) r = (r & 0x0000FFFFu) | ((((__float_as_uint(hi) >> 16) | 0x40u)) << 16);
  return r;
}

__device__ __forceinline__ uint16_t bf16_rn(float f) {
  return (uint16_t)(bf16x2_rn(f, 0.0f) & 0xFFFFu);
}

template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kBytes = 4;
  static constexpr int kPerWord = 1;
  __device__ static __forceinline__ float lane(uint32_t w, int) { return __uint_as_float(w); }
  __device__ static __forceinline__ uint32_t pack_word(const float* f) { return __float_as_uint(f[0]); }
  template <int W>
  __device__ static __forceinline__ void unpack(const Vec<W>& v, float* f) {
#pragma unroll
    for (int k = 0; k < W; ++k) f[k] = __uint_as_float(v.w[k]);
  }
  template <int W>
  __device__ static __forceinline__ Vec<W> pack(const float* f) {
    Vec<W> v;
#pragma unroll
    for (int k = 0; k < W; ++k) v.w[k] = __float_as_uint(f[k]);
    return v;
  }
  __device__ static __forceinline__ float load(const void* p, size_t i) {
    return static_cast<const float*>(p)[i];
  }
  __device__ static __forceinline__ void store(void* p, size_t i, float f) {
    static_cast<float*>(p)[i] = f;
  }
  __device__ static __forceinline__ void copy(const void* s, void* d, size_t i) {
    static_cast<uint32_t*>(d)[i] = static_cast<const uint32_t*>(s)[i];
  }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static constexpr int kPerWord = 2;
  // lane 0 is the low half of the word, lane 1 the high half
  __device__ static __forceinline__ float lane(uint32_t w, int l) {
    return __uint_as_float(l == 0 ? (w << 16) : (w & 0xFFFF0000u));
  }
  __device__ static __forceinline__ uint32_t pack_word(const float* f) { return bf16x2_rn(f[0], f[1]); }
  template <int W>
  __device__ static __forceinline__ void unpack(const Vec<W>& v, float* f) {
#pragma unroll
    for (int k = 0; k < W; ++k) {
      f[2 * k] = __uint_as_float(v.w[k] << 16);
      f[2 * k + 1] = __uint_as_float(v.w[k] & 0xFFFF0000u);
    }
  }
  template <int W>
  __device__ static __forceinline__ Vec<W> pack(const float* f) {
    Vec<W> v;
#pragma unroll
    for (int k = 0; k < W; ++k) v.w[k] = bf16x2_rn(f[2 * k], f[2 * k + 1]);
    return v;
  }
  __device__ static __forceinline__ float load(const void* p, size_t i) {
    return __uint_as_float((uint32_t)static_cast<const uint16_t*>(p)[i] << 16);
  }
  __device__ static __forceinline__ void store(void* p, size_t i, float f) {
    static_cast<uint16_t*>(p)[i] = bf16_rn(f);
  }
  __device__ static __forceinline__ void copy(const void* s, void* d, size_t i) {
    static_cast<uint16_t*>(d)[i] = static_cast<const uint16_t*>(s)[i];
  }
};

// ---- reductions over ranks ---------------------------------------------------

__host__ __device__ constexpr int pow2_below(int n) {
  int p = 1;
  while (p * 2 < n) p *= 2;
  return p;
}

// Pairwise tree over x[LO, HI): split at the largest power of two below the
// length, e.g. 5 ranks -> ((x0+x1)+(x2+x3))+x4.
template <int LO, int HI>
struct Tree {
  __device__ static __forceinline__ float sum(const float* x) {
    if constexpr (HI - LO == 1) {
      return x[LO];
    } else {
      constexpr int mid = LO + pow2_below(HI - LO);
      return __fadd_rn(Tree<LO, mid>::sum(x), Tree<mid, HI>::sum(x));
    }
  }
};

// Running state of one output lane.  Used in rank order: init(x_0), then
// add(x_1), ..., add(x_{R-1}).
template <int RED>
struct Acc {
  float v;
  bool nan;
  __device__ __forceinline__ void init(float x) {
    v = x;
    nan = (x != x);
  }
  __device__ __forceinline__ void add(float x) {
    if constexpr (RED == kRedSum) {
      v = __fadd_rn(v, x);
    } else {
      nan |= (x != x);
      if (RED == kRedMax ? (x > v) : (x < v)) v = x;
    }
  }
  __device__ __forceinline__ float result(int mean_div) const {
    if constexpr (RED == kRedSum) {
      return mean_div > 0 ? __fdiv_rn(v, (float)mean_div) : v;
    } else {
      return nan ? __uint_as_float(kCanonicalNaN) : v;
    }
  }
};

template <int NS, int RED, bool FAST>
__device__ __forceinline__ float reduce_lane(const float (&x)[NS], int mean_div) {
  if constexpr (RED == kRedSum && FAST) {
    float s = Tree<0, NS>::sum(x);
    return mean_div > 0 ? __fdiv_rn(s, (float)mean_div) : s;
  } else {
    Acc<RED> a;
    a.init(x[0]);
#pragma unroll
    for (int q = 1; q < NS; ++q) a.add(x[q]);
    return a.result(mean_div);
  }
}

// ---- the pass ----------------------------------------------------------------

// Per-segment views of the argument block.
struct SegView {
  const MultiPtrArgs& a;
  int seg;
  size_t soff, doff;  // element offsets of this segment
  int a2a_hi, a2a_lo;  // all-to-all: seg / R and seg % R, worked out once
  __device__ __forceinline__ SegView(const MultiPtrArgs& a_, int seg_, size_t soff_, size_t doff_)
      : a(a_), seg(seg_), soff(soff_), doff(doff_), a2a_hi(0), a2a_lo(0) {
    if (a.a2a_ranks > 0) {
      a2a_hi = seg / a.a2a_ranks;
      a2a_lo = seg - a2a_hi * a.a2a_ranks;
    }
  }
  __device__ __forceinline__ const void* src(int q, int eb) const {
    if (a.a2a_ranks > 0)  // chunk (seg % R) of rank (seg / R)
      return static_cast<const char*>(a.src[a2a_hi]) + (size_t)a2a_lo * a.n * eb;
    const void* base = a.src_per_seg ? a.src[seg] : a.src[q];
    return static_cast<const char*>(base) + soff * eb;
  }
  __device__ __forceinline__ void* dst(int d, int eb) const {
    if (a.a2a_ranks > 0)  // slot (seg / R) of rank (seg % R)
      return static_cast<char*>(a.dst[a2a_lo]) + (size_t)a2a_hi * a.n * eb;
    void* base = a.dst_per_seg ? a.dst[seg] : a.dst[d];
    return static_cast<char*>(base) + doff * eb;
  }
  __device__ __forceinline__ int ndst() const {
    return (a.dst_per_seg || a.a2a_ranks > 0) ? 1 : a.ndst;
  }
};

// NS > 0: compile-time number of sources (U vectors per thread in flight per
// source); NS == 0: runtime count (any R up to kMaxRanks), sources loaded in
// groups of G and folded in rank order.  W: 32-bit words per vector (4 or 8);
// the host picks 8 only when every address is 32-byte aligned.
template <typename T, int NS, int RED, bool FAST, int U, int W, int G = 8>
__global__ void RCC_BOUNDS mp_kernel(const __grid_constant__ MultiPtrArgs a) {
  pdl_wait_then_release();
  using E = Elem<T>;
  constexpr int EPV = W * E::kPerWord;  // elements per vector
  constexpr int VB = 4 * W;             // bytes per vector
  constexpr int EB = E::kBytes;
  const SegView sv{a, (int)blockIdx.y, (size_t)blockIdx.y * a.src_seg_stride,
                   (size_t)blockIdx.y * a.dst_seg_stride};
  const int ndst = sv.ndst();
  const size_t nv = a.vec_ok >= VB ? a.n / EPV : 0;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t nthreads = (size_t)gridDim.x * blockDim.x;

  if constexpr (NS > 0) {
    const char* sp[NS];
#pragma unroll
    for (int q = 0; q < NS; ++q) sp[q] = static_cast<const char*>(sv.src(q, EB));

    // cyclic: CTAs sweep the range together with a grid-wide stride;
    // blocked: each CTA walks its own contiguous share
    const size_t tile = (size_t)blockDim.x * U;
    size_t first, end, stride;
    if (RCC_BLOCKED) {
      const size_t share = (nv + gridDim.x - 1) / gridDim.x;
      const size_t chunk = (share + tile - 1) / tile * tile;
      first = (size_t)blockIdx.x * chunk + threadIdx.x;
      end = (size_t)(blockIdx.x + 1) * chunk < nv ? (size_t)(blockIdx.x + 1) * chunk : nv;
      stride = tile;
    } else {
      first = (size_t)blockIdx.x * tile + threadIdx.x;
      end = nv;
      stride = nthreads * U;
    }
    for (size_t base = first; base < end; base += stride) {
      Vec<W> v[U][NS];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const size_t idx = base + (size_t)u * blockDim.x;
        if (idx < end) {
#pragma unroll
          for (int q = 0; q < NS; ++q) v[u][q] = ld_vec<W>(sp[q] + idx * VB);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const size_t idx = base + (size_t)u * blockDim.x;
        if (idx < end) {
          Vec<W> out;
          if constexpr (RED == kRedCopy) {
            out = v[u][0];
          } else {
            // word by word: unpack one 32-bit word of every rank, reduce its
            // lanes, pack; only one word's lanes are live at a time
#pragma unroll
            for (int k = 0; k < W; ++k) {
              float r[E::kPerWord];
#pragma unroll
              for (int l = 0; l < E::kPerWord; ++l) {
                float x[NS];
#pragma unroll
                for (int q = 0; q < NS; ++q) x[q] = E::lane(v[u][q].w[k], l);
                r[l] = reduce_lane<NS, RED, FAST>(x, a.mean_div);
              }
              out.w[k] = E::pack_word(r);
            }
          }
          for (int d = 0; d < ndst; ++d)
            st_vec<W>(static_cast<char*>(sv.dst(d, EB)) + idx * VB, out);
        }
      }
    }
  } else {
    // runtime rank count: rank order fold in groups of G sources, each
    // group's loads all issued before any of it is folded
    const int R = a.nsrc;
    for (size_t idx = tid; idx < nv; idx += nthreads) {
      Acc<RED> acc[EPV];
      for (int q0 = 0; q0 < R; q0 += G) {
        Vec<W> v[G];
#pragma unroll
        for (int k = 0; k < G; ++k)
          if (q0 + k < R)
            v[k] = ld_vec<W>(static_cast<const char*>(sv.src(q0 + k, EB)) + idx * VB);
#pragma unroll
        for (int k = 0; k < G; ++k) {
          if (q0 + k < R) {
            float f[EPV];
            E::template unpack<W>(v[k], f);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
              if (q0 + k == 0)
                acc[e].init(f[e]);
              else
                acc[e].add(f[e]);
            }
          }
        }
      }
      float r[EPV];
#pragma unroll
      for (int e = 0; e < EPV; ++e) r[e] = acc[e].result(a.mean_div);
      const Vec<W> out = E::template pack<W>(r);
      for (int d = 0; d < ndst; ++d)
        st_vec<W>(static_cast<char*>(sv.dst(d, EB)) + idx * VB, out);
    }
  }

  // scalar elements: the ragged tail after the vectors, or everything when
  // some address is not 16-byte aligned
  for (size_t i = nv * EPV + tid; i < a.n; i += nthreads) {
    if constexpr (RED == kRedCopy) {
      const void* s = sv.src(0, EB);
      for (int d = 0; d < ndst; ++d) E::copy(s, sv.dst(d, EB), i);
    } else if constexpr (NS > 0) {
      float x[NS];
#pragma unroll
      for (int q = 0; q < NS; ++q) x[q] = E::load(sv.src(q, EB), i);
      const float y = reduce_lane<NS, RED, FAST>(x, a.mean_div);
      for (int d = 0; d < ndst; ++d) E::store(sv.dst(d, EB), i, y);
    } else {
      Acc<RED> acc;
      acc.init(E::load(sv.src(0, EB), i));
      for (int q = 1; q < a.nsrc; ++q) acc.add(E::load(sv.src(q, EB), i));
      const float y = acc.result(a.mean_div);
      for (int d = 0; d < ndst; ++d) E::store(sv.dst(d, EB), i, y);
    }
  }
}

// ---- segments whose offsets break vector alignment --------------------------
// reduce_scatter, all_gather and all_to_all address rank buffers at offsets of
// s * n elements.  When n is such that those offsets are not multiples of 16
// bytes (while the buffers themselves are aligned), the common vector path
// above would fall back to scalars.  Instead, within each segment, the side
// that carries most of the traffic is aligned by skipping `head` elements
// (done as scalars), and the other side goes through shared memory, so every
// global access stays coalesced:
//   staged_reduce_kernel  sources aligned (reduce_scatter: R reads per write):
//                         vector loads, reduce, tile to shared memory, then
//                         vector stores from each destination's first vector
//                         boundary in the tile (element stores at its ends);
//   staged_copy_kernel    destinations aligned (all_gather, all_to_all): vector
//                         loads from the source's vector boundary at or below
//                         the tile into shared memory, then vector stores to
//                         every destination read back at the source's shift.
// Either way both global sides move whole vectors; the shift between them is
// taken in shared memory.
// kStageU vectors per thread per tile.
constexpr int kStageU = 2;

// Elements [lo, hi) of one segment, one element per thread, as the tail loop
// of mp_kernel.
template <typename T, int NS, int RED, bool FAST>
__device__ __forceinline__ void scalar_range(const MultiPtrArgs& a, const SegView& sv, int ndst,
                                             size_t lo, size_t hi, size_t tid,
                                             size_t nthreads) {
  using E = Elem<T>;
  constexpr int EB = E::kBytes;
  for (size_t i = lo + tid; i < hi; i += nthreads) {
    if constexpr (RED == kRedCopy) {
      const void* s = sv.src(0, EB);
      for (int d = 0; d < ndst; ++d) E::copy(s, sv.dst(d, EB), i);
    } else if constexpr (NS > 0) {
      float x[NS];
#pragma unroll
      for (int q = 0; q < NS; ++q) x[q] = E::load(sv.src(q, EB), i);
      const float y = reduce_lane<NS, RED, FAST>(x, a.mean_div);
      for (int d = 0; d < ndst; ++d) E::store(sv.dst(d, EB), i, y);
    } else {
      Acc<RED> acc;
      acc.init(E::load(sv.src(0, EB), i));
      for (int q = 1; q < a.nsrc; ++q) acc.add(E::load(sv.src(q, EB), i));
      const float y = acc.result(a.mean_div);
      for (int d = 0; d < ndst; ++d) E::store(sv.dst(d, EB), i, y);
    }
  }
}

// The staged kernels' tile in shared memory, word-major: word j of vector v
// at words[j][v].  A thread that writes its whole vector, or reads back the W
// words that start at any element offset, then touches consecutive banks
// across the warp.
template <int W>
struct StageTile {
  static constexpr int kVecs = kThreads * kStageU + 1;  // one spare for a shifted window
  uint32_t words[W][kVecs];

  __device__ __forceinline__ void put(int v, const Vec<W>& x) {
#pragma unroll
    for (int k = 0; k < W; ++k) words[k][v] = x.w[k];
  }
  __device__ __forceinline__ uint32_t word(int p) const { return words[p % W][p / W]; }

  // Reads of whole vectors at one element shift `sh` (the same for every
  // vector of a segment): the vector that starts at tile element sh + v*EPV
  // takes words v*W + ph + i (i = 0..W, ph the shift in words), which sit at
  // words[(ph + i) % W][v + (ph + i) / W].  The W + 1 word offsets are worked
  // out once; each read is then one add and one shared load per word.
  struct Shift {
    int at[W + 1];  // byte offset of word i for vector 0
    bool odd;       // a 2-byte element shift of one half word: funnel shifts
  };
  template <int EB>
  __device__ __forceinline__ static Shift shift(int sh) {
    Shift f;
    const int ph = EB == 4 ? sh : sh >> 1;
    f.odd = EB == 2 && (sh & 1);
#pragma unroll
    for (int i = 0; i <= W; ++i) f.at[i] = (((ph + i) % W) * kVecs + (ph + i) / W) * 4;
    return f;
  }
  __device__ __forceinline__ Vec<W> get(int v, const Shift& f) const {
    const char* base = reinterpret_cast<const char*>(&words[0][0]) + v * 4;
    Vec<W> x;
    if (!f.odd) {
#pragma unroll
      for (int k = 0; k < W; ++k) x.w[k] = *reinterpret_cast<const uint32_t*>(base + f.at[k]);
    } else {
      uint32_t lo = *reinterpret_cast<const uint32_t*>(base + f.at[0]);
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const uint32_t hi = *reinterpret_cast<const uint32_t*>(base + f.at[k + 1]);
        x.w[k] = __funnelshift_r(lo, hi, 16);
        lo = hi;
      }
    }
    return x;
  }
  // One element's raw bits at tile element `e`.
  template <int EB>
  __device__ __forceinline__ uint32_t elem(int e) const {
    if constexpr (EB == 4) {
      return word(e);
    } else {
      return (word(e >> 1) >> (16 * (e & 1))) & 0xFFFFu;
    }
  }
};

// Stores raw element bits b (EB bytes) at element index i of p.
template <int EB>
__device__ __forceinline__ void put_elem(void* p, size_t i, uint32_t b) {
  if constexpr (EB == 4) {
    static_cast<uint32_t*>(p)[i] = b;
  } else {
    static_cast<uint16_t*>(p)[i] = (uint16_t)b;
  }
}

template <int EB>
__device__ __forceinline__ uint32_t get_elem(const void* p, size_t i) {
  if constexpr (EB == 4) {
    return static_cast<const uint32_t*>(p)[i];
  } else {
    return static_cast<const uint16_t*>(p)[i];
  }
}

// Element offset of address p from the VB-byte boundary below it.
template <int VB, int EB>
__device__ __forceinline__ int vec_phase(const void* p) {
  return (int)((reinterpret_cast<uintptr_t>(p) % VB) / EB);
}

template <typename T, int NS, int RED, bool FAST, int W>
__global__ void __launch_bounds__(kThreads)
    staged_reduce_kernel(const __grid_constant__ MultiPtrArgs a) {
  pdl_wait_then_release();
  using E = Elem<T>;
  constexpr int EPV = W * E::kPerWord;
  constexpr int VB = 4 * W;
  constexpr int EB = E::kBytes;
  constexpr int NV = kThreads * kStageU;
  constexpr int TILE = NV * EPV;
  __shared__ StageTile<W> tile;
  const SegView sv{a, (int)blockIdx.y, (size_t)blockIdx.y * a.src_seg_stride,
                   (size_t)blockIdx.y * a.dst_seg_stride};
  const int ndst = sv.ndst();
  // every source of the segment has the same offset from a VB-aligned base
  const uintptr_t anchor = reinterpret_cast<uintptr_t>(sv.src(0, EB));
  size_t head = ((VB - anchor % VB) % VB) / EB;
  if (head > a.n) head = a.n;
  const size_t ntiles = (a.n - head) / TILE;
  for (size_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const size_t e0 = head + t * TILE;
#pragma unroll
    for (int u = 0; u < kStageU; ++u) {
      const int slot = u * kThreads + threadIdx.x;
      const size_t off = (e0 + (size_t)slot * EPV) * EB;
      Vec<W> out;
      if constexpr (NS > 0) {
        Vec<W> v[NS];
#pragma unroll
        for (int q = 0; q < NS; ++q) v[q] = ld_vec<W>(static_cast<const char*>(sv.src(q, EB)) + off);
#pragma unroll
        for (int k = 0; k < W; ++k) {
          float r[E::kPerWord];
#pragma unroll
          for (int l = 0; l < E::kPerWord; ++l) {
            float x[NS];
#pragma unroll
            for (int q = 0; q < NS; ++q) x[q] = E::lane(v[q].w[k], l);
            r[l] = reduce_lane<NS, RED, FAST>(x, a.mean_div);
          }
          out.w[k] = E::pack_word(r);
        }
      } else {
        Acc<RED> acc[EPV];
        for (int q0 = 0; q0 < a.nsrc; q0 += 8) {
          Vec<W> v[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (q0 + k < a.nsrc) v[k] = ld_vec<W>(static_cast<const char*>(sv.src(q0 + k, EB)) + off);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (q0 + k < a.nsrc) {
              float f[EPV];
              E::template unpack<W>(v[k], f);
#pragma unroll
              for (int e = 0; e < EPV; ++e) {
                if (q0 + k == 0)
                  acc[e].init(f[e]);
                else
                  acc[e].add(f[e]);
              }
            }
          }
        }
        float r[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) r[e] = acc[e].result(a.mean_div);
        out = E::template pack<W>(r);
      }
      tile.put(slot, out);
    }
    __syncthreads();
    // Each destination gets vector stores from its first VB boundary in the
    // tile on (read from the tile at that shift), and element stores for the
    // partial vectors at the tile's two ends.
    for (int d = 0; d < ndst; ++d) {
      char* dst = static_cast<char*>(sv.dst(d, EB));
      const int lead = (EPV - vec_phase<VB, EB>(dst + e0 * EB)) % EPV;
      const int nvec = (TILE - lead) / EPV;
      const auto sh = StageTile<W>::template shift<EB>(lead);
      for (int k = threadIdx.x; k < nvec; k += kThreads)
        st_vec<W>(dst + (e0 + lead + (size_t)k * EPV) * EB, tile.get(k, sh));
      const int tail0 = lead + nvec * EPV;
      for (int e = threadIdx.x; e < lead + (TILE - tail0); e += kThreads) {
        const int te = e < lead ? e : tail0 + (e - lead);
        put_elem<EB>(dst, e0 + te, tile.template elem<EB>(te));
      }
    }
    __syncthreads();
  }
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t nthreads = (size_t)gridDim.x * blockDim.x;
  scalar_range<T, NS, RED, FAST>(a, sv, ndst, 0, head, tid, nthreads);
  scalar_range<T, NS, RED, FAST>(a, sv, ndst, head + ntiles * TILE, a.n, tid, nthreads);
}

template <typename T, int W>
__global__ void __launch_bounds__(kThreads) staged_copy_kernel(const __grid_constant__ MultiPtrArgs a) {
  pdl_wait_then_release();
  using E = Elem<T>;
  constexpr int EPV = W * E::kPerWord;
  constexpr int VB = 4 * W;
  constexpr int EB = E::kBytes;
  constexpr int NV = kThreads * kStageU;
  constexpr int TILE = NV * EPV;
  __shared__ StageTile<W> tile;
  const SegView sv{a, (int)blockIdx.y, (size_t)blockIdx.y * a.src_seg_stride,
                   (size_t)blockIdx.y * a.dst_seg_stride};
  const int ndst = sv.ndst();
  const char* src = static_cast<const char*>(sv.src(0, EB));
  // every destination of the segment has the same offset from a VB-aligned base
  const uintptr_t anchor = reinterpret_cast<uintptr_t>(sv.dst(0, EB));
  size_t head = ((VB - anchor % VB) % VB) / EB;
  if (head > a.n) head = a.n;
  const size_t ntiles = (a.n - head) / TILE;
  for (size_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const size_t e0 = head + t * TILE;
    // source vectors from the VB boundary at or below element e0 (`lag`
    // elements before it) until the tile is covered; a vector that reaches
    // outside the segment is read element by element
    const int lag = vec_phase<VB, EB>(src + e0 * EB);
    const int nsv = NV + (lag ? 1 : 0);
    // every load of the thread is issued before any is written to the tile
    Vec<W> x[kStageU + 1];
#pragma unroll
    for (int u = 0; u <= kStageU; ++u) {
      const int j = u * kThreads + threadIdx.x;
      if (j >= nsv) continue;
      const long long s0 = (long long)e0 - lag + (long long)j * EPV;
      if (s0 >= 0 && s0 + EPV <= (long long)a.n) {
        x[u] = ld_vec<W>(src + s0 * EB);
      } else {
#pragma unroll
        for (int k = 0; k < W; ++k) x[u].w[k] = 0u;
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const long long i = s0 + e;
          if (i >= 0 && i < (long long)a.n) {
            const uint32_t b = get_elem<EB>(src, (size_t)i);
            x[u].w[e * EB / 4] |= b << (8 * ((e * EB) % 4));
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u <= kStageU; ++u) {
      const int j = u * kThreads + threadIdx.x;
      if (j < nsv) tile.put(j, x[u]);
    }
    __syncthreads();
    const auto sh = StageTile<W>::template shift<EB>(lag);
#pragma unroll
    for (int u = 0; u < kStageU; ++u) {
      const int k = u * kThreads + threadIdx.x;
      const Vec<W> out = tile.get(k, sh);
      const size_t off = (e0 + (size_t)k * EPV) * EB;
      for (int d = 0; d < ndst; ++d) st_vec<W>(static_cast<char*>(sv.dst(d, EB)) + off, out);
    }
    __syncthreads();
  }
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t nthreads = (size_t)gridDim.x * blockDim.x;
  scalar_range<T, 1, kRedCopy, false>(a, sv, ndst, 0, head, tid, nthreads);
  scalar_range<T, 1, kRedCopy, false>(a, sv, ndst, head + ntiles * TILE, a.n, tid, nthreads);
}

// ---- host-side dispatch -------------------------------------------------------

// 16-byte vectors per thread in flight for each source count: enough loads
// outstanding per thread (U * NS >= 4..8) to cover HBM latency.  32-byte
// vectors halve U.
constexpr int unroll_for(int ns, int red) {
  return red == kRedCopy ? RCC_COPY_U : ns <= 2 ? 4 : ns <= 4 ? 2 : 1;
}

inline int sm_count() {
  static int cached = -1;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int dev = 0;
  cudaGetDevice(&dev);
  static int cached_dev = -1;
  if (cached < 0 || cached_dev != dev) {
    cudaDeviceGetAttribute(&cached, cudaDevAttrMultiProcessorCount, dev);
    cached_dev = dev;
  }
  return cached;
}

inline int resident_blocks(const void* fn) {
  static std::mutex mu;
  static std::unordered_map<const void*, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(fn);
  if (it != cache.end()) return it->second;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, 0);
  if (per_sm < 1) per_sm = 1;
  cache[fn] = per_sm;
  return per_sm;
}

// Widest vector the addresses allow (RCC_VEC_BYTES=16 caps it at 16 bytes).
inline int vec_cap() {
  static int cap = [] {
    const char* v = std::getenv("RCC_VEC_BYTES");
    return (v && std::atoi(v) == 16) ? 16 : 32;
  }();
  return cap;
}

// UO > 0 overrides the vectors per thread per iteration.
template <typename T, int NS, int RED, bool FAST, int W, int G = 8, int UO = 0>
cudaError_t launch_w(int nseg, const MultiPtrArgs& a, cudaStream_t stream) {
  constexpr int U0 = NS > 0 ? unroll_for(NS, RED) * 4 / W : 1;
  constexpr int U = UO > 0 ? UO : (U0 > 0 ? U0 : 1);
  constexpr int EPV = W * Elem<T>::kPerWord;
  auto fn = mp_kernel<T, NS, RED, FAST, U, W, G>;
  const size_t nv = a.vec_ok >= 4 * W ? a.n / EPV : 0;
  const size_t tail = a.n - nv * EPV;
  size_t want = (nv + (size_t)kThreads * U - 1) / ((size_t)kThreads * U);
  const size_t want_tail = (tail + kThreads - 1) / kThreads;
  if (want_tail > want) want = want_tail;
  if (want < 1) want = 1;
  // up to RCC_WAVES waves of resident blocks across all segments
  size_t cap = (size_t)resident_blocks((const void*)fn) * sm_count() * RCC_WAVES / (size_t)nseg;
  if (cap < 1) cap = 1;
  const unsigned gx = (unsigned)(want < cap ? want : cap);
  return launch_kernel(fn, dim3(gx, (unsigned)nseg), dim3(kThreads), 0, stream, a);
}

// A launch with more than one vector per thread (copies, and reductions over
// one or two sources) takes half as many when its default grid stays below
// the wave cap: twice the CTAs, so the last partial wave is half as long.  At
// 8 ranks, broadcast and all_gather of 2^22 / 2^23 fp32 went from 0.77 / 0.91
// to 0.90 / 0.98 of the copy peak (two-rank reductions gained 0-4%); at 2^26
// (a capped grid) the default measured 1.015 against 0.999, so capped grids
// keep it.
template <typename T, int NS, int RED, bool FAST, int W>
cudaError_t launch_unrolled_w(int nseg, const MultiPtrArgs& a, cudaStream_t stream) {
  constexpr int U0 = unroll_for(NS, RED) * 4 / W;
  if constexpr (U0 > 1) {
    constexpr int EPV = W * Elem<T>::kPerWord;
    const size_t nv = a.n / EPV;
    const size_t want = (nv + (size_t)kThreads * U0 - 1) / ((size_t)kThreads * U0);
    const size_t cap = (size_t)resident_blocks((const void*)mp_kernel<T, NS, RED, FAST, U0, W, 8>) *
                       sm_count() * RCC_WAVES / (size_t)nseg;
    if (want < cap) return launch_w<T, NS, RED, FAST, W, 8, U0 / 2>(nseg, a, stream);
  }
  return launch_w<T, NS, RED, FAST, W>(nseg, a, stream);
}

// A runtime source count (NS == 0, more than 8 ranks) always takes 16-byte
// vectors: with 32-byte ones its 8-source groups need about 100 registers (2
// CTAs per SM), and at 9-64 ranks reduce and reduce_scatter measured 0.88-1.01
// of the copy peak against 0.91-1.10 with 16-byte vectors (all_reduce alike).
// 9-12 sources load as one group of 12 (one load round trip instead of two:
// reduce and reduce_scatter at 9 ranks 0.93 / 0.91 -> 1.01 / 1.01); other
// counts in groups of 8 (a group of 12 or 16 holds too many registers for
// the occupancy that 16 ranks and up want: 1.09 -> 0.98 at 16).
template <typename T, int NS, int RED, bool FAST>
cudaError_t launch_ns(int nseg, const MultiPtrArgs& a, cudaStream_t stream) {
  if constexpr (NS > 0) {
    if (a.vec_ok >= 32 && vec_cap() >= 32)
      return launch_unrolled_w<T, NS, RED, FAST, 8>(nseg, a, stream);
    if (a.vec_ok >= 16) return launch_unrolled_w<T, NS, RED, FAST, 4>(nseg, a, stream);
    return launch_w<T, NS, RED, FAST, 4>(nseg, a, stream);
  } else {
    if (a.nsrc <= 12) return launch_w<T, 0, RED, FAST, 4, 12>(nseg, a, stream);
    return launch_w<T, 0, RED, FAST, 4, 8>(nseg, a, stream);
  }
}

// grid for the staged kernels: one CTA per tile up to RCC_WAVES waves
template <typename KernelFn>
unsigned staged_grid(KernelFn fn, size_t n, size_t tile, int nseg) {
  size_t want = n / tile;
  if (want < 1) want = 1;
  size_t cap = (size_t)resident_blocks((const void*)fn) * sm_count() * RCC_WAVES / (size_t)nseg;
  if (cap < 1) cap = 1;
  return (unsigned)(want < cap ? want : cap);
}

template <typename T, int NS, int RED, bool FAST, int W>
cudaError_t launch_staged_reduce_w(int nseg, const MultiPtrArgs& a, cudaStream_t stream) {
  auto fn = staged_reduce_kernel<T, NS, RED, FAST, W>;
  const size_t tile = (size_t)kThreads * kStageU * W * Elem<T>::kPerWord;
  return launch_kernel(fn, dim3(staged_grid(fn, a.n, tile, nseg), (unsigned)nseg), dim3(kThreads),
                       0, stream, a);
}

// bf16 takes 16-byte vectors here: with 32-byte ones a thread reduces and
// stages twice the elements per vector, and the pass measured 0.72 of the
// copy peak against 0.87 (8 ranks, odd shards).  So does a runtime source
// count: with 32-byte vectors the kernel needs 107 registers (2 CTAs per SM),
// and a 12-rank reduce_scatter with odd shards measured 0.60 against 0.88.
template <typename T, int NS, int RED, bool FAST>
cudaError_t launch_staged_reduce_ns(int nseg, const MultiPtrArgs& a, cudaStream_t stream) {
  if constexpr (NS > 0 && Elem<T>::kBytes == 4) {
    if (a.vec_ok >= 32 && vec_cap() >= 32)
      return launch_staged_reduce_w<T, NS, RED, FAST, 8>(nseg, a, stream);
  }
  return launch_staged_reduce_w<T, NS, RED, FAST, 4>(nseg, a, stream);
}

template <typename T>
cudaError_t launch_staged_copy(int nseg, const MultiPtrArgs& a, cudaStream_t stream) {
  if (a.vec_ok >= 32 && vec_cap() >= 32) {
    auto fn = staged_copy_kernel<T, 8>;
    const size_t tile = (size_t)kThreads * kStageU * 8 * Elem<T>::kPerWord;
    return launch_kernel(fn, dim3(staged_grid(fn, a.n, tile, nseg), (unsigned)nseg),
                         dim3(kThreads), 0, stream, a);
  }
  auto fn = staged_copy_kernel<T, 4>;
  const size_t tile = (size_t)kThreads * kStageU * 4 * Elem<T>::kPerWord;
  return launch_kernel(fn, dim3(staged_grid(fn, a.n, tile, nseg), (unsigned)nseg), dim3(kThreads),
                       0, stream, a);
}

// ---- one reduction of one element type: the unit each build object holds --------
// DT 0 = fp32, 1 = bf16.  FAST (pairwise-tree sums) covers 4..8 sources only;
// the dispatcher sends every other source count to the rank-order unit, where
// the tree and the fold are the same sum (1..3 sources) or the fold is the
// defined order (runtime count).
template <int DT>
struct ElemOf {
  using type = float;
};
template <>
struct ElemOf<1> {
  using type = __nv_bfloat16;
};

template <int DT, int RED, bool FAST>
cudaError_t launch_part(int nseg, const MultiPtrArgs& a, cudaStream_t stream) {
  using T = typename ElemOf<DT>::type;
  if constexpr (RED == kRedCopy) {
    if (a.stage == kStageDestinations) return launch_staged_copy<T>(nseg, a, stream);
    if (a.stage != kStageNone) return cudaErrorInvalidValue;
    return launch_ns<T, 1, kRedCopy, false>(nseg, a, stream);
  } else if constexpr (FAST) {
    static_assert(RED == kRedSum, "only sums have a tree order");
    if (a.stage == kStageSources) {
      switch (a.nsrc) {
        case 4: return launch_staged_reduce_ns<T, 4, RED, true>(nseg, a, stream);
        case 5: return launch_staged_reduce_ns<T, 5, RED, true>(nseg, a, stream);
        case 6: return launch_staged_reduce_ns<T, 6, RED, true>(nseg, a, stream);
        case 7: return launch_staged_reduce_ns<T, 7, RED, true>(nseg, a, stream);
        case 8: return launch_staged_reduce_ns<T, 8, RED, true>(nseg, a, stream);
        default: return cudaErrorInvalidValue;
      }
    }
    if (a.stage != kStageNone || a.src_per_seg) return cudaErrorInvalidValue;
    switch (a.nsrc) {
      case 4: return launch_ns<T, 4, RED, true>(nseg, a, stream);
      case 5: return launch_ns<T, 5, RED, true>(nseg, a, stream);
      case 6: return launch_ns<T, 6, RED, true>(nseg, a, stream);
      case 7: return launch_ns<T, 7, RED, true>(nseg, a, stream);
      case 8: return launch_ns<T, 8, RED, true>(nseg, a, stream);
      default: return cudaErrorInvalidValue;
    }
  } else {
    if (a.stage == kStageSources) {
      switch (a.nsrc) {
        case 1: return launch_staged_reduce_ns<T, 1, RED, false>(nseg, a, stream);
        case 2: return launch_staged_reduce_ns<T, 2, RED, false>(nseg, a, stream);
        case 3: return launch_staged_reduce_ns<T, 3, RED, false>(nseg, a, stream);
        case 4: return launch_staged_reduce_ns<T, 4, RED, false>(nseg, a, stream);
        case 5: return launch_staged_reduce_ns<T, 5, RED, false>(nseg, a, stream);
        case 6: return launch_staged_reduce_ns<T, 6, RED, false>(nseg, a, stream);
        case 7: return launch_staged_reduce_ns<T, 7, RED, false>(nseg, a, stream);
        case 8: return launch_staged_reduce_ns<T, 8, RED, false>(nseg, a, stream);
        default: return launch_staged_reduce_ns<T, 0, RED, false>(nseg, a, stream);
      }
    }
    if (a.stage != kStageNone || a.src_per_seg) return cudaErrorInvalidValue;
    switch (a.nsrc) {
      case 1: return launch_ns<T, 1, RED, false>(nseg, a, stream);
      case 2: return launch_ns<T, 2, RED, false>(nseg, a, stream);
      case 3: return launch_ns<T, 3, RED, false>(nseg, a, stream);
      case 4: return launch_ns<T, 4, RED, false>(nseg, a, stream);
      case 5: return launch_ns<T, 5, RED, false>(nseg, a, stream);
      case 6: return launch_ns<T, 6, RED, false>(nseg, a, stream);
      case 7: return launch_ns<T, 7, RED, false>(nseg, a, stream);
      case 8: return launch_ns<T, 8, RED, false>(nseg, a, stream);
      default: return launch_ns<T, 0, RED, false>(nseg, a, stream);
    }
  }
}

}  // namespace mp
}  // namespace rcc
