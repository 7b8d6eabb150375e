/*
 * rcc_oracle_omp.cpp -- a second CPU baseline for the benchmark: the fp32
 * rank-order all_reduce of the oracle's deterministic mode, with the element
 * loop spread over host threads by OpenMP.
 *
 * TEST INFRASTRUCTURE ONLY, and not part of the oracle's reference path: no
 * test compares anything against it.  Only the benchmark's CPU-baseline leg
 * loads it, to report what all host cores reach beside the single-threaded
 * oracle.  It shares no code with the CUDA library.
 *
 * Per element i (ruCCL README §2 all_reduce; §5: sum and mean):
 *   acc = x_0[i]; acc = fl32(acc + x_r[i]) for r = 1..R-1 (sum, mean);
 *   mean: fl32(acc / R);
 *   max/min: acc replaced only by a strictly greater (smaller) value, any NaN
 *   gives the quiet NaN 0x7FC00000.
 * Every rank's output receives the result.
 */
#include <cstddef>
#include <cstdint>
#include <cstring>

extern "C" int orc_omp_all_reduce_f32(int R, const float* const* send, float* const* recv,
                                      size_t n, int op, int threads) {
  if (R < 1 || op < 0 || op > 3 || threads < 1) return -1;
  const long long count = static_cast<long long>(n);
#pragma omp parallel for num_threads(threads) schedule(static)
  for (long long i = 0; i < count; ++i) {
    float acc = send[0][i];
    bool nan = acc != acc;
    for (int r = 1; r < R; ++r) {
      const float x = send[r][i];
      if (op <= 1) {
        acc = acc + x;
      } else {
        nan = nan || (x != x);
        if (op == 2 ? (x > acc) : (x < acc)) acc = x;
      }
    }
    if (op == 1) acc = acc / static_cast<float>(R);
    if (op >= 2 && nan) {
      const uint32_t q = 0x7FC00000u;
      std::memcpy(&acc, &q, 4);
    }
    for (int r = 0; r < R; ++r) recv[r][i] = acc;
  }
  return 0;
}
