// The gathered-entry plan of late (reuse) steps with blocks of 32, built once
// per support after the CSR schedule (WISE, "Attention Routing Stabilizes
// Early: Working-Set Inference for Recurrent Language Models", Appendix B
// "Sparse-kernel implementation": the schedule is built once after discovery
// and reused by every late step). One warp per 128-row tile: the union of its
// four query blocks' lists in ascending order, four key blocks per entry,
// with the mask of which query block lists which slot (gather.cuh) -- the
// entries the late-step scheduler would otherwise form on every claim.
#include <stdint.h>

#include "gather.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace wise {

__global__ void __launch_bounds__(256) gather_plan_kernel(const GatherPlanLaunch g) {
  const int lane = threadIdx.x & 31;
  const int64_t u = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t n_units = (int64_t)g.bh_count * g.n_qtiles;
  if (u >= n_units) return;
  const int bh = (int)(u / g.n_qtiles), t = (int)(u % g.n_qtiles);
  // CSR rows of query blocks 4t .. 4t + nq - 1 (row_ptr entries 0 .. nq)
  const int qb0 = 4 * t;
  const int nq = min(4, g.nb - qb0);
  const int64_t row0 = (int64_t)bh * g.nb + qb0;
  const int32_t rpv = (lane <= nq) ? __ldg(g.row_ptr + row0 + lane) : 0;
  int32_t a[4], b[4], v0[4];
  bool bad = false;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    a[q] = __shfl_sync(0xffffffffu, rpv, q);
    b[q] = __shfl_sync(0xffffffffu, rpv, q + 1);
    if (q >= nq) {
      a[q] = b[q] = 0;
    } else if (a[q] < 0 || a[q] > b[q] || (int64_t)b[q] > g.col_cap) {
      bad = true;
      a[q] = b[q] = 0;
    }
    v0[q] = (a[q] + lane < b[q]) ? __ldg(g.col_idx + a[q] + lane) : INT32_MAX;
  }
  const uint32_t w0 = gather_list_bits(g.col_idx, a[0], b[0], qb0 + 0, v0[0], lane, bad);
  const uint32_t w1 = gather_list_bits(g.col_idx, a[1], b[1], qb0 + 1, v0[1], lane, bad);
  const uint32_t w2 = gather_list_bits(g.col_idx, a[2], b[2], qb0 + 2, v0[2], lane, bad);
  const uint32_t w3 = gather_list_bits(g.col_idx, a[3], b[3], qb0 + 3, v0[3], lane, bad);
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(g.err, kErrBadSupport);
  uint32_t rem = w0 | w1 | w2 | w3;
  uint32_t* dst = g.entries + 4 * plan_entry_index(bh, t, g.n_qtiles);
  // at most t + 1 entries: the lists hold key blocks 0 .. 4t + 3 only
  int cnt = 0;
  while (cnt <= t && __any_sync(0xffffffffu, rem != 0u)) {
    int kb[4] = {0, 0, 0, 0};
    const uint32_t mask = gather_take_entry(rem, w0, w1, w2, w3, lane, kb);
    if (lane < 4) {
      const uint32_t word = (lane == 0) ? ((uint32_t)kb[0] | ((uint32_t)kb[1] << 16))
                            : (lane == 1) ? ((uint32_t)kb[2] | ((uint32_t)kb[3] << 16))
                            : (lane == 2) ? mask
                                          : 0u;
      dst[4 * cnt + lane] = word;
    }
    ++cnt;
  }
  if (lane == 0) g.counts[u] = cnt;
}

cudaError_t launch_gather_plan(const GatherPlanLaunch& g, cudaStream_t stream) {
  const int64_t n_units = (int64_t)g.bh_count * g.n_qtiles;
  if (n_units <= 0) return cudaSuccess;
  gather_plan_kernel<<<(unsigned)((n_units + 7) / 8), 256, 0, stream>>>(g);
  return cudaGetLastError();
}

}  // namespace wise
