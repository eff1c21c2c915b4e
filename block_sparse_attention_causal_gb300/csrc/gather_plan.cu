// The gathered-entry plan of late (reuse) steps with blocks of 32, built once
// per support after the CSR schedule (WISE, "Attention Routing Stabilizes
// Early: Working-Set Inference for Recurrent Language Models", Appendix B
// "Sparse-kernel implementation": the schedule is built once after discovery
// and reused by every late step). One warp per 128-row tile: the union of its
// four query blocks' lists in ascending order, four key blocks per entry,
// with the mask of which query block lists which slot -- the entries that
// the late-step scheduler would otherwise form one at a time on every claim
// (gather.cuh).
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace wise {

// Entries of the longest tile (key blocks 0 .. 1023, four per entry).
constexpr int kPlanMaxEntries = 256;

// Lane l's word of the key blocks listed by one CSR row (query block qb), as
// gather_list_bits, with each admissible value's bit OR-ed into the warp's
// words in shared memory (wrow, zeroed) instead of one shuffle round per
// target word.
__device__ __forceinline__ uint32_t plan_list_bits(const int32_t* col_idx, int32_t a, int32_t b, int qb, int32_t v,
                                                   int lane, bool& bad, uint32_t* wrow) {
  int32_t prev = -1;
  for (int32_t base = a; base < b; base += 32) {
    if (base != a) v = (base + lane < b) ? __ldg(col_idx + base + lane) : INT32_MAX;
    const bool in = base + lane < b;
    int32_t pv = __shfl_up_sync(0xffffffffu, v, 1);
    if (lane == 0) pv = prev;
    const bool ok = in && v >= 0 && v > pv && v <= qb;
    if (in && !ok) bad = true;
    if (ok) atomicOr(&wrow[v >> 5], 1u << (v & 31));
    prev = __shfl_sync(0xffffffffu, v, 31);
  }
  __syncwarp();
  return wrow[lane];
}

// One warp per 128-row tile. The union of the four lists is ranked at once:
// the set bits of lane l's word follow the set bits of lanes < l, so bit i of
// lane l is the (prefix + k)-th block of the union in ascending order; it
// goes to slot r % 4 of entry r / 4, and the query blocks listing it set
// that entry's mask bits (OR-ed in shared memory).
__global__ void __launch_bounds__(256) gather_plan_kernel(const GatherPlanLaunch g) {
  __shared__ uint32_t words_s[8][4][32];
  __shared__ uint32_t mask_s[8][kPlanMaxEntries];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t u = (int64_t)blockIdx.x * 8 + wid;
  const int64_t n_units = (int64_t)g.bh_count * g.n_qtiles;
  if (u >= n_units) return;
  const int bh = (int)(u / g.n_qtiles), t = (int)(u % g.n_qtiles);
#pragma unroll
  for (int j = 0; j < 4; ++j) words_s[wid][j][lane] = 0u;
  __syncwarp();
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
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) w[q] = plan_list_bits(g.col_idx, a[q], b[q], qb0 + q, v0[q], lane, bad, words_s[wid][q]);
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(g.err, kErrBadSupport);
  const uint32_t un = w[0] | w[1] | w[2] | w[3];
  // rank of this lane's first block in the union
  const int pc = __popc(un);
  int incl = pc;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  // the lists hold key blocks 0 .. 4t + 3, at most t + 1 entries
  const int ne = min((total + 3) / 4, t + 1);
  uint32_t* mk = mask_s[wid];
  for (int e = lane; e < ne; e += 32) mk[e] = 0u;
  __syncwarp();
  uint16_t* half = reinterpret_cast<uint16_t*>(g.entries + 4 * plan_entry_index(bh, t, g.n_qtiles));
  int r = incl - pc;
  for (uint32_t x = un; x != 0u; x &= x - 1u, ++r) {
    const int i = __ffs(x) - 1;
    const int e = r >> 2, c = r & 3;
    if (e >= ne) break;
    half[8 * e + c] = (uint16_t)(32 * lane + i);
    uint32_t m = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) m |= ((w[q] >> i) & 1u) << (4 * q + c);
    atomicOr(&mk[e], m);
    // slots past the union's end repeat its last block (masked for every row)
    if (r == total - 1)
      for (int cc = c + 1; cc < 4; ++cc) half[8 * e + cc] = (uint16_t)(32 * lane + i);
  }
  __syncwarp();
  uint32_t* ent = g.entries + 4 * plan_entry_index(bh, t, g.n_qtiles);
  for (int e = lane; e < ne; e += 32) {
    ent[4 * e + 2] = mk[e];
    ent[4 * e + 3] = 0u;
  }
  if (lane == 0) g.counts[u] = ne;
}

cudaError_t launch_gather_plan(const GatherPlanLaunch& g, cudaStream_t stream) {
  const int64_t n_units = (int64_t)g.bh_count * g.n_qtiles;
  if (n_units <= 0) return cudaSuccess;
  gather_plan_kernel<<<(unsigned)((n_units + 7) / 8), 256, 0, stream>>>(g);
  return cudaGetLastError();
}

}  // namespace wise
