// Working-set selection on the GPU: §5.1 Eq 6 of "Attention Routing
// Stabilizes Early: Working-Set Inference for Recurrent Language Models"
// (WISE) plus the CSR schedule of its Appendix B "Sparse-kernel
// implementation".
//
//  select_rows_kernel : one warp per (batch, head, query block) row. For each
//      window step it finds the Eq 6 support without sorting: masses become
//      int64 fixed point (2^-52 units); a bitwise search finds the largest
//      value v* whose "mass of all blocks >= v*" still reaches eta; then
//      k = |{> v*}| + ceil((eta - sum{> v*}) / v*) and v* is the k-th mass in
//      (mass desc, index asc) order. Near-ties within the tolerance of v* are
//      resolved toward lower indices with ballots in index order. Element jj
//      of lane l is block 32*jj + l, so the ballot at step jj is word jj of
//      the row's support bitmask (kept by lane jj). Steps are OR-ed, then the
//      sink / diagonal blocks added.
//  scan_rows_kernel   : exclusive scan of the row counts -> row_ptr, nnz.
//  emit_rows_kernel   : bitmask -> ascending col_idx at row_ptr[row].
//  order_units_kernel : late-step work order: per L2 group of (batch, head)
//      slices, units sorted by number of listed blocks, heaviest first.
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace wise {

struct SelectParams {
  const float* mass;  // [W, BH, nb, nb]
  int32_t window;
  int32_t bh_count;
  int32_t nb;
  int32_t nwords;       // ceil(nb / 32)
  int64_t target_fx;    // eta in fixed point
  int64_t tol_fx;       // tie tolerance in fixed point
  uint32_t flags;
  uint32_t* bits;       // [rows, nwords]
  int32_t* counts;      // [rows]
  int32_t* row_ptr;     // [rows + 1]
  int32_t* col_idx;
  int64_t col_cap;
  int32_t* nnz;
  int32_t* tile_order;
  int32_t npairs;
  int32_t qb_per_unit;  // query blocks per work unit (256 / block)
  int32_t group_heads;
  uint32_t* err;
};

__device__ __forceinline__ int64_t warp_sum64(int64_t v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
__device__ __forceinline__ int warp_sum32(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// 8 warps per CTA, one row per warp; NJ rounds of 32 blocks cover nb <= 32 NJ.
template <int NJ>
__global__ void __launch_bounds__(256) select_rows_kernel(const SelectParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t rows = (int64_t)p.bh_count * p.nb;
  if (row >= rows) return;
  const int bh = (int)(row / p.nb);
  const int q = (int)(row % p.nb);
  const int nadm = q + 1;  // admissible key blocks 0..q
  uint32_t word = 0;  // word `lane` of the row's union bitmask
  for (int w = 0; w < p.window; ++w) {
    const float* src = p.mass + (((int64_t)w * p.bh_count + bh) * p.nb + q) * p.nb;
    int64_t fx[NJ];
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
      const int b = jj * 32 + lane;  // coalesced load order: jj-major
      fx[jj] = (b < nadm) ? __double2ll_rn((double)__ldg(src + b) * 4503599627370496.0) : INT64_MIN;
    }
    int64_t total_pos = 0, max_pos = 0;
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
      total_pos += (fx[jj] > 0) ? fx[jj] : 0;
      max_pos = max(max_pos, fx[jj]);
    }
    total_pos = warp_sum64(total_pos);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) max_pos = max(max_pos, (int64_t)__shfl_xor_sync(0xffffffffu, max_pos, off));
    uint32_t sel_word_mine = 0;  // the word this lane will hold (word index = lane)
    if (total_pos < p.target_fx) {
      // Eq 6 cannot reach eta: every admissible block.
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) {
        const uint32_t bal = __ballot_sync(0xffffffffu, fx[jj] != INT64_MIN);
        if (lane == jj) sel_word_mine = bal;
      }
    } else {
      // largest v with sum_{fx >= v} fx >= target (v > 0 since target > 0);
      // v <= the largest mass, so bits above its top bit stay zero
      int64_t v = 0;
      for (int bit = 63 - __clzll(max_pos); bit >= 0; --bit) {
        const int64_t cand = v | (int64_t(1) << bit);
        int64_t sacc = 0;
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) sacc += (fx[jj] >= cand) ? fx[jj] : 0;
        sacc = warp_sum64(sacc);
        if (sacc >= p.target_fx) v = cand;
      }
      int64_t s_gt = 0;
      int c_gt = 0, c_above = 0;
      const int64_t hi = v + p.tol_fx, lo = v - p.tol_fx;
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) {
        s_gt += (fx[jj] > v) ? fx[jj] : 0;
        c_gt += (fx[jj] > v) ? 1 : 0;
        c_above += (fx[jj] > hi) ? 1 : 0;
      }
      s_gt = warp_sum64(s_gt);
      c_gt = warp_sum32(c_gt);
      c_above = warp_sum32(c_above);
      const int64_t need = p.target_fx - s_gt;  // > 0
      const int m = (int)((need + v - 1) / v);
      const int k = c_gt + m;
      int slots = k - c_above;  // filled from the near-tie group, lowest index first
      int taken = 0;
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) {
        const bool above = fx[jj] != INT64_MIN && fx[jj] > hi;
        const bool near = fx[jj] != INT64_MIN && fx[jj] >= lo && fx[jj] <= hi;
        const uint32_t nb_bal = __ballot_sync(0xffffffffu, near);
        // rank of this lane's near block among near blocks of lower index
        const int rank = taken + __popc(nb_bal & ((1u << lane) - 1u));
        const bool pick = above || (near && rank < slots);
        taken += __popc(nb_bal);
        const uint32_t bal = __ballot_sync(0xffffffffu, pick);
        if (lane == jj) sel_word_mine = bal;
      }
    }
    word |= sel_word_mine;
  }
  // Readings of this library: sink block 0 and diagonal block q.
  if ((p.flags & 1u) && lane == 0) word |= 1u;
  if ((p.flags & 2u) && lane == (q >> 5)) word |= 1u << (q & 31);
  const int cnt = warp_sum32(__popc(word));
  if (lane < p.nwords) p.bits[row * p.nwords + lane] = word;
  if (lane == 0) p.counts[row] = cnt;
}

// Single CTA: exclusive scan of counts into row_ptr.
__global__ void __launch_bounds__(1024) scan_rows_kernel(const SelectParams p) {
  __shared__ int64_t warp_tot[32];
  const int64_t rows = (int64_t)p.bh_count * p.nb;
  const int tid = threadIdx.x;
  const int64_t per = (rows + 1023) / 1024;
  const int64_t r0 = min(rows, tid * per), r1 = min(rows, r0 + per);
  int64_t local = 0;
  for (int64_t r = r0; r < r1; ++r) local += p.counts[r];
  // block-wide exclusive scan of `local`
  const int lane = tid & 31, warp = tid >> 5;
  int64_t inc = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int64_t t = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  int64_t base = inc - local + (warp > 0 ? warp_tot[warp - 1] : 0);
  for (int64_t r = r0; r < r1; ++r) {
    p.row_ptr[r] = (int32_t)base;
    base += p.counts[r];
  }
  if (tid == 1023) {
    p.row_ptr[rows] = (int32_t)base;
    if (p.nnz) *p.nnz = (int32_t)base;
    if (base > p.col_cap) atomicOr(p.err, kErrBadSupport);
  }
}

// One warp per row: write the set bits of the row's bitmask in ascending order.
__global__ void __launch_bounds__(256) emit_rows_kernel(const SelectParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t rows = (int64_t)p.bh_count * p.nb;
  if (row >= rows) return;
  const uint32_t word = (lane < p.nwords) ? p.bits[row * p.nwords + lane] : 0u;
  const int c = __popc(word);
  int excl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, excl, off);
    if (lane >= off) excl += y;
  }
  excl -= c;
  const int64_t start = p.row_ptr[row];
  if (start + p.counts[row] > p.col_cap) return;  // flagged by the scan
  uint32_t w = word;
  int64_t pos = start + excl;
  while (w) {
    const int bit = __ffs(w) - 1;
    p.col_idx[pos++] = lane * 32 + bit;
    w &= w - 1;
  }
}

// One CTA per L2 group: rank units by cost (listed blocks), heaviest first,
// ties by unit index.
__global__ void __launch_bounds__(256) order_units_kernel(const SelectParams p) {
  extern __shared__ int32_t cost[];
  const int g = blockIdx.x;
  const int h0 = g * p.group_heads;
  const int gsize = min(p.group_heads, p.bh_count - h0);
  const int units = gsize * p.npairs;
  for (int u = threadIdx.x; u < units; u += blockDim.x) {
    const int bh = h0 + u / p.npairs, pr = u % p.npairs;
    int c = 0;
    for (int j = 0; j < p.qb_per_unit; ++j) {
      const int qb = pr * p.qb_per_unit + j;
      if (qb < p.nb) c += p.counts[(int64_t)bh * p.nb + qb];
    }
    cost[u] = c;
  }
  __syncthreads();
  const int64_t gbase = (int64_t)h0 * p.npairs;
  for (int u = threadIdx.x; u < units; u += blockDim.x) {
    const int c = cost[u];
    int pos = 0;
    for (int v = 0; v < units; ++v) {
      const int cv = cost[v];
      pos += (cv > c || (cv == c && v < u)) ? 1 : 0;
    }
    const int bh = h0 + u / p.npairs, pr = u % p.npairs;
    p.tile_order[gbase + pos] = bh * p.npairs + pr;
  }
}

cudaError_t launch_select(const SelectLaunch& s, cudaStream_t stream) {
  SelectParams p;
  p.mass = s.mass;
  p.window = s.window;
  p.bh_count = s.bh_count;
  p.nb = s.nb;
  p.nwords = (s.nb + 31) / 32;
  p.target_fx = s.target_fx;
  p.tol_fx = s.tol_fx;
  p.flags = s.flags;
  p.bits = s.bits;
  p.counts = s.counts;
  p.row_ptr = s.row_ptr;
  p.col_idx = s.col_idx;
  p.col_cap = s.col_cap;
  p.nnz = s.nnz;
  p.tile_order = s.tile_order;
  p.npairs = s.npairs;
  p.qb_per_unit = s.qb_per_unit;
  p.group_heads = s.group_heads;
  p.err = s.err;
  const int64_t rows = (int64_t)s.bh_count * s.nb;
  const unsigned grid_rows = (unsigned)((rows + 7) / 8);
  const int rounds = (s.nb + 31) / 32;
  if (rounds <= 1) select_rows_kernel<1><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 2) select_rows_kernel<2><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 4) select_rows_kernel<4><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 8) select_rows_kernel<8><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 16) select_rows_kernel<16><<<grid_rows, 256, 0, stream>>>(p);
  else select_rows_kernel<32><<<grid_rows, 256, 0, stream>>>(p);
  scan_rows_kernel<<<1, 1024, 0, stream>>>(p);
  emit_rows_kernel<<<grid_rows, 256, 0, stream>>>(p);
  if (s.tile_order) {
    const int groups = (s.bh_count + s.group_heads - 1) / s.group_heads;
    const size_t shm = (size_t)s.group_heads * s.npairs * sizeof(int32_t);
    if (shm > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(order_units_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm);
      if (e != cudaSuccess) return e;
    }
    order_units_kernel<<<groups, 256, shm, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace wise
