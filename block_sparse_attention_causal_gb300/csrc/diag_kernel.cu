// Support diagnostics of WISE ("Attention Routing Stabilizes Early:
// Working-Set Inference for Recurrent Language Models"):
//
//  * retained future attention mass (Appendix B, "Evaluation metrics"): for a
//    late step's unrestricted block masses r_qb (§5.1 Eq 5), the share of each
//    query block's mass that falls inside the frozen support, sum over b in B_q
//    of r_qb, and its mean over the query blocks of each batch element;
//  * rolling working-set stability (Appendix C.2 Eq 24): the Jaccard index
//    |A intersect B| / |A union B| of two supports, taken over all active
//    (head, query block, key block) entries of each batch element.
//
// Both are memory-bound reductions over KBs to MBs: one warp per CSR row,
// then one CTA per batch element for a deterministic tree reduction.
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace wise {
namespace {

constexpr int kDiagWarps = 8;  // rows per CTA in the per-row kernels

__device__ __forceinline__ bool row_range(const int32_t* row_ptr, int64_t row, int64_t cap, int32_t& a, int32_t& b) {
  a = __ldg(row_ptr + row);
  b = __ldg(row_ptr + row + 1);
  if (a < 0 || b < a || (int64_t)b > cap) {
    a = b = 0;
    return false;
  }
  return true;
}

// r = sum of the row's listed admissible key blocks of the mass row (fp64
// accumulation, fixed lane order, so repeated calls give identical bits).
__global__ void __launch_bounds__(kDiagWarps * 32) retained_rows_kernel(DiagLaunch d) {
  const int64_t row = (int64_t)blockIdx.x * kDiagWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= d.rows) return;
  const int q = (int)(row % d.nb);
  const float* r = d.mass + row * d.nb;
  int32_t a, b;
  bool bad = !row_range(d.row_ptr_a, row, d.col_cap, a, b);
  double s = 0.0;
  for (int32_t j = a + lane; j < b; j += 32) {
    const int32_t c = __ldg(d.col_idx_a + j);
    if (c >= 0 && c <= q) s += (double)__ldg(r + c);
    else bad = true;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(d.err, kErrBadSupport);
  if (lane == 0) d.row_value[row] = (float)s;
}

// Per row: |A intersect B| and |A union B| of the two supports' key-block sets,
// from two bitmasks of up to 1024 blocks in shared memory (entries outside
// the admissible range are reported and skipped; duplicates count once).
__global__ void __launch_bounds__(kDiagWarps * 32) jaccard_rows_kernel(DiagLaunch d) {
  __shared__ uint32_t bits[kDiagWarps][2][32];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kDiagWarps + w;
  if (row >= d.rows) return;
  const int q = (int)(row % d.nb);
  bits[w][0][lane] = 0u;
  bits[w][1][lane] = 0u;
  __syncwarp();
  bool bad = false;
  for (int side = 0; side < 2; ++side) {
    const int32_t* rp = side ? d.row_ptr_b : d.row_ptr_a;
    const int32_t* ci = side ? d.col_idx_b : d.col_idx_a;
    int32_t a, b;
    bad |= !row_range(rp, row, side ? d.col_cap_b : d.col_cap, a, b);
    for (int32_t j = a + lane; j < b; j += 32) {
      const int32_t c = __ldg(ci + j);
      if (c >= 0 && c <= q) atomicOr(&bits[w][side][c >> 5], 1u << (c & 31));
      else bad = true;
    }
  }
  __syncwarp();
  int inter = __popc(bits[w][0][lane] & bits[w][1][lane]);
  int uni = __popc(bits[w][0][lane] | bits[w][1][lane]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    inter += __shfl_xor_sync(0xffffffffu, inter, off);
    uni += __shfl_xor_sync(0xffffffffu, uni, off);
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(d.err, kErrBadSupport);
  if (lane == 0) {
    d.row_counts[2 * row] = inter;
    d.row_counts[2 * row + 1] = uni;
  }
}

// One CTA per batch element: tree reductions over its heads x nb rows.
// Retained mass: mean of the rows' values. Jaccard: sums of the counts and
// their ratio (1 when both supports are empty).
__global__ void __launch_bounds__(256) batch_reduce_kernel(DiagLaunch d, int jaccard) {
  __shared__ double sh_v[256];
  __shared__ long long sh_i[256], sh_u[256];
  const int64_t per_batch = d.rows / d.batch;
  const int64_t r0 = (int64_t)blockIdx.x * per_batch;
  double v = 0.0;
  long long in = 0, un = 0;
  for (int64_t i = threadIdx.x; i < per_batch; i += blockDim.x) {
    if (jaccard) {
      in += d.row_counts[2 * (r0 + i)];
      un += d.row_counts[2 * (r0 + i) + 1];
    } else {
      v += (double)d.row_value[r0 + i];
    }
  }
  sh_v[threadIdx.x] = v;
  sh_i[threadIdx.x] = in;
  sh_u[threadIdx.x] = un;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      sh_v[threadIdx.x] += sh_v[threadIdx.x + s];
      sh_i[threadIdx.x] += sh_i[threadIdx.x + s];
      sh_u[threadIdx.x] += sh_u[threadIdx.x + s];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (jaccard) {
      if (d.batch_counts) {
        d.batch_counts[2 * blockIdx.x] = sh_i[0];
        d.batch_counts[2 * blockIdx.x + 1] = sh_u[0];
      }
      if (d.batch_value) d.batch_value[blockIdx.x] = sh_u[0] ? (double)sh_i[0] / (double)sh_u[0] : 1.0;
    } else if (d.batch_value) {
      d.batch_value[blockIdx.x] = per_batch ? sh_v[0] / (double)per_batch : 0.0;
    }
  }
}

}  // namespace

cudaError_t launch_retained_mass(const DiagLaunch& d, cudaStream_t stream) {
  const int64_t grid = (d.rows + kDiagWarps - 1) / kDiagWarps;
  retained_rows_kernel<<<(unsigned)grid, kDiagWarps * 32, 0, stream>>>(d);
  if (d.batch_value) batch_reduce_kernel<<<(unsigned)d.batch, 256, 0, stream>>>(d, 0);
  return cudaGetLastError();
}

cudaError_t launch_jaccard(const DiagLaunch& d, cudaStream_t stream) {
  const int64_t grid = (d.rows + kDiagWarps - 1) / kDiagWarps;
  jaccard_rows_kernel<<<(unsigned)grid, kDiagWarps * 32, 0, stream>>>(d);
  if (d.batch_value || d.batch_counts) batch_reduce_kernel<<<(unsigned)d.batch, 256, 0, stream>>>(d, 1);
  return cudaGetLastError();
}

}  // namespace wise
