// Working-set selection on the GPU: §5.1 Eq 6 of "Attention Routing
// Stabilizes Early: Working-Set Inference for Recurrent Language Models"
// (WISE) plus the CSR schedule of its Appendix B "Sparse-kernel
// implementation".
//
//  select_rows_kernel : one warp per (batch, head, query block) row. For each
//      window step it finds the Eq 6 support without sorting (select_step.cuh:
//      int64 fixed point, a search for the k-th mass, near-ties toward lower
//      indices). Element jj of lane l is block 32*jj + l, so the ballot at
//      step jj is word jj of the row's support bitmask (kept by lane jj).
//      Steps are OR-ed, then the sink / diagonal blocks added.
//      The same kernel builds the two early-static controls of WISE's
//      Appendix B ("Intervention controls") from one step's masses and a
//      reference working set: MassMatched (Eqs 20-21) replaces eta by the
//      row's mass covered by the reference, summed in the same fixed point;
//      SizeMatched (Eq 22) keeps the reference's block count k and finds the
//      k-th mass with a bitwise search on counts instead of sums.
//  finalize_kernel    : row_ptr (each CTA adds up the counts before its rows),
//      nnz, ascending col_idx from the bitmasks, and the late-step work order:
//      every unit of the launch sorted by number of listed blocks, heaviest
//      first (ties by unit index), so that no heavy unit starts near the end
//      of a sparse step. Shapes whose ranking does not fit in one CTA's
//      shared memory are ranked per group of (batch, head) slices.
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"
#include "select_step.cuh"

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
  int32_t units_per_bh;
  int32_t qb_per_unit;  // query blocks per work unit (128 / block)
  int32_t group_heads;
  int32_t mode;                // 0: Eq 6 with eta; 1: MassMatched; 2: SizeMatched
  const int32_t* ref_row_ptr;  // reference working set (modes 1 and 2)
  const int32_t* ref_col_idx;
  int64_t ref_cap;
  uint32_t* err;
};

// 8 warps per CTA, one row per warp; NJ rounds of 32 blocks cover nb <= 32 NJ.
template <int NJ>
__global__ void __launch_bounds__(256) select_rows_kernel(const SelectParams p) {
  __shared__ uint32_t refbits[8][32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * 8 + wid;
  const int64_t rows = (int64_t)p.bh_count * p.nb;
  if (row >= rows) return;
  const int bh = (int)(row / p.nb);
  const int q = (int)(row % p.nb);
  const int nadm = q + 1;  // admissible key blocks 0..q
  // Controls: the reference row as a bitmask (entries outside 0..q flagged and
  // skipped; repeated entries count once); in_ref[jj] is this lane's block.
  bool in_ref[NJ];
  int ref_k = 0;
  if (p.mode != 0) {
    refbits[wid][lane] = 0u;
    __syncwarp();
    int32_t a = __ldg(p.ref_row_ptr + row), b = __ldg(p.ref_row_ptr + row + 1);
    bool bad = false;
    if (a < 0 || b < a || (int64_t)b > p.ref_cap) {
      a = b = 0;
      bad = true;
    }
    for (int32_t j = a + lane; j < b; j += 32) {
      const int32_t c = __ldg(p.ref_col_idx + j);
      if (c >= 0 && c <= q) atomicOr(&refbits[wid][c >> 5], 1u << (c & 31));
      else bad = true;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.err, kErrBadSupport);
    __syncwarp();
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) in_ref[jj] = (refbits[wid][jj] >> lane) & 1u;
    ref_k = warp_sum32(__popc(refbits[wid][lane]));
  }
  uint32_t word = 0;  // word `lane` of the row's union bitmask
  for (int w = 0; w < p.window; ++w) {
    const float* src = p.mass + (((int64_t)w * p.bh_count + bh) * p.nb + q) * p.nb;
    int64_t fx[NJ];
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
      const int b = jj * 32 + lane;  // coalesced load order: jj-major
      fx[jj] = (b < nadm) ? mass_fx(__ldg(src + b)) : INT64_MIN;
    }
    uint32_t sel_word_mine = 0;  // the word this lane will hold (word index = lane)
    int64_t target = p.target_fx;
    if (p.mode == 1) {  // MassMatched: the mass the reference covers at this step
      int64_t t = 0;
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) t += (in_ref[jj] && fx[jj] > 0) ? fx[jj] : 0;
      target = warp_sum_u63(t);
    }
    if ((p.mode == 1 && target <= 0) || (p.mode == 2 && ref_k == 0)) {
      // an empty reference (or one without mass) selects nothing
    } else if (p.mode == 2) {
      // SizeMatched: the ref_k largest masses; v = the largest value with at
      // least ref_k admissible blocks >= v
      int64_t v = 0;
      if (ref_k < nadm) {
        if (NJ == 1) {
          // one value per lane: v = the largest value with >= ref_k values >= it
          int c = 0;
#pragma unroll 8
          for (int j = 0; j < 32; ++j) c += (__shfl_sync(0xffffffffu, fx[0], j) >= fx[0]) ? 1 : 0;
          v = warp_max64((fx[0] != INT64_MIN && c >= ref_k) ? fx[0] : 0);
        } else {
          int64_t max_pos = 0;
#pragma unroll
          for (int jj = 0; jj < NJ; ++jj) max_pos = max(max_pos, fx[jj]);
          max_pos = warp_max64(max_pos);
          for (int bit = 63 - __clzll(max_pos > 0 ? max_pos : 1); bit >= 0; --bit) {
            const int64_t cand = v | (int64_t(1) << bit);
            int cnt = 0;
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) cnt += (fx[jj] >= cand) ? 1 : 0;
            if (warp_sum32(cnt) >= ref_k) v = cand;
          }
        }
      }
      int c_above = 0;
      const int64_t hi = v + p.tol_fx, lo = v - p.tol_fx;
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) c_above += (fx[jj] != INT64_MIN && fx[jj] > hi) ? 1 : 0;
      c_above = warp_sum32(c_above);
      const int k = min(ref_k, nadm);
      int slots = k - c_above;  // filled from the near-tie group, lowest index first
      int taken = 0;
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) {
        const bool above = fx[jj] != INT64_MIN && fx[jj] > hi;
        const bool near = fx[jj] != INT64_MIN && fx[jj] >= lo && fx[jj] <= hi;
        const uint32_t nb_bal = __ballot_sync(0xffffffffu, near);
        const int rank = taken + __popc(nb_bal & ((1u << lane) - 1u));
        const bool pick = above || (near && rank < slots);
        taken += __popc(nb_bal);
        const uint32_t bal = __ballot_sync(0xffffffffu, pick);
        if (lane == jj) sel_word_mine = bal;
      }
    } else {
      sel_word_mine = eq6_step_word<NJ>(fx, target, p.tol_fx, lane);
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

constexpr int kChunkRows = 256;  // rows per finalize CTA (one per thread)

// Rank the units of one group of (batch, head) slices by cost (listed
// blocks), heaviest first, ties by unit index, and write their global order:
// a stable counting sort.
// Shared memory: cost[units] | start[maxc + 1], maxc = nb * qb_per_unit.
__device__ void order_group(const SelectParams& p, int g, int32_t* sh) {
  const int h0 = g * p.group_heads;
  const int gsize = min(p.group_heads, p.bh_count - h0);
  const int units = gsize * p.units_per_bh;
  const int maxc = p.nb * p.qb_per_unit;
  int32_t* cost = sh;
  int32_t* start = sh + units;
  for (int c = threadIdx.x; c <= maxc; c += blockDim.x) start[c] = 0;
  __syncthreads();
  for (int u = threadIdx.x; u < units; u += blockDim.x) {
    const int bh = h0 + u / p.units_per_bh, pr = u % p.units_per_bh;
    int c = 0;
    for (int j = 0; j < p.qb_per_unit; ++j) {
      const int qb = pr * p.qb_per_unit + j;
      if (qb < p.nb) c += p.counts[(int64_t)bh * p.nb + qb];
    }
    c = min(max(c, 0), maxc);
    cost[u] = c;
    atomicAdd(&start[c], 1);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    // start[c] = number of units with a larger cost (exclusive scan from the top)
    int run = 0;
    for (int top = maxc; top >= 0; top -= 32) {
      const int c = top - lane;
      const int h = (c >= 0) ? start[c] : 0;
      int inc = h;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
      }
      if (c >= 0) start[c] = run + inc - h;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    __syncwarp();
    // place the units in index order, 32 at a time; equal costs keep index order
    const int64_t gbase = (int64_t)h0 * p.units_per_bh;
    for (int b = 0; b < units; b += 32) {
      const int u = b + lane;
      const int c = (u < units) ? cost[u] : -1;
      const uint32_t peers = __match_any_sync(0xffffffffu, c);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int base = (u < units) ? start[c] : 0;
      __syncwarp();
      if (u < units) {
        p.tile_order[gbase + base + rank] = h0 * p.units_per_bh + u;
        if (rank == 0) start[c] = base + __popc(peers);
      }
      __syncwarp();
    }
  }
}

// Finalize, one launch: CTAs [0, n_chunks) each take kChunkRows rows, add up
// the counts of every earlier row themselves (no separate scan pass), write
// their row_ptr entries and emit their rows' column lists in ascending order;
// the remaining CTAs build the late-step work order, one group each.
__global__ void __launch_bounds__(kChunkRows) finalize_kernel(const SelectParams p, int n_chunks) {
  extern __shared__ int32_t sh[];
  __shared__ int64_t red[kChunkRows / 32];
  __shared__ int32_t start_s[kChunkRows];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if ((int)blockIdx.x >= n_chunks) {
    order_group(p, blockIdx.x - n_chunks, sh);
    return;
  }
  const int64_t rows = (int64_t)p.bh_count * p.nb;
  const int64_t r0 = (int64_t)blockIdx.x * kChunkRows;
  // counts of all rows before this chunk
  int64_t pre = 0;
  for (int64_t r = tid; r < r0; r += kChunkRows) pre += p.counts[r];
  pre = warp_sum64(pre);
  if (lane == 0) red[warp] = pre;
  __syncthreads();
  int64_t prefix = 0;
#pragma unroll
  for (int w = 0; w < kChunkRows / 32; ++w) prefix += red[w];
  __syncthreads();
  // exclusive scan of this chunk's counts
  const int64_t r = r0 + tid;
  const int c = (r < rows) ? p.counts[r] : 0;
  int inc = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  int64_t wpre = 0;
  for (int w = 0; w < warp; ++w) wpre += red[w];
  const int64_t start = prefix + wpre + inc - c;
  if (r < rows) p.row_ptr[r] = (int32_t)start;
  start_s[tid] = (int32_t)start;
  if (r == rows - 1) {
    p.row_ptr[rows] = (int32_t)(start + c);
    if (p.nnz) *p.nnz = (int32_t)(start + c);
    if (start + c > p.col_cap) atomicOr(p.err, kErrBadSupport);
  }
  __syncthreads();
  // emit: one warp per row, lane j holds bitmask word j; a warp's rows are
  // i = warp + 8k, and all their words are loaded before the first is used
  // (one round of memory latency instead of one per row)
  constexpr int kRowsPerWarp = kChunkRows / (kChunkRows / 32);
  uint32_t words[kRowsPerWarp];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int64_t row = r0 + warp + k * (kChunkRows / 32);
    words[k] = (row < rows && lane < p.nwords) ? __ldg(p.bits + row * p.nwords + lane) : 0u;
  }
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int i = warp + k * (kChunkRows / 32);
    const int64_t row = r0 + i;
    if (row >= rows) break;
    const uint32_t word = words[k];
    const int wc = __popc(word);
    int excl = wc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, excl, off);
      if (lane >= off) excl += y;
    }
    const int total = __shfl_sync(0xffffffffu, excl, 31);
    excl -= wc;
    const int64_t st = start_s[i];
    if (st + total > p.col_cap) continue;  // flagged above
    uint32_t w = word;
    int64_t pos = st + excl;
    while (w) {
      const int bit = __ffs(w) - 1;
      p.col_idx[pos++] = lane * 32 + bit;
      w &= w - 1;
    }
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
  p.units_per_bh = s.units_per_bh;
  p.qb_per_unit = s.qb_per_unit;
  // ranking groups: all slices in one group when its counting sort fits in
  // shared memory (cost per unit + one counter per cost value)
  {
    constexpr size_t kOrderSmem = 200u * 1024u;
    const size_t fixed = ((size_t)s.nb * s.qb_per_unit + 1) * sizeof(int32_t);
    const size_t per_slice = (size_t)s.units_per_bh * sizeof(int32_t);
    int64_t g = s.bh_count;
    if (fixed + per_slice * (size_t)g > kOrderSmem) g = (int64_t)((kOrderSmem - fixed) / per_slice);
    p.group_heads = (int32_t)(g < 1 ? 1 : g);
  }
  p.mode = s.mode;
  p.ref_row_ptr = s.ref_row_ptr;
  p.ref_col_idx = s.ref_col_idx;
  p.ref_cap = s.ref_cap;
  p.err = s.err;
  const int64_t rows = (int64_t)s.bh_count * s.nb;
  const unsigned grid_rows = (unsigned)((rows + 7) / 8);
  const int rounds = (s.nb + 31) / 32;
  if (s.finalize_only) {
    // the row bitmasks and counts come from the discovery epilogue
  } else if (rounds <= 1) select_rows_kernel<1><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 2) select_rows_kernel<2><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 4) select_rows_kernel<4><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 8) select_rows_kernel<8><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 16) select_rows_kernel<16><<<grid_rows, 256, 0, stream>>>(p);
  else select_rows_kernel<32><<<grid_rows, 256, 0, stream>>>(p);
  const int n_chunks = (int)((rows + kChunkRows - 1) / kChunkRows);
  const int groups = s.tile_order ? (s.bh_count + p.group_heads - 1) / p.group_heads : 0;
  const size_t shm =
      s.tile_order ? ((size_t)p.group_heads * s.units_per_bh + (size_t)s.nb * s.qb_per_unit + 1) * sizeof(int32_t) : 0;
  if (shm > 40 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm);
    if (e != cudaSuccess) return e;
  }
  finalize_kernel<<<n_chunks + groups, kChunkRows, shm, stream>>>(p, n_chunks);
  return cudaGetLastError();
}

}  // namespace wise
