// Working-set selection on the GPU: §5.1 Eq 6 of "Attention Routing
// Stabilizes Early: Working-Set Inference for Recurrent Language Models"
// (WISE) plus the CSR schedule of its Appendix B "Sparse-kernel
// implementation".
//
//  select_steps_kernel : Eq 6, one warp per (row, window step) with the row's
//      window warps in one CTA. The row's masses (lane l holds blocks
//      32*jj + l) are cut at the k-th mass on their float keys where the
//      2^-52 fixed point is exact (select_keys.cuh), else in the fixed point
//      (select_step.cuh); near-ties go toward lower indices. The ballot at
//      round jj is word jj of the step support (kept by lane jj); the steps
//      are OR-ed in shared memory, then the sink / diagonal blocks added.
//      CTAs run the query blocks from the last down (longest rows first).
//  select_rows_kernel  : the two early-static controls of WISE's Appendix B
//      ("Intervention controls") from one step's masses and a reference
//      working set, one warp per row: MassMatched (Eqs 20-21) replaces eta
//      by the row's mass covered by the reference, summed in the same fixed
//      point; SizeMatched (Eq 22) keeps the reference's block count k and
//      finds the k-th mass with a bitwise search on counts instead of sums.
//  finalize_kernel     : a dependent launch after either. row_ptr (a chunk
//      of rows sums the counts of all earlier rows from one bulk copy when it
//      starts early in the rows, else takes them from the chunks before it by
//      a decoupled look-back), nnz, ascending col_idx from the bitmasks, and
//      the late-step work order: every unit of the launch sorted by number of
//      listed blocks, heaviest first (ties by unit index), so that no heavy
//      unit starts near the end of a sparse step. Shapes whose ranking does
//      not fit in one CTA's shared memory are ranked per group of (batch,
//      head) slices.
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"
#include "select_keys.cuh"
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
  int32_t order_segs;          // segments of a group's units, one warp and one counter table each
  int32_t direct_rows;         // chunks starting at most this many rows in sum the earlier counts directly
  int32_t mode;                // 0: Eq 6 with eta; 1: MassMatched; 2: SizeMatched
  const int32_t* ref_row_ptr;  // reference working set (modes 1 and 2)
  const int32_t* ref_col_idx;
  int64_t ref_cap;
  uint64_t* lb;      // look-back state of the row_ptr scan (zeroed before finalize)
  int32_t lb_words;  // its size in 64-bit words
  uint32_t* err;
};

// Word `lane` of one row's Eq 6 step support at window step w, with NJ rounds
// of 32 blocks covering the row's q + 1 admissible blocks.
template <int NJ>
__device__ __forceinline__ uint32_t step_eq6(const SelectParams& p, int bh, int q, int w, int lane) {
  const int nadm = q + 1;
  const float* src = p.mass + (((int64_t)w * p.bh_count + bh) * p.nb + q) * p.nb;
  float m[NJ];
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) {
    const int b = jj * 32 + lane;  // coalesced load order: jj-major
    m[jj] = (b < nadm) ? __ldg(src + b) : 0.f;
  }
  uint32_t key[NJ];
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) key[jj] = (jj * 32 + lane < nadm) ? mass_key(m[jj]) : 0u;
  {
    // the usual case: the cut among masses in [2^-29, 2^10), decided on the
    // keys alone. A row of one round that needs more than 8 values (a flat
    // row) takes the single pass over all 32 below instead.
    uint32_t word;
    if (eq6_step_word_keys<NJ, (NJ == 1 ? 8 : kExtractLimit)>(key, p.target_fx, p.tol_fx, lane, word)) return word;
  }
  int64_t fx[NJ];
  // every admissible mass of the row in [2^-29, 2^10): the fixed point is a
  // plain shift; otherwise the general rounding
  bool exact = true;
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj)
    exact &= (jj * 32 + lane >= nadm) || mass_fx_exact(__float_as_uint(m[jj]));
  if (__all_sync(0xffffffffu, exact)) {
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj)
      fx[jj] = (jj * 32 + lane < nadm) ? mass_fx_exact_bits(__float_as_uint(m[jj])) : INT64_MIN;
  } else {
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) fx[jj] = (jj * 32 + lane < nadm) ? mass_fx(m[jj]) : INT64_MIN;
  }
  return eq6_step_word<NJ>(fx, key, p.target_fx, p.tol_fx, lane);
}

// The same with the fewest rounds that cover the row (a row near the start
// of the sequence costs less than one near its end).
template <int NJ>
__device__ __forceinline__ uint32_t step_eq6_any(const SelectParams& p, int bh, int q, int w, int lane) {
  const int nadm = q + 1;
  if (NJ == 1 || nadm <= 32) return step_eq6<1>(p, bh, q, w, lane);
  if (NJ == 2 || nadm <= 64) return step_eq6<(NJ < 2 ? NJ : 2)>(p, bh, q, w, lane);
  if (NJ == 4 || nadm <= 128) return step_eq6<(NJ < 4 ? NJ : 4)>(p, bh, q, w, lane);
  if (NJ == 8 || nadm <= 256) return step_eq6<(NJ < 8 ? NJ : 8)>(p, bh, q, w, lane);
  if (NJ == 16 || nadm <= 512) return step_eq6<(NJ < 16 ? NJ : 16)>(p, bh, q, w, lane);
  return step_eq6<NJ>(p, bh, q, w, lane);
}

// Eq 6 over the window: one warp per (row, window step), window warps per
// row; a CTA takes one query block q of rows_per_cta (batch, head) slices.
// blockIdx.y runs over q from the last query block down, so the CTAs with
// the longest rows (q + 1 admissible blocks) start first and the short ones
// fill the end of the launch. Each warp ORs its step support into the row's
// words in shared memory; the row's step-0 warp then adds the sink /
// diagonal blocks and writes the row's bitmask and count.
template <int NJ>
__global__ void __launch_bounds__(256, (NJ <= 8) ? 4 : 1) select_steps_kernel(const SelectParams p, int rows_per_cta) {
  __shared__ uint32_t rowbits[8][32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  // the finalize launch may be scheduled now; it waits for this grid to
  // finish (and its writes to be visible) before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the finalize kernel that follows starts from a cleared look-back state
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < p.lb_words; i += blockDim.x) p.lb[i] = 0ull;
  const int r_local = wid / p.window, w = wid - r_local * p.window;
  const int q = p.nb - 1 - (int)blockIdx.y;
  const int bh = (int)blockIdx.x * rows_per_cta + r_local;
  const bool live = r_local < rows_per_cta && bh < p.bh_count;
  const int64_t row = (int64_t)bh * p.nb + q;
  if (w == 0 && r_local < rows_per_cta) rowbits[r_local][lane] = 0u;
  __syncthreads();
  if (live) {
    const uint32_t word = step_eq6_any<NJ>(p, bh, q, w, lane);
    if (word) atomicOr(&rowbits[r_local][lane], word);
  }
  __syncthreads();
  if (!live || w != 0) return;
  uint32_t word = rowbits[r_local][lane];
  // Readings of this library: sink block 0 and diagonal block q.
  if ((p.flags & 1u) && lane == 0) word |= 1u;
  if ((p.flags & 2u) && lane == (q >> 5)) word |= 1u << (q & 31);
  const int cnt = warp_sum32(__popc(word));
  if (lane < p.nwords) p.bits[row * p.nwords + lane] = word;
  if (lane == 0) p.counts[row] = cnt;
}

// The early-static controls (one step, window 1): 8 warps per CTA, one row
// per warp; NJ rounds of 32 blocks cover nb <= 32 NJ.
template <int NJ>
__global__ void __launch_bounds__(256) select_rows_kernel(const SelectParams p) {
  __shared__ uint32_t refbits[8][32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  // the finalize kernel that follows starts from a cleared look-back state
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < p.lb_words; i += blockDim.x) p.lb[i] = 0ull;
  const int64_t row = (int64_t)blockIdx.x * 8 + wid;
  const int64_t rows = (int64_t)p.bh_count * p.nb;
  if (row >= rows) return;
  const int bh = (int)(row / p.nb);
  const int q = (int)(row % p.nb);
  const int nadm = q + 1;  // admissible key blocks 0..q
  uint32_t word = 0;  // word `lane` of the row's union bitmask
  {
    // Controls: the reference row as a bitmask (entries outside 0..q flagged
    // and skipped; repeated entries count once); in_ref[jj] is this lane's
    // block.
    bool in_ref[NJ];
    int ref_k = 0;
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
    for (int w = 0; w < p.window; ++w) {
      const float* src = p.mass + (((int64_t)w * p.bh_count + bh) * p.nb + q) * p.nb;
      int64_t fx[NJ];
      uint32_t key[NJ];
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) {
        const int bb = jj * 32 + lane;  // coalesced load order: jj-major
        const float m = (bb < nadm) ? __ldg(src + bb) : 0.f;
        fx[jj] = (bb < nadm) ? mass_fx(m) : INT64_MIN;
        key[jj] = (bb < nadm) ? mass_key(m) : 0u;
      }
      uint32_t sel_word_mine = 0;  // the word this lane will hold (word index = lane)
      int64_t target = 0;
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
        sel_word_mine = eq6_step_word<NJ>(fx, key, target, p.tol_fx, lane);
      }
      word |= sel_word_mine;
    }
  }
  // Readings of this library: sink block 0 and diagonal block q.
  if ((p.flags & 1u) && lane == 0) word |= 1u;
  if ((p.flags & 2u) && lane == (q >> 5)) word |= 1u << (q & 31);
  const int cnt = warp_sum32(__popc(word));
  if (lane < p.nwords) p.bits[row * p.nwords + lane] = word;
  if (lane == 0) p.counts[row] = cnt;
}

constexpr int kChunkRows = kSelectChunkRows;  // rows per finalize CTA (one per thread)
constexpr int kOrderWarps = kChunkRows / 32;
constexpr int kEmitStage = 1024;  // column entries staged per warp in the emit

// Look-back state of the row_ptr scan: one word per chunk of kChunkRows
// rows (flag in the top two bits: 1 = the chunk's own total, 2 = the total
// of every row up to and including the chunk). It sits after the bitmasks
// and counts in the workspace and is zeroed by the selection kernel (or, for
// a finalize-only launch, by a memset) before the finalize kernel runs.
constexpr uint64_t kLbAggregate = 1ull << 62, kLbInclusive = 2ull << 62, kLbValue = (1ull << 62) - 1;


__device__ __forceinline__ uint64_t ld_acquire_gpu(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Rank the units of one group of (batch, head) slices by cost (listed
// blocks), heaviest first, ties by unit index, and write their global order:
// a stable counting sort. The units are split into order_segs contiguous
// segments (8, 16 or 32), each with its own counter table: the counts per
// cost value of the segment's units, then the first position of the
// segment's units of every cost. Warp w serves segments w, w + 8, ..., one
// round of 32 units of each at a time, so the rounds of its segments
// overlap instead of waiting on each other.
// Shared memory: cost[units] | hist[order_segs][maxc + 1] | start[maxc + 1],
// maxc = nb * qb_per_unit.
__device__ void order_group(const SelectParams& p, int g, int32_t* sh) {
  constexpr int kMaxSpw = 4;  // segments per warp
  const int h0 = g * p.group_heads;
  const int gsize = min(p.group_heads, p.bh_count - h0);
  const int units = gsize * p.units_per_bh;
  const int maxc = p.nb * p.qb_per_unit;
  const int nc = maxc + 1;
  const int nseg = p.order_segs;
  const int spw = nseg / kOrderWarps;
  int32_t* cost = sh;
  __shared__ int32_t top_cost;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) top_cost = 0;
  // costs: the listed blocks of the unit's query blocks (at most four); each
  // thread requests a batch of counts before it uses any, so its loads
  // overlap instead of waiting on each other
  const int64_t row0 = (int64_t)h0 * p.nb;
  const int per_unit = p.qb_per_unit;
  if (per_unit == 1) {
    // one query block per unit: the group's rows in order, raw (clamped
    // where they are read). Taken by the TMA unit in bulk when aligned: a
    // single SM's own loads of this many counts wait on its few outstanding
    // misses.
    const int32_t* src = p.counts + row0;
    const uint32_t bytes = (uint32_t)units * 4u;
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(cost)) & 15u) == 0 && (bytes & 15u) == 0) {
      if (tid == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);
        fence_mbar_init();
      }
      __syncthreads();
      if (tid == 0) {
        constexpr uint32_t kPiece = 16384;
        mbar_arrive_expect_tx(&bar, bytes);
        for (uint32_t off = 0; off < bytes; off += kPiece) {
          const uint32_t n = min(kPiece, bytes - off);
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                  smem_u32(reinterpret_cast<uint8_t*>(cost) + off)),
              "l"(reinterpret_cast<const uint8_t*>(src) + off), "r"(n), "r"(smem_u32(&bar))
              : "memory");
        }
      }
      mbar_wait<7>(&bar, 0, &abort_flag, p.err);
    } else {
      constexpr int kBatch = 32;
      for (int base = 0; base < units; base += kBatch * (int)blockDim.x) {
        int v[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int u = base + k * (int)blockDim.x + tid;
          v[k] = (u < units) ? __ldg(src + u) : 0;
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int u = base + k * (int)blockDim.x + tid;
          if (u < units) cost[u] = v[k];
        }
      }
    }
  } else {
    constexpr int kBatch = 16;
    for (int base = 0; base < units; base += kBatch * (int)blockDim.x) {
      int v[kBatch][4];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int u = base + k * (int)blockDim.x + tid;
        const int bh = u / p.units_per_bh, pr = u % p.units_per_bh;
        const int nq = (u < units) ? min(per_unit, p.nb - pr * per_unit) : 0;
        const int32_t* src = p.counts + row0 + (int64_t)bh * p.nb + pr * per_unit;
#pragma unroll
        for (int j = 0; j < 4; ++j) v[k][j] = (j < nq) ? __ldg(src + j) : 0;
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int u = base + k * (int)blockDim.x + tid;
        if (u < units) cost[u] = min(max(v[k][0] + v[k][1] + v[k][2] + v[k][3], 0), maxc);
      }
    }
  }
  __syncthreads();
  const int64_t gbase = (int64_t)h0 * p.units_per_bh;
  int32_t* hist = cost + units;
  int32_t* start = hist + nseg * nc;
  for (int c = tid; c < nseg * nc; c += blockDim.x) hist[c] = 0;
  __syncthreads();
  const int seg = (units + nseg - 1) / nseg;
  int my_top = 0;
  for (int b = 0; b < seg; b += 32) {
#pragma unroll
    for (int k = 0; k < kMaxSpw; ++k) {
      if (k < spw) {
        const int sg = warp + kOrderWarps * k;
        const int lo = min(units, sg * seg), hi = min(units, lo + seg);
        const int u = lo + b + lane;
        if (u < hi) {
          const int c = min(max(cost[u], 0), maxc);
          atomicAdd(&hist[sg * nc + c], 1);
          my_top = max(my_top, c);
        }
      }
    }
  }
  my_top = (int)__reduce_max_sync(0xffffffffu, (uint32_t)my_top);
  if (lane == 0) atomicMax(&top_cost, my_top);
  __syncthreads();
  const int tc = top_cost;
  // start[c] = number of units with a larger cost (exclusive scan from the top)
  for (int c = tid; c <= tc; c += blockDim.x) {
    int t = 0;
    for (int w = 0; w < nseg; ++w) t += hist[w * nc + c];
    start[c] = t;
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int top = tc; top >= 0; top -= 32) {
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
  }
  __syncthreads();
  // first position of segment w's units of cost c
  for (int c = tid; c <= tc; c += blockDim.x) {
    int run = start[c];
    for (int w = 0; w < nseg; ++w) {
      const int h = hist[w * nc + c];
      hist[w * nc + c] = run;
      run += h;
    }
  }
  __syncthreads();
  // place each segment's units in index order, 32 at a time; equal costs
  // keep index order. The reads of all of the warp's segments come before
  // any of their writes (each segment has its own table).
  for (int b = 0; b < seg; b += 32) {
    int cs[kMaxSpw], us[kMaxSpw], bases[kMaxSpw];
    uint32_t peers[kMaxSpw];
#pragma unroll
    for (int k = 0; k < kMaxSpw; ++k) {
      const int sg = warp + kOrderWarps * k;
      const int lo = min(units, sg * seg), hi = min(units, lo + seg);
      us[k] = lo + b + lane;
      cs[k] = (k < spw && us[k] < hi) ? min(max(cost[us[k]], 0), maxc) : -1;
    }
#pragma unroll
    for (int k = 0; k < kMaxSpw; ++k) peers[k] = (k < spw) ? __match_any_sync(0xffffffffu, cs[k]) : 0u;
#pragma unroll
    for (int k = 0; k < kMaxSpw; ++k)
      bases[k] = (cs[k] >= 0) ? hist[(warp + kOrderWarps * k) * nc + cs[k]] : 0;
    __syncwarp();
#pragma unroll
    for (int k = 0; k < kMaxSpw; ++k) {
      if (cs[k] >= 0) {
        const int rank = __popc(peers[k] & ((1u << lane) - 1u));
        p.tile_order[gbase + bases[k] + rank] = (int32_t)(gbase + us[k]);
        if (rank == 0) hist[(warp + kOrderWarps * k) * nc + cs[k]] = bases[k] + __popc(peers[k]);
      }
    }
    __syncwarp();
  }
}

// Finalize, one launch: CTA k < n_chunks takes the k-th chunk of kChunkRows
// rows, gets the count of all earlier rows from the chunks before it
// (decoupled look-back: a chunk publishes its own total at once and the
// running total as soon as it knows it), writes its row_ptr entries and
// emits its rows' column lists in ascending order; the remaining CTAs build
// the late-step work order, one group each. CTAs are dispatched in index
// order, so every chunk a CTA waits for is already running (the usual
// assumption of a single-pass scan); the wait is bounded all the same.
__global__ void __launch_bounds__(kChunkRows, 1) finalize_kernel(const SelectParams p, int n_chunks, uint64_t* lb) {
  extern __shared__ __align__(16) int32_t sh[];
  __shared__ int32_t red[kOrderWarps];
  __shared__ int32_t start_s[kChunkRows];
  __shared__ int32_t cnt_s[kChunkRows];
  __shared__ int64_t s_prefix;
  __shared__ int64_t red64[kOrderWarps];
  __shared__ uint64_t pre_bar;
  __shared__ int pre_abort;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // launched early after the Eq 6 kernel: wait until its bitmasks, counts
  // and cleared look-back state are complete and visible (a no-op after an
  // ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if ((int)blockIdx.x >= n_chunks) {
    order_group(p, blockIdx.x - n_chunks, sh);
    return;
  }
  uint64_t* state = lb;
  const int64_t rows = (int64_t)p.bh_count * p.nb;
  const int chunk = (int)blockIdx.x;
  const int64_t r0 = (int64_t)chunk * kChunkRows;
  const int nrows = (int)min((int64_t)kChunkRows, rows - r0);
  const int64_t r = r0 + tid;
  const int c = (tid < nrows) ? __ldg(p.counts + r) : 0;
  // the chunk's bit words, read coalesced into shared memory (row stride
  // nwords + 1, so that the lanes of a warp reading consecutive rows' words
  // hit distinct banks); behind them, the warps' staging areas for the emit
  const int nw = p.nwords, stride = nw + 1;
  uint32_t* bits_s = reinterpret_cast<uint32_t*>(sh);
  uint32_t* stage = bits_s + kChunkRows * stride;
  {
    const uint32_t* src = p.bits + r0 * nw;
    const int total = nrows * nw;
#pragma unroll 4
    for (int i = tid; i < total; i += kChunkRows) {
      const int rr = i / nw;
      bits_s[rr * stride + (i - rr * nw)] = __ldg(src + i);
    }
  }
  // A chunk that starts within the first direct_rows rows sums the counts of
  // all earlier rows itself (one bulk copy into shared memory) instead of
  // waiting for the chunks before it; the others look back.
  int32_t* pre_s = reinterpret_cast<int32_t*>(stage + kOrderWarps * kEmitStage);
  const bool direct = chunk > 0 && r0 <= (int64_t)p.direct_rows &&
                      (reinterpret_cast<uintptr_t>(p.counts) & 15u) == 0;
  if (direct && tid == 0) {
    pre_abort = 0;
    mbar_init(&pre_bar, 1);
    fence_mbar_init();
    const uint32_t bytes = (uint32_t)r0 * 4u;
    constexpr uint32_t kPiece = 16384;
    mbar_arrive_expect_tx(&pre_bar, bytes);
    for (uint32_t off = 0; off < bytes; off += kPiece) {
      const uint32_t n = min(kPiece, bytes - off);
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              smem_u32(reinterpret_cast<uint8_t*>(pre_s) + off)),
          "l"(reinterpret_cast<const uint8_t*>(p.counts) + off), "r"(n), "r"(smem_u32(&pre_bar))
          : "memory");
    }
  }
  cnt_s[tid] = c;
  // exclusive scan of this chunk's counts
  int inc = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  int wpre = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kOrderWarps; ++w) {
    wpre += (w < warp) ? red[w] : 0;
    total += red[w];
  }
  if (direct) {
    mbar_wait<8>(&pre_bar, 0, &pre_abort, p.err);
    int part = 0;
    for (int i = tid; i < (int)r0; i += kChunkRows) part += pre_s[i];
    part = warp_sum32(part);
    if (lane == 0) red64[warp] = part;
    __syncthreads();
    if (tid == 0) {
      int64_t prefix = 0;
#pragma unroll
      for (int w = 0; w < kOrderWarps; ++w) prefix += red64[w];
      st_release_gpu(state + chunk, kLbInclusive | (uint64_t)(prefix + total));
      s_prefix = prefix;
    }
  } else if (warp == 0) {
    // look back over the chunks before this one, 32 at a time
    if (lane == 0)
      st_release_gpu(state + chunk, (chunk == 0 ? kLbInclusive : kLbAggregate) | (uint64_t)total);
    int64_t prefix = 0;
    int j = chunk - 1;
    const uint64_t t0 = global_timer_ns();
    bool timed_out = false;
    while (j >= 0 && !timed_out) {
      const int idx = j - lane;
      uint64_t st = (idx >= 0) ? ld_acquire_gpu(state + idx) : kLbInclusive;
      // wait until every chunk of this window up to the nearest finished one has published
      const uint32_t incl = __ballot_sync(0xffffffffu, (st >> 62) == 2u);
      const int stop = incl ? __ffs(incl) - 1 : 31;  // nearest chunk with a running total
      const uint32_t unready = __ballot_sync(0xffffffffu, (st >> 62) == 0u) & ((stop == 31) ? 0xffffffffu
                                                                                   : ((2u << stop) - 1u));
      if (unready) {
        if (global_timer_ns() - t0 > kWaitLimitNs) timed_out = true;
        continue;
      }
      int64_t v = (lane <= stop) ? (int64_t)(st & kLbValue) : 0;
      prefix += warp_sum64(v);
      if (incl) break;
      j -= 32;
    }
    if (timed_out && lane == 0) atomicOr(p.err, kErrTimeout);
    if (lane == 0) {
      if (chunk > 0) st_release_gpu(state + chunk, kLbInclusive | (uint64_t)(prefix + total));
      s_prefix = prefix;
    }
  }
  __syncthreads();
  const int64_t prefix = s_prefix;
  const int64_t start = prefix + wpre + inc - c;
  if (r < rows) p.row_ptr[r] = (int32_t)start;
  start_s[tid] = (int32_t)start;
  if (r == rows - 1) {
    p.row_ptr[rows] = (int32_t)(start + c);
    if (p.nnz) *p.nnz = (int32_t)(start + c);
    if (start + c > p.col_cap) atomicOr(p.err, kErrBadSupport);
  }
  __syncthreads();
  // emit: warp w writes the column lists of rows 32 w .. 32 w + 31, which
  // are contiguous in col_idx. Each lane expands its row's set bits, in
  // ascending order, into the warp's staging area; the warp then copies the
  // area out with consecutive lanes on consecutive entries. A warp whose
  // lists exceed the area or the capacity writes each row directly instead
  // (a row over capacity is flagged above and skipped). A lane writes at
  // most its row's count.
  {
    const int i = 32 * warp + lane;
    const bool have = i < nrows;
    const int64_t my_start = have ? start_s[i] : 0;
    const int my_cnt = have ? cnt_s[i] : 0;
    const int64_t ws = __shfl_sync(0xffffffffu, my_start, 0);
    const int wn = warp_sum32(my_cnt);
    if (32 * warp < nrows) {
      const uint32_t* rowbits = bits_s + i * stride;
      if (ws + wn <= p.col_cap && wn <= kEmitStage) {
        uint32_t* st = stage + warp * kEmitStage;
        if (have) {
          int off = (int)(my_start - ws);
          const int lim = off + my_cnt;
          for (int j = 0; j < nw; ++j) {
            uint32_t x = rowbits[j];
            while (x && off < lim) {
              st[off++] = 32u * j + __ffs(x) - 1;
              x &= x - 1;
            }
          }
        }
        __syncwarp();
        for (int e = lane; e < wn; e += 32) p.col_idx[ws + e] = (int32_t)st[e];
      } else if (have) {
        int64_t pos = my_start;
        const int64_t end = pos + my_cnt;
        if (end <= p.col_cap) {
          for (int j = 0; j < nw; ++j) {
            uint32_t x = rowbits[j];
            while (x && pos < end) {
              p.col_idx[pos++] = 32 * j + __ffs(x) - 1;
              x &= x - 1;
            }
          }
        }
      }
    }
  }
}

cudaError_t launch_select(const SelectLaunch& s, cudaStream_t stream) {
  SelectParams p = {};
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
  // shared memory (cost per unit + per-segment and total counters per cost
  // value); 32 segments when their counters take at most half of it, else
  // 16 or 8
  {
    constexpr size_t kOrderSmem = 200u * 1024u;
    const size_t nc = (size_t)s.nb * s.qb_per_unit + 1;
    int segs = 4 * kOrderWarps;
    while (segs > kOrderWarps && nc * sizeof(int32_t) * (segs + 1) > kOrderSmem / 2) segs >>= 1;
    const size_t fixed = nc * sizeof(int32_t) * (segs + 1);
    const size_t per_slice = (size_t)s.units_per_bh * sizeof(int32_t);
    int64_t g = s.bh_count;
    if (fixed + per_slice * (size_t)g > kOrderSmem) g = (int64_t)((kOrderSmem - fixed) / per_slice);
    p.group_heads = (int32_t)(g < 1 ? 1 : g);
    p.order_segs = segs;
  }
  p.mode = s.mode;
  p.ref_row_ptr = s.ref_row_ptr;
  p.ref_col_idx = s.ref_col_idx;
  p.ref_cap = s.ref_cap;
  p.err = s.err;
  const int64_t rows = (int64_t)s.bh_count * s.nb;
  p.lb = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(s.bits) + select_lookback_offset(rows, p.nwords));
  p.lb_words = (int32_t)(select_lookback_bytes(rows) / 8);
  const unsigned grid_rows = (unsigned)((rows + 7) / 8);
  const int rounds = (s.nb + 31) / 32;
  // Eq 6: window warps per row, as many rows per CTA as fit in 8 warps
  const int rpc = (s.window >= 1 && s.window <= 8) ? 8 / s.window : 1;
  const dim3 grid_steps((unsigned)((s.bh_count + rpc - 1) / rpc), (unsigned)s.nb);
  const unsigned threads_steps = (unsigned)(32 * s.window * rpc);
  if (s.finalize_only) {
    // the row bitmasks and counts come from the discovery epilogue
    cudaError_t e = cudaMemsetAsync(p.lb, 0, (size_t)p.lb_words * 8, stream);
    if (e != cudaSuccess) return e;
  } else if (s.mode == 0) {
    if (rounds <= 1) select_steps_kernel<1><<<grid_steps, threads_steps, 0, stream>>>(p, rpc);
    else if (rounds <= 2) select_steps_kernel<2><<<grid_steps, threads_steps, 0, stream>>>(p, rpc);
    else if (rounds <= 4) select_steps_kernel<4><<<grid_steps, threads_steps, 0, stream>>>(p, rpc);
    else if (rounds <= 8) select_steps_kernel<8><<<grid_steps, threads_steps, 0, stream>>>(p, rpc);
    else if (rounds <= 16) select_steps_kernel<16><<<grid_steps, threads_steps, 0, stream>>>(p, rpc);
    else select_steps_kernel<32><<<grid_steps, threads_steps, 0, stream>>>(p, rpc);
  } else if (rounds <= 1) select_rows_kernel<1><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 2) select_rows_kernel<2><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 4) select_rows_kernel<4><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 8) select_rows_kernel<8><<<grid_rows, 256, 0, stream>>>(p);
  else if (rounds <= 16) select_rows_kernel<16><<<grid_rows, 256, 0, stream>>>(p);
  else select_rows_kernel<32><<<grid_rows, 256, 0, stream>>>(p);
  const int n_chunks = (int)((rows + kChunkRows - 1) / kChunkRows);
  const int groups = s.tile_order ? (s.bh_count + p.group_heads - 1) / p.group_heads : 0;
  const size_t shm_order = s.tile_order ? ((size_t)p.group_heads * s.units_per_bh +
                                           (size_t)(p.order_segs + 1) * ((size_t)s.nb * s.qb_per_unit + 1)) *
                                              sizeof(int32_t)
                                        : 0;
  // chunks within the first kDirectRows rows sum the earlier counts directly
  constexpr int64_t kDirectRows = 16384;
  p.direct_rows = (int32_t)(rows < kDirectRows ? rows : kDirectRows);
  const size_t shm_chunk =
      ((size_t)kChunkRows * (p.nwords + 1) + (size_t)kOrderWarps * kEmitStage + (size_t)p.direct_rows) *
      sizeof(uint32_t);
  const size_t shm = shm_order > shm_chunk ? shm_order : shm_chunk;
  if (shm > 40 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shm);
    if (e != cudaSuccess) return e;
  }
  // after the Eq 6 kernel, finalize is a programmatic dependent launch: its
  // CTAs are scheduled while the last Eq 6 CTAs run
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_chunks + groups));
  cfg.blockDim = dim3(kChunkRows);
  cfg.dynamicSmemBytes = shm;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = (!s.finalize_only && s.mode == 0) ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, finalize_kernel, p, n_chunks, p.lb);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace wise
