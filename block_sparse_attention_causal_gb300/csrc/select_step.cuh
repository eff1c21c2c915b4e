// One step of the working-set selection of WISE ("Attention Routing
// Stabilizes Early: Working-Set Inference for Recurrent Language Models"),
// §5.1 Eq 6, for one (batch, head, query block) row, run by one warp. Shared
// by the selection kernel and the discovery epilogue that selects while it
// writes the block masses, so both give the same bits.
//
// Masses are int64 fixed point (2^-52 units). Element jj of lane l is key
// block 32 jj + l (INT64_MIN past the admissible range). Without sorting, a
// search finds the largest value v* whose "mass of all blocks >= v*" still
// reaches the target; then k = |{> v*}| + ceil((target - sum{> v*}) / v*)
// and v* is the k-th mass in (mass desc, index asc) order. Blocks within the
// tolerance of v* are taken toward lower indices. If the admissible mass
// cannot reach the target, every admissible block is taken.
#pragma once
#include <stdint.h>

namespace wise {

__device__ __forceinline__ int64_t warp_sum64(int64_t v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
// Warp sum of lane values in [0, 2^63 / 32): three 21-bit slices summed with
// the hardware reduction (each slice sum < 2^26), then recombined exactly.
__device__ __forceinline__ int64_t warp_sum_u63(int64_t v) {
  const uint64_t u = static_cast<uint64_t>(v);
  const uint32_t a = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(u & 0x1FFFFFu));
  const uint32_t b = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>((u >> 21) & 0x1FFFFFu));
  const uint32_t c = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(u >> 42));
  return static_cast<int64_t>(a) + (static_cast<int64_t>(b) << 21) + (static_cast<int64_t>(c) << 42);
}
__device__ __forceinline__ int64_t warp_max64(int64_t v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, (int64_t)__shfl_xor_sync(0xffffffffu, v, off));
  return v;
}
__device__ __forceinline__ int warp_sum32(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// A mass in the selection's fixed point (round to nearest).
__device__ __forceinline__ int64_t mass_fx(float m) { return __double2ll_rn((double)m * 4503599627370496.0); }

// Word `lane` of the row's step support (bit i = key block 32 lane + i) for
// a positive target mass; tol is the tie tolerance (both fixed point).
// COMPACT keeps the one-pass loop rolled (a small instruction footprint for
// callers that share the SM with instruction-heavy warps).
template <int NJ, bool COMPACT = false>
__device__ __forceinline__ uint32_t eq6_step_word(const int64_t (&fx)[NJ], int64_t target, int64_t tol, int lane) {
  int64_t total_pos = 0, max_pos = 0;
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) {
    total_pos += (fx[jj] > 0) ? fx[jj] : 0;
    max_pos = max(max_pos, fx[jj]);
  }
  total_pos = warp_sum64(total_pos);
  max_pos = warp_max64(max_pos);
  uint32_t sel_word_mine = 0;  // the word this lane will hold (word index = lane)
  if (total_pos < target) {
    // Eq 6 cannot reach the target: every admissible block.
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
      const uint32_t bal = __ballot_sync(0xffffffffu, fx[jj] != INT64_MIN);
      if (lane == jj) sel_word_mine = bal;
    }
    return sel_word_mine;
  }
  // largest v with sum_{fx >= v} fx >= target (v > 0 since target > 0);
  // v <= the largest mass, so bits above its top bit stay zero
  int64_t v = 0;
  if (NJ == 1) {
    // one value per lane: v = the largest value x with sum{>= x} >= target
    // (the value the bitwise search below converges to)
    const int64_t mine = fx[0];
    int64_t acc = 0;
    if (COMPACT) {
#pragma unroll 1
      for (int j = 0; j < 32; ++j) {
        const int64_t o = __shfl_sync(0xffffffffu, mine, j);
        acc += (o >= mine && o > 0) ? o : 0;
      }
    } else {
#pragma unroll 8
      for (int j = 0; j < 32; ++j) {
        const int64_t o = __shfl_sync(0xffffffffu, mine, j);
        acc += (o >= mine && o > 0) ? o : 0;
      }
    }
    v = warp_max64((mine > 0 && acc >= target) ? mine : 0);
  } else {
    for (int bit = 63 - __clzll(max_pos); bit >= 0; --bit) {
      const int64_t cand = v | (int64_t(1) << bit);
      int64_t sacc = 0;
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) sacc += (fx[jj] >= cand) ? fx[jj] : 0;
      sacc = warp_sum_u63(sacc);
      if (sacc >= target) v = cand;
    }
  }
  int64_t s_gt = 0;
  int c_gt = 0, c_above = 0;
  const int64_t hi = v + tol, lo = v - tol;
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) {
    s_gt += (fx[jj] > v) ? fx[jj] : 0;
    c_gt += (fx[jj] > v) ? 1 : 0;
    c_above += (fx[jj] > hi) ? 1 : 0;
  }
  s_gt = warp_sum64(s_gt);
  c_gt = warp_sum32(c_gt);
  c_above = warp_sum32(c_above);
  const int64_t need = target - s_gt;  // > 0
  const int m = (int)((need + v - 1) / v);
  const int k = c_gt + m;
  const int slots = k - c_above;  // filled from the near-tie group, lowest index first
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
  return sel_word_mine;
}

}  // namespace wise
