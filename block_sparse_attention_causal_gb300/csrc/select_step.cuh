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

// A mass in the selection's fixed point: round(m * 2^52), ties to even, in
// integer arithmetic on the float's fields (no FP64 work, which is slow on
// this GPU). With m = M * 2^(e - 150) (M the 24-bit significand), m * 2^52 =
// M * 2^(e - 98): exact for e >= 98 (masses >= 2^-29), a rounded right
// shift below. Values past 2^63 saturate; NaN gives 0. Masses are expected
// in [0, 1].
__device__ __forceinline__ int64_t mass_fx_bits(uint32_t b) {
  const uint32_t e = (b >> 23) & 0xffu;
  const uint32_t frac = b & 0x7fffffu;
  if (e == 0xffu) return frac ? 0 : ((b >> 31) ? -INT64_MAX : INT64_MAX);
  const uint32_t sig = e ? (frac | 0x800000u) : frac;
  const int sh = (int)(e ? e : 1u) - 98;
  int64_t v;
  if (sh >= 0) {
    v = (sh > 39) ? INT64_MAX : (int64_t)((uint64_t)sig << sh);
  } else {
    const int r = min(-sh, 26);
    const uint32_t q = sig >> r, rem = sig & ((1u << r) - 1u), half = 1u << (r - 1);
    v = (int64_t)(q + ((rem > half || (rem == half && (q & 1u))) ? 1u : 0u));
  }
  return (b >> 31) ? -v : v;
}
__device__ __forceinline__ int64_t mass_fx(float m) { return mass_fx_bits(__float_as_uint(m)); }

// Whether mass_fx_bits is the plain shift M << (e - 98) for this float: a
// positive mass in [2^-29, 2^10), where the fixed point is exact.
__device__ __forceinline__ bool mass_fx_exact(uint32_t b) { return b >= (98u << 23) && b < (137u << 23); }
__device__ __forceinline__ int64_t mass_fx_exact_bits(uint32_t b) {
  return (int64_t)((uint64_t)((b & 0x7fffffu) | 0x800000u) << ((b >> 23) - 98u));
}

// Ordering key of a mass for the cut search: its float bits when it is
// positive (the bits of positive floats order like their values, and
// mass_fx_bits is non-decreasing in them), 0 otherwise.
__device__ __forceinline__ uint32_t mass_key(float m) { return (m > 0.f) ? __float_as_uint(m) : 0u; }

// Word `lane` of the row's step support (bit i = key block 32 lane + i) for
// a positive target mass; tol is the tie tolerance (both fixed point). fx
// holds the fixed-point masses (INT64_MIN past the admissible range).
//
// v* (the k-th mass) is the fixed-point value at which the cumulative mass,
// taken in descending order, first reaches the target: the largest v with
// sum{fx >= v} >= target. The callers find v* (eq6_cut_value below); this
// part forms the support from it.
template <int NJ>
__device__ __forceinline__ uint32_t eq6_word_from_cut(const int64_t (&fx)[NJ], int64_t v, int64_t target,
                                                      int64_t tol, int lane, bool gt_known = false,
                                                      int64_t s_gt_known = 0, int c_gt_known = 0) {
  uint32_t sel_word_mine = 0;  // the word this lane will hold (word index = lane)
  const int64_t hi = v + tol, lo = v - tol;
  int64_t s_gt = s_gt_known;
  int c_gt = c_gt_known, c_above = 0, c_near = 0;
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) {
    if (!gt_known) {
      s_gt += (fx[jj] > v) ? fx[jj] : 0;
      c_gt += (fx[jj] > v) ? 1 : 0;
    }
    c_above += (fx[jj] > hi) ? 1 : 0;
    c_near += (fx[jj] != INT64_MIN && fx[jj] >= lo && fx[jj] <= hi) ? 1 : 0;
  }
  if (!gt_known) {
    s_gt = warp_sum_u63(s_gt);
    c_gt = (int)__reduce_add_sync(0xffffffffu, (uint32_t)c_gt);
  }
  c_above = (int)__reduce_add_sync(0xffffffffu, (uint32_t)c_above);
  c_near = (int)__reduce_add_sync(0xffffffffu, (uint32_t)c_near);
  // m = ceil(need / v) blocks of mass v complete the target; 1 <= m <= the
  // number of blocks at v (usually 1), so an estimate corrected by exact
  // integer products replaces a 64-bit division
  const int64_t need = target - s_gt;  // > 0
  int m = (int)fminf(fmaxf((float)need / (float)v, 1.f), 4096.f);
  while (m > 1 && (int64_t)(m - 1) * v >= need) --m;
  while ((int64_t)m * v < need) ++m;
  const int k = c_gt + m;
  const int slots = k - c_above;  // filled from the near-tie group, lowest index first
  if (slots >= c_near) {
    // the whole near-tie group is taken (the usual case: v alone)
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
      const bool pick = fx[jj] != INT64_MIN && fx[jj] >= lo;
      const uint32_t bal = __ballot_sync(0xffffffffu, pick);
      if (lane == jj) sel_word_mine = bal;
    }
    return sel_word_mine;
  }
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

// Every admissible block (Eq 6 cannot reach the target).
template <int NJ>
__device__ __forceinline__ uint32_t eq6_all_admissible(const int64_t (&fx)[NJ], int lane) {
  uint32_t sel_word_mine = 0;
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) {
    const uint32_t bal = __ballot_sync(0xffffffffu, fx[jj] != INT64_MIN);
    if (lane == jj) sel_word_mine = bal;
  }
  return sel_word_mine;
}

// v* for rows of up to 32 blocks (one value per lane): each lane sums the
// masses >= its own.
template <bool COMPACT>
__device__ __forceinline__ int64_t eq6_cut_one_round(int64_t mine, int64_t target) {
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
  return warp_max64((mine > 0 && acc >= target) ? mine : 0);
}

// The selection kernel's step: key holds the masses' ordering keys (mass_key;
// 0 past the admissible range). Rows of more than 32 blocks take the
// distinct largest keys one at a time (a warp max and a warp count per
// value), which ends after a few values on the concentrated rows the method
// produces; after kExtractLimit values without reaching the target, a
// bitwise search over the 31-bit keys finds the crossing instead
// (K* = the largest key K with sum{key >= K} fx >= target; since fx is
// non-decreasing in the key, v* = fx(K*)).
constexpr int kExtractLimit = 24;

// Compare-exchange keeping a >= b.
__device__ __forceinline__ void cx_desc(uint32_t& a, uint32_t& b) {
  const uint32_t hi = max(a, b), lo = min(a, b);
  a = hi;
  b = lo;
}
// Each lane's keys in descending order (a sorting network).
template <int NJ>
__device__ __forceinline__ void sort_desc(uint32_t (&q)[NJ]) {
#pragma unroll
  for (int k = 2; k <= NJ; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
      for (int i = 0; i < NJ; ++i) {
        const int l = i ^ j;
        if (l > i) {
          if ((i & k) == 0) cx_desc(q[i], q[l]);
          else cx_desc(q[l], q[i]);
        }
      }
}

template <int NJ>
__device__ __forceinline__ uint32_t eq6_step_word(const int64_t (&fx)[NJ], const uint32_t (&key)[NJ],
                                                  int64_t target, int64_t tol, int lane) {
  int64_t total_pos = 0;
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) total_pos += (fx[jj] > 0) ? fx[jj] : 0;
  if (warp_sum_u63(total_pos) < target) return eq6_all_admissible<NJ>(fx, lane);
  if (NJ == 1) return eq6_word_from_cut<NJ>(fx, eq6_cut_one_round<false>(fx[0], target), target, tol, lane);
  // the lane's keys in descending order: its largest remaining one is q[0]
  uint32_t q[NJ];
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) q[jj] = key[jj];
  sort_desc<NJ>(q);
  const uint32_t kmax_all = __reduce_max_sync(0xffffffffu, q[0]);
  uint32_t top = kmax_all;
  int64_t cum = 0;
  int cnt = 0;
#pragma unroll 1
  for (int it = 0; it < kExtractLimit && top != 0u; ++it) {
    const bool hit = q[0] == top;
    const uint32_t c = __reduce_add_sync(0xffffffffu, hit ? 1u : 0u);
    const int64_t f = mass_fx_bits(top);
    if (cum + (int64_t)c * f >= target) {
      // v* = f; above 2^23 (masses >= 2^-29) the fixed point is exact, so
      // the values greater than v* are exactly the ones taken so far
      if (f >= (int64_t(1) << 23)) return eq6_word_from_cut<NJ>(fx, f, target, tol, lane, true, cum, cnt);
      return eq6_word_from_cut<NJ>(fx, f, target, tol, lane);
    }
    cum += (int64_t)c * f;
    cnt += (int)c;
    if (hit) {
#pragma unroll
      for (int jj = 0; jj + 1 < NJ; ++jj) q[jj] = q[jj + 1];
      q[NJ - 1] = 0u;
    }
    top = __reduce_max_sync(0xffffffffu, q[0]);
  }
  // bitwise search over the keys
  uint32_t kk = 0u;
  for (int bit = 31 - __clz(kmax_all); bit >= 0; --bit) {
    const uint32_t cand = kk | (1u << bit);
    int64_t sacc = 0;
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) sacc += (key[jj] >= cand) ? fx[jj] : 0;
    if (warp_sum_u63(sacc) >= target) kk = cand;
  }
  return eq6_word_from_cut<NJ>(fx, mass_fx_bits(kk), target, tol, lane);
}

// The same step with a small footprint, for the discovery epilogue that
// selects while it writes the masses (its warps share the SM with
// instruction-heavy warps and run with few registers): the loops stay
// rolled and v* comes from a bitwise search over the fixed-point values.
template <int NJ>
__device__ __forceinline__ uint32_t eq6_step_word_compact(const int64_t (&fx)[NJ], int64_t target, int64_t tol,
                                                          int lane) {
  int64_t total_pos = 0, max_pos = 0;
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) {
    total_pos += (fx[jj] > 0) ? fx[jj] : 0;
    max_pos = max(max_pos, fx[jj]);
  }
  if (warp_sum_u63(total_pos) < target) return eq6_all_admissible<NJ>(fx, lane);
  int64_t v = 0;
  if (NJ == 1) {
    v = eq6_cut_one_round<true>(fx[0], target);
  } else {
    max_pos = warp_max64(max_pos);
    for (int bit = 63 - __clzll(max_pos); bit >= 0; --bit) {
      const int64_t cand = v | (int64_t(1) << bit);
      int64_t sacc = 0;
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) sacc += (fx[jj] >= cand) ? fx[jj] : 0;
      if (warp_sum_u63(sacc) >= target) v = cand;
    }
  }
  return eq6_word_from_cut<NJ>(fx, v, target, tol, lane);
}

}  // namespace wise
