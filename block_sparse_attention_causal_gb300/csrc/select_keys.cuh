// The selection kernel's usual case of one step of the working-set
// selection of WISE ("Attention Routing Stabilizes Early: Working-Set
// Inference for Recurrent Language Models", §5.1 Eq 6): the cut decided on
// the masses' ordering keys alone, for rows whose k-th mass lies where the
// fixed point of select_step.cuh is exact. Gives the same bits as
// eq6_step_word; rows it cannot decide go there.
#pragma once
#include <stdint.h>

#include "select_step.cuh"

namespace wise {

// The float bits of x * 2^-52 rounded down (ROUND_UP false) or up, for x in
// [2^23, 2^62): with e the position of x's leading one, the float's
// significand is x >> (e - 23) and its biased exponent e + 75. Keys in
// [2^-29, 2^10) map back to their fixed point exactly (mass_fx_exact_bits),
// so key >= fx_to_key<true>(x) <=> fixed point >= x and
// key <= fx_to_key<false>(x) <=> fixed point <= x.
template <bool ROUND_UP>
__device__ __forceinline__ uint32_t fx_to_key(int64_t x) {
  const uint64_t u = static_cast<uint64_t>(x);
  const int e = 63 - __clzll(x);
  const int sh = e - 23;
  uint32_t k = ((uint32_t)(e + 75) << 23) + ((uint32_t)(u >> sh) & 0x7fffffu);
  if (ROUND_UP && (u & ((uint64_t(1) << sh) - 1u))) ++k;
  return k;
}

// A positive int64 as a float, near enough for an estimate (no 64-bit
// conversion instruction, which runs on the FP64 pipe).
__device__ __forceinline__ float approx_float(int64_t x) {
  const uint64_t u = static_cast<uint64_t>(x);
  return __uint2float_rz((uint32_t)(u >> 32)) * 4294967296.f + __uint2float_rz((uint32_t)u);
}

// eq6_word_from_cut in the key domain: v* = v (its key range [k_lo, k_hi]
// is the near-tie group v* +- tol), with c_gt blocks above v* whose masses
// leave `need` of the target to blocks of mass v*.
template <int NJ>
__device__ __forceinline__ uint32_t eq6_word_from_key_cut(const uint32_t (&key)[NJ], uint32_t k_lo, uint32_t k_hi,
                                                          int64_t v, int64_t need, int c_gt, int lane) {
  uint32_t sel_word_mine = 0;
  uint32_t c_both = 0;  // blocks above the group (low half), in it (high half)
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj)
    c_both += (key[jj] > k_hi) ? 1u : ((key[jj] >= k_lo) ? 0x10000u : 0u);
  c_both = __reduce_add_sync(0xffffffffu, c_both);
  const int c_above = (int)(c_both & 0xffffu), c_near = (int)(c_both >> 16);
  // m = ceil(need / v) blocks of mass v, 1 <= m <= the blocks at v
  int m = 1;
  if (need > v) {
    m = (int)fminf(fmaxf(__fdividef(approx_float(need), approx_float(v)), 1.f), 4096.f);
    while (m > 1 && (int64_t)(m - 1) * v >= need) --m;
    while ((int64_t)m * v < need) ++m;
  }
  const int slots = c_gt + m - c_above;  // taken from the group, lowest index first
  if (slots >= c_near) {
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
      const uint32_t bal = __ballot_sync(0xffffffffu, key[jj] >= k_lo);
      if (lane == jj) sel_word_mine = bal;
    }
    return sel_word_mine;
  }
  int taken = 0;
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) {
    const bool above = key[jj] > k_hi;
    const bool near = !above && key[jj] >= k_lo;
    const uint32_t nb_bal = __ballot_sync(0xffffffffu, near);
    const int rank = taken + __popc(nb_bal & ((1u << lane) - 1u));
    taken += __popc(nb_bal);
    const uint32_t bal = __ballot_sync(0xffffffffu, above || (near && rank < slots));
    if (lane == jj) sel_word_mine = bal;
  }
  return sel_word_mine;
}

// The selection kernel's step on the ordering keys alone (no fixed-point
// array), for rows whose cut lies where the fixed point is exact: there it
// is a strictly increasing function of the key, so every comparison with
// v* +- tol is a comparison of keys, and the sums are exact sums of the
// values taken. The distinct largest keys are taken one at a time, as in
// eq6_step_word. Returns false, having decided nothing, when the row needs
// the general path: a mass at or above 2^10, the crossing not reached within
// LIMIT values at or above 2^-29 (rows whose admissible mass cannot reach
// the target among them), or v* +- tol outside [2^-29, 2^10).
template <int NJ, int LIMIT>
__device__ __forceinline__ bool eq6_step_word_keys(const uint32_t (&key)[NJ], int64_t target, int64_t tol, int lane,
                                                   uint32_t& word) {
  uint32_t q[NJ];
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) q[jj] = key[jj];
  sort_desc<NJ>(q);
  uint32_t top = __reduce_max_sync(0xffffffffu, q[0]);
  if (top >= (137u << 23) || tol < 0) return false;
  int64_t cum = 0;
  int cnt = 0;
#pragma unroll 1
  for (int it = 0; it < LIMIT && top >= (98u << 23); ++it) {
    const bool hit = q[0] == top;
    const uint32_t c = __reduce_add_sync(0xffffffffu, hit ? 1u : 0u);
    const int64_t f = mass_fx_exact_bits(top);
    if (cum + (int64_t)c * f >= target) {
      const int64_t lo = f - tol, hi = f + tol;
      if (lo <= (int64_t(1) << 23) || hi >= (int64_t(1) << 62)) return false;
      word = eq6_word_from_key_cut<NJ>(key, fx_to_key<true>(lo), fx_to_key<false>(hi), f, target - cum, cnt, lane);
      return true;
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
  return false;
}

}  // namespace wise
