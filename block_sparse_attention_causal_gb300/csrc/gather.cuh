// Gathered entries of late (reuse) steps with blocks of 32: the working set of
// WISE ("Attention Routing Stabilizes Early: Working-Set Inference for
// Recurrent Language Models", §5.2 Eqs 7-8, CSR of Appendix B "Sparse-kernel
// implementation") on 128-row tiles. A tile holds four 32-row query blocks;
// an entry takes the next four key blocks of the union of their four lists,
// in ascending order, with the 4 x 4 mask of which query block lists which
// slot. Formed once per support by the plan kernel, or by the late-step
// scheduler on every claim when there is no plan. Both run these functions
// with a whole warp.
#pragma once
#include <stdint.h>

namespace wise {

// Lane l's word of the key blocks listed by one CSR row (query block qb):
// bit i is key block 32 l + i. [a, b) is the row's range in col_idx, v the
// list's first 32 values (one per lane, INT32_MAX past b). Values outside
// [0, qb] are skipped; they and values that do not ascend set `bad`.
__device__ __forceinline__ uint32_t gather_list_bits(const int32_t* col_idx, int32_t a, int32_t b, int qb, int32_t v,
                                                     int lane, bool& bad) {
  uint32_t word = 0u;
  int32_t prev = -1;
  for (int32_t base = a; base < b; base += 32) {
    if (base != a) v = (base + lane < b) ? __ldg(col_idx + base + lane) : INT32_MAX;
    const bool in = base + lane < b;
    int32_t pv = __shfl_up_sync(0xffffffffu, v, 1);
    if (lane == 0) pv = prev;
    const bool ok = in && v >= 0 && v > pv && v <= qb;
    if (in && !ok) bad = true;
    // OR each value's bit into the word of the lane that owns it, one
    // target word per round
    uint32_t pend = __ballot_sync(0xffffffffu, ok);
    while (pend != 0u) {
      const int tgt = __shfl_sync(0xffffffffu, v >> 5, __ffs(pend) - 1);
      const bool mine = ok && (v >> 5) == tgt;
      const uint32_t grp = __ballot_sync(0xffffffffu, mine);
      const uint32_t bits = __reduce_or_sync(0xffffffffu, mine ? (1u << (v & 31)) : 0u);
      if (lane == tgt) word |= bits;
      pend &= ~grp;
    }
    prev = __shfl_sync(0xffffffffu, v, 31);
  }
  return word;
}

// Takes the next (up to) four blocks of `rem` (this lane's word of the union
// not yet taken) into kb[0..3]; returns the slot mask (bit 4j + c: query
// block j of the tile lists slot c's block). w0..w3 are this lane's words of
// the four query blocks' lists. Slots past the end of the union repeat the
// last block and are masked for every row. Call only while some lane's rem
// is non-zero.
__device__ __forceinline__ uint32_t gather_take_entry(uint32_t& rem, uint32_t w0, uint32_t w1, uint32_t w2,
                                                      uint32_t w3, int lane, int (&kb)[4]) {
  uint32_t mask = 0u;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t who = __ballot_sync(0xffffffffu, rem != 0u);
    if (who == 0u) {
      kb[c] = kb[c > 0 ? c - 1 : 0];
    } else {
      const int src = __ffs(who) - 1;
      const int bit = (rem != 0u) ? __ffs(rem) - 1 : 0;
      const uint32_t qm = ((w0 >> bit) & 1u) | (((w1 >> bit) & 1u) << 1) | (((w2 >> bit) & 1u) << 2) |
                          (((w3 >> bit) & 1u) << 3);
      if (lane == src) rem &= rem - 1u;
      const int bsrc = __shfl_sync(0xffffffffu, bit, src);
      const uint32_t qsrc = __shfl_sync(0xffffffffu, qm, src);
      kb[c] = 32 * src + bsrc;
      mask |= ((qsrc & 1u) << c) | (((qsrc >> 1) & 1u) << (4 + c)) | (((qsrc >> 2) & 1u) << (8 + c)) |
              (((qsrc >> 3) & 1u) << (12 + c));
    }
  }
  return mask;
}

}  // namespace wise
