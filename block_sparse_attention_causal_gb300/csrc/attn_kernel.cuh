// Causal flash attention on sm_103a tensor cores (tcgen05 + TMEM + TMA), used
// for both WISE steps that touch Q/K/V:
//
//  * discover (SPARSE = false): unrestricted causal attention, §3 Eq 2 of
//    "Attention Routing Stabilizes Early: Working-Set Inference for Recurrent
//    Language Models" (WISE), optionally with the §5.1 Eq 5 block masses;
//  * reuse    (SPARSE = true): attention restricted to the CSR block support,
//    §5.2 Eqs 7-8 -- only listed key blocks are loaded and multiplied.
//
// Persistent: one CTA per SM pulls work units (two 128-row query tiles,
// "streams", of one (batch, head)) from the work order, heaviest first. While one unit's epilogue
// runs, the next unit's Q/K/V loads and first MMAs proceed. Warp roles (384
// threads, three warpgroups):
//   warp 0      TMA producer: Q tiles once, then K/V blocks into an NST ring
//   warp 1      TMEM allocator + MMA issuer of stream 0 (single thread)
//   warp 2      MMA issuer of stream 1 (single thread)
//   warp 3      idle (the control warpgroup gives its registers away)
//   warps 4-7   softmax warpgroup of stream 0 (one query row per thread)
//   warps 8-11  softmax warpgroup of stream 1
// Registers are moved from the control warpgroup (96 each) to the softmax
// warpgroups (200 each): 128*96 + 256*200 <= 384*168, the launch allocation.
// Both MMA threads walk the ascending union of the two streams' key-block
// lists; a K/V block read by both streams is loaded once. Per stream, S = Q K^T goes
// to its own TMEM columns; the softmax warps turn S into P (bf16, written
// back over S) and the MMA thread accumulates O += P V from TMEM. While one
// stream's warps run the softmax, the tensor core works on the other stream.
// The running row max is only moved (and O rescaled) when it grows by more
// than 2^8, so most tiles skip the O correction.
#pragma once
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace wise {

// Work counters of the persistent kernels: each launch takes one slot of this
// ring (chosen by the host launcher), its CTAs pull work units from `next`
// with atomics, and the last CTA to finish resets the slot for a later launch.
struct SchedSlot {
  unsigned int next;
  unsigned int done;
};
constexpr int kSchedSlots = 256;
static __device__ SchedSlot g_sched[kSchedSlots];

template <int D, int BN, bool SPARSE>
struct AttnCfg {
  static_assert(D == 64 || D == 96 || D == 128, "head_dim");
  static_assert(BN == 64 || BN == 128, "block");
  static constexpr int CH = (D == 96) ? 32 : 64;         // elements per swizzled smem row
  static constexpr int NCH = D / CH;                     // TMA boxes per tile
  static constexpr uint32_t SWZ = (CH == 64) ? 2u : 4u;  // descriptor code: 128B / 64B swizzle
  static constexpr uint32_t ROWB = CH * 2;               // bytes per swizzled row
  static constexpr uint32_t Q_BYTES = 128u * D * 2u;
  static constexpr uint32_t KV_BYTES = (uint32_t)BN * D * 2u;
  static constexpr uint32_t SMEM_BUDGET = 230400u;
  static constexpr int MAX_NB = 1024;
  // per-warp partial block masses of the Eq 5 epilogue, [2 streams][4 warps][nb]
  static constexpr uint32_t PART_BYTES = SPARSE ? 0u : 2u * 4u * MAX_NB * 4u;
  static constexpr int NST_FIT = (int)((SMEM_BUDGET - 2u * Q_BYTES - PART_BYTES) / (2u * KV_BYTES));
  static constexpr int NST = NST_FIT > 4 ? 4 : NST_FIT;  // K/V ring depth
  static_assert(NST >= 2, "ring");
  static constexpr int THREADS = 384;
  static constexpr uint32_t REGS_CONTROL = 104, REGS_SOFTMAX = 200, REGS_LAUNCH = 168;
  // setmaxnreg.inc waits for registers released by setmaxnreg.dec: the split
  // must fit in what the CTA was launched with (checked against ptxas -v).
  static_assert(128 * REGS_CONTROL + 256 * REGS_SOFTMAX <= THREADS * REGS_LAUNCH, "register split");
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = 2u * Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + NST * KV_BYTES;
  static constexpr uint32_t OFF_PART = OFF_V + NST * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_PART + PART_BYTES;
  static constexpr int RING = 4;  // work units published to the consumer roles
  // q_full[2] kv_full[NST] kv_empty[NST] s_full[2] p_full[2] o_final[2] drain
  // ring_full[RING] ring_empty[RING]
  static constexpr int NBAR = 2 + 2 * NST + 2 + 2 + 2 + 1 + 2 * RING;
  // tmem base (+0), abort flag (+4), softmax lock (+8), ring of unit ids (+16)
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16u + 4u * RING + 1024u;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM columns: S/P of stream i at s_col(i), O of stream i at o_col(i)
  __host__ __device__ static constexpr uint32_t s_col(int i) { return i ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t o_col(int i) { return i ? 384u : 256u; }
  static constexpr int ENT_PER_TILE = 128 / BN;  // key blocks per 128 rows
};

// Entries (key blocks) of one 128-row query tile in ascending order. Dense:
// the causal range. Sparse: the union of the CSR lists of the query blocks
// inside the tile (one for BN = 128, two for BN = 64); bit j of `mask` says
// whether query block j of the tile lists the entry. List values that are not
// strictly ascending or not admissible (b > q) are skipped and reported.
struct TileCursor {
  const int32_t* col;
  int32_t pos[2], end[2], last[2], maxv[2];
  int32_t head[2];
  int32_t next_dense, dense_end;
  bool sparse, bad;

  __device__ __forceinline__ int32_t adv(int j) {
    while (pos[j] < end[j]) {
      const int32_t v = __ldg(col + pos[j]);
      ++pos[j];
      if (v > last[j] && v <= maxv[j]) {
        last[j] = v;
        return v;
      }
      bad = true;
    }
    return INT32_MAX;
  }

  __device__ __forceinline__ void init_empty() {
    sparse = false;
    next_dense = 0;
    dense_end = 0;
    bad = false;
  }
  __device__ __forceinline__ void init_dense(int t, const AttnParams& p, int bn) {
    sparse = false;
    bad = false;
    next_dense = 0;
    const int rows_end = min(128 * (t + 1), p.n);
    dense_end = (rows_end - 1) / bn + 1;
  }
  __device__ __forceinline__ void init_sparse(int t, int bh, const AttnParams& p, int ent_per_tile) {
    sparse = true;
    bad = false;
    col = p.col_idx;
    for (int j = 0; j < 2; ++j) {
      pos[j] = end[j] = 0;
      last[j] = -1;
      maxv[j] = -1;
      const int qb = t * ent_per_tile + j;
      if (j < ent_per_tile && qb < p.nb) {
        const int64_t r = (int64_t)bh * p.nb + qb;
        const int32_t a = __ldg(p.row_ptr + r), b = __ldg(p.row_ptr + r + 1);
        if (a >= 0 && a <= b && (int64_t)b <= p.col_cap) {
          pos[j] = a;
          end[j] = b;
          maxv[j] = qb;
        } else {
          bad = true;
        }
      }
    }
    head[0] = adv(0);
    head[1] = adv(1);
  }
  __device__ __forceinline__ bool next(int32_t& blk, uint32_t& mask) {
    if (!sparse) {
      if (next_dense >= dense_end) return false;
      blk = next_dense++;
      mask = 3u;
      return true;
    }
    if (head[0] == INT32_MAX && head[1] == INT32_MAX) return false;
    blk = min(head[0], head[1]);
    mask = (head[0] == blk ? 1u : 0u) | (head[1] == blk ? 2u : 0u);
    if (head[0] == blk) head[0] = adv(0);
    if (head[1] == blk) head[1] = adv(1);
    return true;
  }
};

// Ascending union of the two streams' entries; `who` bit i = stream i uses it.
struct PairCursor {
  TileCursor c[2];
  int32_t head[2];
  __device__ __forceinline__ void start() {
    uint32_t m;
    for (int i = 0; i < 2; ++i)
      if (!c[i].next(head[i], m)) head[i] = INT32_MAX;
  }
  __device__ __forceinline__ bool next(int32_t& blk, uint32_t& who) {
    if (head[0] == INT32_MAX && head[1] == INT32_MAX) return false;
    blk = min(head[0], head[1]);
    who = (head[0] == blk ? 1u : 0u) | (head[1] == blk ? 2u : 0u);
    uint32_t m;
    for (int i = 0; i < 2; ++i)
      if (head[i] == blk && !c[i].next(head[i], m)) head[i] = INT32_MAX;
    return true;
  }
};

// Default order of work units: (batch, head) slices in groups sized so the
// group's K/V stays in L2, heavier (later) query tiles first inside a group.
__device__ __forceinline__ int64_t default_unit(int64_t x, const AttnParams& p) {
  const int64_t g_heads = p.group_heads;
  const int64_t per_group = g_heads * p.npairs;
  const int64_t g = x / per_group, w = x % per_group;
  const int64_t gsize = min(g_heads, (int64_t)p.bh_count - g * g_heads);
  const int64_t pr = p.npairs - 1 - w / gsize;
  const int64_t bh = g * g_heads + w % gsize;
  return bh * p.npairs + pr;
}

__device__ __forceinline__ int64_t lam_tile_offset(int bh, int t, const AttnParams& p, int ept) {
  const int64_t before = (int64_t)ept * t * (t + 1) / 2;
  const int64_t total = (int64_t)ept * p.n_qtiles * (p.n_qtiles + 1) / 2;
  return ((int64_t)bh * total + before) * 128;
}

__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint32_t* err) {
  int dummy_abort = 0;
  return mbar_wait(bar, parity, &dummy_abort, err);
}

template <int D, int BN, bool SPARSE>
__global__ void __launch_bounds__(384, 1)
    wise_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = AttnCfg<D, BN, SPARSE>;
  constexpr int NST = C::NST;
  constexpr uint32_t ROWB = C::ROWB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ[2] = {smem + C::OFF_Q, smem + C::OFF_Q + C::Q_BYTES};
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 2;
  uint64_t* kv_empty = kv_full + NST;
  uint64_t* s_full = kv_empty + NST;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_final = p_full + 2;
  uint64_t* drain = o_final + 2;
  uint64_t* ring_full = drain + 1;
  uint64_t* ring_empty = ring_full + C::RING;
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  int* sm_lock = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&q_full[0], 1);
    mbar_init(&q_full[1], 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 2);  // one release per MMA thread
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);  // one elected arrival per softmax warp
      mbar_init(&o_final[i], 1);
    }
    mbar_init(drain, 2);
    *sm_lock = 0;
    for (int j = 0; j < C::RING; ++j) {
      mbar_init(&ring_full[j], 1);
      mbar_init(&ring_empty[j], 2 + 8);  // both MMA threads + one arrival per softmax warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_base_slot;

  // Work distribution: the producer thread pulls positions x of the work
  // order from the launch's counter (greedy, heaviest units first) and
  // publishes the unit ids through a shared-memory ring; every other role
  // reads the same sequence from the ring. -1 ends the sequence, -2 marks a
  // malformed schedule entry (skipped).
  struct Unit {
    int bh, tile[2];
    bool has1;
  };
  auto decode = [&](int id, Unit& u) {
    u.bh = id / p.npairs;
    const int pair = id % p.npairs;
    u.tile[0] = 2 * pair;
    u.tile[1] = 2 * pair + 1;
    u.has1 = u.tile[1] < p.n_qtiles;
  };
  // consumer side: next unit id from the ring (-1 at the end or on abort)
  auto ring_take = [&](int& ci, bool warp_vote) -> int {
    const int slot = ci % C::RING;
    bool okw = mbar_wait(&ring_full[slot], (ci / C::RING) & 1, abort_flag, p.err);
    if (warp_vote) okw = __all_sync(0xffffffffu, okw);
    if (!okw) return -1;
    const int id = ring[slot];
    if (warp_vote) {
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&ring_empty[slot]);
    } else {
      mbar_arrive(&ring_empty[slot]);
    }
    ++ci;
    return id;
  };
  auto make_cursor = [&](TileCursor& c, const Unit& u, int i) {
    if (i == 1 && !u.has1) {
      c.init_empty();
    } else if (SPARSE) {
      c.init_sparse(u.tile[i], u.bh, p, C::ENT_PER_TILE);
    } else {
      c.init_dense(u.tile[i], p, BN);
    }
  };

  if (warp < 4) {
   setmaxnreg_dec<C::REGS_CONTROL>();
   if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t nq[2] = {0u, 0u};  // Q loads per stream (one per unit using it)
      int k = 0;                  // K/V loads issued (ring position)
      bool ok = true;
      SchedSlot* sched = &g_sched[p.sched_slot];
      for (int pi = 0; ok; ++pi) {
        const int slot = pi % C::RING;
        if (pi >= C::RING && !(ok = mbar_wait(&ring_empty[slot], ((pi / C::RING) - 1) & 1, abort_flag, p.err)))
          break;
        const unsigned int x = atomicAdd(&sched->next, 1u);
        int id = -1;
        if ((int64_t)x < p.n_units) {
          const int64_t v = (SPARSE && p.tile_order != nullptr) ? (int64_t)__ldg(p.tile_order + x) : default_unit(x, p);
          id = (v >= 0 && v < p.n_units) ? (int)v : -2;
          if (id == -2) atomicOr(p.err, kErrBadSupport);
        }
        ring[slot] = id;
        mbar_arrive(&ring_full[slot]);
        if (id == -1) break;
        if (id < 0) continue;
        Unit u;
        decode(id, u);
        for (int i = 0; i < (u.has1 ? 2 : 1) && ok; ++i) {
          // the previous unit that used Q_i has finished all its MMAs
          if (nq[i] > 0 && !(ok = mbar_wait(&o_final[i], (nq[i] - 1) & 1, abort_flag, p.err))) break;
          const int row = u.bh * p.n + u.tile[i] * 128;
          mbar_arrive_expect_tx(&q_full[i], C::Q_BYTES);
          for (int c = 0; c < C::NCH; ++c) tma_load_2d(sQ[i] + c * 128 * ROWB, &tm_q, &q_full[i], c * C::CH, row);
          ++nq[i];
        }
        PairCursor pc;
        make_cursor(pc.c[0], u, 0);
        make_cursor(pc.c[1], u, 1);
        pc.start();
        int32_t blk;
        uint32_t who;
        while (ok && pc.next(blk, who)) {
          const int s = k % NST;
          if (k >= NST && !(ok = mbar_wait(&kv_empty[s], ((k / NST) - 1) & 1, abort_flag, p.err))) break;
          const int row = u.bh * p.n + blk * BN;
          uint8_t* sk = smem + C::OFF_K + s * C::KV_BYTES;
          uint8_t* sv = smem + C::OFF_V + s * C::KV_BYTES;
          mbar_arrive_expect_tx(&kv_full[s], 2 * C::KV_BYTES);
          for (int c = 0; c < C::NCH; ++c) tma_load_2d(sk + c * BN * ROWB, &tm_k, &kv_full[s], c * C::CH, row);
          for (int c = 0; c < C::NCH; ++c) tma_load_2d(sv + c * BN * ROWB, &tm_v, &kv_full[s], c * C::CH, row);
          ++k;
        }
        if (pc.c[0].bad || pc.c[1].bad) atomicOr(p.err, kErrBadSupport);
      }
      // No copy into this CTA's shared memory may outlive the CTA.
      for (int j = (k > NST ? k - NST : 0); j < k; ++j) {
        const int s = j % NST;
        const uint32_t ph = (j / NST) & 1;
        mbar_wait_drain(&kv_full[s], ph, p.err);
      }
      for (int i = 0; i < 2; ++i)
        if (nq[i] > 0) mbar_wait_drain(&q_full[i], (nq[i] - 1) & 1, p.err);
    }
    __syncwarp();
   } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per stream (warp 1: stream 0, warp 2: stream 1), so
    // that one stream's waits overlap the other's MMA issue. Both walk the
    // union of the unit's key blocks: a block the stream does not use is
    // released at once, a used one after the stream's PV MMA on it.
    if (lane == 0) {
      const int i = warp - 1;
      constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BN, 0, 0);
      constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, 0, 1);
      bool ok = true;
      uint32_t nq = 0u;    // units using this stream (q_full / o_final phases)
      uint32_t n_pt = 0u;  // P tiles consumed (p_full phases)
      uint32_t n_pv = 0u;  // PV MMAs in the current unit (accumulate flag)
      bool pending = false;
      int pend_slot = 0;

      auto flush_pv = [&]() -> bool {
        if (!mbar_wait(&p_full[i], n_pt & 1, abort_flag, p.err)) return false;
        ++n_pt;
        tc_fence_after();
        const uint32_t vbase = smem_u32(smem + C::OFF_V + pend_slot * C::KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bdesc = smem_desc(vbase + kk * 16 * ROWB, BN * ROWB, 8 * ROWB, C::SWZ);
          umma_ts(tbase + C::o_col(i), tbase + C::s_col(i) + kk * 8, bdesc, IDESC_O, (n_pv | kk) != 0);
        }
        ++n_pv;
        umma_commit(&kv_empty[pend_slot]);
        pending = false;
        return true;
      };

      int k = 0;
      int ci = 0;
      while (ok) {
        const int id = ring_take(ci, false);
        if (id == -1) break;
        if (id < 0) continue;
        Unit u;
        decode(id, u);
        const bool active = (i == 0) || u.has1;
        PairCursor pc;
        make_cursor(pc.c[0], u, 0);
        make_cursor(pc.c[1], u, 1);
        pc.start();
        bool q_ready = false;
        n_pv = 0;
        int32_t blk;
        uint32_t who;
        while (ok && pc.next(blk, who)) {
          const int s = k % NST;
          const uint32_t ph = (k / NST) & 1;
          if (pending && !(ok = flush_pv())) break;
          // waiting for the block also keeps this thread from releasing a
          // slot's next use before the other thread released this one
          if (!(ok = mbar_wait(&kv_full[s], ph, abort_flag, p.err))) break;
          if (who & (1u << i)) {
            if (!q_ready) {
              if (!(ok = mbar_wait(&q_full[i], nq & 1, abort_flag, p.err))) break;
              q_ready = true;
            }
            tc_fence_after();
            const uint32_t qa = smem_u32(sQ[i]);
            const uint32_t ka = smem_u32(smem + C::OFF_K + s * C::KV_BYTES);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int c = kk / (C::CH / 16), w = kk % (C::CH / 16);
              const uint64_t adesc = smem_desc(qa + c * 128 * ROWB + w * 32, 16, 8 * ROWB, C::SWZ);
              const uint64_t bdesc = smem_desc(ka + c * BN * ROWB + w * 32, 16, 8 * ROWB, C::SWZ);
              umma_ss(tbase + C::s_col(i), adesc, bdesc, IDESC_S, kk > 0);
            }
            umma_commit(&s_full[i]);
            pending = true;
            pend_slot = s;
          } else {
            mbar_arrive(&kv_empty[s]);
          }
          ++k;
        }
        if (ok && pending) ok = flush_pv();
        // Close the unit for this stream: its Q load has landed (so the next
        // load into the buffer cannot overlap it) and o_final fires once every
        // MMA this thread issued has completed.
        if (ok && active) {
          if (!q_ready) ok = mbar_wait(&q_full[i], nq & 1, abort_flag, p.err);
          umma_commit(&o_final[i]);
          ++nq;
        }
      }
      umma_commit(drain);  // every MMA of this thread done before TMEM is released
      mbar_wait_drain(drain, 0, p.err);
    }
    __syncwarp();
   }
  } else {
    setmaxnreg_inc<C::REGS_SOFTMAX>();
    // ------------------------------------------------------------ softmax
    const int i = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row within the query tile = TMEM lane
    const uint32_t trow = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t tS = trow + C::s_col(i);
    const uint32_t tO = trow + C::o_col(i);
    const float sl2 = p.scale_log2;
    const bool want_mass = (!SPARSE) && (p.mass != nullptr);
    const int half = (BN == 64) ? (r >> 6) : 0;
    float* part = reinterpret_cast<float*>(smem + C::OFF_PART) + i * 4 * C::MAX_NB;
    uint32_t n_s = 0;   // S tiles consumed (s_full phases)
    uint32_t nq = 0;    // units processed (o_final phases)
    bool ok = true;
    int ci = 0;
    while (ok) {
      const int id = ring_take(ci, true);
      if (id == -1) break;
      if (id < 0) continue;
      Unit u;
      decode(id, u);
      if (i == 1 && !u.has1) continue;
      const int bh = u.bh;
      const int t = u.tile[i];
      const int qpos = t * 128 + r;
      const bool row_valid = qpos < p.n;
      float* lam = want_mass ? p.lam + lam_tile_offset(bh, t, p, C::ENT_PER_TILE) + r : nullptr;

      TileCursor cur;
      make_cursor(cur, u, i);
      // l: fp32 row sum (for LSE and the block masses); lt: sum of the
      // bf16-rounded P that the tensor core multiplies (normalises O, so the
      // output is an exact weighted mean of the rounded weights)
      float m_ref = -INFINITY, l = 0.f, lt = 0.f;
      uint32_t cnt = 0;
      int32_t blk;
      uint32_t mask;
      while (cur.next(blk, mask)) {
        ok = mbar_wait(&s_full[i], n_s & 1, abort_flag, p.err);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++n_s;
        tc_fence_after();
        // Dense steps: only one softmax warpgroup computes at a time, so the
        // other stream's MMAs run while this one works (ping-pong) and the two
        // never split the SM's issue slots. (Sparse steps, whose two streams
        // often have different blocks, run faster without the lock.)
        if (!SPARSE) {
          if (r == 0) {
            for (;;) {
              if (*reinterpret_cast<volatile int*>(sm_lock) == 0 && atomicCAS(sm_lock, 0, 1) == 0) break;
              __nanosleep(20);
            }
          }
          named_bar_sync(3 + i, 128);
        }
        const int kbase = blk * BN;
        const bool row_on = (mask >> half) & 1u;
        // columns c <= limit are admissible (causal mask M, working-set mask R)
        const int limit = row_on ? ((kbase + BN - 1 > qpos) ? qpos - kbase : BN) : -1;
        const bool full = limit >= BN - 1;
        // The whole S row (BN columns) is read from TMEM once; the row max and
        // then P are computed from registers.
        uint32_t s[BN / 32][32];
#pragma unroll
        for (int cc = 0; cc < BN / 32; ++cc) tmem_ld_x32(tS + cc * 32, s[cc]);
#pragma unroll
        for (int cc = 0; cc < BN / 32; ++cc) tmem_wait_ld(s[cc]);
        if (!full) {
#pragma unroll
          for (int cc = 0; cc < BN / 32; ++cc)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              s[cc][j] = (cc * 32 + j <= limit) ? s[cc][j] : __float_as_uint(-INFINITY);
        }
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int cc = 0; cc < BN / 32; ++cc)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            mx4[j & 3] = fmax3(mx4[j & 3], __uint_as_float(s[cc][2 * j]), __uint_as_float(s[cc][2 * j + 1]));
        float mx = fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]) * sl2;
        float factor = 1.f;
        bool resc = false;
        if (cnt == 0) {
          m_ref = mx;
        } else if (mx > m_ref + 8.f) {
          factor = fast_exp2(m_ref - mx);
          m_ref = mx;
          resc = true;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        // P = 2^(s*scale*log2e - m) as bf16 pairs, written over S. Packed f32x2
        // FMA for the exponent argument, a packed add for the fp32 row sum and
        // mixed bf16+f32 adds for the sum of the rounded P (two independent
        // accumulators each). Masked entries hold -inf and give exactly 0.
        const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_use, -m_use);
        uint64_t rs2[2] = {0ull, 0ull}, rt2[2] = {0ull, 0ull};
#pragma unroll
        for (int cc = 0; cc < BN / 32; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float e0, e1;
            f2_unpack(ffma2(f2_pack(__uint_as_float(s[cc][2 * j]), __uint_as_float(s[cc][2 * j + 1])), sc2, nm2),
                      e0, e1);
            const float p0 = fast_exp2(e0);
            const float p1 = fast_exp2(e1);
            pk[j] = pack_bf16x2(p0, p1);
            rs2[j & 1] = fadd2(rs2[j & 1], f2_pack(p0, p1));
            add_bf16x2_to(rt2[j & 1], pk[j]);
          }
          tmem_st_x16(tS + cc * 16, pk);
        }
        float rs, rt;
        {
          float a0, a1, b0, b1;
          f2_unpack(fadd2(rs2[0], rs2[1]), a0, a1);
          f2_unpack(fadd2(rt2[0], rt2[1]), b0, b1);
          rs = a0 + a1;
          rt = b0 + b1;
        }
        l = l * factor + rs;
        lt = lt * factor + rt;
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld_x32(tO + cc * 32, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * factor);
            tmem_st_x32(tO + cc * 32, o);
          }
        }
        tmem_wait_st();
        if (!SPARSE) {
          named_bar_sync(3 + i, 128);
          if (r == 0) atomicExch(sm_lock, 0);
        }
        if (want_mass) lam[(size_t)cnt * 128] = (rs > 0.f) ? m_use + fast_log2(rs) : -INFINITY;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[i]);
        ++cnt;
      }

      // ------------------------------------------------------------ epilogue
      if (ok) {  // the unit's MMAs are complete (waited even without entries: keeps phases in step)
        ok = mbar_wait(&o_final[i], nq & 1, abort_flag, p.err);
        ok = __all_sync(0xffffffffu, ok);
        ++nq;
        tc_fence_after();
      }
      if (ok) {
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        const float inv_l = (lt > 0.f) ? 1.f / lt : 0.f;
        const size_t grow = (size_t)bh * p.n + qpos;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          if (cnt > 0) {
            tmem_ld_x32(tO + cc * 32, o);
            tmem_wait_ld(o);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = 0u;
          }
          if (row_valid) {
            if (p.out_f32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + grow * D + cc * 32);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                dst[j] = make_float4(__uint_as_float(o[4 * j]) * inv_l, __uint_as_float(o[4 * j + 1]) * inv_l,
                                     __uint_as_float(o[4 * j + 2]) * inv_l, __uint_as_float(o[4 * j + 3]) * inv_l);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + grow * D + cc * 32);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(o[8 * j + 0]) * inv_l, __uint_as_float(o[8 * j + 1]) * inv_l);
                v.y = pack_bf16x2(__uint_as_float(o[8 * j + 2]) * inv_l, __uint_as_float(o[8 * j + 3]) * inv_l);
                v.z = pack_bf16x2(__uint_as_float(o[8 * j + 4]) * inv_l, __uint_as_float(o[8 * j + 5]) * inv_l);
                v.w = pack_bf16x2(__uint_as_float(o[8 * j + 6]) * inv_l, __uint_as_float(o[8 * j + 7]) * inv_l);
                dst[j] = v;
              }
            }
          }
        }
        const float lse2 = (l > 0.f) ? m_use + fast_log2(l) : -INFINITY;
        if (p.lse != nullptr && row_valid) p.lse[grow] = lse2 * 0.69314718055994531f;
        if (want_mass) {
          // Eq 5: r_qb = (1/B) sum over the block's rows of 2^(lam_ib - lse2_i).
#pragma unroll 1
          for (uint32_t e = 0; e < cnt; ++e) {
            float a = (row_valid && l > 0.f) ? fast_exp2(lam[(size_t)e * 128] - lse2) : 0.f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            if (lane == 0) part[quarter * p.nb + e] = a;
          }
          named_bar_sync(1 + i, 128);
          constexpr int QB_PER_TILE = C::ENT_PER_TILE;
          for (int qq = 0; qq < QB_PER_TILE; ++qq) {
            const int qb = t * QB_PER_TILE + qq;
            if (qb >= p.nb) break;
            float* dst = p.mass + ((size_t)bh * p.nb + qb) * p.nb;
            for (int e = r; e < p.nb; e += 128) {
              float v = 0.f;
              if (e < (int)cnt) {
                if (BN == 128) {
                  v = (part[0 * p.nb + e] + part[1 * p.nb + e]) + (part[2 * p.nb + e] + part[3 * p.nb + e]);
                } else {
                  v = part[(2 * qq) * p.nb + e] + part[(2 * qq + 1) * p.nb + e];
                }
                v *= (1.f / BN);
              }
              dst[e] = v;
            }
          }
          named_bar_sync(1 + i, 128);  // partials are reused by the next unit
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    // every CTA has pulled its last position: the last one out resets the slot
    __threadfence();
    if (atomicAdd(&g_sched[p.sched_slot].done, 1u) == gridDim.x - 1) {
      g_sched[p.sched_slot].next = 0u;
      g_sched[p.sched_slot].done = 0u;
      __threadfence();
    }
  }
}

}  // namespace wise
