// Causal flash attention on sm_103a tensor cores (tcgen05 + TMEM + TMA), used
// for both WISE steps that touch Q/K/V:
//
//  * discover (SPARSE = false): unrestricted causal attention, §3 Eq 2 of
//    "Attention Routing Stabilizes Early: Working-Set Inference for Recurrent
//    Language Models" (WISE), optionally with the §5.1 Eq 5 block masses;
//  * reuse    (SPARSE = true): attention restricted to the CSR block support,
//    §5.2 Eqs 7-8 -- only listed key blocks are loaded and multiplied.
//
// Persistent: one CTA per SM pulls work units (one 128-row query tile of one
// (batch, head)) from the work order, heaviest first. The key blocks of all
// units a CTA takes form one continuous stream of "entries"; the pipeline runs
// across unit boundaries. Warp roles (512 threads, four warpgroups):
//   warp 0      scheduler: claims units, walks their key-block lists, and
//               publishes one record per entry in a shared-memory ring
//   warp 1      TMA loads of Q (once per unit), K (ring of NK slots) and V
//               (ring of NV slots)
//   warp 2      issues the S = Q K^T MMAs (one elected lane)
//   warp 3      TMEM allocator; issues the O += P V MMAs (one elected lane)
//   warps 4-7   softmax warpgroup 0: key columns [0, BN/2) of every row
//   warps 8-11  softmax warpgroup 1: key columns [BN/2, BN)
//   warps 12-15 epilogue: O normalisation and store, LSE, block masses
// TMEM holds three S buffers and the O accumulator. S for entry j+1 and j+2
// is computed while the softmax works on entry j; P (bf16) is written over
// S_j and consumed from TMEM by the PV MMA, after which S_{j+3} reuses the
// buffer. The two softmax warpgroups split each score row and exchange row
// maxima through shared memory. The running row max is only moved (and O
// rescaled) when it grows by more than 2^8, so most entries skip the O
// correction.
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

// Flags of an entry record.
enum : uint32_t {
  kEntFirst = 1u,   // first entry of its unit
  kEntLast = 2u,    // last entry of its unit
  kEntEnd = 4u,     // no more entries: the CTA's work is done
  kEntQbuf = 8u,    // Q buffer of the unit
  kEntRows0 = 16u,  // the rows of query block 0 of the tile list this key block
  kEntRows1 = 32u,  // ... of query block 1 (BN = 64 only)
};

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
  static constexpr int THREADS = 512;
  static constexpr int NSB = 3;       // S buffers in TMEM
  static constexpr int META = 32;     // entry records in flight
  static constexpr int URING = 8;     // unit records in flight (epilogue)
  static constexpr int HB = BN / 2;   // key columns per softmax warpgroup
  static constexpr int MAX_NB = 1024;
  static constexpr int ENT_PER_TILE = 128 / BN;  // query blocks per 128-row tile
  // shared memory: Q[2] | K[NK] | V[NV] | xch | stats | part | meta | units | barriers | misc
  static constexpr uint32_t XCH_BYTES = 2u * 2u * 128u * 4u;    // row-max exchange, two tiles
  static constexpr uint32_t STATS_BYTES = 2u * 5u * 128u * 4u;  // per-row m, l, lt of two units
  static constexpr uint32_t PART_BYTES = SPARSE ? 0u : 4u * 64u * 4u;
  static constexpr uint32_t META_BYTES = META * 16u;
  static constexpr uint32_t URING_BYTES = URING * 8u;
  static constexpr int NBAR_FIXED = 2 + 2 + 3 * NSB + 2 + 2 + 2 + 2 * URING + 2;
  static constexpr uint32_t SMEM_LIMIT = 232448u;  // 227 KB per CTA
  static constexpr uint32_t FIXED = 2u * Q_BYTES + XCH_BYTES + STATS_BYTES + PART_BYTES + META_BYTES + URING_BYTES +
                                    (NBAR_FIXED + 16) * 8u + 32u + 1024u;
  static constexpr int SLOTS_FIT = (int)((SMEM_LIMIT - FIXED) / KV_BYTES);
  static constexpr int NK = SLOTS_FIT >= 8 ? 4 : (SLOTS_FIT + 1) / 2;
  static constexpr int NV = SLOTS_FIT >= 8 ? 4 : SLOTS_FIT / 2;
  static_assert(NK >= 2 && NV >= 2, "K/V rings");
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = 2u * Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr uint32_t OFF_XCH = OFF_V + NV * KV_BYTES;
  static constexpr uint32_t OFF_STATS = OFF_XCH + XCH_BYTES;
  static constexpr uint32_t OFF_PART = OFF_STATS + STATS_BYTES;
  static constexpr uint32_t OFF_META = OFF_PART + PART_BYTES;
  static constexpr uint32_t OFF_URING = OFF_META + META_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_URING + URING_BYTES;
  static constexpr int NBAR = NBAR_FIXED + 2 * NK + 2 * NV;
  // tmem base (+0), abort flag (+4), entries whose PV was issued (+8),
  // softmax abort entry (+12), epilogue abort unit (+16)
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 32u + 1024u;  // + alignment slack
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
  static constexpr uint32_t TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t s_col(int b) { return 128u * (uint32_t)b; }
  static constexpr uint32_t O_COL = 384;
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

// Default order of work units: (batch, head) slices in groups sized so the
// group's K/V stays in L2, heavier (later) query tiles first inside a group.
__device__ __forceinline__ int64_t default_unit(int64_t x, const AttnParams& p) {
  const int64_t g_heads = p.group_heads;
  const int64_t per_group = g_heads * p.n_qtiles;
  const int64_t g = x / per_group, w = x % per_group;
  const int64_t gsize = min(g_heads, (int64_t)p.bh_count - g * g_heads);
  const int64_t t = p.n_qtiles - 1 - w / gsize;
  const int64_t bh = g * g_heads + w % gsize;
  return bh * p.n_qtiles + t;
}

// First float of tile t's Eq 5 scratch: per entry, two halves of 128 rows.
__device__ __forceinline__ int64_t lam_tile_offset(int bh, int t, const AttnParams& p, int ept) {
  const int64_t before = (int64_t)ept * t * (t + 1) / 2;
  const int64_t total = (int64_t)ept * p.n_qtiles * (p.n_qtiles + 1) / 2;
  return ((int64_t)bh * total + before) * 256;
}

__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint32_t* err) {
  int dummy_abort = 0;
  return mbar_wait(bar, parity, &dummy_abort, err);
}

// Entry records: word 0 is the tag (entry index + 1), written last.
struct EntryRec {
  uint32_t tag;
  uint32_t krow;   // global row of the key block's first key (TMA coordinate)
  uint32_t unit;   // unit id = bh * n_qtiles + tile
  uint32_t info;   // flags | block index << 8
};

// Wait until record j is published; false on abort/timeout or if the ring
// was overrun (which the scheduler's flow control rules out). The spin is out
// of line; the common case (already published) is one load and a compare.
static __device__ __noinline__ bool wait_entry_slow(EntryRec* r, uint32_t j, volatile int* abort_flag, uint32_t* err) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    const uint32_t tag = ld_acquire_smem(&r->tag);
    if (tag == j + 1u) return true;
    if (tag > j + 1u) {
      *abort_flag = 1;
      atomicOr(err, kErrTimeout);
      return false;
    }
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_entry(EntryRec* ring, int meta, uint32_t j, EntryRec& out,
                                           volatile int* abort_flag, uint32_t* err) {
  EntryRec* r = ring + (j % (uint32_t)meta);
  if (ld_acquire_smem(&r->tag) != j + 1u && !wait_entry_slow(r, j, abort_flag, err)) return false;
  out.tag = j + 1u;
  out.krow = r->krow;
  out.unit = r->unit;
  out.info = r->info;
  return true;
}

// O row segment [tO, tO + ncols) *= factor (the lazy rescale, rare).
static __device__ __noinline__ void rescale_o(uint32_t tO, int ncols, float factor) {
  for (int c = 0; c < ncols; c += 8) {
    uint32_t o[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]), "=r"(o[4]), "=r"(o[5]), "=r"(o[6]), "=r"(o[7])
                 : "r"(tO + c)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(o[0]), "+r"(o[1]), "+r"(o[2]), "+r"(o[3]), "+r"(o[4]), "+r"(o[5]), "+r"(o[6]), "+r"(o[7])
                 :
                 : "memory");
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * factor);
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(tO + c), "r"(o[0]),
                 "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                 : "memory");
  }
}

template <int D, int BN, bool SPARSE>
__global__ void __launch_bounds__(512, 1)
    wise_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = AttnCfg<D, BN, SPARSE>;
  constexpr int NK = C::NK, NV = C::NV, NSB = C::NSB, META = C::META, URING = C::URING;
  constexpr uint32_t ROWB = C::ROWB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;              // [2]
  uint64_t* q_empty = q_full + 2;       // [2]
  uint64_t* s_full = q_empty + 2;       // [NSB]
  uint64_t* p_full = s_full + NSB;      // [NSB]
  uint64_t* pv_done = p_full + NSB;     // [NSB]
  uint64_t* o_final = pv_done + NSB;    // [1]
  uint64_t* o_free = o_final + 1;       // [1]
  uint64_t* st_full = o_free + 1;       // [2]
  uint64_t* st_empty = st_full + 2;     // [2]
  uint64_t* u_full = st_empty + 2;      // [URING]
  uint64_t* u_empty = u_full + URING;   // [URING]
  uint64_t* drain = u_empty + URING;    // [2]
  uint64_t* k_full = drain + 2;         // [NK]
  uint64_t* k_empty = k_full + NK;      // [NK]
  uint64_t* v_full = k_empty + NK;      // [NV]
  uint64_t* v_empty = v_full + NV;      // [NV]
  EntryRec* meta = reinterpret_cast<EntryRec*>(smem + C::OFF_META);
  int32_t* uring = reinterpret_cast<int32_t*>(smem + C::OFF_URING);  // {unit id, entries}
  float* xch = reinterpret_cast<float*>(smem + C::OFF_XCH);
  float* stats = reinterpret_cast<float*>(smem + C::OFF_STATS);
  float* part = reinterpret_cast<float*>(smem + C::OFF_PART);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  uint32_t* tmem_base_slot = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  uint32_t* pv_issued = misc + 2;
  int* sm_abort = reinterpret_cast<int*>(misc + 3);
  int* ep_abort = reinterpret_cast<int*>(misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&st_full[i], 8);   // one arrival per softmax warp
      mbar_init(&st_empty[i], 4);  // one arrival per epilogue warp
    }
    for (int b = 0; b < NSB; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 8);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(o_final, 1);
    mbar_init(o_free, 4);
    for (int j = 0; j < URING; ++j) {
      mbar_init(&u_full[j], 1);
      mbar_init(&u_empty[j], 4);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int j = 0; j < META; ++j) meta[j].tag = 0u;
    *abort_flag = 0;
    *pv_issued = 0u;
    *sm_abort = INT32_MAX;
    *ep_abort = INT32_MAX;
    fence_mbar_init();
  }
  if (warp == 3) {
    tmem_alloc(tmem_base_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_base_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ scheduler
    if (lane == 0) {
      SchedSlot* sched = &g_sched[p.sched_slot];
      uint32_t j = 0;  // entries published
      int u = 0;       // units published
      int uq = 0;      // units with at least one entry
      bool ok = true;
      // publish one entry record, after the flow control allows slot j
      auto publish = [&](uint32_t krow, uint32_t unit, uint32_t info) -> bool {
        if (j >= (uint32_t)META) {
          const uint64_t t0 = global_timer_ns();
          for (uint32_t it = 0; j >= ld_acquire_smem(pv_issued) + (uint32_t)META; ++it) {
            if ((it & 63u) == 63u) {
              if (*abort_flag) return false;
              if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(p.err, kErrTimeout);
                return false;
              }
            }
            __nanosleep(64);
          }
        }
        EntryRec* r = meta + (j % (uint32_t)META);
        r->krow = krow;
        r->unit = unit;
        r->info = info;
        st_release_smem(&r->tag, j + 1u);
        ++j;
        return true;
      };
      while (ok) {
        const unsigned int x = atomicAdd(&sched->next, 1u);
        int id = -1;
        if ((int64_t)x < p.n_units) {
          const int64_t v = (SPARSE && p.tile_order != nullptr) ? (int64_t)__ldg(p.tile_order + x) : default_unit(x, p);
          id = (v >= 0 && v < p.n_units) ? (int)v : -2;
          if (id == -2) {
            atomicOr(p.err, kErrBadSupport);
            continue;
          }
        }
        if (id == -1) break;
        const int bh = id / p.n_qtiles, t = id % p.n_qtiles;
        TileCursor cur;
        if (SPARSE) cur.init_sparse(t, bh, p, C::ENT_PER_TILE);
        else cur.init_dense(t, p, BN);
        const uint32_t qbuf = (uq & 1) ? kEntQbuf : 0u;
        int cnt = 0;
        int32_t blk, pblk = -1;
        uint32_t mask, pmask = 0;
        while (cur.next(blk, mask)) {
          if (cnt > 0) {
            const uint32_t info = (cnt == 1 ? kEntFirst : 0u) | qbuf | (pmask << 4) | ((uint32_t)pblk << 8);
            if (!(ok = publish((uint32_t)(bh * p.n + pblk * BN), (uint32_t)id, info))) break;
          }
          pblk = blk;
          pmask = mask;
          ++cnt;
        }
        if (!ok) break;
        if (cnt > 0) {
          const uint32_t info = (cnt == 1 ? kEntFirst : 0u) | kEntLast | qbuf | (pmask << 4) | ((uint32_t)pblk << 8);
          if (!(ok = publish((uint32_t)(bh * p.n + pblk * BN), (uint32_t)id, info))) break;
          ++uq;
        }
        if (cur.bad) atomicOr(p.err, kErrBadSupport);
        const int slot = u % URING;
        if (u >= URING && !(ok = mbar_wait(&u_empty[slot], ((u / URING) - 1) & 1, abort_flag, p.err))) break;
        uring[2 * slot] = id;
        uring[2 * slot + 1] = cnt;
        mbar_arrive(&u_full[slot]);
        ++u;
      }
      if (ok) ok = publish(0u, 0u, kEntEnd);
      if (ok) {
        const int slot = u % URING;
        if (u < URING || mbar_wait(&u_empty[slot], ((u / URING) - 1) & 1, abort_flag, p.err)) {
          uring[2 * slot] = -1;
          uring[2 * slot + 1] = 0;
          mbar_arrive(&u_full[slot]);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ TMA loads
    // Q (at the first entry of each unit), K and V. K runs KLEAD entries ahead
    // of V: entry j's K is needed for S_j, which precedes the softmax and PV_j,
    // which need V_j. The whole warp runs the loop; one elected lane issues.
    const bool leader = elect_one();
    constexpr int KLEAD = (NK - 1 < 2) ? NK - 1 : 2;
    if (leader) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    uint32_t nq[2] = {0u, 0u};  // Q loads per buffer
    uint32_t jk = 0, jv = 0;    // K and V loads issued
    bool k_end = false, ok = true;
    while (ok) {
      // K for entry jk while it is at most KLEAD ahead of V
      while (ok && !k_end && jk <= jv + KLEAD) {
        EntryRec e;
        ok = __all_sync(0xffffffffu, wait_entry(meta, META, jk, e, abort_flag, p.err));
        if (!ok) break;
        if (e.info & kEntEnd) {
          k_end = true;
          break;
        }
        if (e.info & kEntFirst) {
          const int qb = (e.info & kEntQbuf) ? 1 : 0;
          // the previous unit in this buffer has finished its S MMAs
          if (nq[qb] > 0) ok = __all_sync(0xffffffffu, mbar_wait(&q_empty[qb], (nq[qb] - 1) & 1, abort_flag, p.err));
          if (!ok) break;
          const int bh = (int)e.unit / p.n_qtiles, t = (int)e.unit % p.n_qtiles;
          const int row = bh * p.n + t * 128;
          uint8_t* sq = smem + C::OFF_Q + qb * C::Q_BYTES;
          if (leader) {
            mbar_arrive_expect_tx(&q_full[qb], C::Q_BYTES);
            for (int c = 0; c < C::NCH; ++c) tma_load_2d(sq + c * 128 * ROWB, &tm_q, &q_full[qb], c * C::CH, row);
          }
          ++nq[qb];
        }
        const int s = (int)(jk % NK);
        if (jk >= (uint32_t)NK) ok = __all_sync(0xffffffffu, mbar_wait(&k_empty[s], ((jk / NK) - 1) & 1, abort_flag, p.err));
        if (!ok) break;
        uint8_t* dst = smem + C::OFF_K + s * C::KV_BYTES;
        if (leader) {
          mbar_arrive_expect_tx(&k_full[s], C::KV_BYTES);
          for (int c = 0; c < C::NCH; ++c) tma_load_2d(dst + c * BN * ROWB, &tm_k, &k_full[s], c * C::CH, (int)e.krow);
        }
        ++jk;
        __syncwarp();
      }
      if (!ok || jv == jk) break;  // jv == jk only once the entry stream has ended
      // V for entry jv (its record is already published)
      EntryRec e;
      ok = __all_sync(0xffffffffu, wait_entry(meta, META, jv, e, abort_flag, p.err));
      if (!ok) break;
      const int s = (int)(jv % NV);
      if (jv >= (uint32_t)NV) ok = __all_sync(0xffffffffu, mbar_wait(&v_empty[s], ((jv / NV) - 1) & 1, abort_flag, p.err));
      if (!ok) break;
      uint8_t* dst = smem + C::OFF_V + s * C::KV_BYTES;
      if (leader) {
        mbar_arrive_expect_tx(&v_full[s], C::KV_BYTES);
        for (int c = 0; c < C::NCH; ++c) tma_load_2d(dst + c * BN * ROWB, &tm_v, &v_full[s], c * C::CH, (int)e.krow);
      }
      ++jv;
      __syncwarp();
    }
    // No copy into this CTA's shared memory may outlive the CTA.
    if (leader) {
      for (uint32_t i = (jk > (uint32_t)NK ? jk - NK : 0u); i < jk; ++i)
        mbar_wait_drain(&k_full[i % NK], (i / NK) & 1, p.err);
      for (uint32_t i = (jv > (uint32_t)NV ? jv - NV : 0u); i < jv; ++i)
        mbar_wait_drain(&v_full[i % NV], (i / NV) & 1, p.err);
      for (int qb = 0; qb < 2; ++qb)
        if (nq[qb] > 0) mbar_wait_drain(&q_full[qb], (nq[qb] - 1) & 1, p.err);
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 2 issues S_j = Q K_j^T, warp 3 issues O += P_j V_j. Each whole warp
    // runs its loop (barrier waits and descriptor arithmetic stay warp-uniform)
    // and one elected lane issues the MMAs and their commits: single-lane
    // issue loops lose most of their issue slots to the softmax warps sharing
    // the SM sub-partition. Both walk the entry records in order. S_{j+NSB}
    // reuses the TMEM buffer of P_j and is issued once PV_j has completed.
    const bool leader = elect_one();
    if (warp == 2) {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BN, 0, 0);
      uint32_t nq[2] = {0u, 0u};  // units per Q buffer whose S MMAs began
      bool ok = true;
      for (uint32_t j = 0; ok; ++j) {
        EntryRec e;
        ok = __all_sync(0xffffffffu, wait_entry(meta, META, j, e, abort_flag, p.err));
        if (!ok || (e.info & kEntEnd)) break;
        const int qb = (e.info & kEntQbuf) ? 1 : 0;
        const int b = (int)(j % NSB);
        if (j >= (uint32_t)NSB) ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[b], ((j / NSB) - 1) & 1, abort_flag, p.err));
        if (ok && (e.info & kEntFirst)) ok = __all_sync(0xffffffffu, mbar_wait(&q_full[qb], nq[qb] & 1, abort_flag, p.err));
        const int s = (int)(j % NK);
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&k_full[s], (j / NK) & 1, abort_flag, p.err));
        if (!ok) break;
        tc_fence_after();
        const uint64_t qd = smem_desc(smem_u32(smem + C::OFF_Q + qb * C::Q_BYTES), 16, 8 * ROWB, C::SWZ);
        const uint64_t kd = smem_desc(smem_u32(smem + C::OFF_K + s * C::KV_BYTES), 16, 8 * ROWB, C::SWZ);
        const uint32_t dS = tbase + C::s_col(b);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int c = kk / (C::CH / 16), w = kk % (C::CH / 16);
            // descriptor start addresses advance in 16-byte units
            umma_ss(dS, qd + (uint64_t)((c * 128 * ROWB + w * 32) >> 4), kd + (uint64_t)((c * BN * ROWB + w * 32) >> 4),
                    IDESC_S, kk > 0);
          }
          umma_commit(&s_full[b]);
          umma_commit(&k_empty[s]);
          if (e.info & kEntLast) umma_commit(&q_empty[qb]);  // the unit's last read of its Q buffer
        }
        if (e.info & kEntLast) ++nq[qb];
        __syncwarp();
      }
      if (leader) {
        umma_commit(&drain[0]);  // every MMA of this thread done before TMEM is released
        mbar_wait_drain(&drain[0], 0, p.err);
      }
    } else {
      constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, 0, 1);
      uint32_t units = 0u;  // units whose PV MMAs began
      bool ok = true;
      for (uint32_t j = 0; ok; ++j) {
        EntryRec e;
        ok = __all_sync(0xffffffffu, wait_entry(meta, META, j, e, abort_flag, p.err));
        if (!ok || (e.info & kEntEnd)) break;
        const int b = (int)(j % NSB);
        const int sv = (int)(j % NV);
        const bool first = (e.info & kEntFirst) != 0u;
        ok = __all_sync(0xffffffffu, mbar_wait(&p_full[b], (j / NSB) & 1, abort_flag, p.err));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&v_full[sv], (j / NV) & 1, abort_flag, p.err));
        // the epilogue has read the previous unit's O out of TMEM
        if (ok && first && units > 0) ok = __all_sync(0xffffffffu, mbar_wait(o_free, (units - 1) & 1, abort_flag, p.err));
        if (!ok) break;
        tc_fence_after();
        const uint64_t vd = smem_desc(smem_u32(smem + C::OFF_V + sv * C::KV_BYTES), BN * ROWB, 8 * ROWB, C::SWZ);
        const uint32_t aP = tbase + C::s_col(b);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            umma_ts(tbase + C::O_COL, aP + kk * 8, vd + (uint64_t)((kk * 16 * ROWB) >> 4), IDESC_O,
                    (first && kk == 0) ? 0u : 1u);
          umma_commit(&v_empty[sv]);
          umma_commit(&pv_done[b]);
          if (e.info & kEntLast) umma_commit(o_final);
          st_release_smem(pv_issued, j + 1u);
        }
        if (e.info & kEntLast) ++units;
        __syncwarp();
      }
      if (leader) {
        umma_commit(&drain[1]);
        mbar_wait_drain(&drain[1], 0, p.err);
      }
    }
    __syncwarp();
  } else if (warp < 12) {
    // ------------------------------------------------------------ softmax
    const int h = (warp - 4) >> 2;       // which half of the key columns
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;   // row within the query tile = TMEM lane
    const uint32_t trow = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    const bool want_mass = (!SPARSE) && (p.mass != nullptr);
    const int half = (BN == 64) ? (r >> 6) : 0;
    constexpr int NC = C::HB / 32;       // 32-column chunks per half row
    constexpr int DH = D / 2;            // O columns this warpgroup rescales
    float m_ref = -INFINITY, l = 0.f, lt = 0.f;
    uint32_t cnt = 0, su = 0;
    int t = 0, bh = 0;
    float* lam = nullptr;
    for (uint32_t j = 0;; ++j) {
      EntryRec e;
      bool ok = wait_entry(meta, META, j, e, abort_flag, p.err);
      ok = __all_sync(0xffffffffu, ok);
      // every thread reads the same record; the end is taken after the
      // exchange barrier below so that all 256 threads leave together
      const bool end = ok && (e.info & kEntEnd);
      const int b = (int)(j % NSB);
      if (ok && !end) ok = mbar_wait(&s_full[b], (j / NSB) & 1, abort_flag, p.err);
      ok = __all_sync(0xffffffffu, ok);
      if (ok && !end && (e.info & kEntFirst)) {
        bh = (int)e.unit / p.n_qtiles;
        t = (int)e.unit % p.n_qtiles;
        m_ref = -INFINITY;
        l = 0.f;
        lt = 0.f;
        cnt = 0;
        lam = want_mass ? p.lam + lam_tile_offset(bh, t, p, C::ENT_PER_TILE) + h * 128 + r : nullptr;
      }
      const uint32_t tS = trow + C::s_col(b);
      uint32_t s[NC][32];
      float mxh = -INFINITY;
      int limit = -1;
      if (ok && !end) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < NC; ++cc) tmem_ld_x32(tS + h * C::HB + cc * 32, s[cc]);
#pragma unroll
        for (int cc = 0; cc < NC; ++cc) tmem_wait_ld(s[cc]);
        const int kbase = (int)(e.info >> 8) * BN;
        const int qpos = t * 128 + r;
        const bool row_on = (e.info >> (4 + half)) & 1u;
        // columns c <= limit of the tile are admissible (causal mask M, working-set mask R)
        limit = row_on ? ((kbase + BN - 1 > qpos) ? qpos - kbase : BN) : -1;
        if (limit < h * C::HB + C::HB - 1) {
#pragma unroll
          for (int cc = 0; cc < NC; ++cc)
#pragma unroll
            for (int q = 0; q < 32; ++q)
              s[cc][q] = (h * C::HB + cc * 32 + q <= limit) ? s[cc][q] : __float_as_uint(-INFINITY);
        }
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int cc = 0; cc < NC; ++cc)
#pragma unroll
          for (int q = 0; q < 16; ++q)
            mx4[q & 3] = fmax3(mx4[q & 3], __uint_as_float(s[cc][2 * q]), __uint_as_float(s[cc][2 * q + 1]));
        mxh = fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
      } else if (lane == 0) {
        atomicMin(sm_abort, (int)j);
      }
      // both halves' loads of S are complete before either writes P over it
      tc_fence_before();
      xch[(j & 1) * 256 + h * 128 + r] = mxh;
      named_bar_sync(1, 256);
      if (end || *reinterpret_cast<volatile int*>(sm_abort) <= (int)j) break;
      tc_fence_after();
      const float mx = fmaxf(mxh, xch[(j & 1) * 256 + (1 - h) * 128 + r]) * sl2;
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
      for (int cc = 0; cc < NC; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          float e0, e1;
          f2_unpack(ffma2(f2_pack(__uint_as_float(s[cc][2 * q]), __uint_as_float(s[cc][2 * q + 1])), sc2, nm2), e0,
                    e1);
          const float p0 = fast_exp2(e0);
          const float p1 = fast_exp2(e1);
          pk[q] = pack_bf16x2(p0, p1);
          rs2[q & 1] = fadd2(rs2[q & 1], f2_pack(p0, p1));
          add_bf16x2_to(rt2[q & 1], pk[q]);
        }
        tmem_st_x16(tS + h * (C::HB / 2) + cc * 16, pk);
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
        // O of this unit holds PV up to entry j-1: wait for the last one
        const uint32_t jb = j - 1u;
        bool okw = mbar_wait(&pv_done[jb % NSB], (jb / NSB) & 1, abort_flag, p.err);
        okw = __all_sync(0xffffffffu, okw);
        if (okw) {
          tc_fence_after();
          rescale_o(trow + C::O_COL + h * DH, DH, factor);
        } else if (lane == 0) {
          atomicMin(sm_abort, (int)j + 1);
        }
      }
      tmem_wait_st();
      if (want_mass) lam[(size_t)cnt * 256] = (rs > 0.f) ? m_use + fast_log2(rs) : -INFINITY;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
      ++cnt;
      if (e.info & kEntLast) {
        // per-row statistics of the unit for the epilogue
        const int sb = (int)(su & 1);
        bool okw = (su < 2) || mbar_wait(&st_empty[sb], ((su >> 1) - 1) & 1, abort_flag, p.err);
        okw = __all_sync(0xffffffffu, okw);
        if (okw) {
          float* st = stats + sb * 5 * 128;
          if (h == 0) st[r] = m_ref;
          st[(1 + h) * 128 + r] = l;
          st[(3 + h) * 128 + r] = lt;
        }
        __syncwarp();
        if (lane == 0) {
          if (okw) mbar_arrive(&st_full[sb]);
          else atomicMin(sm_abort, (int)j + 1);
        }
        ++su;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t tO = tbase + (static_cast<uint32_t>(quarter * 32) << 16) + C::O_COL;
    const bool want_mass = (!SPARSE) && (p.mass != nullptr);
    uint32_t eu = 0;  // units with entries processed (o_final / stats phases)
    for (int u = 0;; ++u) {
      const int slot = u % URING;
      bool ok = mbar_wait(&u_full[slot], (u / URING) & 1, abort_flag, p.err);
      ok = __all_sync(0xffffffffu, ok);
      int id = -1, cnt = 0;
      if (ok) {
        id = uring[2 * slot];
        cnt = uring[2 * slot + 1];
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&u_empty[slot]);
      const bool end = ok && id < 0;  // every epilogue thread reads the same record
      if (end) cnt = 0;
      const int bh = ok ? id / p.n_qtiles : 0, t = ok ? id % p.n_qtiles : 0;
      const int qpos = t * 128 + r;
      const bool row_valid = qpos < p.n;
      const size_t grow = (size_t)bh * p.n + qpos;
      float m = 0.f, lsum = 0.f, ltsum = 0.f;
      if (ok && cnt > 0) {
        const int sb = (int)(eu & 1);
        ok = mbar_wait(&st_full[sb], (eu >> 1) & 1, abort_flag, p.err);
        if (ok) {
          const float* st = stats + sb * 5 * 128;
          m = st[r];
          lsum = st[128 + r] + st[256 + r];
          ltsum = st[384 + r] + st[512 + r];
        }
        ok = __all_sync(0xffffffffu, ok);
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(&st_empty[sb]);
        if (ok) ok = mbar_wait(o_final, eu & 1, abort_flag, p.err);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (!ok && lane == 0) atomicMin(ep_abort, u);
      named_bar_sync(2, 128);
      if (end || *reinterpret_cast<volatile int*>(ep_abort) <= u) break;
      const float inv_l = (ltsum > 0.f) ? 1.f / ltsum : 0.f;
      if (cnt > 0) tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        if (cnt > 0) {
          tmem_ld_x32(tO + cc * 32, o);
          tmem_wait_ld(o);
          if (cc == D / 32 - 1) {
            // O is out of TMEM: the next unit's PV may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) o[q] = 0u;
        }
        if (row_valid) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + grow * D + cc * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(__uint_as_float(o[4 * q]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                                   __uint_as_float(o[4 * q + 2]) * inv_l, __uint_as_float(o[4 * q + 3]) * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + grow * D + cc * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv_l, __uint_as_float(o[8 * q + 1]) * inv_l);
              v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv_l, __uint_as_float(o[8 * q + 3]) * inv_l);
              v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv_l, __uint_as_float(o[8 * q + 5]) * inv_l);
              v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv_l, __uint_as_float(o[8 * q + 7]) * inv_l);
              dst[q] = v;
            }
          }
        }
      }
      const float lse2 = (lsum > 0.f) ? m + fast_log2(lsum) : -INFINITY;
      if (p.lse != nullptr && row_valid) p.lse[grow] = lse2 * 0.69314718055994531f;
      if (want_mass) {
        // Eq 5: r_qb = (1/B) * sum over the block's rows of 2^(lam_ib - lse2_i),
        // lam summed over the two column halves. Entries go through `part`
        // 64 at a time; blocks past the unit's entries are zero.
        const float* lam = p.lam + lam_tile_offset(bh, t, p, C::ENT_PER_TILE) + r;
        for (int c0 = 0; c0 < cnt; c0 += 64) {
          const int c1 = min(cnt, c0 + 64);
          for (int e = c0; e < c1; ++e) {
            float a = 0.f;
            if (row_valid && lsum > 0.f)
              a = fast_exp2(lam[(size_t)e * 256] - lse2) + fast_exp2(lam[(size_t)e * 256 + 128] - lse2);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            if (lane == 0) part[quarter * 64 + (e - c0)] = a;
          }
          named_bar_sync(2, 128);
          const int e = c0 + (r & 63);
          if (e < c1) {
            if (BN == 128) {
              if (r < 64) {
                const float v = (part[e - c0] + part[64 + e - c0]) + (part[128 + e - c0] + part[192 + e - c0]);
                p.mass[((size_t)bh * p.nb + t) * p.nb + e] = v * (1.f / BN);
              }
            } else {
              const int qq = r >> 6;
              const int qb = 2 * t + qq;
              if (qb < p.nb) {
                const float v = part[(2 * qq) * 64 + e - c0] + part[(2 * qq + 1) * 64 + e - c0];
                p.mass[((size_t)bh * p.nb + qb) * p.nb + e] = v * (1.f / BN);
              }
            }
          }
          named_bar_sync(2, 128);  // part is reused by the next chunk
        }
        for (int qq = 0; qq < C::ENT_PER_TILE; ++qq) {
          const int qb = t * C::ENT_PER_TILE + qq;
          if (qb >= p.nb) break;
          float* dst = p.mass + ((size_t)bh * p.nb + qb) * p.nb;
          for (int e = cnt + r; e < p.nb; e += 128) dst[e] = 0.f;
        }
      }
      if (cnt > 0) ++eu;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 3) {
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
