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
// (batch, head)) from the work order, heaviest first. Each CTA runs two
// independent query-tile streams; while the softmax of one stream works on its
// scores, the tensor core runs the other stream's MMAs. The key blocks
// ("entries") of both streams are published in one record ring, alternating
// between the streams while both have work.
//
// Warp roles (512 threads, four warpgroups):
//   warp 0      scheduler: claims units, walks their key-block lists and
//               publishes one record per entry (plus an end marker per stream)
//   warp 1      TMA loads of Q (per unit, one buffer per stream), K and V
//   warps 2, 3  MMA issue for stream 0 / stream 1 (warp 3 also allocates
//               TMEM): for each record of the stream, O_s += P_s V, then
//               S_s = Q_s K^T of the stream's next entry
//   warps 4-7   softmax of stream 0, one score row per thread
//   warps 8-11  softmax of stream 1
//   warps 12-15 epilogue of both streams: O normalisation and store, LSE,
//               block masses
// Entries are 128 keys wide for blocks of 128 and of 32, 64 keys for blocks
// of 64. With blocks of 32, a discovery entry is a contiguous 128-key span
// (four key blocks, with one Eq 5 partial sum per block and row), and a
// sparse entry gathers any four key blocks listed by the tile's four query
// blocks (32-row TMA boxes), with a per-(query block, slot) mask; each
// softmax warp owns one 32-row query block, so the mask is warp-uniform.
// TMEM: S_0 | S_1 | O_0 | O_1. P (bf16) is written over S_s by the softmax
// and read from TMEM by the PV MMA; the next S_s of the same stream is issued
// by the same thread right after that PV MMA, and tcgen05 MMAs issued by one
// thread execute in issue order. The commit that signals S_s also covers
// every earlier MMA, so when the softmax sees S_s its O_s already holds all
// previous entries and can be rescaled in place. The running row max only
// moves (and O is rescaled) when it grows by more than 2^8.
#pragma once
#include <stdint.h>

#include "gather.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "select_step.cuh"

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

// Flags of an entry record (low byte of `info`; the key block index is above).
enum : uint32_t {
  kEntFirst = 1u,   // first entry of its unit
  kEntLast = 2u,    // last entry of its unit
  kEntMark = 4u,    // end marker: the stream has no more entries
  kEntStream = 8u,  // the record belongs to stream 1 (else stream 0)
  kEntRows0 = 16u,  // query block 0 of the tile lists this key block
  kEntRows1 = 32u,  // ... query block 1 (BN = 64 only)
};

// Entry records: word 0 is the tag (record index + 1), written last; tag and
// info are read together with one 64-bit acquire load.
struct __align__(16) EntryRec {
  uint32_t tag;
  uint32_t info;   // flags | query-block bits << 4 | block index << 8
  uint32_t krow;   // global row of the key block's first key in K/V (TMA coordinate)
  uint32_t unit;   // unit id = bh * n_qtiles + tile
};
// Record of a gathered entry (sparse steps with blocks of 32): up to four
// listed key blocks in ascending order; unused slots repeat the last block
// and are masked for every row.
struct __align__(16) GatherRec {
  uint32_t tag;
  uint32_t info;    // flags | slot mask << 8: bit 4j + c = query block j of the tile lists slot c's block
  uint32_t krow;    // key blocks of slots 0 and 1 (16 bits each)
  uint32_t unit;    // unit id = bh * n_qtiles + tile
  uint32_t kb23;    // key blocks of slots 2 and 3
  uint32_t kvrow0;  // first K/V row of the unit's key/value head
  uint32_t pad[2];
};
__device__ __forceinline__ int gather_kb(const GatherRec& e, int c) {
  const uint32_t w = (c < 2) ? e.krow : e.kb23;
  return (int)((c & 1) ? (w >> 16) : (w & 0xffffu));
}

template <bool B, class T, class F>
struct pick_type {
  using type = T;
};
template <class T, class F>
struct pick_type<false, T, F> {
  using type = F;
};

template <int D, int BN, bool SPARSE>
struct AttnCfg {
  static_assert(D == 64 || D == 96 || D == 128, "head_dim");
  static_assert(BN == 32 || BN == 64 || BN == 128, "block");
  static constexpr int KW = (BN == 32) ? 128 : BN;       // keys per entry (one K/V tile)
  static constexpr bool GATHER = SPARSE && BN == 32;      // entries gather four listed 32-key blocks
  using Rec = typename pick_type<GATHER, GatherRec, EntryRec>::type;
  static constexpr int CH = (D == 96) ? 32 : 64;         // elements per swizzled smem row
  static constexpr int NCH = D / CH;                     // TMA boxes per tile
  static constexpr uint32_t SWZ = (CH == 64) ? 2u : 4u;  // descriptor code: 128B / 64B swizzle
  static constexpr uint32_t ROWB = CH * 2;               // bytes per swizzled row
  static constexpr uint32_t Q_BYTES = 128u * D * 2u;
  static constexpr uint32_t KV_BYTES = (uint32_t)KW * D * 2u;
  static constexpr int THREADS = 512;
  static constexpr int META = GATHER ? 16 : 32;  // entry records in flight
  static constexpr int MAX_NB = 1024;
  static constexpr int ENT_PER_TILE = 128 / BN;  // query blocks per 128-row tile
  // per stream: lse2[128], inv_l[128], unit, entries (+ padding)
  static constexpr int ST_STRIDE = 2 * 128 + 8;
  static constexpr uint32_t STATS_BYTES = 2u * ST_STRIDE * 4u;
  static constexpr uint32_t META_BYTES = META * (uint32_t)sizeof(Rec);
  static constexpr int NBAR_FIXED = 8 * 2 + 2 + 8;
  static constexpr uint32_t MISC_BYTES = 64;
  static constexpr uint32_t SMEM_LIMIT = 232448u;  // 227 KB per CTA
  static constexpr uint32_t FIXED = 2u * Q_BYTES + STATS_BYTES + META_BYTES + MISC_BYTES + (NBAR_FIXED + 16) * 8u;
  static constexpr int SLOTS_FIT = (int)((SMEM_LIMIT - FIXED) / KV_BYTES);
  static constexpr int NK = ((SLOTS_FIT + 1) / 2 > 4) ? 4 : (SLOTS_FIT + 1) / 2;
  static constexpr int NV = (SLOTS_FIT / 2 > 4) ? 4 : SLOTS_FIT / 2;
  static_assert(NK >= 2 && NV >= 2, "K/V rings");
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = 2u * Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr uint32_t OFF_STATS = OFF_V + NV * KV_BYTES;
  static constexpr uint32_t OFF_META = OFF_STATS + STATS_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_META + META_BYTES;
  static constexpr int NBAR = NBAR_FIXED + 2 * NK + 2 * NV;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8u;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + MISC_BYTES;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
  static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && KV_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(OFF_META % 16 == 0, "records");
  static constexpr uint32_t TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t s_col(int s) { return 128u * (uint32_t)s; }
  __host__ __device__ static constexpr uint32_t o_col(int s) { return 256u + (uint32_t)(s * D); }
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

// First float of tile t's Eq 5 scratch: per entry, one value per row.
__device__ __forceinline__ int64_t lam_tile_offset(int bh, int t, const AttnParams& p, int ept) {
  const int64_t before = (int64_t)ept * t * (t + 1) / 2;
  const int64_t total = (int64_t)ept * p.n_qtiles * (p.n_qtiles + 1) / 2;
  return ((int64_t)bh * total + before) * 128;
}

template <int TAG>
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint32_t* err) {
  int dummy_abort = 0;
  return mbar_wait<TAG>(bar, parity, &dummy_abort, err);
}

// Wait until record j is published; false on abort/timeout or if the ring
// was overrun (which the scheduler's flow control rules out). The spin is out
// of line; the common case (already published) is one load and a compare.
template <int TAG, class R>
static __device__ __noinline__ bool wait_entry_slow(R* r, uint32_t j, volatile int* abort_flag, uint32_t* err) {
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
__device__ __forceinline__ void read_rest(const EntryRec* r, EntryRec& out) {
  out.krow = r->krow;
  out.unit = r->unit;
}
__device__ __forceinline__ void read_rest(const GatherRec* r, GatherRec& out) {
  out.krow = r->krow;
  out.unit = r->unit;
  out.kb23 = r->kb23;
  out.kvrow0 = r->kvrow0;
}
// FULL: also read the rest of the record (tag and info always).
template <int TAG, bool FULL, class R>
__device__ __forceinline__ bool wait_entry(R* ring, int meta, uint32_t j, R& out, volatile int* abort_flag,
                                           uint32_t* err) {
  R* r = ring + (j % (uint32_t)meta);
  uint64_t ti = ld_acquire_smem_b64(&r->tag);
  if ((uint32_t)ti != j + 1u) {
    if (!wait_entry_slow<TAG>(r, j, abort_flag, err)) return false;
    ti = ld_acquire_smem_b64(&r->tag);
  }
  out.tag = j + 1u;
  out.info = (uint32_t)(ti >> 32);
  if (FULL) read_rest(r, out);
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

// Output rows of a unit with no entries (a sparse tile whose query blocks list
// nothing): O = 0 and LSE = -inf.
static __device__ __noinline__ void write_empty_unit(int id, const AttnParams& p, int d) {
  const int bh = id / p.n_qtiles, t = id % p.n_qtiles;
  for (int rr = 0; rr < 128; ++rr) {
    const int qpos = t * 128 + rr;
    if (qpos >= p.n) break;
    const size_t grow = (size_t)bh * p.n + qpos;
    if (p.out_f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + grow * d);
      for (int c = 0; c < d / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + grow * d);
      for (int c = 0; c < d / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (p.lse != nullptr) p.lse[grow] = -INFINITY;
  }
}

__device__ __forceinline__ void sched_slot_done(const AttnParams& p) {
  // every CTA has pulled its last position (all claims are made by one
  // thread, which calls this after its last claim): the last one out resets
  // the slot
  __threadfence();
  if (atomicAdd(&g_sched[p.sched_slot].done, 1u) == gridDim.x - 1) {
    g_sched[p.sched_slot].next = 0u;
    g_sched[p.sched_slot].done = 0u;
    __threadfence();
  }
}

// Eq 6 step support of mass row (bh, q), fused into discovery: one warp,
// the same fixed-point step as the selection kernel. The row's masses were
// stored by this CTA's epilogue warps (read through L2 after their barrier).
template <int NJ>
static __device__ __noinline__ void select_row_fused(const AttnParams& p, int bh, int q, int lane) {
  const int64_t row = (int64_t)bh * p.nb + q;
  const float* src = p.mass + row * p.nb;
  int64_t fx[NJ];
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) {
    const int b = jj * 32 + lane;
    fx[jj] = (b <= q) ? mass_fx(__ldcg(src + b)) : INT64_MIN;
  }
  uint32_t word = eq6_step_word_compact<NJ>(fx, p.sel_target_fx, p.sel_tol_fx, lane);
  uint32_t* dst = p.sel_bits + row * p.sel_nwords;
  if (!p.sel_first && lane < p.sel_nwords) word |= __ldcg(dst + lane);  // union with the window's earlier steps
  if (p.sel_last) {
    // sink block 0 and diagonal block q
    if ((p.sel_flags & 1u) && lane == 0) word |= 1u;
    if ((p.sel_flags & 2u) && lane == (q >> 5)) word |= 1u << (q & 31);
    const int cnt = warp_sum32(__popc(word));
    if (lane == 0) p.sel_counts[row] = cnt;
  }
  if (lane < p.sel_nwords) dst[lane] = word;
}
static __device__ __forceinline__ void select_row_fused_any(const AttnParams& p, int bh, int q, int lane) {
  if (p.sel_nwords <= 1) select_row_fused<1>(p, bh, q, lane);
  else if (p.sel_nwords <= 2) select_row_fused<2>(p, bh, q, lane);
  else if (p.sel_nwords <= 4) select_row_fused<4>(p, bh, q, lane);
  else select_row_fused<8>(p, bh, q, lane);
}

// ------------------------------------------------ gathered entries (B = 32)

// The scheduler of sparse steps with blocks of 32, run by the whole warp.
// With a plan (gather_plan.cu), a claimed unit's entries are read from it,
// one per lane, 32 at a time. Without one, the unit's four CSR rows become
// per-lane bit words and each entry takes the next four blocks of their
// union in ascending order, with the 4 x 4 mask of which query block lists
// which slot (gather.cuh). Flow control and the order of the two streams'
// records are those of the scheduler of the other variants.
template <class C>
__device__ __forceinline__ void gather_scheduler(const AttnParams& p, const CUtensorMap* tm_q, GatherRec* meta,
                                                 uint32_t* qpos0, uint32_t* qpos1, volatile int* abort_flag,
                                                 int lane, int d) {
  constexpr uint32_t FULLM = 0xffffffffu;
  constexpr uint32_t AHEAD = 10u;
  static_assert(AHEAD + 4u <= (uint32_t)C::META, "record ring");
  SchedSlot* sched = &g_sched[p.sched_slot];
  uint32_t j = 0;  // records published
  // publish record j once j < min(qpos0, qpos1) + AHEAD (lane 0 waits and writes)
  auto publish = [&](uint32_t info, uint32_t krow, uint32_t unit, uint32_t kb23, uint32_t kvrow0) -> bool {
    int good = 1;
    if (lane == 0) {
      if (j >= AHEAD) {
        const uint64_t t0 = global_timer_ns();
        for (uint32_t it = 0; j >= min(ld_acquire_smem(qpos0), ld_acquire_smem(qpos1)) + AHEAD; ++it) {
          if ((it & 63u) == 63u) {
            if (*abort_flag) {
              good = 0;
              break;
            }
            if (global_timer_ns() - t0 > kWaitLimitNs) {
              *abort_flag = 1;
              atomicOr(p.err, kErrTimeout);
              good = 0;
              break;
            }
          }
          __nanosleep(64);
        }
      }
      if (good) {
        GatherRec* r = meta + (j % (uint32_t)C::META);
        r->info = info;
        r->krow = krow;
        r->unit = unit;
        r->kb23 = kb23;
        r->kvrow0 = kvrow0;
        st_release_smem(&r->tag, j + 1u);
      }
    }
    ++j;
    return __shfl_sync(FULLM, good, 0) != 0;
  };
  struct GCur {
    uint32_t w0, w1, w2, w3;  // this lane's word of the blocks listed by query blocks 0-3 of the tile
    uint32_t rem;             // ... of their union, not yet published
    int unit, cnt;
    uint32_t kvrow0;  // first K/V row of the unit's key/value head
    bool alive;
    // with a plan: the unit's entries (this lane holds entry 32 k + lane of
    // the current group of 32) and their number
    const uint32_t* pe;
    int ne;
    uint32_t e0, e1, e2;
  };
  const bool planned = p.plan_counts != nullptr;
  GCur sc0, sc1;
  // a CTA's first two work-order positions are fixed (2b and 2b + 1); the
  // counter hands out the positions after the first 2 x gridDim
  uint32_t nclaim = 0;
  auto claim = [&](GCur& sc) -> bool {
    for (;;) {
      int stop = 0;
      unsigned int x = 0u;
      if (lane == 0) {
        stop = *abort_flag;
        if (!stop) x = (nclaim < 2u) ? 2u * blockIdx.x + nclaim : 2u * gridDim.x + atomicAdd(&sched->next, 1u);
      }
      ++nclaim;
      if (__shfl_sync(FULLM, stop, 0)) return false;
      x = __shfl_sync(FULLM, x, 0);
      if ((int64_t)x >= p.n_units) return false;
      const int64_t v = (p.tile_order != nullptr) ? (int64_t)__ldg(p.tile_order + x) : default_unit(x, p);
      if (v < 0 || v >= p.n_units) {
        if (lane == 0) atomicOr(p.err, kErrBadSupport);
        continue;
      }
      const int id = (int)v;
      const int bh = id / p.n_qtiles, t = id % p.n_qtiles;
      if (lane == 0)
        for (int c = 0; c < C::NCH; ++c) tma_prefetch_l2_2d(tm_q, c * C::CH, bh * p.n + t * 128);
      sc.kvrow0 = (uint32_t)(((bh / p.heads) * (p.heads / p.kv_group) + (bh % p.heads) / p.kv_group) * p.n);
      if (planned) {
        // the unit's count and its first 32 entries, read together (tile t
        // has room for t + 1 entries)
        const uint32_t* pe = p.plan_entries + 4 * plan_entry_index(bh, t, p.n_qtiles);
        const int ne = __ldg(p.plan_counts + id);
        uint4 ev = make_uint4(0u, 0u, 0u, 0u);
        if (lane <= t) ev = __ldg(reinterpret_cast<const uint4*>(pe) + lane);
        if (ne <= 0 || ne > t + 1) {
          if (ne != 0 && lane == 0) atomicOr(p.err, kErrBadSupport);
          if (lane == 0) write_empty_unit(id, p, d);
          __syncwarp();
          continue;
        }
        sc.pe = pe;
        sc.ne = ne;
        sc.e0 = ev.x;
        sc.e1 = ev.y;
        sc.e2 = ev.z;
        sc.unit = id;
        sc.cnt = 0;
        return true;
      }
      // CSR rows of query blocks 4t .. 4t + nq - 1 (row_ptr entries 0 .. nq)
      const int qb0 = 4 * t;
      const int nq = min(4, p.nb - qb0);
      const int64_t row0 = (int64_t)bh * p.nb + qb0;
      const int32_t rpv = (lane <= nq) ? __ldg(p.row_ptr + row0 + lane) : 0;
      int32_t a[4], b[4], v0[4];
      bool bad = false;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[q] = __shfl_sync(FULLM, rpv, q);
        b[q] = __shfl_sync(FULLM, rpv, q + 1);
        if (q >= nq) {
          a[q] = b[q] = 0;
        } else if (a[q] < 0 || a[q] > b[q] || (int64_t)b[q] > p.col_cap) {
          bad = true;
          a[q] = b[q] = 0;
        }
        v0[q] = (a[q] + lane < b[q]) ? __ldg(p.col_idx + a[q] + lane) : INT32_MAX;
      }
      sc.w0 = gather_list_bits(p.col_idx, a[0], b[0], qb0 + 0, v0[0], lane, bad);
      sc.w1 = gather_list_bits(p.col_idx, a[1], b[1], qb0 + 1, v0[1], lane, bad);
      sc.w2 = gather_list_bits(p.col_idx, a[2], b[2], qb0 + 2, v0[2], lane, bad);
      sc.w3 = gather_list_bits(p.col_idx, a[3], b[3], qb0 + 3, v0[3], lane, bad);
      sc.rem = sc.w0 | sc.w1 | sc.w2 | sc.w3;
      if (__any_sync(FULLM, bad) && lane == 0) atomicOr(p.err, kErrBadSupport);
      if (!__any_sync(FULLM, sc.rem != 0u)) {
        if (lane == 0) write_empty_unit(id, p, d);
        __syncwarp();
        continue;
      }
      sc.unit = id;
      sc.cnt = 0;
      return true;
    }
  };
  // publish stream s's next entry; claim its next unit after the last one
  auto step = [&](GCur& sc, uint32_t sflag) -> bool {
    uint32_t mask, kb01, kb23;
    bool more;
    if (planned) {
      const int c = sc.cnt;
      if (c > 0 && (c & 31) == 0) {
        // the next 32 of a long tile's entries
        uint4 ev = make_uint4(0u, 0u, 0u, 0u);
        if (c + lane < sc.ne) ev = __ldg(reinterpret_cast<const uint4*>(sc.pe) + c + lane);
        sc.e0 = ev.x;
        sc.e1 = ev.y;
        sc.e2 = ev.z;
      }
      kb01 = __shfl_sync(FULLM, sc.e0, c & 31);
      kb23 = __shfl_sync(FULLM, sc.e1, c & 31);
      mask = __shfl_sync(FULLM, sc.e2, c & 31) & 0xffffu;
      more = c + 1 < sc.ne;
    } else {
      int kb[4] = {0, 0, 0, 0};
      mask = gather_take_entry(sc.rem, sc.w0, sc.w1, sc.w2, sc.w3, lane, kb);
      kb01 = (uint32_t)kb[0] | ((uint32_t)kb[1] << 16);
      kb23 = (uint32_t)kb[2] | ((uint32_t)kb[3] << 16);
      more = __any_sync(FULLM, sc.rem != 0u);
    }
    const uint32_t info = (sc.cnt == 0 ? kEntFirst : 0u) | (more ? 0u : kEntLast) | sflag | (mask << 8);
    if (!publish(info, kb01, (uint32_t)sc.unit, kb23, sc.kvrow0)) return false;
    ++sc.cnt;
    if (more) return true;
    sc.alive = claim(sc);
    return sc.alive || publish(kEntMark | sflag, 0u, 0u, 0u, 0u);
  };
  bool ok = true;
  sc0.alive = claim(sc0);
  if (!sc0.alive) ok = publish(kEntMark, 0u, 0u, 0u, 0u);
  sc1.alive = ok && claim(sc1);
  if (ok && !sc1.alive) ok = publish(kEntMark | kEntStream, 0u, 0u, 0u, 0u);
  int s = 0;
  while (ok && (sc0.alive || sc1.alive)) {
    if (s == 0 && !sc0.alive) s = 1;
    else if (s == 1 && !sc1.alive) s = 0;
    ok = s ? step(sc1, kEntStream) : step(sc0, 0u);
    s ^= 1;
  }
}

// TMA loads of one K or V tile (KV_BYTES, announced on `bar` by the caller):
// one box per 64 (or 32) columns of the head dimension (map `tm`); for
// gathered entries, four 32-row boxes per column chunk (map `tm`), one per
// slot at the slot's key block, or one 128-row box (map `tm4`) when the four
// blocks are consecutive.
template <class C>
__device__ __forceinline__ void load_kv_tile(uint8_t* dst, const CUtensorMap* tm, const CUtensorMap* tm4,
                                             uint64_t* bar, const EntryRec& e) {
  for (int c = 0; c < C::NCH; ++c) tma_load_2d(dst + c * C::KW * C::ROWB, tm, bar, c * C::CH, (int)e.krow);
}
template <class C>
__device__ __forceinline__ void load_kv_tile(uint8_t* dst, const CUtensorMap* tm, const CUtensorMap* tm4,
                                             uint64_t* bar, const GatherRec& e) {
  const int kb0 = gather_kb(e, 0);
  if (gather_kb(e, 1) == kb0 + 1 && gather_kb(e, 2) == kb0 + 2 && gather_kb(e, 3) == kb0 + 3) {
    for (int c = 0; c < C::NCH; ++c)
      tma_load_2d(dst + c * C::KW * C::ROWB, tm4, bar, c * C::CH, (int)e.kvrow0 + 32 * kb0);
    return;
  }
#pragma unroll
  for (int sl = 0; sl < 4; ++sl) {
    const int row = (int)e.kvrow0 + 32 * gather_kb(e, sl);
    for (int c = 0; c < C::NCH; ++c) tma_load_2d(dst + (c * C::KW + sl * 32) * C::ROWB, tm, bar, c * C::CH, row);
  }
}

template <int D, int BN, bool SPARSE>
__global__ void __launch_bounds__(512, 1)
    wise_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_k4,
                     const __grid_constant__ CUtensorMap tm_v4, const AttnParams p) {
  using C = AttnCfg<D, BN, SPARSE>;
  constexpr int NK = C::NK, NV = C::NV, META = C::META;
  constexpr uint32_t ROWB = C::ROWB;
  extern __shared__ __align__(1024) uint8_t smem[];
  // 128B-swizzled TMA tiles need 1024-byte aligned destinations
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) {
      atomicOr(p.err, kErrInternal);
      sched_slot_done(p);
    }
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;           // [2] Q of the stream's unit loaded
  uint64_t* q_empty = q_full + 2;    // [2] last S MMA of the stream's unit done
  uint64_t* s_full = q_empty + 2;    // [2] S_s computed
  uint64_t* p_full = s_full + 2;     // [2] P_s written (4 softmax warps)
  uint64_t* o_final = p_full + 2;    // [2] last PV MMA of the stream's unit done
  uint64_t* o_free = o_final + 2;    // [2] O_s read out by the epilogue (4 warps)
  uint64_t* st_full = o_free + 2;    // [2] unit statistics written (4 softmax warps)
  uint64_t* st_empty = st_full + 2;  // [2] unit statistics consumed (4 epilogue warps)
  uint64_t* drain = st_empty + 2;    // [2] all MMAs of issuer s done
  uint64_t* comp_full = drain + 2;   // [8] completion word n % 8 written (phase n / 8)
  uint64_t* k_full = comp_full + 8;  // [NK]
  uint64_t* k_empty = k_full + NK;   // [NK]
  uint64_t* v_full = k_empty + NK;   // [NV]
  uint64_t* v_empty = v_full + NV;   // [NV]
  using Rec = typename C::Rec;
  Rec* meta = reinterpret_cast<Rec*>(smem + C::OFF_META);
  float* stats = reinterpret_cast<float*>(smem + C::OFF_STATS);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  uint32_t* tmem_base_slot = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  uint32_t* qpos0 = misc + 2;
  int* ep_bad = reinterpret_cast<int*>(misc + 3);
  uint32_t* qpos1 = misc + 4;
  uint32_t* comp_tail = misc + 5;
  uint32_t* marks_seen = misc + 6;  // [2] softmax warps of stream s past its end marker
  // completed units in the order their last PV MMA was issued: word n % 8 =
  // (n + 1) << 2 | end flag << 1 | stream, announced on comp_full[n % 8]
  uint32_t* comp = misc + 8;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4);
      mbar_init(&o_final[s], 1);
      mbar_init(&o_free[s], 4);
      mbar_init(&st_full[s], 4);
      mbar_init(&st_empty[s], 4);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    for (int i = 0; i < 8; ++i) mbar_init(&comp_full[i], 1);
    for (int i = 0; i < NK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int j = 0; j < META; ++j) meta[j].tag = 0u;
    *abort_flag = 0;
    *qpos0 = 0u;
    *qpos1 = 0u;
    *comp_tail = 0u;
    marks_seen[0] = 0u;
    marks_seen[1] = 0u;
    *ep_bad = 0;
    for (int i = 0; i < 8; ++i) comp[i] = 0u;
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
  // Registers per thread: 80 (warps 0-3) + 184 (two softmax warpgroups) + 64
  // (epilogue), in sum the 512 x 128 of the launch; each warpgroup sets its
  // count at the top of its branch.
  if (warp < 4) {
  setmaxnreg_dec<80>();
  if (warp == 0) {
    // ------------------------------------------------------------ scheduler
    if constexpr (C::GATHER) {
      gather_scheduler<C>(p, &tm_q, meta, qpos0, qpos1, abort_flag, lane, D);
    } else if (lane == 0) {
      SchedSlot* sched = &g_sched[p.sched_slot];
      uint32_t j = 0;  // records published
      bool ok = true;
      // Publish record j once j < min(qpos0, qpos1) + AHEAD, where qpos_s is
      // one past the last record whose PV MMA stream s's issuer has issued,
      // raised to "no limit" only once all four softmax warps of stream s
      // have read its end marker (they scan the records up to it after the
      // issuer has finished). Every reader (softmax, loader, issuers) is at
      // or beyond that minimum, so the ring is never overrun. AHEAD is also the claim horizon: units
      // are taken from the shared work counter only a few records before
      // they are needed, which keeps the CTAs' finishing times close. It
      // must exceed the issuers' read-ahead (their next record can be three
      // records past the minimum's stream position plus one marker).
      constexpr uint32_t AHEAD = 10u;
      static_assert(AHEAD + 4u <= (uint32_t)META, "record ring");
      auto publish = [&](uint32_t krow, uint32_t unit, uint32_t info) -> bool {
        if (j >= AHEAD) {
          const uint64_t t0 = global_timer_ns();
          for (uint32_t it = 0; j >= min(ld_acquire_smem(qpos0), ld_acquire_smem(qpos1)) + AHEAD; ++it) {
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
        r->info = info;
        r->krow = krow;
        r->unit = unit;
        st_release_smem(&r->tag, j + 1u);
        ++j;
        return true;
      };
      // per-stream state in two named structs (no runtime-indexed arrays:
      // those would live in local memory)
      struct StreamCur {
        TileCursor cur;
        int unit, cnt;
        uint32_t kvrow0;  // first K/V row of the unit's key/value head
        int32_t pblk;
        uint32_t pmask;
        bool alive;
      };
      StreamCur sc0, sc1;
      // Late steps: a CTA's first two work-order positions are fixed (2b and
      // 2b + 1), which saves the launch-wide atomic at the start; the counter
      // hands out the positions after the first 2 x gridDim.
      uint32_t nclaim = SPARSE ? 0u : 2u;
      // claim the next unit with at least one entry for stream s
      auto claim = [&](StreamCur& sc) -> bool {
        for (;;) {
          if (*abort_flag) return false;
          const unsigned int x = (nclaim < 2u) ? 2u * blockIdx.x + nclaim
                                               : (SPARSE ? 2u * gridDim.x : 0u) + atomicAdd(&sched->next, 1u);
          ++nclaim;
          if ((int64_t)x >= p.n_units) return false;
          const int64_t v = (SPARSE && p.tile_order != nullptr) ? (int64_t)__ldg(p.tile_order + x) : default_unit(x, p);
          if (v < 0 || v >= p.n_units) {
            atomicOr(p.err, kErrBadSupport);
            continue;
          }
          const int id = (int)v;
          const int bh = id / p.n_qtiles, t = id % p.n_qtiles;
          // Q of the unit into L2 ahead of its TMA load, while the CSR is read
          for (int c = 0; c < C::NCH; ++c) tma_prefetch_l2_2d(&tm_q, c * C::CH, bh * p.n + t * 128);
          if (SPARSE) sc.cur.init_sparse(t, bh, p, C::ENT_PER_TILE);
          else sc.cur.init_dense(t, p, C::KW);
          if (!sc.cur.next(sc.pblk, sc.pmask)) {
            if (sc.cur.bad) atomicOr(p.err, kErrBadSupport);
            write_empty_unit(id, p, D);
            continue;
          }
          sc.unit = id;
          sc.cnt = 0;
          // the key/value head of query head bh (grouped-query attention)
          sc.kvrow0 = (uint32_t)(((bh / p.heads) * (p.heads / p.kv_group) + (bh % p.heads) / p.kv_group) * p.n);
          return true;
        }
      };
      // publish stream s's next entry; claim its next unit after the last one
      auto step = [&](StreamCur& sc, uint32_t sflag) -> bool {
        int32_t nblk;
        uint32_t nmask;
        const bool more = sc.cur.next(nblk, nmask);
        const uint32_t info = (sc.cnt == 0 ? kEntFirst : 0u) | (more ? 0u : kEntLast) | sflag | (sc.pmask << 4) |
                              ((uint32_t)sc.pblk << 8);
        if (!publish(sc.kvrow0 + (uint32_t)(sc.pblk * C::KW), (uint32_t)sc.unit, info)) return false;
        if (more) {
          sc.pblk = nblk;
          sc.pmask = nmask;
          ++sc.cnt;
          return true;
        }
        if (sc.cur.bad) atomicOr(p.err, kErrBadSupport);
        sc.alive = claim(sc);
        return sc.alive || publish(0u, 0u, kEntMark | sflag);
      };
      if (SPARSE) {
        // The reads behind the CTA's first two claims, both units at once:
        // their work-order entries, then their CSR row starts, then a
        // prefetch of their first column entries. Each claim below then
        // finds its data in L1 instead of waiting on three dependent loads
        // in turn, and the launch's first records are published sooner.
        int64_t u[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int64_t x = 2 * (int64_t)blockIdx.x + i;
          u[i] = (x >= p.n_units) ? -1 : (p.tile_order != nullptr) ? (int64_t)__ldg(p.tile_order + x) : default_unit(x, p);
        }
        int32_t a[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const bool in = u[i] >= 0 && u[i] < p.n_units;
          const int64_t r = in ? (u[i] / p.n_qtiles) * p.nb + (u[i] % p.n_qtiles) * C::ENT_PER_TILE : 0;
          a[i] = in ? __ldg(p.row_ptr + r) : -1;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (a[i] >= 0 && (int64_t)a[i] < p.col_cap)
            asm volatile("prefetch.global.L1 [%0];" ::"l"(p.col_idx + a[i]));
      }
      sc0.alive = claim(sc0);
      if (!sc0.alive) ok = publish(0u, 0u, kEntMark);
      sc1.alive = ok && claim(sc1);
      if (ok && !sc1.alive) ok = publish(0u, 0u, kEntMark | kEntStream);
      int s = 0;
      while (ok && (sc0.alive || sc1.alive)) {
        if (s == 0 && !sc0.alive) s = 1;
        else if (s == 1 && !sc1.alive) s = 0;
        ok = s ? step(sc1, kEntStream) : step(sc0, 0u);
        s ^= 1;
      }
    }
    // The CTA's claims are over: release its hold on the launch's work
    // counter now. Done at the very end of the CTA instead, the counter's
    // atomic (all CTAs of a late step finish within a few microseconds of each
    // other) added about 11 us to every sparse launch.
    if (lane == 0) sched_slot_done(p);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ TMA loads
    // Records in order; K runs up to KLEAD records ahead of V (the MMA thread
    // needs K of a stream's next entry right after V of its current one).
    // The whole warp runs the loop; one elected lane issues.
    const bool leader = elect_one();
    constexpr uint32_t KLEAD = 2;
    if (leader) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      if (C::GATHER) {
        tma_prefetch_desc(&tm_k4);
        tma_prefetch_desc(&tm_v4);
      }
    }
    uint32_t nq0 = 0u, nq1 = 0u;  // Q loads per stream
    uint32_t rk = 0, rv = 0;    // next record for K / V
    uint32_t nk = 0, nv = 0;    // K / V loads issued
    int kends = 0, vends = 0;   // end markers passed
    bool ok = true;
    while (ok && vends < 2) {
      // K only if its record is already published: V (of an earlier record)
      // must never wait behind an unpublished record
      const bool k_turn = kends < 2 && rk < rv + KLEAD &&
                          (rk == rv || ld_acquire_smem(&meta[rk % (uint32_t)META].tag) == rk + 1u);
      Rec e;
      ok = __all_sync(0xffffffffu, wait_entry<2, true>(meta, META, k_turn ? rk : rv, e, abort_flag, p.err));
      if (!ok) break;
      if (k_turn) {
        ++rk;
        if (e.info & kEntMark) {
          ++kends;
          continue;
        }
        const int s = (e.info & kEntStream) ? 1 : 0;
        if (e.info & kEntFirst) {
          // the stream's previous unit has finished its S MMAs
          const uint32_t nqs = s ? nq1 : nq0;
          if (nqs > 0) ok = __all_sync(0xffffffffu, mbar_wait<2>(&q_empty[s], (nqs - 1) & 1, abort_flag, p.err));
          if (!ok) break;
          const int bh = (int)e.unit / p.n_qtiles, t = (int)e.unit % p.n_qtiles;
          uint8_t* sq = smem + C::OFF_Q + s * C::Q_BYTES;
          if (leader) {
            mbar_arrive_expect_tx(&q_full[s], C::Q_BYTES);
            for (int c = 0; c < C::NCH; ++c)
              tma_load_2d(sq + c * 128 * ROWB, &tm_q, &q_full[s], c * C::CH, bh * p.n + t * 128);
          }
          if (s) ++nq1;
          else ++nq0;
        }
        const int slot = (int)(nk % NK);
        if (nk >= (uint32_t)NK)
          ok = __all_sync(0xffffffffu, mbar_wait<2>(&k_empty[slot], ((nk / NK) - 1) & 1, abort_flag, p.err));
        if (!ok) break;
        uint8_t* dst = smem + C::OFF_K + slot * C::KV_BYTES;
        if (leader) {
          mbar_arrive_expect_tx(&k_full[slot], C::KV_BYTES);
          load_kv_tile<C>(dst, &tm_k, &tm_k4, &k_full[slot], e);
        }
        ++nk;
      } else {
        ++rv;
        if (e.info & kEntMark) {
          ++vends;
          continue;
        }
        const int slot = (int)(nv % NV);
        if (nv >= (uint32_t)NV)
          ok = __all_sync(0xffffffffu, mbar_wait<2>(&v_empty[slot], ((nv / NV) - 1) & 1, abort_flag, p.err));
        if (!ok) break;
        uint8_t* dst = smem + C::OFF_V + slot * C::KV_BYTES;
        if (leader) {
          mbar_arrive_expect_tx(&v_full[slot], C::KV_BYTES);
          load_kv_tile<C>(dst, &tm_v, &tm_v4, &v_full[slot], e);
        }
        ++nv;
      }
      __syncwarp();
    }
    // No copy into this CTA's shared memory may outlive the CTA.
    if (leader) {
      for (uint32_t i = (nk > (uint32_t)NK ? nk - NK : 0u); i < nk; ++i)
        mbar_wait_drain<2>(&k_full[i % NK], (i / NK) & 1, p.err);
      for (uint32_t i = (nv > (uint32_t)NV ? nv - NV : 0u); i < nv; ++i)
        mbar_wait_drain<2>(&v_full[i % NV], (i / NV) & 1, p.err);
      if (nq0 > 0) mbar_wait_drain<2>(&q_full[0], (nq0 - 1) & 1, p.err);
      if (nq1 > 0) mbar_wait_drain<2>(&q_full[1], (nq1 - 1) & 1, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ MMA issue
    // Warp 2 issues the MMAs of stream 0, warp 3 those of stream 1. For each
    // record of its stream: O_s += P_s V once the softmax has written P_s,
    // then S_s = Q_s K^T of the stream's next record, both from the same
    // elected thread, so the S MMA executes after the PV MMA that reads P_s
    // from the same TMEM columns. Records of the other stream are skipped but
    // counted: K and V slots are assigned in record order. The whole warp
    // runs the loop (waits stay warp-uniform); one elected lane issues.
    const int s = warp - 2;
    const uint32_t sflag = s ? kEntStream : 0u;
    const bool leader = elect_one();
    constexpr uint32_t IDESC_S = idesc_bf16_f32(128, C::KW, 0, 0);
    constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, 0, 1);
    const uint64_t qd = smem_desc(smem_u32(smem + C::OFF_Q + s * C::Q_BYTES), 16, 8 * ROWB, C::SWZ);
    const uint64_t kd_base = smem_desc(smem_u32(smem + C::OFF_K), 16, 8 * ROWB, C::SWZ);
    const uint64_t vd_base = smem_desc(smem_u32(smem + C::OFF_V), C::KW * ROWB, 8 * ROWB, C::SWZ);
    const uint32_t dS = tbase + C::s_col(s);
    const uint32_t dO = tbase + C::o_col(s);
    uint32_t* qpos = s ? qpos1 : qpos0;
    uint32_t scan = 0u, ord = 0u;  // next record to read; K/V records read so far
    uint32_t nqs = 0u, npv = 0u, nun = 0u;
    bool ok = true;
    // the stream's next record (index i, K/V ordinal o); false at its end
    // marker or on abort (then ok is false too)
    auto next_own = [&](Rec& e, uint32_t& i, uint32_t& o) -> bool {
      for (;;) {
        if (!__all_sync(0xffffffffu, wait_entry<3, false>(meta, META, scan, e, abort_flag, p.err))) {
          ok = false;
          return false;
        }
        const uint32_t idx = scan++;
        if (e.info & kEntMark) {
          if ((e.info & kEntStream) == sflag) return false;
          continue;
        }
        const uint32_t oo = ord++;
        if ((e.info & kEntStream) == sflag) {
          i = idx;
          o = oo;
          return true;
        }
      }
    };
    // operands of S_s for the record with K/V ordinal o are in shared memory
    auto wait_s = [&](const Rec& e, uint32_t o) -> bool {
      if (e.info & kEntFirst) {
        if (!__all_sync(0xffffffffu, mbar_wait<3>(&q_full[s], nqs & 1, abort_flag, p.err))) return false;
        ++nqs;
      }
      return __all_sync(0xffffffffu, mbar_wait<3>(&k_full[o % NK], (o / NK) & 1, abort_flag, p.err));
    };
    // S_s = Q_s K^T for the record with K/V ordinal o (operands waited for)
    auto issue_s = [&](const Rec& e, uint32_t o) {
      const int slot = (int)(o % NK);
      // descriptor start addresses advance in 16-byte units
      const uint64_t kd = kd_base + (uint64_t)((slot * C::KV_BYTES) >> 4);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int c = kk / (C::CH / 16), w = kk % (C::CH / 16);
          umma_ss(dS, qd + (uint64_t)((c * 128 * ROWB + w * 32) >> 4), kd + (uint64_t)((c * C::KW * ROWB + w * 32) >> 4),
                  IDESC_S, kk > 0);
        }
        umma_commit(&s_full[s]);
        umma_commit(&k_empty[slot]);
        if (e.info & kEntLast) umma_commit(&q_empty[s]);  // the unit's last read of its Q buffer
      }
      __syncwarp();
    };
    // announce a completed unit (or, with end = 2, this issuer's end) to the epilogue
    auto announce = [&](uint32_t end) {
      const uint32_t n = atomicAdd(comp_tail, 1u);
      comp[n % 8u] = ((n + 1u) << 2) | end | (uint32_t)s;
      mbar_arrive(&comp_full[n % 8u]);
    };
    Rec cur;
    uint32_t ci = 0u, co = 0u;
    bool have = next_own(cur, ci, co);
    if (have) {
      ok = wait_s(cur, co);
      if (ok) {
        tc_fence_after();
        issue_s(cur, co);
      }
    }
    while (ok && have) {
      // While the softmax works on the current record: read the next record
      // and wait for every operand except P, so that the PV MMA and the next
      // S MMA issue back to back once P is written.
      Rec nxt;
      uint32_t ni = 0u, no = 0u;
      const bool have_next = next_own(nxt, ni, no);
      if (!ok) break;
      const bool first = (cur.info & kEntFirst) != 0u;
      const int vslot = (int)(co % NV);
      ok = __all_sync(0xffffffffu, mbar_wait<3>(&v_full[vslot], (co / NV) & 1, abort_flag, p.err));
      // the epilogue has read the stream's previous O out of TMEM
      if (ok && first && nun > 0) ok = __all_sync(0xffffffffu, mbar_wait<3>(&o_free[s], (nun - 1) & 1, abort_flag, p.err));
      if (ok && have_next) ok = wait_s(nxt, no);
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait<3>(&p_full[s], npv & 1, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      const uint64_t vd = vd_base + (uint64_t)((vslot * C::KV_BYTES) >> 4);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < C::KW / 16; ++kk)
          umma_ts(dO, dS + kk * 8, vd + (uint64_t)((kk * 16 * ROWB) >> 4), IDESC_O, (first && kk == 0) ? 0u : 1u);
        umma_commit(&v_empty[vslot]);
        if (cur.info & kEntLast) {
          umma_commit(&o_final[s]);
          announce(0u);
        }
        atomicMax(qpos, ci + 1u);
      }
      ++npv;
      if (first) ++nun;
      __syncwarp();
      if (have_next) issue_s(nxt, no);
      cur = nxt;
      ci = ni;
      co = no;
      have = have_next;
    }
    if (leader) {
      announce(2u);  // also after an abort: the epilogue stops at both ends
      umma_commit(&drain[s]);  // every MMA of this thread done before TMEM is released
      mbar_wait_drain<3>(&drain[s], 0, p.err);
    }
    __syncwarp();
  }
  } else if (warp < 12) {
    setmaxnreg_inc<184>();
    // ------------------------------------------------------------ softmax
    const int s = (warp - 4) >> 2;  // stream
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row within the query tile = TMEM lane
    const uint32_t trow = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t tS = trow + C::s_col(s);
    const uint32_t tO = trow + C::o_col(s);
    const float sl2 = p.scale_log2;
    const bool want_mass = (!SPARSE) && (p.mass != nullptr);
    const int half = (BN == 64) ? (r >> 6) : 0;
    constexpr int NC = C::KW / 32;  // 32-column chunks of a score row
    // blocks of 32 in discovery: the fp32 row sum is taken per 32-column
    // chunk (one Eq 5 partial sum per key block). Only discovery with masses
    // runs this variant: without masses, blocks of 32 use the kernel for
    // blocks of 128 (the same arithmetic as gathered sparse steps).
    constexpr bool CHUNK_SUMS = (BN == 32) && !SPARSE;
    float* st = stats + s * C::ST_STRIDE;
    float m_ref = -INFINITY, l = 0.f, lt = 0.f;
    uint32_t cnt = 0, ne = 0, nst = 0;
    int t = 0, bh = 0;
    float* lam = nullptr;
    for (uint32_t rec = 0;; ++rec) {
      Rec e;
      bool ok = __all_sync(0xffffffffu, wait_entry<4, C::GATHER>(meta, META, rec, e, abort_flag, p.err));
      if (!ok) break;
      if ((((e.info & kEntStream) != 0u) ? 1 : 0) != s) continue;
      if (e.info & kEntMark) {
        // the last of the stream's softmax warps to get here releases the
        // stream's hold on the scheduler
        if (lane == 0 && atomicAdd(&marks_seen[s], 1u) == 3u) atomicMax(s ? qpos1 : qpos0, 0x7fffffffu);
        break;
      }
      ok = __all_sync(0xffffffffu, mbar_wait<4>(&s_full[s], ne & 1, abort_flag, p.err));
      if (!ok) break;
      if (e.info & kEntFirst) {
        e.unit = meta[rec % (uint32_t)META].unit;  // ordered after the tag's acquire load
        bh = (int)e.unit / p.n_qtiles;
        t = (int)e.unit % p.n_qtiles;
        m_ref = -INFINITY;
        l = 0.f;
        lt = 0.f;
        cnt = 0;
        lam = want_mass ? p.lam + lam_tile_offset(bh, t, p, C::ENT_PER_TILE) + (CHUNK_SUMS ? 4 * r : r) : nullptr;
      }
      tc_fence_after();
      uint32_t v[NC][32];
#pragma unroll
      for (int cc = 0; cc < NC; ++cc) tmem_ld_x32(tS + cc * 32, v[cc]);
#pragma unroll
      for (int cc = 0; cc < NC; ++cc) tmem_wait_ld(v[cc]);
      if constexpr (C::GATHER) {
        // this warp's rows are query block qb = 4t + quarter; slot c holds
        // key block kb_c: all columns if qb lists it and kb_c < qb, columns
        // 0..lane if kb_c == qb (causal mask M), none if qb does not list it
        // (working-set mask R)
        const uint32_t mq = (e.info >> (8 + 4 * quarter)) & 0xfu;
        const int qb = 4 * t + quarter;
        int lim[4];
        bool any = false;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const bool on = (mq >> c) & 1u;
          const bool diag = gather_kb(e, c) == qb;
          lim[c] = on ? (diag ? lane : 31) : -1;
          any |= !on || diag;
        }
        if (any) {
#pragma unroll
          for (int cc = 0; cc < NC; ++cc)
#pragma unroll
            for (int q = 0; q < 32; ++q) v[cc][q] = (q <= lim[cc]) ? v[cc][q] : __float_as_uint(-INFINITY);
        }
      } else {
        const int kbase = (int)(e.info >> 8) * C::KW;
        const int qpos = t * 128 + r;
        const bool row_on = (e.info >> (4 + half)) & 1u;
        // columns c <= limit of the tile are admissible (causal mask M, working-set mask R)
        const int limit = row_on ? ((kbase + C::KW - 1 > qpos) ? qpos - kbase : C::KW) : -1;
        if (limit < C::KW - 1) {
#pragma unroll
          for (int cc = 0; cc < NC; ++cc)
#pragma unroll
            for (int q = 0; q < 32; ++q) v[cc][q] = (cc * 32 + q <= limit) ? v[cc][q] : __float_as_uint(-INFINITY);
        }
      }
      // row max: eight independent 3-input max chains
      float mx8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mx8[q] = -INFINITY;
#pragma unroll
      for (int cc = 0; cc < NC; ++cc)
#pragma unroll
        for (int q = 0; q < 16; ++q)
          mx8[q & 7] = fmax3(mx8[q & 7], __uint_as_float(v[cc][2 * q]), __uint_as_float(v[cc][2 * q + 1]));
      const float mx =
          fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])) * sl2;
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
      float rsc[NC];  // per-chunk fp32 sums (CHUNK_SUMS)
#pragma unroll
      for (int cc = 0; cc < NC; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          float e0, e1;
          f2_unpack(ffma2(f2_pack(__uint_as_float(v[cc][2 * q]), __uint_as_float(v[cc][2 * q + 1])), sc2, nm2), e0,
                    e1);
          const float p0 = fast_exp2(e0);
          const float p1 = fast_exp2(e1);
          pk[q] = pack_bf16x2(p0, p1);
          rs2[q & 1] = fadd2(rs2[q & 1], f2_pack(p0, p1));
          add_bf16x2_to(rt2[q & 1], pk[q]);
        }
        tmem_st_x16(tS + cc * 16, pk);
        if constexpr (CHUNK_SUMS) {
          float a0, a1;
          f2_unpack(fadd2(rs2[0], rs2[1]), a0, a1);
          rsc[cc] = a0 + a1;
          rs2[0] = rs2[1] = 0ull;
        }
      }
      float rs, rt;
      {
        float a0, a1, b0, b1;
        f2_unpack(fadd2(rs2[0], rs2[1]), a0, a1);
        f2_unpack(fadd2(rt2[0], rt2[1]), b0, b1);
        rs = a0 + a1;
        rt = b0 + b1;
      }
      if constexpr (CHUNK_SUMS) rs = (rsc[0] + rsc[1]) + (rsc[2] + rsc[3]);
      l = l * factor + rs;
      lt = lt * factor + rt;
      // O_s holds every PV MMA up to the previous entry (the S_s commit
      // covers them); rows whose max jumped are rescaled in place
      if (__any_sync(0xffffffffu, resc)) rescale_o(tO, D, factor);
      tmem_wait_st();
      if (want_mass) {
        if constexpr (CHUNK_SUMS) {
          // lam_ib of the entry's four key blocks: one float4 per row
          float4 lv;
          lv.x = (rsc[0] > 0.f) ? m_use + fast_log2(rsc[0]) : -INFINITY;
          lv.y = (rsc[1] > 0.f) ? m_use + fast_log2(rsc[1]) : -INFINITY;
          lv.z = (rsc[2] > 0.f) ? m_use + fast_log2(rsc[2]) : -INFINITY;
          lv.w = (rsc[3] > 0.f) ? m_use + fast_log2(rsc[3]) : -INFINITY;
          reinterpret_cast<float4*>(lam)[(size_t)cnt * 128] = lv;
        } else {
          lam[(size_t)cnt * 128] = (rs > 0.f) ? m_use + fast_log2(rs) : -INFINITY;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[s]);
      ++ne;
      ++cnt;
      if (e.info & kEntLast) {
        // per-row results of the unit for the epilogue
        ok = (nst == 0) || __all_sync(0xffffffffu, mbar_wait<4>(&st_empty[s], (nst - 1) & 1, abort_flag, p.err));
        if (!ok) break;
        st[r] = (l > 0.f) ? m_use + fast_log2(l) : -INFINITY;
        st[128 + r] = (lt > 0.f) ? 1.f / lt : 0.f;
        if (quarter == 0 && lane == 0) {
          reinterpret_cast<int*>(st)[256] = bh * p.n_qtiles + t;
          reinterpret_cast<int*>(st)[257] = (int)cnt;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&st_full[s]);
        ++nst;
      }
    }
  } else {
    setmaxnreg_dec<64>();
    // ------------------------------------------------------------ epilogue
    // Serves the units of both streams in the order the MMA thread issued
    // their last PV MMA (the order in which their O accumulators complete).
    // All four warps walk the same completion list; named barrier 2 keeps
    // them together around the shared statistics and the mass partials.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const bool want_mass = (!SPARSE) && (p.mass != nullptr);
    uint32_t served0 = 0u, served1 = 0u;  // units served per stream
    int ends = 0;
    for (uint32_t n = 0;; ++n) {
      // next completed unit: its completion word is published through an
      // mbarrier (the waiting threads sleep instead of polling shared memory)
      bool ok = __all_sync(0xffffffffu, mbar_wait<5>(&comp_full[n % 8u], (n / 8u) & 1u, abort_flag, p.err));
      const uint32_t w = ok ? comp[n % 8u] : 0u;
      if (ok && (w >> 2) != n + 1u) {  // overrun, which the O hand-off rules out
        *abort_flag = 1;
        atomicOr(p.err, kErrTimeout);
        ok = false;
      }
      ok = __all_sync(0xffffffffu, ok);
      const bool end = ok && (w & 2u);
      const int s = (int)(w & 1u);
      float* st = stats + s * C::ST_STRIDE;
      int id = -1, cnt = 0;
      float lse2 = 0.f, inv_l = 0.f;
      float lrow[4] = {0.f, 0.f, 0.f, 0.f};  // lse2 of rows 4 lane .. 4 lane + 3 (mass reduction)
      const uint32_t served = s ? served1 : served0;
      if (ok && !end) {
        ok = __all_sync(0xffffffffu, mbar_wait<5>(&st_full[s], served & 1, abort_flag, p.err));
        if (ok) {
          id = reinterpret_cast<const int*>(st)[256];
          cnt = reinterpret_cast<const int*>(st)[257];
          lse2 = st[r];
          inv_l = st[128 + r];
          if (want_mass && BN != 32) {
#pragma unroll
            for (int i = 0; i < 4; ++i) lrow[i] = st[4 * lane + i];
          }
          // everything the unit needs from the statistics is in registers:
          // the stream's next unit may write them (its softmax waits for
          // this only at its last entry)
          __syncwarp();
          if (lane == 0) mbar_arrive(&st_empty[s]);
          ok = __all_sync(0xffffffffu, mbar_wait<5>(&o_final[s], served & 1, abort_flag, p.err));
        }
      }
      if (!ok && lane == 0) atomicOr(ep_bad, 1);
      named_bar_sync(2, 128);  // every warp has read the statistics
      if (*reinterpret_cast<volatile int*>(ep_bad)) break;
      if (end) {
        if (++ends == 2) break;  // both issuers have finished
        continue;
      }
      const int bh = id / p.n_qtiles, t = id % p.n_qtiles;
      const int qpos = t * 128 + r;
      const bool row_valid = qpos < p.n;
      const size_t grow = (size_t)bh * p.n + qpos;
      const uint32_t tO = tbase + (static_cast<uint32_t>(quarter * 32) << 16) + C::o_col(s);
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < D / 16; ++cc) {
        uint32_t o[16];
        tmem_ld_x16(tO + cc * 16, o);
        tmem_wait_ld16(o);
        if (cc == D / 16 - 1) {
          // O is out of TMEM: the stream's next PV may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&o_free[s]);
        }
        if (row_valid) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + grow * D + cc * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_float4(__uint_as_float(o[4 * q]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                                   __uint_as_float(o[4 * q + 2]) * inv_l, __uint_as_float(o[4 * q + 3]) * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + grow * D + cc * 16);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
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
      if (p.lse != nullptr && row_valid) p.lse[grow] = lse2 * 0.69314718055994531f;
      if (want_mass) {
        // Eq 5: r_qb = (1/B) * sum over the block's rows of 2^(lam_ib - lse2_i).
        const float* lamt = p.lam + lam_tile_offset(bh, t, p, C::ENT_PER_TILE);
        if constexpr (BN == 32) {
          // warp `quarter` owns query block 4t + quarter (its 32 rows, one per
          // lane); an entry holds four key blocks, one float4 per row. The
          // four sums are reduced together: after the exchanges, lanes
          // 8c .. 8c + 7 hold the sum of key block c.
          const int qb = 4 * t + quarter;
          const float l2 = (row_valid && lse2 > -INFINITY) ? lse2 : INFINITY;
          const float4* lam4 = reinterpret_cast<const float4*>(lamt) + r;
          const bool hi4 = (lane & 16) != 0, hi3 = (lane & 8) != 0;
#pragma unroll 4
          for (int e = 0; e < cnt; ++e) {
            const float4 lv = lam4[(size_t)e * 128];
            const float a0 = fast_exp2(lv.x - l2), a1 = fast_exp2(lv.y - l2);
            const float a2 = fast_exp2(lv.z - l2), a3 = fast_exp2(lv.w - l2);
            float k0 = hi4 ? a2 : a0, k1 = hi4 ? a3 : a1;
            k0 += __shfl_xor_sync(0xffffffffu, hi4 ? a0 : a2, 16);
            k1 += __shfl_xor_sync(0xffffffffu, hi4 ? a1 : a3, 16);
            float k = hi3 ? k1 : k0;
            k += __shfl_xor_sync(0xffffffffu, hi3 ? k0 : k1, 8);
            k += __shfl_xor_sync(0xffffffffu, k, 4);
            k += __shfl_xor_sync(0xffffffffu, k, 2);
            k += __shfl_xor_sync(0xffffffffu, k, 1);
            // the last span can reach past the sequence's last key block
            const int kb = 4 * e + (lane >> 3);
            if ((lane & 7) == 0 && qb < p.nb && kb < p.nb) p.mass[((size_t)bh * p.nb + qb) * p.nb + kb] = k * (1.f / 32);
          }
        } else {
          // Warp `quarter` takes entries quarter, quarter + 4, ...; lane l reads
          // rows 4l..4l+3 of an entry as one float4, so the loads of different
          // entries do not wait on each other, and a (half-)warp reduction gives
          // the block's sum. lse2 of the rows comes from the statistics area.
          float l2[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = 4 * lane + i;
            // rows past n, or with no admissible key, contribute nothing
            l2[i] = (t * 128 + row < p.n && lrow[i] > -INFINITY) ? lrow[i] : INFINITY;
          }
#pragma unroll 4
          for (int e = quarter; e < cnt; e += 4) {
            const float4 lv = *reinterpret_cast<const float4*>(lamt + (size_t)e * 128 + 4 * lane);
            float a = (fast_exp2(lv.x - l2[0]) + fast_exp2(lv.y - l2[1])) + (fast_exp2(lv.z - l2[2]) + fast_exp2(lv.w - l2[3]));
            if (BN == 128) {
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
              if (lane == 0) p.mass[((size_t)bh * p.nb + t) * p.nb + e] = a * (1.f / BN);
            } else {
              // lanes 0-15 hold rows 0-63 (query block 2t), lanes 16-31 rows 64-127
#pragma unroll
              for (int off = 8; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
              const int qb = 2 * t + (lane >> 4);
              if ((lane & 15) == 0 && qb < p.nb) p.mass[((size_t)bh * p.nb + qb) * p.nb + e] = a * (1.f / BN);
            }
          }
        }
        // blocks past the tile's last entry (beyond the causal range)
        const int covered = (BN == 32) ? 4 * cnt : cnt;
        for (int qq = 0; qq < C::ENT_PER_TILE; ++qq) {
          const int qb = t * C::ENT_PER_TILE + qq;
          if (qb >= p.nb) break;
          float* dst = p.mass + ((size_t)bh * p.nb + qb) * p.nb;
          for (int e = covered + r; e < p.nb; e += 128) dst[e] = 0.f;
        }
        if (p.sel_bits != nullptr) {
          // the unit's mass rows are complete once all four warps stored
          // their part; warp j then selects the tile's query block j
          named_bar_sync(3, 128);
          const int qb = t * C::ENT_PER_TILE + quarter;
          if (quarter < C::ENT_PER_TILE && qb < p.nb) select_row_fused_any(p, bh, qb, lane);
        }
      }
      if (s) ++served1;
      else ++served0;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 3) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

}  // namespace wise
