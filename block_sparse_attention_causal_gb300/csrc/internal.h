// Internal host/device interfaces shared by the translation units of libwise.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace wise {

struct AttnParams {
  int32_t bh_count;     // batch * heads
  int32_t heads;        // query heads per batch element
  int32_t kv_group;     // query heads per key/value head (1 without grouped-query attention)
  int32_t n;            // sequence length
  int32_t nb;           // n / BN key (and query) blocks
  int32_t n_qtiles;     // ceil(n / 128): work units (query tiles) per (batch, head)
  int32_t group_heads;  // (batch, head) slices per L2 group in the default order
  float scale_log2;     // softmax scale * log2(e)
  int32_t out_f32;      // O dtype: 0 bf16, 1 f32
  void* o;
  float* lse;           // optional
  float* mass;          // optional [bh, nb, nb] (discover only)
  float* lam;           // per-row, per-entry, per-half log2-sum-exp scratch (mass only)
  const int32_t* row_ptr;
  const int32_t* col_idx;
  int64_t col_cap;
  const int32_t* tile_order;  // optional unit order (reuse only)
  int64_t n_units;
  uint32_t* err;
  uint32_t sched_slot;  // work-counter slot of this launch
  // Selection fused into discovery with masses (one step of the window):
  // each completed mass row's Eq 6 step support is written (first step) or
  // OR-ed into sel_bits; the last step adds the sink / diagonal blocks and
  // writes the row counts. Off when sel_bits is null.
  uint32_t* sel_bits;   // [bh * nb, sel_nwords]
  int32_t* sel_counts;  // [bh * nb]
  int64_t sel_target_fx, sel_tol_fx;
  int32_t sel_nwords;
  int32_t sel_first, sel_last;
  uint32_t sel_flags;
  // Sparse steps with blocks of 32: the tiles' gathered entries, built once
  // per support (gather_plan.cu). Without them (null) the scheduler forms
  // each claimed tile's entries from its four CSR rows.
  const int32_t* plan_counts;    // [n_units] entries per tile
  const uint32_t* plan_entries;  // 4 words per entry, at plan_entry_index(bh, t, n_qtiles)
};

// Gathered-entry plan of sparse steps with blocks of 32: per work unit (one
// 128-row tile of one (batch, head) slice) its entry count, then, 16-byte
// aligned, the entries of each slice as a triangle: tile t has at most t + 1
// (its query blocks admit key blocks 0 .. 4t + 3, four per entry). An entry
// is four words: key blocks of slots 0 | 1 << 16, of slots 2 | 3 << 16, the
// slot mask (bit 4j + c: query block j of the tile lists slot c's block), 0.
__host__ __device__ inline int64_t plan_entry_index(int64_t bh, int64_t t, int64_t n_qtiles) {
  return bh * (n_qtiles * (n_qtiles + 1) / 2) + t * (t + 1) / 2;
}
__host__ __device__ inline int64_t plan_counts_bytes(int64_t n_units) { return (n_units * 4 + 15) / 16 * 16; }
__host__ __device__ inline int64_t plan_bytes(int64_t bh, int64_t n_qtiles) {
  return plan_counts_bytes(bh * n_qtiles) + plan_entry_index(bh, 0, n_qtiles) * 16;
}

struct GatherPlanLaunch {
  const int32_t* row_ptr;
  const int32_t* col_idx;
  int64_t col_cap;
  int32_t bh_count, nb, n_qtiles;
  int32_t* counts;
  uint32_t* entries;
  uint32_t* err;
};
cudaError_t launch_gather_plan(const GatherPlanLaunch& g, cudaStream_t stream);

struct SelectLaunch {
  const float* mass;
  int32_t window, bh_count, nb;
  int64_t target_fx, tol_fx;
  uint32_t flags;
  uint32_t* bits;
  int32_t* counts;
  int32_t* row_ptr;
  int32_t* col_idx;
  int64_t col_cap;
  int32_t* nnz;
  int32_t* tile_order;
  int32_t units_per_bh, qb_per_unit;
  int32_t mode;                // 0: Eq 6; 1: MassMatched; 2: SizeMatched (window 1)
  int32_t finalize_only;       // bits and counts are already built (fused selection)
  const int32_t* ref_row_ptr;  // reference working set of the controls
  const int32_t* ref_col_idx;
  int64_t ref_cap;
  uint32_t* err;
};

// Launch the attention kernel for one head dimension (defined in
// attn_d{64,96,128}.cu). maps = {Q, K, V, K128, V128} tensor maps (the last
// two with 128-row boxes, for consecutive gathered blocks of 32).
cudaError_t launch_attn_d64(int block, bool sparse, const CUtensorMap* maps, const AttnParams& p, cudaStream_t st);
cudaError_t launch_attn_d96(int block, bool sparse, const CUtensorMap* maps, const AttnParams& p, cudaStream_t st);
cudaError_t launch_attn_d128(int block, bool sparse, const CUtensorMap* maps, const AttnParams& p, cudaStream_t st);

cudaError_t launch_select(const SelectLaunch& s, cudaStream_t stream);

// Selection workspace layout: the row bitmasks [rows][nwords] and counts
// [rows] (int32), then, 16-byte aligned, the look-back state of the row_ptr
// scan (one 64-bit word per chunk of kSelectChunkRows rows plus a ticket).
constexpr int kSelectChunkRows = 256;
__host__ __device__ inline int64_t select_lookback_offset(int64_t rows, int64_t nwords) {
  return ((rows * nwords + rows) * 4 + 15) / 16 * 16;
}
__host__ __device__ inline int64_t select_lookback_bytes(int64_t rows) {
  return ((rows + kSelectChunkRows - 1) / kSelectChunkRows) * 8 + 16;
}

// Support diagnostics (diag_kernel.cu): retained future attention mass and
// the Jaccard index of two supports.
struct DiagLaunch {
  int64_t rows;  // batch * heads * nb CSR rows
  int32_t nb, batch;
  int64_t col_cap;           // col_idx entries of support A that may be read
  int64_t col_cap_b;         // ... of support B
  const float* mass;         // [rows, nb] (retained mass)
  const int32_t* row_ptr_a;  // support A (the only one for retained mass)
  const int32_t* col_idx_a;
  const int32_t* row_ptr_b;  // support B (Jaccard)
  const int32_t* col_idx_b;
  float* row_value;          // [rows] retained mass per row
  int32_t* row_counts;       // [rows][2] |A intersect B|, |A union B| per row
  double* batch_value;       // [batch] mean retained mass or Jaccard index (optional)
  long long* batch_counts;   // [batch][2] summed counts (optional)
  uint32_t* err;
};
cudaError_t launch_retained_mass(const DiagLaunch& d, cudaStream_t stream);
cudaError_t launch_jaccard(const DiagLaunch& d, cudaStream_t stream);

}  // namespace wise
