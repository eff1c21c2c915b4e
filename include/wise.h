/*
 * wise.h -- C ABI of the GB300 (sm_103a) WISE block-sparse causal attention
 * library: discover early, select a block support once, reuse it late.
 *
 * The operations follow "Attention Routing Stabilizes Early: Working-Set
 * Inference for Recurrent Language Models" (WISE, arXiv 2609.27373):
 *
 *   wise_attn_discover   §3 Eq 2 (unrestricted causal attention during the
 *                        first t_d recurrent steps) plus §5.1 Eq 5 (block
 *                        mass r_qb) fused into the same kernel;
 *   wise_select_support  §5.1 Eq 6 (per-step cumulative-mass block support,
 *                        unioned over the discovery window) and Appendix B
 *                        "Sparse-kernel implementation" (support stored as a
 *                        GPU-resident CSR of row offsets and block indices,
 *                        built once after discovery);
 *   wise_attn_sparse     §5.2 Eqs 7-8 (late-step attention restricted to the
 *                        reused support; Q/K/V and the within-support softmax
 *                        are recomputed on every call);
 *   wise_select_control  the MassMatched and SizeMatched controls of
 *                        Appendix B Eqs 20-22;
 *   wise_support_retained_mass, wise_support_jaccard
 *                        the support diagnostics of Appendix B ("retained
 *                        future attention mass") and Appendix C.2 Eq 24
 *                        (rolling working-set Jaccard stability).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Tensors are dense, row-major, in device memory owned by the caller:
 *     Q, O       : [batch, heads, seq_len, head_dim], head_dim contiguous;
 *     K, V       : [batch, kv_heads, seq_len, head_dim] (kv_heads = heads
 *                  unless the descriptor asks for grouped-query attention);
 *     LSE        : [batch, heads, seq_len] float32, natural-log
 *                  log-sum-exp of the scaled scores of each query row;
 *     block mass : [batch, heads, nb, nb] float32, nb = seq_len / block,
 *                  row q = query block, column b = key block (zero for b > q).
 *   Q, K, V are bf16. O is bf16 or float32 (wise_attn_desc.out_dtype).
 * - Masking is causal: key j is admissible for query i iff j <= i; key block
 *   b is admissible for query block q iff b <= q. One call is one attention
 *   layer.
 * - Supported shapes: head_dim in {64, 96, 128}; block in {32, 64, 128}
 *   (32 is the pages' default support granularity; the kernels work on
 *   128-row query tiles, i.e. four query blocks of 32 share one tile);
 *   seq_len a positive multiple of block with seq_len / block <= 1024;
 *   batch * heads >= 1. Base pointers of Q/K/V/O must be 16-byte aligned.
 * - The library never allocates or frees memory. Its only state lives in
 *   fixed device arrays of the library image: one error word per GPU, a ring
 *   of 256 work counters that attention launches take in turn (each launch
 *   leaves its counter at zero when it ends), and the scratch array of
 *   wise_select_support_noalloc. Calls are asynchronous and ordered on the
 *   given stream (a cudaStream_t; NULL means the legacy default stream).
 * - Calls may be recorded into a CUDA graph (stream capture) and replayed.
 *   The attention kernels each hold a work-counter slot for the length of a
 *   launch; eager launches and recorded ones draw from separate halves of the
 *   slots, so replays and eager calls on other streams can run side by side.
 *   One graph must not be replayed on two streams at once.
 * - Argument, shape and alignment errors are reported before any launch and
 *   nothing is written. A failed launch returns WISE_ERR_CUDA. Kernel-side
 *   problems (a malformed support list, a wait that timed out) are recorded in
 *   the device error word and read back with wise_device_status().
 */
#ifndef WISE_H_
#define WISE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WISE_ABI_VERSION 5

typedef struct CUstream_st* wise_stream_t; /* same type as cudaStream_t */

typedef enum wise_status {
  WISE_OK = 0,
  WISE_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad shape, bad eta, ...   */
  WISE_ERR_UNSUPPORTED = 2,      /* valid but not built (head_dim, block)   */
  WISE_ERR_ALIGNMENT = 3,        /* a tensor base is not 16-byte aligned     */
  WISE_ERR_WORKSPACE = 4,        /* workspace missing or too small           */
  WISE_ERR_BAD_SUPPORT = 5,      /* support CSR malformed / over capacity    */
  WISE_ERR_CUDA = 6,             /* CUDA runtime or driver error             */
  WISE_ERR_DEVICE_TIMEOUT = 7    /* a kernel wait exceeded its time limit    */
} wise_status;

typedef enum wise_dtype { WISE_BF16 = 0, WISE_F32 = 1 } wise_dtype;

/* Support flags (readings of this library, not part of Eq 6 itself). */
#define WISE_SUPPORT_SINK 1u /* add key block 0, which holds the first token  */
#define WISE_SUPPORT_DIAG 2u /* add the diagonal key block b = q              */

typedef struct wise_attn_desc {
  int32_t batch;
  int32_t heads;
  int32_t seq_len;       /* n */
  int32_t head_dim;      /* d_h */
  int32_t block;         /* B, the support block size (query and key blocks) */
  float softmax_scale;   /* 0 => 1/sqrt(head_dim), the scale of Eq 2 */
  int32_t out_dtype;     /* wise_dtype of O */
  int32_t kv_heads;      /* key/value heads; 0 => heads. Grouped-query
                          * attention when kv_heads < heads: kv_heads must
                          * divide heads, and query head h reads key/value
                          * head h / (heads / kv_heads). Masses and supports
                          * stay per query head. */
} wise_attn_desc;

/* ABI version (WISE_ABI_VERSION) and a static string for a status code. */
int wise_abi_version(void);
const char* wise_status_str(int status);

/* Bytes of workspace wise_attn_discover needs when block_mass != NULL
 * (per-row, per-key-block partial log-sum-exp values); 0 when the
 * descriptor is invalid. */
size_t wise_attn_discover_workspace(const wise_attn_desc* desc);

/*
 * wise_attn_discover -- one early (discovery) recurrent step.
 * Computes O = softmax(Q K^T * scale + M) V with the causal mask M (§3 Eq 2)
 * and, when block_mass != NULL, the block masses of §5.1 Eq 5:
 *     r_qb = (1/B) * sum_{i in query block q} sum_{j in key block b} A_ij,
 * written as [batch, heads, nb, nb] float32 (every entry is written; entries
 * with b > q are zero, and each row sums to 1 up to rounding).
 *   q, k, v     : bf16 inputs (device).
 *   o           : output (device), dtype desc->out_dtype.
 *   lse         : optional float32 [batch, heads, seq_len] (device) or NULL.
 *   block_mass  : optional float32 masses (device) or NULL.
 *   workspace   : device buffer of wise_attn_discover_workspace(desc) bytes
 *                 when block_mass != NULL; ignored otherwise. Its contents
 *                 are scratch and need no initialisation.
 * Returns WISE_OK or an error status (nothing launched on error).
 */
int wise_attn_discover(const wise_attn_desc* desc, const void* q, const void* k, const void* v,
                       void* o, float* lse, float* block_mass, void* workspace,
                       size_t workspace_bytes, wise_stream_t stream);

/* Number of work units of the late-step kernel: the length of the
 * tile_order schedule (one unit = 128 consecutive query rows of one
 * (batch, head)); 0 when the descriptor is invalid. */
int64_t wise_schedule_units(const wise_attn_desc* desc);

/* Maximum number of CSR entries a support can hold:
 * batch * heads * nb * (nb + 1) / 2 (every admissible block). */
int64_t wise_support_capacity(const wise_attn_desc* desc);

/* Bytes of workspace wise_select_support needs for `window` mass tensors. */
size_t wise_select_workspace(const wise_attn_desc* desc, int32_t window);

/*
 * wise_select_support -- build the reused working set once after discovery.
 * For every (batch, head, query block q) and each of the `window` mass
 * tensors (the last min(4, t_d) discovery steps, §5.1 Eq 6 / Appendix B
 * Eq 18), takes the smallest set of admissible key blocks (b <= q) whose
 * cumulative mass reaches eta, blocks ordered by descending mass; the
 * support is the union over the window, plus key block 0 if
 * WISE_SUPPORT_SINK and block q if WISE_SUPPORT_DIAG is set in `flags`.
 * Cumulative sums run in int64 fixed point (2^-52 units, masses rounded to
 * nearest even); near-ties within 1e-6 of the k-th mass go to the lower
 * block index; if the admissible mass never reaches eta every admissible
 * block is taken.
 *   block_mass : float32 [window, batch, heads, nb, nb] (device).
 *   window     : 1..8.   eta: 0 < eta < 1.
 *   row_ptr    : int32 [batch*heads*nb + 1] (device), rows ordered
 *                (batch, head, query block); row_ptr[0] = 0.
 *   col_idx    : int32 [col_capacity] (device), ascending key blocks per
 *                row. col_capacity must be >= wise_support_capacity(desc).
 *   tile_order : int32 [wise_schedule_units(desc)] (device) or NULL: the
 *                late-step work order (execution metadata for
 *                wise_attn_sparse: units with more listed blocks first,
 *                ties by unit index).
 *   nnz        : int32 [1] (device) or NULL: total number of entries.
 *   workspace  : wise_select_workspace(desc, window) bytes (device).
 */
int wise_select_support(const wise_attn_desc* desc, const float* block_mass, int32_t window,
                        double eta, uint32_t flags, int32_t* row_ptr, int32_t* col_idx,
                        int64_t col_capacity, int32_t* tile_order, int32_t* nnz,
                        void* workspace, size_t workspace_bytes, wise_stream_t stream);

/*
 * wise_attn_discover_select -- one discovery step of the selection window
 * with that step's part of wise_select_support done in the same launch.
 * (§5.1 Eq 6 / Appendix B Eq 18, streamed: the step supports are OR-ed into
 * per-row bitmasks as the step's block masses are produced, so the window's
 * mass tensors need not be kept, and no separate selection launch runs.)
 * Computes what wise_attn_discover computes (O, LSE, the block masses into
 * block_mass, which is required here). Then, for every query-block row, it
 * takes the row's Eq 6 step support with exactly the arithmetic of
 * wise_select_support, and:
 *   - at step 0 writes it into the row's bitmask in select_state;
 *   - at later steps ORs it in;
 *   - at step window - 1 also adds the WISE_SUPPORT_SINK / _DIAG blocks of
 *     `flags` and records the row's block count.
 * After the last step, wise_select_finalize turns select_state into the CSR
 * and work order. The steps of a window must run in order on one stream. The
 * result is bit-identical to wise_select_support on the window's masses.
 *   step, window : 0 <= step < window <= 8.   eta: 0 < eta < 1.
 *   block_mass   : float32 [batch, heads, nb, nb] (device), this step's masses.
 *   workspace    : wise_attn_discover_workspace(desc) bytes (device).
 *   select_state : wise_select_workspace(desc, window) bytes (device, 16-byte
 *                  aligned), kept by the caller across the window's steps;
 *                  needs no initialisation (step 0 overwrites it).
 * Supports nb <= 256 (WISE_ERR_UNSUPPORTED beyond: use wise_select_support).
 */
int wise_attn_discover_select(const wise_attn_desc* desc, const void* q, const void* k, const void* v,
                              void* o, float* lse, float* block_mass, void* workspace,
                              size_t workspace_bytes, double eta, uint32_t flags, int32_t step,
                              int32_t window, void* select_state, size_t select_state_bytes,
                              wise_stream_t stream);

/*
 * wise_select_finalize -- the CSR schedule of the support accumulated by a
 * window of wise_attn_discover_select steps (Appendix B "Sparse-kernel
 * implementation"): row_ptr, ascending col_idx, nnz and the late-step work
 * order, with the same meaning, layouts and checks as in
 * wise_select_support.
 */
int wise_select_finalize(const wise_attn_desc* desc, const void* select_state, size_t select_state_bytes,
                         int32_t* row_ptr, int32_t* col_idx, int64_t col_capacity, int32_t* tile_order,
                         int32_t* nnz, wise_stream_t stream);

/*
 * wise_select_support_noalloc -- wise_select_support for callers that cannot
 * allocate device memory. (Not an operation of the paper: the same selection
 * as wise_select_support, only the scratch memory comes from elsewhere.)
 * Some callers cannot call cudaMalloc or hand out a workspace: engines whose
 * memory plan is fixed before they run, runtimes that own every byte of
 * device memory through their own pool, and code that must not call the
 * allocator on its path because cudaMalloc / cudaFree can synchronise the
 * device. This variant takes the
 * same arguments minus the workspace and uses a 2 MiB scratch array that is
 * part of the library image instead, so it allocates nothing.
 *   - The scratch is held by every GPU that loads the library until the
 *     process exits; shapes needing more than 2 MiB of selection workspace
 *     (wise_select_workspace(desc, window) > 2 MiB: about 8 bytes per
 *     (batch, head, query block) row plus 4 bytes per 32 key blocks, i.e.
 *     up to ~260 000 rows when seq_len / block <= 32 and ~58 000 rows at
 *     seq_len / block = 256) return WISE_ERR_WORKSPACE without launching.
 *   - The first call on a device looks up the scratch address for that
 *     device (cudaGetSymbolAddress); make that first call before any stream
 *     capture on the device.
 *   - All calls share the one scratch array, which keeps the last call's
 *     contents (nothing in it needs to start at zero): calls whose kernels
 *     overlap on the GPU (different streams without ordering) race on it and
 *     must be serialised by the caller.
 * Arguments, outputs and status codes are those of wise_select_support.
 */
int wise_select_support_noalloc(const wise_attn_desc* desc, const float* block_mass, int32_t window,
                                double eta, uint32_t flags, int32_t* row_ptr, int32_t* col_idx,
                                int64_t col_capacity, int32_t* tile_order, int32_t* nnz,
                                wise_stream_t stream);

/*
 * wise_attn_sparse -- one late (reuse) recurrent step, §5.2 Eq 8:
 * O = softmax(Q K^T * scale + M + R) V where R is 0 on the key blocks listed
 * for the query's block and -inf elsewhere (Eq 7); M is causal. Only the
 * listed key blocks are read and computed.
 *   row_ptr, col_idx : the support CSR (device), as written by
 *                wise_select_support or by the caller (same layout; blocks
 *                strictly ascending and <= q within each row).
 *   col_capacity     : number of int32 entries readable at col_idx.
 *   tile_order       : the schedule from wise_select_support, or NULL for
 *                the natural order.
 *   o, lse           : as in wise_attn_discover. A row whose support admits
 *                no key gets O = 0 and LSE = -inf.
 * Entries that break the CSR rules are skipped and flagged in the device
 * error word (WISE_ERR_BAD_SUPPORT); they are never dereferenced out of
 * bounds.
 */
int wise_attn_sparse(const wise_attn_desc* desc, const void* q, const void* k, const void* v,
                     const int32_t* row_ptr, const int32_t* col_idx, int64_t col_capacity,
                     const int32_t* tile_order, void* o, float* lse, wise_stream_t stream);

/*
 * wise_gather_plan_bytes / wise_gather_plan -- for blocks of 32 only: the
 * late steps' gathered entries of every 128-row tile, built once from the
 * support CSR and reused by every late step (WISE Appendix B
 * "Sparse-kernel implementation": the schedule is built once after
 * discovery). A tile holds four 32-row query blocks; an entry is the next
 * four key blocks of the union of their lists, in ascending order, with
 * the mask of which query block lists which of the four. Without a plan,
 * wise_attn_sparse forms the same entries from the CSR on every late step.
 *   wise_gather_plan_bytes : bytes of the plan for desc (0 unless
 *                desc->block == 32): an int32 count per tile, then, 16-byte
 *                aligned, 16 bytes per entry, tile t of each (batch, head)
 *                slice owning room for t + 1 entries.
 *   row_ptr, col_idx, col_capacity : the support CSR (device), as for
 *                wise_attn_sparse; entries breaking its rules are skipped
 *                and flagged (WISE_ERR_BAD_SUPPORT in the device word).
 *   plan, plan_bytes : device buffer (caller-owned, 16-byte aligned), at
 *                least wise_gather_plan_bytes(desc). Every tile's count and
 *                entries are written; it stays valid while the CSR is not
 *                changed.
 * Returns WISE_ERR_UNSUPPORTED for other block sizes, WISE_ERR_WORKSPACE if
 * plan_bytes is too small. One launch on `stream`.
 */
size_t wise_gather_plan_bytes(const wise_attn_desc* desc);
int wise_gather_plan(const wise_attn_desc* desc, const int32_t* row_ptr, const int32_t* col_idx,
                     int64_t col_capacity, void* plan, size_t plan_bytes, wise_stream_t stream);

/*
 * wise_attn_sparse_planned -- wise_attn_sparse (§5.2 Eq 8) over a support
 * whose gathered entries were built by wise_gather_plan from the same CSR
 * (blocks of 32; plan NULL = wise_attn_sparse). The results are the same bits
 * as without the plan: the entries, their order and the arithmetic are the
 * same; the late step only reads them instead of forming them. A plan whose
 * counts exceed a tile's room is flagged (WISE_ERR_BAD_SUPPORT) and its tile
 * is written as empty.
 */
int wise_attn_sparse_planned(const wise_attn_desc* desc, const void* q, const void* k, const void* v,
                             const int32_t* row_ptr, const int32_t* col_idx, int64_t col_capacity,
                             const int32_t* tile_order, const void* plan, void* o, float* lse,
                             wise_stream_t stream);

/*
 * wise_select_control -- the early-static support controls of WISE Appendix B
 * ("Intervention controls"), built from ONE step's masses (the pages use the
 * first recurrent step) and a reference working set (WISE's own):
 *   WISE_CONTROL_MASS_MATCHED (Eqs 20-21): per query block q, the smallest
 *       set of highest-mass admissible blocks of this step whose cumulative
 *       mass reaches m_q, the mass of this step that the reference row covers
 *       (summed in the same 2^-52 fixed point as Eq 6);
 *   WISE_CONTROL_SIZE_MATCHED (Eq 22): the |reference row| highest-mass
 *       admissible blocks of this step (TopK).
 * Order, near-tie rule and output are those of wise_select_support; the
 * Static-95 control (Eq 19) is wise_select_support itself with window 1,
 * eta = 0.95 and the first step's masses.
 *   block_mass   : [batch, heads, nb, nb] float32 masses of the step (device).
 *   mode         : WISE_CONTROL_MASS_MATCHED or WISE_CONTROL_SIZE_MATCHED.
 *   ref_row_ptr, ref_col_idx, ref_capacity : the reference support CSR
 *                  (device); repeated entries count once, entries outside
 *                  0 <= b <= q are skipped and flagged.
 *   flags        : WISE_SUPPORT_SINK / _DIAG blocks added afterwards (0 for
 *                  the pages' definitions).
 *   row_ptr .. nnz, workspace : as in wise_select_support with window = 1
 *                  (workspace of wise_select_workspace(desc, 1) bytes).
 */
enum { WISE_CONTROL_MASS_MATCHED = 1, WISE_CONTROL_SIZE_MATCHED = 2 };
int wise_select_control(const wise_attn_desc* desc, const float* block_mass, int32_t mode,
                        const int32_t* ref_row_ptr, const int32_t* ref_col_idx, int64_t ref_capacity, uint32_t flags,
                        int32_t* row_ptr, int32_t* col_idx, int64_t col_capacity, int32_t* tile_order, int32_t* nnz,
                        void* workspace, size_t workspace_bytes, wise_stream_t stream);

/*
 * wise_support_retained_mass -- retained future attention mass (WISE
 * Appendix B, "Evaluation metrics"): the fraction of a later step's
 * unrestricted attention mass that falls inside a (frozen) support.
 *   block_mass   : [batch, heads, nb, nb] float32 block masses r_qb of the
 *                  later step, as wise_attn_discover writes them (device).
 *   row_ptr, col_idx, col_capacity : the support CSR (device), as for
 *                  wise_attn_sparse.
 *   row_retained : [batch * heads * nb] float32 (device, caller-owned):
 *                  sum over the row's listed key blocks b <= q of r_qb.
 *   batch_mean   : [batch] float64 (device, optional): mean of row_retained
 *                  over the heads x nb rows of each batch element.
 * Entries outside 0 <= b <= q are skipped and flagged (WISE_ERR_BAD_SUPPORT).
 * The row sums are accumulated in float64 in a fixed order, so repeated calls
 * give identical results.
 */
int wise_support_retained_mass(const wise_attn_desc* desc, const float* block_mass, const int32_t* row_ptr,
                                const int32_t* col_idx, int64_t col_capacity, float* row_retained,
                                double* batch_mean, wise_stream_t stream);

/*
 * wise_support_jaccard -- rolling working-set stability (WISE Appendix C.2
 * Eq 24): the Jaccard index of two supports A and B over all active
 * (head, query block, key block) entries of each batch element.
 *   row_ptr_a, col_idx_a, col_capacity_a, row_ptr_b, col_idx_b,
 *   col_capacity_b : two support CSRs of the same shape (device), each with
 *                  the number of col_idx entries that may be read.
 *   row_counts   : [batch * heads * nb][2] int32 (device, caller-owned):
 *                  |A_q intersect B_q| and |A_q union B_q| per row.
 *   batch_counts : [batch][2] int64 (device, optional): their sums.
 *   batch_jaccard: [batch] float64 (device, optional): sum of intersections
 *                  / sum of unions (1 when both supports are empty).
 * Sets, not lists, are compared: repeated entries count once; entries outside
 * 0 <= b <= q are skipped and flagged (WISE_ERR_BAD_SUPPORT).
 */
int wise_support_jaccard(const wise_attn_desc* desc, const int32_t* row_ptr_a, const int32_t* col_idx_a,
                         int64_t col_capacity_a, const int32_t* row_ptr_b, const int32_t* col_idx_b,
                         int64_t col_capacity_b, int32_t* row_counts, int64_t* batch_counts, double* batch_jaccard,
                         wise_stream_t stream);

/* Host-side check of a support CSR (host pointers): row_ptr monotone from 0,
 * every row strictly ascending with 0 <= b <= q, and, if the flags ask for
 * them, block 0 and block q present. Returns WISE_OK or
 * WISE_ERR_BAD_SUPPORT. */
int wise_validate_support(const wise_attn_desc* desc, const int32_t* row_ptr_host,
                          const int32_t* col_idx_host, uint32_t flags);

/* Host-side check of a late-step work order (host pointer): tile_order must
 * hold every unit 0 .. wise_schedule_units(desc) - 1 exactly once, as
 * wise_select_support writes it (Appendix B "Sparse-kernel implementation"
 * fixes the CSR, not an order; the order is this library's schedule). With a
 * duplicated unit two CTAs would compute and write the same rows; a missing
 * unit would never be written. wise_attn_sparse only range-checks the entries
 * it reads. Returns WISE_OK, WISE_ERR_BAD_SUPPORT, or WISE_ERR_INVALID_ARGUMENT
 * for a NULL pointer or a bad descriptor. */
int wise_validate_schedule(const wise_attn_desc* desc, const int32_t* tile_order_host);

/* Self-check of the library's failure handling (no counterpart in the paper).
 * Every wait in the kernels is bounded: when a wait runs out (2 s), the kernel
 * records WISE_ERR_DEVICE_TIMEOUT in the device error word, lets its own
 * copies finish and returns, so the CUDA context stays usable. This call
 * launches one single-thread kernel that waits, through that same wait
 * routine, on a barrier nothing arrives on, with the limit shortened to 20 ms.
 * The wait runs out and the kernel returns; it touches no memory but the
 * error word. Afterwards wise_device_status() reports
 * WISE_ERR_DEVICE_TIMEOUT (and clears the word). Returns WISE_OK once the
 * kernel is queued on `stream`, WISE_ERR_CUDA if the launch failed. */
int wise_wait_expiry_check(wise_stream_t stream);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device: WISE_OK, WISE_ERR_BAD_SUPPORT, WISE_ERR_DEVICE_TIMEOUT, or
 * WISE_ERR_CUDA if the synchronisation itself failed. */
int wise_device_status(wise_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* WISE_H_ */
