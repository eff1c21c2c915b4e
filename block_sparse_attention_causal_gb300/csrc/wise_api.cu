// C ABI of libwise (declared in include/wise.h): argument validation, TMA
// descriptor encoding, workspace sizing, dispatch to the kernels, and the
// device error word.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"
#include "ptx.cuh"
#include "wise.h"

// The one piece of library state: a per-device word that kernels OR error
// bits into (bounded-wait timeouts, malformed supports).
__device__ uint32_t g_wise_error_word;

namespace wise {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxBlocks = 1024;
constexpr size_t kL2GroupBytes = 32ull << 20;  // K/V bytes kept hot per group of heads

std::mutex g_mu;
uint32_t* g_err_ptr[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

// Device address of g_wise_error_word on the current device (looked up once).
uint32_t* error_word() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wise_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_err_ptr[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

// 2D view [rows = batch*heads*seq_len, head_dim] of a bf16 tensor; boxes of
// `box_rows` rows and 64 (128B swizzle) or 32 (64B swizzle, head_dim 96)
// columns.
int encode_map(CUtensorMap* m, const void* ptr, int64_t rows, int d, int box_rows) {
  auto enc = encoder();
  if (!enc) return WISE_ERR_CUDA;
  const int ch = (d == 96) ? 32 : 64;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {(cuuint32_t)ch, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, ch == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? WISE_OK : WISE_ERR_UNSUPPORTED;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_desc(const wise_attn_desc* d) {
  if (!d) return WISE_ERR_INVALID_ARGUMENT;
  if (d->batch < 1 || d->heads < 1 || d->seq_len < 1 || d->block < 1) return WISE_ERR_INVALID_ARGUMENT;
  if (d->kv_heads < 0 || (d->kv_heads > 0 && d->heads % d->kv_heads != 0)) return WISE_ERR_INVALID_ARGUMENT;
  if (d->out_dtype != WISE_BF16 && d->out_dtype != WISE_F32) return WISE_ERR_INVALID_ARGUMENT;
  if (!(d->softmax_scale >= 0.f) || isinf(d->softmax_scale)) return WISE_ERR_INVALID_ARGUMENT;
  if (d->seq_len % d->block != 0) return WISE_ERR_INVALID_ARGUMENT;
  if (d->head_dim != 64 && d->head_dim != 96 && d->head_dim != 128) return WISE_ERR_UNSUPPORTED;
  if (d->block != 32 && d->block != 64 && d->block != 128) return WISE_ERR_UNSUPPORTED;
  if (d->seq_len / d->block > kMaxBlocks) return WISE_ERR_UNSUPPORTED;
  const int64_t rows = (int64_t)d->batch * d->heads * d->seq_len;
  if (rows + 256 > INT32_MAX) return WISE_ERR_UNSUPPORTED;
  return WISE_OK;
}

struct Shape {
  int64_t bh;
  int n, d, bn, nb, n_qtiles, group_heads;
  int heads, kv_heads;  // kv_heads divides heads (grouped-query attention)
  int64_t n_units;
};

Shape shape_of(const wise_attn_desc* d) {
  Shape s;
  s.bh = (int64_t)d->batch * d->heads;
  s.n = d->seq_len;
  s.d = d->head_dim;
  s.bn = d->block;
  s.nb = d->seq_len / d->block;
  s.n_qtiles = (d->seq_len + 127) / 128;
  s.heads = d->heads;
  s.kv_heads = d->kv_heads > 0 ? d->kv_heads : d->heads;
  // K/V bytes per query head (query heads that share a key/value head share it)
  const size_t kv_per_head = (size_t)2 * d->seq_len * d->head_dim * 2 * s.kv_heads / s.heads;
  int64_t g = (int64_t)(kL2GroupBytes / (kv_per_head > 0 ? kv_per_head : 1));
  if (g < 1) g = 1;
  if (g > s.bh) g = s.bh;
  s.group_heads = (int)g;
  s.n_units = s.bh * s.n_qtiles;
  return s;
}

size_t lam_bytes(const Shape& s) {
  const int64_t ept = 128 / s.bn;
  const int64_t per_bh = ept * (int64_t)s.n_qtiles * (s.n_qtiles + 1) / 2;
  return (size_t)(s.bh * per_bh * 128 * sizeof(float));
}

int64_t fixed_point(double x);

// One step of a selection window fused into discovery (see AttnParams).
struct FusedSelect {
  uint32_t* bits;
  int32_t* counts;
  int64_t target_fx, tol_fx;
  int32_t nwords, first, last;
  uint32_t flags;
};

int launch_attention(const wise_attn_desc* desc, const void* q, const void* k, const void* v, void* o, float* lse,
                     float* mass, void* ws, const int32_t* row_ptr, const int32_t* col_idx, int64_t col_cap,
                     const int32_t* tile_order, bool sparse, cudaStream_t stream,
                     const FusedSelect* fs = nullptr, const void* plan = nullptr) {
  const Shape s = shape_of(desc);
  uint32_t* err = error_word();
  if (!err) return WISE_ERR_CUDA;
  // Q, K, V, and K, V with 128-row boxes (consecutive gathered blocks; the
  // same maps as K, V for the other variants)
  CUtensorMap maps[5];
  const int64_t rows = s.bh * s.n;
  const int64_t kv_rows = (int64_t)desc->batch * s.kv_heads * s.n;
  // K/V boxes: one key block (64 or 128 rows); blocks of 32 use 128-row
  // boxes in discovery and one 32-row box per gathered block in sparse steps
  const int kv_box = (s.bn == 32) ? (sparse ? 32 : 128) : s.bn;
  int st = encode_map(&maps[0], q, rows, s.d, 128);
  if (st == WISE_OK) st = encode_map(&maps[1], k, kv_rows, s.d, kv_box);
  if (st == WISE_OK) st = encode_map(&maps[2], v, kv_rows, s.d, kv_box);
  if (st == WISE_OK) st = encode_map(&maps[3], k, kv_rows, s.d, kv_box == 32 ? 128 : kv_box);
  if (st == WISE_OK) st = encode_map(&maps[4], v, kv_rows, s.d, kv_box == 32 ? 128 : kv_box);
  if (st != WISE_OK) return st;
  AttnParams p;
  memset(&p, 0, sizeof(p));
  p.bh_count = (int32_t)s.bh;
  p.heads = s.heads;
  p.kv_group = s.heads / s.kv_heads;
  p.n = s.n;
  p.nb = s.nb;
  p.n_qtiles = s.n_qtiles;
  p.group_heads = s.group_heads;
  const float scale = desc->softmax_scale > 0.f ? desc->softmax_scale : 1.0f / sqrtf((float)s.d);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out_f32 = desc->out_dtype == WISE_F32;
  p.o = o;
  p.lse = lse;
  p.mass = mass;
  p.lam = static_cast<float*>(ws);
  p.row_ptr = row_ptr;
  p.col_idx = col_idx;
  p.col_cap = col_cap;
  p.tile_order = tile_order;
  p.n_units = s.n_units;
  p.err = err;
  if (plan) {
    p.plan_counts = static_cast<const int32_t*>(plan);
    p.plan_entries = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(plan) +
                                                        plan_counts_bytes(s.n_units));
  }
  if (fs) {
    p.sel_bits = fs->bits;
    p.sel_counts = fs->counts;
    p.sel_target_fx = fs->target_fx;
    p.sel_tol_fx = fs->tol_fx;
    p.sel_nwords = fs->nwords;
    p.sel_first = fs->first;
    p.sel_last = fs->last;
    p.sel_flags = fs->flags;
  }
  // The launch's work-counter ticket, one sequence shared by every attention
  // kernel (launches on different streams may run at the same time, so each
  // must hold its own slot); bit 31 marks a launch recorded into a CUDA graph
  static std::atomic<uint32_t> eager_tickets{0}, graph_tickets{0};
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return WISE_ERR_CUDA;
  p.sched_slot = (cap == cudaStreamCaptureStatusActive) ? (0x80000000u | (graph_tickets.fetch_add(1u) & 0x7fffffffu))
                                                        : (eager_tickets.fetch_add(1u) & 0x7fffffffu);
  cudaError_t e;
  switch (s.d) {
    case 64: e = launch_attn_d64(s.bn, sparse, maps, p, stream); break;
    case 96: e = launch_attn_d96(s.bn, sparse, maps, p, stream); break;
    default: e = launch_attn_d128(s.bn, sparse, maps, p, stream); break;
  }
  return e == cudaSuccess ? WISE_OK : WISE_ERR_CUDA;
}

int64_t fixed_point(double x) { return llrint(x * 4503599627370496.0); }  // x * 2^52, nearest even

// Fixed scratch of wise_select_support_noalloc: the per-row support bitmasks
// and counts that wise_select_support keeps in its caller's workspace. It is
// part of the library image, so every GPU that loads the library holds these
// bytes until the process exits; calls share it.
constexpr size_t kNoAllocScratchBytes = 2u << 20;
static __device__ __align__(256) uint8_t g_select_scratch[kNoAllocScratchBytes];
uint8_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_select_scratch on the current device. The name is only
// a host-side stand-in, so the address is looked up once per device (with that
// device current) and cached.
uint8_t* select_scratch() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
  }
  return g_scratch_ptr[dev];
}

// Self-check of the bounded wait: one thread waits on an mbarrier that
// nothing arrives on, through the same wait routine as the attention kernels
// but with a 20 ms limit. The wait expires, kErrTimeout is recorded, and the
// kernel returns (no copy or MMA is in flight, so nothing needs draining).
constexpr uint64_t kSelfCheckWaitNs = 20000000ull;
__global__ void wait_expiry_kernel(uint32_t* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  mbar_wait<6, kSelfCheckWaitNs>(&bar, 0, &abort_flag, err);
}

}  // namespace
}  // namespace wise

using namespace wise;

extern "C" {

int wise_abi_version(void) { return WISE_ABI_VERSION; }

const char* wise_status_str(int status) {
  switch (status) {
    case WISE_OK: return "ok";
    case WISE_ERR_INVALID_ARGUMENT: return "invalid argument";
    case WISE_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case WISE_ERR_ALIGNMENT: return "tensor base address not 16-byte aligned";
    case WISE_ERR_WORKSPACE: return "workspace missing or too small";
    case WISE_ERR_BAD_SUPPORT: return "malformed support (CSR) or schedule";
    case WISE_ERR_CUDA: return "CUDA error";
    case WISE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

size_t wise_attn_discover_workspace(const wise_attn_desc* desc) {
  if (check_desc(desc) != WISE_OK) return 0;
  return lam_bytes(shape_of(desc));
}

int64_t wise_schedule_units(const wise_attn_desc* desc) {
  if (check_desc(desc) != WISE_OK) return 0;
  return shape_of(desc).n_units;
}

int64_t wise_support_capacity(const wise_attn_desc* desc) {
  if (check_desc(desc) != WISE_OK) return 0;
  const Shape s = shape_of(desc);
  return s.bh * (int64_t)s.nb * (s.nb + 1) / 2;
}

size_t wise_select_workspace(const wise_attn_desc* desc, int32_t window) {
  if (check_desc(desc) != WISE_OK || window < 1 || window > 8) return 0;
  const Shape s = shape_of(desc);
  const int64_t rows = s.bh * s.nb;
  const int64_t words = (s.nb + 31) / 32;
  return (size_t)(select_lookback_offset(rows, words) + select_lookback_bytes(rows) + 256);
}

int wise_attn_discover(const wise_attn_desc* desc, const void* q, const void* k, const void* v, void* o, float* lse,
                       float* block_mass, void* workspace, size_t workspace_bytes, wise_stream_t stream) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (!q || !k || !v || !o) return WISE_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return WISE_ERR_ALIGNMENT;
  if ((lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) || (block_mass && (reinterpret_cast<uintptr_t>(block_mass) & 3u)))
    return WISE_ERR_ALIGNMENT;
  if (block_mass) {
    const size_t need = lam_bytes(shape_of(desc));
    if (!workspace || workspace_bytes < need) return WISE_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return WISE_ERR_ALIGNMENT;
  }
  return launch_attention(desc, q, k, v, o, lse, block_mass, workspace, nullptr, nullptr, 0, nullptr, false,
                          reinterpret_cast<cudaStream_t>(stream));
}

int wise_attn_sparse(const wise_attn_desc* desc, const void* q, const void* k, const void* v, const int32_t* row_ptr,
                     const int32_t* col_idx, int64_t col_capacity, const int32_t* tile_order, void* o, float* lse,
                     wise_stream_t stream) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (!q || !k || !v || !o || !row_ptr || !col_idx || col_capacity < 0) return WISE_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return WISE_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(row_ptr) & 3u) || (reinterpret_cast<uintptr_t>(col_idx) & 3u) ||
      (tile_order && (reinterpret_cast<uintptr_t>(tile_order) & 3u)) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return WISE_ERR_ALIGNMENT;
  return launch_attention(desc, q, k, v, o, lse, nullptr, nullptr, row_ptr, col_idx, col_capacity, tile_order, true,
                          reinterpret_cast<cudaStream_t>(stream));
}

int wise_attn_sparse_planned(const wise_attn_desc* desc, const void* q, const void* k, const void* v,
                             const int32_t* row_ptr, const int32_t* col_idx, int64_t col_capacity,
                             const int32_t* tile_order, const void* plan, void* o, float* lse,
                             wise_stream_t stream) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (!q || !k || !v || !o || !row_ptr || !col_idx || col_capacity < 0) return WISE_ERR_INVALID_ARGUMENT;
  if (plan && desc->block != 32) return WISE_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (plan && !aligned16(plan)))
    return WISE_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(row_ptr) & 3u) || (reinterpret_cast<uintptr_t>(col_idx) & 3u) ||
      (tile_order && (reinterpret_cast<uintptr_t>(tile_order) & 3u)) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return WISE_ERR_ALIGNMENT;
  return launch_attention(desc, q, k, v, o, lse, nullptr, nullptr, row_ptr, col_idx, col_capacity, tile_order, true,
                          reinterpret_cast<cudaStream_t>(stream), nullptr, plan);
}

size_t wise_gather_plan_bytes(const wise_attn_desc* desc) {
  if (check_desc(desc) != WISE_OK || desc->block != 32) return 0;
  const Shape s = shape_of(desc);
  return (size_t)plan_bytes(s.bh, s.n_qtiles);
}

int wise_gather_plan(const wise_attn_desc* desc, const int32_t* row_ptr, const int32_t* col_idx,
                     int64_t col_capacity, void* plan, size_t plan_bytes_given, wise_stream_t stream) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (desc->block != 32) return WISE_ERR_UNSUPPORTED;
  if (!row_ptr || !col_idx || !plan || col_capacity < 0) return WISE_ERR_INVALID_ARGUMENT;
  if (plan_bytes_given < wise_gather_plan_bytes(desc)) return WISE_ERR_WORKSPACE;
  if (!aligned16(plan) || (reinterpret_cast<uintptr_t>(row_ptr) & 3u) || (reinterpret_cast<uintptr_t>(col_idx) & 3u))
    return WISE_ERR_ALIGNMENT;
  uint32_t* err = error_word();
  if (!err) return WISE_ERR_CUDA;
  const Shape s = shape_of(desc);
  GatherPlanLaunch g;
  g.row_ptr = row_ptr;
  g.col_idx = col_idx;
  g.col_cap = col_capacity;
  g.bh_count = (int32_t)s.bh;
  g.nb = s.nb;
  g.n_qtiles = s.n_qtiles;
  g.counts = static_cast<int32_t*>(plan);
  g.entries = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(plan) + plan_counts_bytes(s.n_units));
  g.err = err;
  return launch_gather_plan(g, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? WISE_OK : WISE_ERR_CUDA;
}

int wise_select_support(const wise_attn_desc* desc, const float* block_mass, int32_t window, double eta,
                        uint32_t flags, int32_t* row_ptr, int32_t* col_idx, int64_t col_capacity, int32_t* tile_order,
                        int32_t* nnz, void* workspace, size_t workspace_bytes, wise_stream_t stream) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (!block_mass || !row_ptr || !col_idx) return WISE_ERR_INVALID_ARGUMENT;
  if (window < 1 || window > 8 || !(eta > 0.0 && eta < 1.0) || (flags & ~3u)) return WISE_ERR_INVALID_ARGUMENT;
  if (col_capacity < wise_support_capacity(desc)) return WISE_ERR_BAD_SUPPORT;
  const size_t need = wise_select_workspace(desc, window);
  if (!workspace || workspace_bytes < need) return WISE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) || (reinterpret_cast<uintptr_t>(block_mass) & 3u) ||
      (reinterpret_cast<uintptr_t>(row_ptr) & 3u) || (reinterpret_cast<uintptr_t>(col_idx) & 3u))
    return WISE_ERR_ALIGNMENT;
  uint32_t* err = error_word();
  if (!err) return WISE_ERR_CUDA;
  const Shape s = shape_of(desc);
  const int64_t rows = s.bh * s.nb;
  const int64_t words = (s.nb + 31) / 32;
  SelectLaunch sl;
  memset(&sl, 0, sizeof(sl));
  sl.mass = block_mass;
  sl.window = window;
  sl.bh_count = (int32_t)s.bh;
  sl.nb = s.nb;
  sl.target_fx = fixed_point(eta);
  sl.tol_fx = fixed_point(1e-6);
  sl.flags = flags;
  sl.bits = static_cast<uint32_t*>(workspace);
  sl.counts = reinterpret_cast<int32_t*>(static_cast<uint32_t*>(workspace) + rows * words);
  sl.row_ptr = row_ptr;
  sl.col_idx = col_idx;
  sl.col_cap = col_capacity;
  sl.nnz = nnz;
  sl.tile_order = tile_order;
  sl.units_per_bh = s.n_qtiles;
  sl.qb_per_unit = 128 / s.bn;
  sl.err = err;
  cudaError_t e = launch_select(sl, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WISE_OK : WISE_ERR_CUDA;
}

// Largest nb of the fused selection (eight 32-block rounds per row in the
// epilogue warps' registers).
constexpr int kFusedSelectMaxBlocks = 256;

int wise_attn_discover_select(const wise_attn_desc* desc, const void* q, const void* k, const void* v, void* o,
                              float* lse, float* block_mass, void* workspace, size_t workspace_bytes, double eta,
                              uint32_t flags, int32_t step, int32_t window, void* select_state,
                              size_t select_state_bytes, wise_stream_t stream) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (!q || !k || !v || !o || !block_mass || !select_state) return WISE_ERR_INVALID_ARGUMENT;
  if (window < 1 || window > 8 || step < 0 || step >= window || !(eta > 0.0 && eta < 1.0) || (flags & ~3u))
    return WISE_ERR_INVALID_ARGUMENT;
  const Shape s = shape_of(desc);
  if (s.nb > kFusedSelectMaxBlocks) return WISE_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return WISE_ERR_ALIGNMENT;
  if ((lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) || (reinterpret_cast<uintptr_t>(block_mass) & 3u) ||
      (reinterpret_cast<uintptr_t>(select_state) & 15u))
    return WISE_ERR_ALIGNMENT;
  const size_t need = lam_bytes(s);
  if (!workspace || workspace_bytes < need) return WISE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return WISE_ERR_ALIGNMENT;
  if (select_state_bytes < wise_select_workspace(desc, window)) return WISE_ERR_WORKSPACE;
  const int64_t rows = s.bh * s.nb;
  const int64_t words = (s.nb + 31) / 32;
  FusedSelect fs;
  fs.bits = static_cast<uint32_t*>(select_state);
  fs.counts = reinterpret_cast<int32_t*>(static_cast<uint32_t*>(select_state) + rows * words);
  fs.target_fx = fixed_point(eta);
  fs.tol_fx = fixed_point(1e-6);
  fs.nwords = (int32_t)words;
  fs.first = step == 0;
  fs.last = step == window - 1;
  fs.flags = flags;
  return launch_attention(desc, q, k, v, o, lse, block_mass, workspace, nullptr, nullptr, 0, nullptr, false,
                          reinterpret_cast<cudaStream_t>(stream), &fs);
}

int wise_select_finalize(const wise_attn_desc* desc, const void* select_state, size_t select_state_bytes,
                         int32_t* row_ptr, int32_t* col_idx, int64_t col_capacity, int32_t* tile_order, int32_t* nnz,
                         wise_stream_t stream) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (!select_state || !row_ptr || !col_idx) return WISE_ERR_INVALID_ARGUMENT;
  if (col_capacity < wise_support_capacity(desc)) return WISE_ERR_BAD_SUPPORT;
  if (select_state_bytes < wise_select_workspace(desc, 1)) return WISE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(select_state) & 15u) || (reinterpret_cast<uintptr_t>(row_ptr) & 3u) ||
      (reinterpret_cast<uintptr_t>(col_idx) & 3u) || (tile_order && (reinterpret_cast<uintptr_t>(tile_order) & 3u)) ||
      (nnz && (reinterpret_cast<uintptr_t>(nnz) & 3u)))
    return WISE_ERR_ALIGNMENT;
  uint32_t* err = error_word();
  if (!err) return WISE_ERR_CUDA;
  const Shape s = shape_of(desc);
  const int64_t rows = s.bh * s.nb;
  const int64_t words = (s.nb + 31) / 32;
  SelectLaunch sl;
  memset(&sl, 0, sizeof(sl));
  sl.window = 1;
  sl.bh_count = (int32_t)s.bh;
  sl.nb = s.nb;
  sl.bits = const_cast<uint32_t*>(static_cast<const uint32_t*>(select_state));
  sl.counts = reinterpret_cast<int32_t*>(sl.bits + rows * words);
  sl.row_ptr = row_ptr;
  sl.col_idx = col_idx;
  sl.col_cap = col_capacity;
  sl.nnz = nnz;
  sl.tile_order = tile_order;
  sl.units_per_bh = s.n_qtiles;
  sl.qb_per_unit = 128 / s.bn;
  sl.finalize_only = 1;
  sl.err = err;
  cudaError_t e = launch_select(sl, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WISE_OK : WISE_ERR_CUDA;
}

int wise_select_support_noalloc(const wise_attn_desc* desc, const float* block_mass, int32_t window, double eta,
                                uint32_t flags, int32_t* row_ptr, int32_t* col_idx, int64_t col_capacity,
                                int32_t* tile_order, int32_t* nnz, wise_stream_t stream) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (!block_mass || !row_ptr || !col_idx) return WISE_ERR_INVALID_ARGUMENT;
  if (window < 1 || window > 8 || !(eta > 0.0 && eta < 1.0) || (flags & ~3u)) return WISE_ERR_INVALID_ARGUMENT;
  if (col_capacity < wise_support_capacity(desc)) return WISE_ERR_BAD_SUPPORT;
  if (wise_select_workspace(desc, window) > kNoAllocScratchBytes) return WISE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(block_mass) & 3u) || (reinterpret_cast<uintptr_t>(row_ptr) & 3u) ||
      (reinterpret_cast<uintptr_t>(col_idx) & 3u))
    return WISE_ERR_ALIGNMENT;
  uint32_t* err = error_word();
  uint8_t* scratch = select_scratch();
  if (!err || !scratch) return WISE_ERR_CUDA;
  const Shape s = shape_of(desc);
  const int64_t rows = s.bh * s.nb;
  const int64_t words = (s.nb + 31) / 32;
  SelectLaunch sl;
  memset(&sl, 0, sizeof(sl));
  sl.mass = block_mass;
  sl.window = window;
  sl.bh_count = (int32_t)s.bh;
  sl.nb = s.nb;
  sl.target_fx = fixed_point(eta);
  sl.tol_fx = fixed_point(1e-6);
  sl.flags = flags;
  // every row writes its bitmask words and its count before they are read,
  // so the shared scratch needs no clearing between calls
  sl.bits = reinterpret_cast<uint32_t*>(scratch);
  sl.counts = reinterpret_cast<int32_t*>(scratch + rows * words * 4);
  sl.row_ptr = row_ptr;
  sl.col_idx = col_idx;
  sl.col_cap = col_capacity;
  sl.nnz = nnz;
  sl.tile_order = tile_order;
  sl.units_per_bh = s.n_qtiles;
  sl.qb_per_unit = 128 / s.bn;
  sl.err = err;
  cudaError_t e = launch_select(sl, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WISE_OK : WISE_ERR_CUDA;
}

int wise_support_retained_mass(const wise_attn_desc* desc, const float* block_mass, const int32_t* row_ptr,
                                const int32_t* col_idx, int64_t col_capacity, float* row_retained, double* batch_mean,
                                wise_stream_t stream) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (!block_mass || !row_ptr || !col_idx || !row_retained || col_capacity < 0) return WISE_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(block_mass) & 3u) || (reinterpret_cast<uintptr_t>(row_ptr) & 3u) ||
      (reinterpret_cast<uintptr_t>(col_idx) & 3u) || (reinterpret_cast<uintptr_t>(row_retained) & 3u) ||
      (batch_mean && (reinterpret_cast<uintptr_t>(batch_mean) & 7u)))
    return WISE_ERR_ALIGNMENT;
  uint32_t* err = error_word();
  if (!err) return WISE_ERR_CUDA;
  const Shape s = shape_of(desc);
  DiagLaunch d;
  memset(&d, 0, sizeof(d));
  d.rows = s.bh * s.nb;
  d.nb = s.nb;
  d.batch = desc->batch;
  d.col_cap = col_capacity;
  d.mass = block_mass;
  d.row_ptr_a = row_ptr;
  d.col_idx_a = col_idx;
  d.row_value = row_retained;
  d.batch_value = batch_mean;
  d.err = err;
  return launch_retained_mass(d, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? WISE_OK : WISE_ERR_CUDA;
}

int wise_support_jaccard(const wise_attn_desc* desc, const int32_t* row_ptr_a, const int32_t* col_idx_a,
                         int64_t col_capacity_a, const int32_t* row_ptr_b, const int32_t* col_idx_b,
                         int64_t col_capacity_b, int32_t* row_counts, int64_t* batch_counts, double* batch_jaccard,
                         wise_stream_t stream) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (!row_ptr_a || !col_idx_a || !row_ptr_b || !col_idx_b || !row_counts || col_capacity_a < 0 ||
      col_capacity_b < 0)
    return WISE_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(row_ptr_a) & 3u) || (reinterpret_cast<uintptr_t>(col_idx_a) & 3u) ||
      (reinterpret_cast<uintptr_t>(row_ptr_b) & 3u) || (reinterpret_cast<uintptr_t>(col_idx_b) & 3u) ||
      (reinterpret_cast<uintptr_t>(row_counts) & 3u) || (batch_counts && (reinterpret_cast<uintptr_t>(batch_counts) & 7u)) ||
      (batch_jaccard && (reinterpret_cast<uintptr_t>(batch_jaccard) & 7u)))
    return WISE_ERR_ALIGNMENT;
  uint32_t* err = error_word();
  if (!err) return WISE_ERR_CUDA;
  const Shape s = shape_of(desc);
  DiagLaunch d;
  memset(&d, 0, sizeof(d));
  d.rows = s.bh * s.nb;
  d.nb = s.nb;
  d.batch = desc->batch;
  d.col_cap = col_capacity_a;
  d.col_cap_b = col_capacity_b;
  d.row_ptr_a = row_ptr_a;
  d.col_idx_a = col_idx_a;
  d.row_ptr_b = row_ptr_b;
  d.col_idx_b = col_idx_b;
  d.row_counts = row_counts;
  d.batch_counts = reinterpret_cast<long long*>(batch_counts);
  d.batch_value = batch_jaccard;
  d.err = err;
  return launch_jaccard(d, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? WISE_OK : WISE_ERR_CUDA;
}

int wise_select_control(const wise_attn_desc* desc, const float* block_mass, int32_t mode,
                        const int32_t* ref_row_ptr, const int32_t* ref_col_idx, int64_t ref_capacity, uint32_t flags,
                        int32_t* row_ptr, int32_t* col_idx, int64_t col_capacity, int32_t* tile_order, int32_t* nnz,
                        void* workspace, size_t workspace_bytes, wise_stream_t stream) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (mode != WISE_CONTROL_MASS_MATCHED && mode != WISE_CONTROL_SIZE_MATCHED) return WISE_ERR_INVALID_ARGUMENT;
  if (!block_mass || !ref_row_ptr || !ref_col_idx || !row_ptr || !col_idx || ref_capacity < 0 || (flags & ~3u))
    return WISE_ERR_INVALID_ARGUMENT;
  if (col_capacity < wise_support_capacity(desc)) return WISE_ERR_BAD_SUPPORT;
  const size_t need = wise_select_workspace(desc, 1);
  if (!workspace || workspace_bytes < need) return WISE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) || (reinterpret_cast<uintptr_t>(block_mass) & 3u) ||
      (reinterpret_cast<uintptr_t>(row_ptr) & 3u) || (reinterpret_cast<uintptr_t>(col_idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(ref_row_ptr) & 3u) || (reinterpret_cast<uintptr_t>(ref_col_idx) & 3u))
    return WISE_ERR_ALIGNMENT;
  uint32_t* err = error_word();
  if (!err) return WISE_ERR_CUDA;
  const Shape s = shape_of(desc);
  const int64_t rows = s.bh * s.nb;
  const int64_t words = (s.nb + 31) / 32;
  SelectLaunch sl;
  memset(&sl, 0, sizeof(sl));
  sl.mass = block_mass;
  sl.window = 1;
  sl.bh_count = (int32_t)s.bh;
  sl.nb = s.nb;
  sl.target_fx = 0;
  sl.tol_fx = fixed_point(1e-6);
  sl.flags = flags;
  sl.bits = static_cast<uint32_t*>(workspace);
  sl.counts = reinterpret_cast<int32_t*>(static_cast<uint32_t*>(workspace) + rows * words);
  sl.row_ptr = row_ptr;
  sl.col_idx = col_idx;
  sl.col_cap = col_capacity;
  sl.nnz = nnz;
  sl.tile_order = tile_order;
  sl.units_per_bh = s.n_qtiles;
  sl.qb_per_unit = 128 / s.bn;
  sl.mode = mode;
  sl.ref_row_ptr = ref_row_ptr;
  sl.ref_col_idx = ref_col_idx;
  sl.ref_cap = ref_capacity;
  sl.err = err;
  cudaError_t e = launch_select(sl, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WISE_OK : WISE_ERR_CUDA;
}

int wise_validate_support(const wise_attn_desc* desc, const int32_t* row_ptr, const int32_t* col_idx,
                          uint32_t flags) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (!row_ptr || (!col_idx && row_ptr[0] != 0)) return WISE_ERR_INVALID_ARGUMENT;
  const Shape s = shape_of(desc);
  const int64_t rows = s.bh * s.nb;
  if (row_ptr[0] != 0) return WISE_ERR_BAD_SUPPORT;
  for (int64_t r = 0; r < rows; ++r) {
    const int32_t a = row_ptr[r], b = row_ptr[r + 1];
    if (b < a) return WISE_ERR_BAD_SUPPORT;
    const int q = (int)(r % s.nb);
    int prev = -1;
    bool has0 = false, hasq = false;
    for (int32_t j = a; j < b; ++j) {
      const int32_t c = col_idx[j];
      if (c <= prev || c > q) return WISE_ERR_BAD_SUPPORT;
      has0 |= (c == 0);
      hasq |= (c == q);
      prev = c;
    }
    if (((flags & WISE_SUPPORT_SINK) && !has0) || ((flags & WISE_SUPPORT_DIAG) && !hasq)) return WISE_ERR_BAD_SUPPORT;
  }
  return WISE_OK;
}

int wise_validate_schedule(const wise_attn_desc* desc, const int32_t* tile_order) {
  int st = check_desc(desc);
  if (st != WISE_OK) return st;
  if (!tile_order) return WISE_ERR_INVALID_ARGUMENT;
  const int64_t units = shape_of(desc).n_units;
  std::vector<uint8_t> seen((size_t)units, 0);
  for (int64_t x = 0; x < units; ++x) {
    const int32_t u = tile_order[x];
    if (u < 0 || u >= units || seen[(size_t)u]) return WISE_ERR_BAD_SUPPORT;
    seen[(size_t)u] = 1;
  }
  return WISE_OK;
}

int wise_wait_expiry_check(wise_stream_t stream) {
  uint32_t* err = error_word();
  if (!err) return WISE_ERR_CUDA;
  wait_expiry_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err);
  return cudaGetLastError() == cudaSuccess ? WISE_OK : WISE_ERR_CUDA;
}

int wise_device_status(wise_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return WISE_ERR_CUDA;
  uint32_t word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_wise_error_word, sizeof(word)) != cudaSuccess) return WISE_ERR_CUDA;
  if (word && cudaMemcpyToSymbol(g_wise_error_word, &zero, sizeof(zero)) != cudaSuccess) return WISE_ERR_CUDA;
  if (word & kErrTimeout) return WISE_ERR_DEVICE_TIMEOUT;
  if (word & kErrInternal) return WISE_ERR_CUDA;
  if (word & kErrBadSupport) return WISE_ERR_BAD_SUPPORT;
  return WISE_OK;
}

}  // extern "C"
