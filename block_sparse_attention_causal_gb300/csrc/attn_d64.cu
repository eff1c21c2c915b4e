// Instantiations of the tcgen05 attention kernel for head_dim = 64.
#include "attn_kernel.cuh"

namespace wise {
namespace {

template <int D, int BN, bool SPARSE>
cudaError_t launch_one(const CUtensorMap* m, const AttnParams& p, cudaStream_t st) {
  using C = AttnCfg<D, BN, SPARSE>;
  static bool configured[64] = {};
  static int sm_count[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(wise_attn_kernel<D, BN, SPARSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  // persistent: one CTA per SM (the shared-memory footprint allows no more).
  // p.sched_slot is the launch's ticket (launch_attention): eager launches
  // take the lower half of the work-counter slots, launches recorded into a
  // CUDA graph the upper half, so a graph's replay never shares a slot with
  // an eager launch running beside it
  AttnParams q = p;
  constexpr uint32_t half = kSchedSlots / 2;
  q.sched_slot = (p.sched_slot >> 31) ? half + (p.sched_slot & 0x7fffffffu) % half : p.sched_slot % half;
  const int64_t grid = p.n_units < sm_count[dev] ? p.n_units : sm_count[dev];
  wise_attn_kernel<D, BN, SPARSE><<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, st>>>(m[0], m[1], m[2], m[3], m[4], q);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_d64(int block, bool sparse, const CUtensorMap* maps, const AttnParams& p, cudaStream_t st) {
  if (block == 128) return sparse ? launch_one<64, 128, true>(maps, p, st) : launch_one<64, 128, false>(maps, p, st);
  // blocks of 32: discovery without masses is the dense kernel of blocks of 128
  if (block == 32)
    return sparse ? launch_one<64, 32, true>(maps, p, st)
                  : (p.mass ? launch_one<64, 32, false>(maps, p, st) : launch_one<64, 128, false>(maps, p, st));
  return sparse ? launch_one<64, 64, true>(maps, p, st) : launch_one<64, 64, false>(maps, p, st);
}

}  // namespace wise
