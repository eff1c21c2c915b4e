// Instantiations of the tcgen05 attention kernel for head_dim = 64.
#include <atomic>

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
  // persistent: one CTA per SM (the shared-memory footprint allows no more);
  // each launch takes the next work-counter slot
  static std::atomic<uint32_t> launches{0};
  AttnParams q = p;
  q.sched_slot = launches.fetch_add(1u) % kSchedSlots;
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
