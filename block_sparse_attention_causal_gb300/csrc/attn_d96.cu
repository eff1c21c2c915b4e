// Instantiations of the tcgen05 attention kernel for head_dim = 96.
#include "attn_kernel.cuh"

namespace wise {
namespace {

template <int D, int BN, bool SPARSE>
cudaError_t launch_one(const CUtensorMap* m, const AttnParams& p, cudaStream_t st) {
  using C = AttnCfg<D, BN>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(wise_attn_kernel<D, BN, SPARSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  wise_attn_kernel<D, BN, SPARSE><<<(unsigned)p.n_units, C::THREADS, C::SMEM_BYTES, st>>>(m[0], m[1], m[2], p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_d96(int block, bool sparse, const CUtensorMap* maps, const AttnParams& p, cudaStream_t st) {
  if (block == 128) return sparse ? launch_one<96, 128, true>(maps, p, st) : launch_one<96, 128, false>(maps, p, st);
  return sparse ? launch_one<96, 64, true>(maps, p, st) : launch_one<96, 64, false>(maps, p, st);
}

}  // namespace wise
