// Split-K sparse decode attention over fp8 (E4M3) K/V storage: the instances
// for head_dim 128, plain and with the per-page attention mass (kernel in
// decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace spd {
namespace {

template <bool kMass>
cudaError_t set_fp8_attrs() {
  cudaError_t e;
  if ((e = set_smem_attrs<__half, 128, 1, kMass, true>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs<__half, 128, 2, kMass, true>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs<__half, 128, 4, kMass, true>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs<__half, 128, 8, kMass, true>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs<__nv_bfloat16, 128, 1, kMass, true>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs<__nv_bfloat16, 128, 2, kMass, true>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs<__nv_bfloat16, 128, 4, kMass, true>()) != cudaSuccess) return e;
  return set_smem_attrs<__nv_bfloat16, 128, 8, kMass, true>();
}

template <typename T, bool kMass>
cudaError_t launch_fp8_g(const TileDecodeParams &p, int G, cudaStream_t st) {
  switch (G) {
    case 1: return launch_one<T, 128, 1, kMass, true>(p, st);
    case 2: return launch_one<T, 128, 2, kMass, true>(p, st);
    case 4: return launch_one<T, 128, 4, kMass, true>(p, st);
    case 8: return launch_one<T, 128, 8, kMass, true>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t prepare_decode_fp8_kernels() {
  cudaError_t e = set_fp8_attrs<false>();
  return e != cudaSuccess ? e : set_fp8_attrs<true>();
}

cudaError_t launch_decode_tiles_fp8(const TileDecodeParams &p, int dtype, int G,
                                    cudaStream_t s) {
  const bool mass = p.page_part != nullptr;
  if (dtype == 0) return mass ? launch_fp8_g<__half, true>(p, G, s) : launch_fp8_g<__half, false>(p, G, s);
  return mass ? launch_fp8_g<__nv_bfloat16, true>(p, G, s)
              : launch_fp8_g<__nv_bfloat16, false>(p, G, s);
}

}  // namespace spd
