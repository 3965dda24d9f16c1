// Split-K sparse decode attention, the instances for launches in which no
// unit selects its pages (the steps that reuse a stored selection): the same
// kernel (decode_kernel.cuh) built without the fused top-k code.
#include "decode_kernel.cuh"

namespace spd {
namespace {

template <typename T, int D, bool kDeep>
cudaError_t prep_reuse_g() {
  cudaError_t e;
  if ((e = set_smem_attrs<T, D, 1, false, false, kDeep, true>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs<T, D, 2, false, false, kDeep, true>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs<T, D, 4, false, false, kDeep, true>()) != cudaSuccess) return e;
  return set_smem_attrs<T, D, 8, false, false, kDeep, true>();
}

template <bool kDeep>
cudaError_t prep_reuse_shape() {
  cudaError_t e;
  if ((e = prep_reuse_g<__half, 64, kDeep>()) != cudaSuccess) return e;
  if ((e = prep_reuse_g<__half, 128, kDeep>()) != cudaSuccess) return e;
  if ((e = prep_reuse_g<__nv_bfloat16, 64, kDeep>()) != cudaSuccess) return e;
  return prep_reuse_g<__nv_bfloat16, 128, kDeep>();
}

}  // namespace

cudaError_t prepare_decode_reuse_kernels() {
  cudaError_t e = prep_reuse_shape<false>();
  return e != cudaSuccess ? e : prep_reuse_shape<true>();
}

cudaError_t launch_decode_tiles_reuse(const TileDecodeParams &p, int dtype, int d, int G,
                                      cudaStream_t s) {
  if (p.deep) return launch_variant<false, true, true>(p, dtype, d, G, s);
  return launch_variant<false, false, true>(p, dtype, d, G, s);
}

}  // namespace spd
