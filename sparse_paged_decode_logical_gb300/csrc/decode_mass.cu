// Split-K sparse decode attention, the instances that also export the
// per-page attention mass (kernel in decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace spd {

cudaError_t prepare_decode_mass_kernels() { return set_smem_attrs_all<true>(); }

cudaError_t launch_decode_tiles_mass(const TileDecodeParams &p, int dtype, int d, int G,
                                     cudaStream_t s) {
  return launch_variant<true>(p, dtype, d, G, s);
}

}  // namespace spd
