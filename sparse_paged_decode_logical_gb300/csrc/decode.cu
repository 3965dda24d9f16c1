// Split-K sparse decode attention: the plain kernel's instances, the cluster
// sizes they can be launched with, and the launch entry (the kernel itself is
// in decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace spd {
namespace {

// [deep][dtype][d == 128][log2 G]: co-schedulable cluster size
int g_max_cluster[2][2][2][4];

template <typename T, int D, int G, bool kDeep>
cudaError_t prep_one(int *max_cluster) {
  cudaError_t e = set_smem_attrs<T, D, G, false, false, kDeep>();
  if (e != cudaSuccess) return e;
  int cs = 8;  // portable cluster size
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(16);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<D, G, false, kDeep>::kAlloc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 16;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int q = 0;
  if (cudaOccupancyMaxPotentialClusterSize(&q, decode_tiles_kernel<T, D, G, false, false, kDeep>,
                                          &cfg) ==
          cudaSuccess &&
      q >= 1)
    cs = q;
  (void)cudaGetLastError();
  *max_cluster = cs;
  return cudaSuccess;
}

template <typename T, int D, bool kDeep>
cudaError_t prep_g(int dt) {
  cudaError_t e;
  int *mc = g_max_cluster[kDeep][dt][D == 128];
  if ((e = prep_one<T, D, 1, kDeep>(&mc[0])) != cudaSuccess) return e;
  if ((e = prep_one<T, D, 2, kDeep>(&mc[1])) != cudaSuccess) return e;
  if ((e = prep_one<T, D, 4, kDeep>(&mc[2])) != cudaSuccess) return e;
  return prep_one<T, D, 8, kDeep>(&mc[3]);
}

template <bool kDeep>
cudaError_t prep_shape() {
  cudaError_t e;
  if ((e = prep_g<__half, 64, kDeep>(0)) != cudaSuccess) return e;
  if ((e = prep_g<__half, 128, kDeep>(0)) != cudaSuccess) return e;
  if ((e = prep_g<__nv_bfloat16, 64, kDeep>(1)) != cudaSuccess) return e;
  return prep_g<__nv_bfloat16, 128, kDeep>(1);
}

}  // namespace

cudaError_t prepare_decode_kernels() {
  cudaError_t e;
  if ((e = prep_shape<false>()) != cudaSuccess) return e;
  if ((e = prep_shape<true>()) != cudaSuccess) return e;
  // the mass-exporting and fp8 instances: same block; their cluster sizes are
  // taken to be the plain kernel's (the fp8 ones need no more shared memory)
  if ((e = prepare_decode_mass_kernels()) != cudaSuccess) return e;
  if ((e = prepare_decode_reuse_kernels()) != cudaSuccess) return e;
  return prepare_decode_fp8_kernels();
}

// Largest power-of-two cluster (<= 16) the decode kernel can be launched with.
int decode_max_cluster(int dtype, int d, int G, bool deep) {
  const int gi = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  const int cs = g_max_cluster[deep ? 1 : 0][dtype ? 1 : 0][d == 128][gi];
  int p2 = 1;
  while (p2 * 2 <= cs && p2 < 16) p2 *= 2;
  return p2;
}

int decode_max_tiles_per_cta() { return kMaxDesc; }

int decode_ring_stages(bool deep) { return deep ? Ring<false, true>::n : Ring<false>::n; }

cudaError_t launch_decode_tiles(const TileDecodeParams &p, int dtype, int d, int G,
                                cudaStream_t s, long long *n) {
  if (p.n_seqs == 0 || p.total_items == 0) return cudaSuccess;
  *n += 1;
  if (p.kv_fp8) return d == 128 ? launch_decode_tiles_fp8(p, dtype, G, s) : cudaErrorInvalidValue;
  if (p.page_part != nullptr) return launch_decode_tiles_mass(p, dtype, d, G, s);
  bool selects = false;  // does any unit of this launch select its pages?
  for (int i = 0; i < p.n_seqs && !selects; ++i) selects = p.seqs[i].topk_n > 0;
  if (!selects) return launch_decode_tiles_reuse(p, dtype, d, G, s);
  if (p.deep) return launch_variant<false, true>(p, dtype, d, G, s);
  return launch_variant<false>(p, dtype, d, G, s);
}

}  // namespace spd
