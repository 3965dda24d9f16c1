// C ABI of the prefill-side block-sparse attention (declared in spd.h):
// argument checks, the workspace layout, and the three launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "prefill.h"
#include "spd.h"

namespace {

constexpr size_t kErrBytes = 256;  // device error word (4 ints), padded

struct PrefillLayout {
  int nb = 0, KB = 0, kblocks = 0, dense = 0, G = 0;
  size_t qbar = 0, kbar = 0, lists = 0, total = 0;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool valid_config(const spd_prefill_config *c) {
  if (!c) return false;
  if (c->num_kv_heads < 1 || c->num_q_heads < 1 || c->num_q_heads % c->num_kv_heads) return false;
  const int G = c->num_q_heads / c->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->dtype != SPD_F16 && c->dtype != SPD_BF16) return false;
  if (c->rank < 1 || c->rank > spd::kPrefillMaxRank) return false;
  if (c->block != spd::kPrefillBlock) return false;
  if (c->token_budget < c->block || c->dense_below < 0) return false;
  return true;
}

spd_status layout(const spd_prefill_config *c, int L, PrefillLayout *z) {
  if (!valid_config(c) || L < 1) return SPD_ERR_INVALID_ARG;
  z->nb = (L + c->block - 1) / c->block;
  if (z->nb > spd::kPrefillMaxBlocks) return SPD_ERR_CAPACITY;
  z->G = c->num_q_heads / c->num_kv_heads;
  z->dense = L < c->dense_below ? 1 : 0;
  z->kblocks = c->token_budget / c->block;
  z->KB = z->dense ? z->nb : (z->kblocks < z->nb ? z->kblocks : z->nb);
  const size_t Hkv = (size_t)c->num_kv_heads, r = (size_t)c->rank, nb = (size_t)z->nb;
  size_t off = kErrBytes;
  z->qbar = off;
  off = round_up(off + Hkv * z->G * nb * r * 4, 256);
  z->kbar = off;
  off = round_up(off + Hkv * nb * r * 4, 256);
  z->lists = off;
  off = round_up(off + Hkv * nb * (size_t)z->KB * 4, 256);
  z->total = off;
  return SPD_OK;
}

bool aligned(const void *p, uintptr_t a) { return p && reinterpret_cast<uintptr_t>(p) % a == 0; }

spd_status enqueue(const spd_prefill_config *cfg, int seq_len, const PrefillLayout &z,
                   const void *q, const void *k, const void *v, const float *w_q,
                   const float *w_k, float *out, int *blocks, void *workspace, spd_stream stream);

// TMA map over Q, K or V ([L][heads][d], 16-bit) for the tensor-core
// attention: {64 channels, d / 64, heads, L}; one box is 64 tokens x 64
// channels of one head, stored in shared memory as 64 rows of 128 bytes with
// the 128-byte swizzle.  Tokens past L read as zero.
bool encode_map(CUtensorMap *m, const void *base, const spd_prefill_config *c, int heads, int L) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t d = (cuuint64_t)c->head_dim, h = (cuuint64_t)heads;
  cuuint64_t dims[4] = {64, d / 64, h, (cuuint64_t)L};
  cuuint64_t strides[3] = {128, d * 2, h * d * 2};
  cuuint32_t box[4] = {64, 1, 1, (cuuint32_t)spd::kPrefillBlock};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(m, c->dtype == SPD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                4, const_cast<void *>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

spd_status spd_prefill_sizes(const spd_prefill_config *cfg, int seq_len,
                             int *blocks_per_query_block, size_t *workspace_bytes) {
  PrefillLayout z;
  const spd_status s = layout(cfg, seq_len, &z);
  if (s != SPD_OK) return s;
  if (blocks_per_query_block) *blocks_per_query_block = z.KB;
  if (workspace_bytes) *workspace_bytes = z.total;
  return SPD_OK;
}

spd_status spd_prefill_block_sparse_attention(const spd_prefill_config *cfg, int seq_len,
                                              const void *q, const void *k, const void *v,
                                              const float *w_q, const float *w_k, float *out,
                                              int *blocks, void *workspace,
                                              size_t workspace_bytes, spd_stream stream) {
  PrefillLayout z;
  spd_status s = layout(cfg, seq_len, &z);
  if (s != SPD_OK) return s;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(w_q, 4) || !aligned(w_k, 4) || !aligned(workspace, 256) ||
      (blocks && !aligned(blocks, 4)))
    return SPD_ERR_INVALID_ARG;
  if (workspace_bytes < z.total) return SPD_ERR_CAPACITY;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, workspace) != cudaSuccess ||
      (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)) {
    (void)cudaGetLastError();
    return SPD_ERR_INVALID_ARG;
  }
  // the workspace's device for the launches, the caller's again afterwards
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return SPD_ERR_CUDA;
  if (prev != a.device && cudaSetDevice(a.device) != cudaSuccess) return SPD_ERR_CUDA;
  const spd_status r = enqueue(cfg, seq_len, z, q, k, v, w_q, w_k, out, blocks, workspace, stream);
  if (prev != a.device) (void)cudaSetDevice(prev);
  return r;
}

}  // extern "C"

namespace {

spd_status enqueue(const spd_prefill_config *cfg, int seq_len, const PrefillLayout &z,
                   const void *q, const void *k, const void *v, const float *w_q,
                   const float *w_k, float *out, int *blocks, void *workspace, spd_stream stream) {
  cudaStream_t st = (cudaStream_t)stream;
  char *ws = static_cast<char *>(workspace);
  if (cudaMemsetAsync(ws, 0, 16, st) != cudaSuccess) return SPD_ERR_CUDA;
  spd::PrefillParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.wq = w_q;
  p.wk = w_k;
  p.out = out;
  p.blocks_out = blocks;
  p.err = reinterpret_cast<int *>(ws);
  p.qbar = reinterpret_cast<float *>(ws + z.qbar);
  p.kbar = reinterpret_cast<float *>(ws + z.kbar);
  p.lists = reinterpret_cast<int *>(ws + z.lists);
  p.L = seq_len;
  p.Hq = cfg->num_q_heads;
  p.Hkv = cfg->num_kv_heads;
  p.G = z.G;
  p.r = cfg->rank;
  p.nb = z.nb;
  p.KB = z.KB;
  p.kblocks = z.kblocks;
  p.dense = z.dense;
  p.score_scale = (float)(1.0 / std::sqrt((double)cfg->head_dim));
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)cfg->head_dim));
  if (spd::prefill_tc_supported(p.G) &&
      (!encode_map(&p.tm_q, q, cfg, p.Hq, seq_len) || !encode_map(&p.tm_k, k, cfg, p.Hkv, seq_len) ||
       !encode_map(&p.tm_v, v, cfg, p.Hkv, seq_len)))
    return SPD_ERR_CUDA;
  return spd::launch_prefill(p, cfg->dtype, cfg->head_dim, st) == cudaSuccess ? SPD_OK
                                                                              : SPD_ERR_CUDA;
}

}  // namespace

extern "C" {

spd_status spd_prefill_check(const void *workspace, spd_stream stream) {
  if (!aligned(workspace, 256)) return SPD_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SPD_ERR_CUDA;
  int w[4] = {0, 0, 0, 0};
  if (cudaMemcpy(w, workspace, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPD_ERR_CUDA;
  return w[0] == 0 ? SPD_OK : SPD_ERR_DEVICE_CHECK;
}

}  // extern "C"
