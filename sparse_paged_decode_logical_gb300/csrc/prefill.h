// Internal interface of the prefill kernels (prefill.cu): block importance,
// block selection and block-sparse causal attention of one prompt.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spd {

constexpr int kPrefillBlock = 64;       // tokens per block (query and key)
constexpr int kPrefillMaxBlocks = 8192;  // blocks of a prompt (the top-k holds this many)
constexpr int kPrefillMaxRank = 64;

struct PrefillParams {
  // Q, K and V for the tensor-core attention: 4-D maps {64 channels, d / 64,
  // heads, L}, boxes of 64 channels x 64 tokens, 128-byte swizzle
  CUtensorMap tm_q, tm_k, tm_v;
  const void *q;         // [L][Hq][d]
  const void *k, *v;     // [L][Hkv][d]
  const float *wq, *wk;  // [Hkv][d][r]
  float *out;            // [L][Hq][d]
  int *blocks_out;       // [Hkv][nb][KB] or null
  float *qbar;           // [Hkv][G][nb][r] block means of q, projected
  float *kbar;           // [Hkv][nb][r]    block means of k, projected
  int *lists;            // [Hkv][nb][KB]   key blocks of every query block, ascending, -1 after
  int *err;              // device error word (4 ints)
  int L, Hq, Hkv, G, r, nb, KB;
  int kblocks;           // key blocks a query block keeps in sparse mode (own block included)
  int dense;             // 1: every causal block
  float score_scale;     // 1 / sqrt(d)
  float scale_log2;      // log2(e) / sqrt(d)
};

// dtype: 0 fp16, 1 bf16; d: 64 or 128.  Each returns cudaGetLastError().
// launch_prefill runs the block means, the selection and the attention, the
// latter on the 5th-generation tensor cores when prefill_tc_supported(G)
// (tm_q / tm_k / tm_v set), else with mma.sync tiles.
cudaError_t launch_prefill(const PrefillParams &p, int dtype, int d, cudaStream_t st);
bool prefill_tc_supported(int G);
cudaError_t launch_prefill_attn_tc(const PrefillParams &p, int dtype, int d, cudaStream_t st);

}  // namespace spd
