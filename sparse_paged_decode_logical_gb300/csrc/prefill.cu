// Prefill-side block-sparse attention for sm_103a ("LServe long-sequence LLM
// serving system", section 3.1: a low-rank estimate of every text block's
// importance, exact attention on the top blocks only, dense attention below
// 32K tokens).
//
// Three kernels per prompt, in stream order:
//   pool    one CTA per (block, kv head): the block's mean key and the mean
//           query of each of the G query heads, projected with W_k / W_q
//           (d x r).  The mean of the low-rank logits over a block pair is
//           the product of the two projected means, so one pass over Q and K
//           replaces the pairwise estimate.
//   select  one CTA per (query block b, kv head): scores of the earlier
//           blocks, s(b, i) = max_g qbar_g(b) . kbar(i) / sqrt(d), and an
//           exact top-k (ties to the lower block) of them; the list is the
//           chosen blocks plus b itself, ascending.  Dense mode, or b below
//           the budget: every block 0..b.
//   attn    (prefill_tc.cu on the 5th-generation tensor cores when G >= 2;
//           this kernel otherwise)
//           one CTA per (query block, query head), 4 warps of 16 queries:
//           the chosen key blocks are staged in shared memory 64 rows at a
//           time and each warp runs the decode kernel's tile math with its
//           16 queries as two 8-column tiles -- S^T = K Q^T and O^T += V^T
//           P^T on tensor cores (mma.sync m16n8k16, fp32 accumulate, P split
//           into a 16-bit high part and the rounding of the rest), an online
//           softmax per query, the causal mask on the query block's own
//           block.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "prefill.h"
#include "ptx.cuh"
#include "spd_internal.h"
#include "topk.cuh"

namespace spd {
namespace {

constexpr int kAttnWarps = 4;  // 4 x 16 queries = one block
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kPoolThreads = 128;

template <typename T> struct PF;
template <> struct PF<__half> {
  static constexpr bool bf = false;
  static __device__ __forceinline__ float f(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from(float x) { return __float2half_rn(x); }
};
template <> struct PF<__nv_bfloat16> {
  static constexpr bool bf = true;
  static __device__ __forceinline__ float f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ void pf_err(int *err, int code, int a, int b, int c) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}

// ---- pool: projected block means -------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kPoolThreads) prefill_pool_kernel(const __grid_constant__ PrefillParams p) {
  __shared__ float mean_s[D];
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x % p.nb, hk = blockIdx.x / p.nb;
  const int c = threadIdx.x;
  const int t0 = b * kPrefillBlock, t1 = min(t0 + kPrefillBlock, p.L);
  const float inv = 1.f / (float)(t1 - t0);
  const T *k = static_cast<const T *>(p.k);
  const T *q = static_cast<const T *>(p.q);
  if (c < D) {
    float acc = 0.f;
    for (int t = t0; t < t1; ++t) acc += PF<T>::f(k[((size_t)t * p.Hkv + hk) * D + c]);
    mean_s[c] = acc * inv;
  }
  __syncthreads();
  if (c < p.r) {
    const float *w = p.wk + (size_t)hk * D * p.r;
    float acc = 0.f;
    for (int x = 0; x < D; ++x) acc = fmaf(mean_s[x], w[(size_t)x * p.r + c], acc);
    p.kbar[((size_t)hk * p.nb + b) * p.r + c] = acc;
  }
  for (int g = 0; g < p.G; ++g) {
    __syncthreads();  // mean_s is rewritten
    const int h = hk * p.G + g;
    if (c < D) {
      float acc = 0.f;
      for (int t = t0; t < t1; ++t) acc += PF<T>::f(q[((size_t)t * p.Hq + h) * D + c]);
      mean_s[c] = acc * inv;
    }
    __syncthreads();
    if (c < p.r) {
      const float *w = p.wq + (size_t)hk * D * p.r;
      float acc = 0.f;
      for (int x = 0; x < D; ++x) acc = fmaf(mean_s[x], w[(size_t)x * p.r + c], acc);
      p.qbar[(((size_t)hk * p.G + g) * p.nb + b) * p.r + c] = acc;
    }
  }
}

// ---- select: block scores and their top-k ----------------------------------
__global__ void __launch_bounds__(kSelThreads) prefill_select_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ __align__(16) uint8_t sel_smem[];
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x % p.nb, hk = blockIdx.x / p.nb;
  const int tid = threadIdx.x;
  int *list = p.lists + ((size_t)hk * p.nb + b) * p.KB;
  int cnt;
  if (p.dense || b + 1 <= p.kblocks) {
    cnt = b + 1;
    for (int j = tid; j <= b; j += kSelThreads) list[j] = j;
  } else if (p.kblocks == 1) {
    cnt = 1;
    if (tid == 0) list[0] = b;
  } else {
    cnt = p.kblocks;
    TopkSmem m = carve_topk_smem(sel_smem);
    if (p.r == 16 && p.G <= 8) {
      // the common rank: the query block's G projected means in shared
      // memory (broadcast reads), each candidate's row as four 16-byte loads
      __shared__ float4 s_q[8 * 4];
      if (tid < p.G * 4)
        s_q[tid] = reinterpret_cast<const float4 *>(
            p.qbar + (((size_t)hk * p.G + tid / 4) * p.nb + b) * 16)[tid % 4];
      __syncthreads();
      const float4 *kb = reinterpret_cast<const float4 *>(p.kbar + (size_t)hk * p.nb * 16);
      for (int i = tid; i < b; i += kSelThreads) {
        float4 kr[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) kr[c] = kb[(size_t)i * 4 + c];
        float best = -CUDART_INF_F;
        for (int g = 0; g < p.G; ++g) {
          float acc = 0.f;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 q = s_q[4 * g + c];
            acc = fmaf(q.x, kr[c].x, acc);
            acc = fmaf(q.y, kr[c].y, acc);
            acc = fmaf(q.z, kr[c].z, acc);
            acc = fmaf(q.w, kr[c].w, acc);
          }
          best = fmaxf(best, acc * p.score_scale);
        }
        m.skey[i] = score_key(best);
      }
    } else {
      for (int i = tid; i < b; i += kSelThreads) {
        float best = -CUDART_INF_F;
        for (int g = 0; g < p.G; ++g) {
          const float *qb = p.qbar + (((size_t)hk * p.G + g) * p.nb + b) * p.r;
          const float *kb = p.kbar + ((size_t)hk * p.nb + i) * p.r;
          float acc = 0.f;
          for (int j = 0; j < p.r; ++j) acc = fmaf(qb[j], kb[j], acc);
          best = fmaxf(best, acc * p.score_scale);
        }
        m.skey[i] = score_key(best);
      }
    }
    __syncthreads();
    const int k = p.kblocks - 1;  // 1 <= k < b
    const int got = topk_core(m.skey, nullptr, b, b, k, list, m);
    __syncthreads();
    if (tid == 0) {
      list[k] = b;  // the query block's own block is always attended
      if (got != k) pf_err(p.err, kDevTopkCount, hk, b, got);
    }
  }
  for (int j = cnt + tid; j < p.KB; j += kSelThreads) list[j] = -1;
  if (p.blocks_out) {
    __syncthreads();  // the list is complete (written by this CTA's threads)
    int *o = p.blocks_out + ((size_t)hk * p.nb + b) * p.KB;
    for (int j = tid; j < p.KB; j += kSelThreads) o[j] = list[j];
  }
}

// ---- attention --------------------------------------------------------------
// Shared memory: K rows and V rows of one key block, each as 4 tiles of 16
// rows stored like the decode kernel's stages (128-byte boxes of 64 16-bit
// channels, 16-byte chunks swizzled by row), then a per-warp P buffer
// [16 keys][16 queries].
template <int D>
struct PfSmem {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTile = kBoxes * 16 * 128;  // one 16-row tile of K or V
  static constexpr int kMat = 4 * kTile;           // 64 rows
  static constexpr int kK = 0, kV = kMat, kP = 2 * kMat;
  static constexpr int kBytes = kP + kAttnWarps * 16 * 16 * 4;
};

template <typename T, int D>
__global__ void __launch_bounds__(kAttnThreads) prefill_attn_kernel(const __grid_constant__ PrefillParams p) {
  using Sm = PfSmem<D>;
  constexpr int MT = D / 16;
  extern __shared__ __align__(1024) uint8_t at_smem[];
  uint8_t *Ks = at_smem + Sm::kK, *Vs = at_smem + Sm::kV;
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x % p.nb, h = blockIdx.x / p.nb;
  const int hk = h / p.G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int t0 = b * kPrefillBlock;
  const int qw = t0 + warp * 16;  // this warp's first query
  float *Pw = reinterpret_cast<float *>(at_smem + Sm::kP) + warp * 256;

  // q^T fragments (B operand) of the warp's two 8-query tiles
  uint32_t qb[D / 16][2][2];
  {
    const uint16_t *q = static_cast<const uint16_t *>(p.q);
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const int t = qw + 8 * n + g8;
      const uint32_t *row = reinterpret_cast<const uint32_t *>(q + ((size_t)t * p.Hq + h) * D);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        qb[kk][n][0] = t < p.L ? row[(kk * 16 + 2 * t4) / 2] : 0u;
        qb[kk][n][1] = t < p.L ? row[(kk * 16 + 2 * t4 + 8) / 2] : 0u;
      }
    }
  }
  float oacc[MT][2][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[m][n][e] = 0.f;
  // running max / partial sums of the lane's 4 queries: [n][column 2t4 + j]
  float mrun[2][2] = {{-CUDART_INF_F, -CUDART_INF_F}, {-CUDART_INF_F, -CUDART_INF_F}};
  float lrun[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  const float sc = p.scale_log2;

  const int *list = p.lists + ((size_t)hk * p.nb + b) * p.KB;
  const int nsel = p.dense ? b + 1 : min(b + 1, p.kblocks);
  const uint16_t *kg = static_cast<const uint16_t *>(p.k);
  const uint16_t *vg = static_cast<const uint16_t *>(p.v);
  for (int li = 0; li < nsel; ++li) {
    const int i = list[li];
    if (i < 0 || i > b) {
      if (tid == 0) pf_err(p.err, kDevBadSelection, h, b, i);
      break;
    }
    __syncthreads();  // every warp is done with the previous block's rows
    // stage K and V rows i*64 .. i*64+63 (zero past the prompt)
    for (int x = tid; x < 64 * (D / 8); x += kAttnThreads) {
      const int r = x / (D / 8), c16 = x % (D / 8);
      const int t = i * kPrefillBlock + r;
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (t < p.L) {
        const size_t src = ((size_t)t * p.Hkv + hk) * D + c16 * 8;
        kv = *reinterpret_cast<const uint4 *>(kg + src);
        vv = *reinterpret_cast<const uint4 *>(vg + src);
      }
      const int rr = r & 15;
      const uint32_t off = (uint32_t)((r >> 4) * Sm::kTile + (c16 >> 3) * 2048) +
                           swz128(rr, c16 & 7);
      *reinterpret_cast<uint4 *>(Ks + off) = kv;
      *reinterpret_cast<uint4 *>(Vs + off) = vv;
    }
    __syncthreads();
    for (int mt = 0; mt < 4; ++mt) {
      const int key0 = i * kPrefillBlock + mt * 16;
      if (key0 > qw + 15) break;  // every later key is after all of this warp's queries
      const uint8_t *kt = Ks + mt * Sm::kTile, *vt = Vs + mt * Sm::kTile;
      // S^T = K Q^T: 16 keys x (2 x 8 queries)
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int chalf = lane >> 4;
        const uint32_t kbase = smem_u32(kt);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t a[4];
          ldmatrix_x4(kbase + (kk >> 2) * 2048 + swz128(row, 2 * (kk & 3) + chalf), a[0], a[1],
                      a[2], a[3]);
          mma_16816<PF<T>::bf>(acc[0], a, qb[kk][0][0], qb[kk][0][1]);
          mma_16816<PF<T>::bf>(acc[1], a, qb[kk][1][0], qb[kk][1][1]);
        }
      }
      // acc[n]: [0] key g8 x query 2t4, [1] key g8 x query 2t4+1, [2]/[3] key g8+8
      const int klo = key0 + g8, khi = key0 + g8 + 8;
      float cfac[2][2];
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const int qa = qw + 8 * n + 2 * t4, qbq = qa + 1;
        const float z0 = (klo <= qa && klo < p.L) ? acc[n][0] * sc : -CUDART_INF_F;
        const float z1 = (klo <= qbq && klo < p.L) ? acc[n][1] * sc : -CUDART_INF_F;
        const float z2 = (khi <= qa && khi < p.L) ? acc[n][2] * sc : -CUDART_INF_F;
        const float z3 = (khi <= qbq && khi < p.L) ? acc[n][3] * sc : -CUDART_INF_F;
        float mx0 = fmaxf(z0, z2), mx1 = fmaxf(z1, z3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(mrun[n][0], mx0), mn1 = fmaxf(mrun[n][1], mx1);
        // (a query with no allowed key so far keeps max -inf and weight 0)
        const float c0 = mrun[n][0] == -CUDART_INF_F ? 0.f : exp2f(mrun[n][0] - mn0);
        const float c1 = mrun[n][1] == -CUDART_INF_F ? 0.f : exp2f(mrun[n][1] - mn1);
        const float p0 = z0 == -CUDART_INF_F ? 0.f : exp2f(z0 - mn0);
        const float p1 = z1 == -CUDART_INF_F ? 0.f : exp2f(z1 - mn1);
        const float p2 = z2 == -CUDART_INF_F ? 0.f : exp2f(z2 - mn0);
        const float p3 = z3 == -CUDART_INF_F ? 0.f : exp2f(z3 - mn1);
        lrun[n][0] = lrun[n][0] * c0 + p0 + p2;
        lrun[n][1] = lrun[n][1] * c1 + p1 + p3;
        mrun[n][0] = mn0;
        mrun[n][1] = mn1;
        cfac[n][0] = c0;
        cfac[n][1] = c1;
        Pw[g8 * 16 + 8 * n + 2 * t4] = p0;
        Pw[g8 * 16 + 8 * n + 2 * t4 + 1] = p1;
        Pw[(g8 + 8) * 16 + 8 * n + 2 * t4] = p2;
        Pw[(g8 + 8) * 16 + 8 * n + 2 * t4 + 1] = p3;
      }
      __syncwarp();
      // O^T += V^T P^T
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          oacc[m][n][0] *= cfac[n][0];
          oacc[m][n][1] *= cfac[n][1];
          oacc[m][n][2] *= cfac[n][0];
          oacc[m][n][3] *= cfac[n][1];
        }
      uint32_t bh[2][2], bl[2][2];  // B = P^T: k = keys 2t4.. / 2t4+8.., n = query g8
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const float pv[4] = {Pw[(2 * t4) * 16 + 8 * n + g8], Pw[(2 * t4 + 1) * 16 + 8 * n + g8],
                             Pw[(2 * t4 + 8) * 16 + 8 * n + g8], Pw[(2 * t4 + 9) * 16 + 8 * n + g8]};
        uint16_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const T th = PF<T>::from(pv[e]);
          hi[e] = *reinterpret_cast<const uint16_t *>(&th);
          const T tl = PF<T>::from(pv[e] - PF<T>::f(th));
          lo[e] = *reinterpret_cast<const uint16_t *>(&tl);
        }
        bh[n][0] = (uint32_t)hi[0] | ((uint32_t)hi[1] << 16);
        bh[n][1] = (uint32_t)hi[2] | ((uint32_t)hi[3] << 16);
        bl[n][0] = (uint32_t)lo[0] | ((uint32_t)lo[1] << 16);
        bl[n][1] = (uint32_t)lo[2] | ((uint32_t)lo[3] << 16);
      }
      {
        const int j = lane >> 3;
        const int row = (lane & 7) + 8 * (j >> 1);
        const uint32_t vbase = smem_u32(vt);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          uint32_t a[4];
          ldmatrix_x4_trans(vbase + (m >> 2) * 2048 + swz128(row, 2 * (m & 3) + (j & 1)), a[0],
                            a[1], a[2], a[3]);
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            mma_16816<PF<T>::bf>(oacc[m][n], a, bh[n][0], bh[n][1]);
            mma_16816<PF<T>::bf>(oacc[m][n], a, bl[n][0], bl[n][1]);
          }
        }
      }
      __syncwarp();  // Pw is rewritten by the next tile
    }
  }
  // the row sums: every lane of a column holds part of it
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
        lrun[n][j] += __shfl_xor_sync(0xffffffffu, lrun[n][j], off);
  // O^T m-tile m: [0] channel 16m + g8 x query 2t4, [1] query 2t4+1, [2]/[3] channel + 8
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int t = qw + 8 * n + 2 * t4 + j;
      if (t >= p.L) continue;
      const float inv = 1.f / lrun[n][j];
      float *o = p.out + ((size_t)t * p.Hq + h) * D;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        o[16 * m + g8] = oacc[m][n][j] * inv;
        o[16 * m + g8 + 8] = oacc[m][n][2 + j] * inv;
      }
    }
}

template <typename T, int D>
cudaError_t launch_t(const PrefillParams &p, cudaStream_t st) {
  const int grid_kv = p.nb * p.Hkv, grid_q = p.nb * p.Hq;
  cudaError_t e = launch_pdl(prefill_pool_kernel<T, D>, grid_kv, kPoolThreads, 0, st, p);
  if (e != cudaSuccess) return e;
  e = launch_pdl(prefill_select_kernel, grid_kv, kSelThreads, (size_t)kTopkSmemBytes, st, p);
  if (e != cudaSuccess) return e;
  if (prefill_tc_supported(p.G)) return launch_prefill_attn_tc(p, PF<T>::bf ? 1 : 0, D, st);
  e = launch_pdl(prefill_attn_kernel<T, D>, grid_q, kAttnThreads, (size_t)PfSmem<D>::kBytes, st,
                 p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams &p, int dtype, int d, cudaStream_t st) {
  if (dtype == 0) return d == 64 ? launch_t<__half, 64>(p, st) : launch_t<__half, 128>(p, st);
  return d == 64 ? launch_t<__nv_bfloat16, 64>(p, st) : launch_t<__nv_bfloat16, 128>(p, st);
}

}  // namespace spd
