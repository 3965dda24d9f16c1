// Block-sparse causal attention of a prompt on the 5th-generation tensor
// cores ("LServe long-sequence LLM serving system", section 3.1: exact
// attention on the chosen key blocks of every query block).
//
// One CTA per (query block b, kv head, group of HC query heads), HC = 2 or 4:
// its HC x 64 query rows are MT = HC / 2 matrices of 128 rows (two heads x
// the block's 64 tokens each).  Per chosen key block i (ascending):
//   S_m  = Q_m . K_i^T         tcgen05.mma, M 128 x N 64 x K d, fp32 in TMEM
//   softmax, one row per thread: tcgen05.ld of its 64 logits, the causal mask
//        on the diagonal block (and keys past the prompt), an online max and
//        sum in fp32 (base 2), P written to shared memory as a 16-bit high
//        part and the 16-bit rounding of the rest (like the decode kernel's
//        P.V), and O's row rescaled in tensor memory when its max moved;
//   O_m += (P_hi + P_lo)_m . V_i  tcgen05.mma, M 128 x N 64 (per half of d)
//        x K 64 keys, fp32 in TMEM.
// Q is staged once in shared memory (128-byte swizzled rows of 64 channels);
// K and V blocks come by TMA (4-D maps over [L][Hkv][d], 64 x 64 boxes,
// 128-byte swizzle) into two buffers, the next block loading while the
// current one is in use.  One thread issues the MMAs and commits them to an
// mbarrier; every wait is bounded, and a CTA that gives up records the error,
// waits (bounded) for what it has in flight and frees its tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "prefill.h"
#include "ptx.cuh"
#include "spd_internal.h"

namespace spd {
namespace {

constexpr uint32_t kTcWait = 1u << 22;  // bounded mbarrier polls

template <typename T> struct TcT;
template <> struct TcT<__half> {
  static constexpr bool bf = false;
  static __device__ __forceinline__ uint16_t bits(float x) {
    const __half h = __float2half_rn(x);
    return *reinterpret_cast<const uint16_t *>(&h);
  }
  static __device__ __forceinline__ float val(uint16_t b) {
    return __half2float(*reinterpret_cast<const __half *>(&b));
  }
};
template <> struct TcT<__nv_bfloat16> {
  static constexpr bool bf = true;
  static __device__ __forceinline__ uint16_t bits(float x) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<const uint16_t *>(&h);
  }
  static __device__ __forceinline__ float val(uint16_t b) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(&b));
  }
};

// Shared memory (offsets from a 1024-byte aligned base).  Every matrix is a
// stack of 64-column sub-tiles of rows x 128 bytes, 128-byte swizzled.
template <int D, int HC>
struct TcSmem {
  static constexpr int MT = HC / 2;            // 128-row matrices of the CTA
  static constexpr int KB = D / 64;            // 64-column sub-tiles of a row
  static constexpr int kQ = 0;                 // [MT][KB][128 x 128 B]
  static constexpr int kKV = kQ + MT * KB * 16384;  // [2 buffers][K, V][KB][64 x 128 B]
  static constexpr int kKVBuf = 2 * KB * 8192;
  static constexpr int kP = kKV + 2 * kKVBuf;  // [MT][hi, lo][128 x 128 B]
  static constexpr int kBars = kP + MT * 2 * 16384;  // uint64 [4]: kv[2], s, pv
  static constexpr int kMisc = kBars + 32;           // tmem base, fail flag
  static constexpr int kBytes = kMisc + 16 + 1024;   // + alignment slack
  // tensor-memory columns: S_m at 64m, O_m at 64 MT + D m
  static constexpr int kCols = MT * (64 + D);
  static constexpr int kAlloc = kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  static_assert(kBytes <= 232448, "shared memory");
};

__device__ __forceinline__ void pf_set_err(int *err, int code, int a, int b, int c) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}

__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kTcWait; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

template <typename T, int D, int HC>
__global__ void __launch_bounds__(HC / 2 * 128) prefill_attn_tc_kernel(const __grid_constant__ PrefillParams p) {
  using Sm = TcSmem<D, HC>;
  constexpr int MT = Sm::MT, KB = Sm::KB;
  constexpr int kThreads = MT * 128;
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Sm::kBars);  // kv[0], kv[1], s, pv
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Sm::kMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m = warp >> 2;                      // this thread's 128-row matrix
  const int row = 32 * (warp & 3) + lane;       // its row there = tensor-memory lane
  const int b = blockIdx.x % p.nb, rest = blockIdx.x / p.nb;
  const int hk = rest % p.Hkv, hg = rest / p.Hkv;
  const int t0 = b * kPrefillBlock;
  // the thread's query: head (of the kv head's group) and token
  const int h_row = hk * p.G + hg * HC + 2 * m + (row >> 6);
  const int t_row = t0 + (row & 63);

  pdl_wait();
  pdl_launch_dependents();
  if (warp == 0) tmem_alloc(tmem_slot, Sm::kAlloc);
  if (tid == 0) {
    for (int x = 0; x < 4; ++x) mbar_init(&bars[x], 1);
    fence_mbar_init();
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
  }
  // ---- Q: the CTA's rows, 16 bytes per thread and step ----
  {
    const uint16_t *q = static_cast<const uint16_t *>(p.q);
    for (int x = tid; x < MT * 128 * (D / 8); x += kThreads) {
      const int mm = x / (128 * (D / 8)), rem = x % (128 * (D / 8));
      const int r = rem / (D / 8), c16 = rem % (D / 8);
      const int t = t0 + (r & 63), h = hk * p.G + hg * HC + 2 * mm + (r >> 6);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < p.L) v = *reinterpret_cast<const uint4 *>(q + ((size_t)t * p.Hq + h) * D + c16 * 8);
      uint8_t *sub = smem + Sm::kQ + (mm * KB + (c16 >> 3)) * 16384;
      *reinterpret_cast<uint4 *>(sub + swz128(r, c16 & 7)) = v;
    }
  }
  fence_proxy_async_smem();  // the MMAs read Q through the async proxy
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int *list = p.lists + ((size_t)hk * p.nb + b) * p.KB;
  const int nsel = p.dense ? b + 1 : min(b + 1, p.kblocks);
  // TMA of key block i into buffer buf: K then V, KB boxes each
  auto load_kv = [&](int i, int buf) {
    uint8_t *kv = smem + Sm::kKV + buf * Sm::kKVBuf;
    mbar_arrive_expect_tx(&bars[buf], 2 * KB * 8192);
    for (int kb = 0; kb < KB; ++kb) {
      tma_load_4d(kv + kb * 8192, &p.tm_k, 0, kb, hk, i * kPrefillBlock, &bars[buf]);
      tma_load_4d(kv + (KB + kb) * 8192, &p.tm_v, 0, kb, hk, i * kPrefillBlock, &bars[buf]);
    }
  };
  int issued[2] = {0, 0};  // (thread 0) loads issued per buffer
  if (tid == 0) {
    for (int li = 0; li < min(2, nsel); ++li) {
      const int i = list[li];
      if (i >= 0 && i <= b) {
        load_kv(i, li);
        ++issued[li];
      }
    }
  }

  const bool bf = TcT<T>::bf;
  const uint32_t idesc_s = umma_idesc_f16(bf, 128, 64, 0, 0);  // Q . K^T: both K-major
  const uint32_t idesc_o = umma_idesc_f16(bf, 128, 64, 0, 1);  // P . V: V MN-major
  const float sc = p.scale_log2;
  float m_run = -CUDART_INF_F, l_run = 0.f;
  int commits = 0;       // (thread 0) MMA commits issued; alternately s and pv
  bool fail = false;
  for (int li = 0; li < nsel && !fail; ++li) {
    const int i = list[li];
    if (i < 0 || i > b) {  // (the selection never yields one: record it and drain)
      if (tid == 0) pf_set_err(p.err, kDevBadSelection, hk, b, i);
      fail = true;
      break;
    }
    const int buf = li & 1;
    uint8_t *kv = smem + Sm::kKV + buf * Sm::kKVBuf;
    // ---- S = Q . K^T ----
    bool ok = true;
    if (tid == 0) {
      ok = tc_wait(&bars[buf], (li >> 1) & 1);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = umma_desc_sw128(
                smem_u32(smem + Sm::kQ + (mm * KB + (kk >> 2)) * 16384) + (kk & 3) * 32, 16, 1024);
            const uint64_t bd =
                umma_desc_sw128(smem_u32(kv + (kk >> 2) * 8192) + (kk & 3) * 32, 16, 1024);
            umma_f16(tmem + 64 * mm, a, bd, idesc_s, kk > 0);
          }
        umma_commit(&bars[2]);
        ++commits;
      }
    }
    ok = tc_wait(&bars[2], li & 1) && ok;
    ok = __all_sync(0xffffffffu, ok);  // the tensor-memory loads below are warp-wide
    tc_fence_after();
    // ---- softmax of this thread's row ----
    float alpha = 1.f;
    if (ok) {
      const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 64 * m;
      uint32_t s[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r16[16];
        tmem_ld16(ta + 16 * c, r16);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) s[16 * c + j] = r16[j];
      }
      const int key0 = i * kPrefillBlock;
      const int lim = min(i == b ? (row & 63) : 63, p.L - 1 - key0);  // last allowed key
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (j <= lim) mx = fmaxf(mx, __uint_as_float(s[j]) * sc);
      const float m_new = fmaxf(m_run, mx);
      alpha = m_run == -CUDART_INF_F ? 0.f : exp2f(m_run - m_new);
      float lsum = 0.f;
      uint8_t *phi = smem + Sm::kP + (2 * m) * 16384, *plo = phi + 16384;
#pragma unroll
      for (int c = 0; c < 8; ++c) {  // 16-byte chunks: keys 8c .. 8c+7
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint16_t hb[2], lb[2];
#pragma unroll
          for (int f = 0; f < 2; ++f) {
            const int j = 8 * c + 2 * e + f;
            const float pj =
                (j <= lim && m_new != -CUDART_INF_F) ? exp2f(__uint_as_float(s[j]) * sc - m_new)
                                                     : 0.f;
            lsum += pj;
            hb[f] = TcT<T>::bits(pj);
            lb[f] = TcT<T>::bits(pj - TcT<T>::val(hb[f]));
          }
          hw[e] = (uint32_t)hb[0] | ((uint32_t)hb[1] << 16);
          lw[e] = (uint32_t)lb[0] | ((uint32_t)lb[1] << 16);
        }
        *reinterpret_cast<uint4 *>(phi + swz128(row, c)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(plo + swz128(row, c)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      l_run = l_run * alpha + lsum;
      m_run = m_new;
    }
    // O's row follows the new max (the previous block's P.V has finished)
    if (li > 0 && __any_sync(0xffffffffu, ok && alpha != 1.f)) {
      const uint32_t to = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 64 * MT + D * m;
#pragma unroll 1
      for (int c = 0; c < D / 16; ++c) {
        uint32_t r16[16];
        tmem_ld16(to + 16 * c, r16);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) r16[j] = __float_as_uint(__uint_as_float(r16[j]) * alpha);
        tmem_st16(to + 16 * c, r16);
      }
      tmem_wait_st();
    }
    fence_proxy_async_smem();  // P was written through the generic proxy
    tc_fence_before();
    fail = __syncthreads_or(!ok);
    tc_fence_after();
    if (fail) break;
    // ---- O += P . V ----
    if (tid == 0) {
#pragma unroll
      for (int mm = 0; mm < MT; ++mm)
#pragma unroll
        for (int half = 0; half < KB; ++half)
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = umma_desc_sw128(
                  smem_u32(smem + Sm::kP + (2 * mm + part) * 16384) + kk * 32, 16, 1024);
              const uint64_t bd =
                  umma_desc_sw128(smem_u32(kv + (KB + half) * 8192) + kk * 2048, 16, 1024);
              umma_f16(tmem + 64 * MT + D * mm + 64 * half, a, bd, idesc_o,
                       li > 0 || part > 0 || kk > 0);
            }
      umma_commit(&bars[3]);
      ++commits;
    }
    ok = tc_wait(&bars[3], li & 1);
    tc_fence_after();
    fail = __syncthreads_or(!ok);
    if (fail) break;
    // the buffer's MMAs are done: it takes block li + 2
    if (tid == 0 && li + 2 < nsel) {
      const int i2 = list[li + 2];
      if (i2 >= 0 && i2 <= b) {
        load_kv(i2, buf);
        ++issued[buf];
      }
    }
  }
  if (fail) {
    // record it (the first error stays), and give what is still in flight one
    // more bounded wait
    if (tid == 0) {
      pf_set_err(p.err, kDevTimeout, hk, b, 0);
      for (int x = 0; x < 2; ++x)
        if (issued[x] > 0) tc_wait(&bars[x], (issued[x] - 1) & 1);
      if (commits > 0) tc_wait(&bars[2 + ((commits - 1) & 1)], ((commits - 1) >> 1) & 1);
    }
  } else {
    // ---- out = O / l (the loads are warp-wide; rows past the prompt store nothing) ----
    const uint32_t to = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 64 * MT + D * m;
    float *o = p.out + ((size_t)t_row * p.Hq + h_row) * D;
    const float inv = 1.f / l_run;
#pragma unroll 1
    for (int c = 0; c < D / 16; ++c) {
      uint32_t r16[16];
      tmem_ld16(to + 16 * c, r16);
      tmem_wait_ld();
      if (t_row < p.L) {
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<float4 *>(o + 16 * c + j) =
              make_float4(__uint_as_float(r16[j]) * inv, __uint_as_float(r16[j + 1]) * inv,
                          __uint_as_float(r16[j + 2]) * inv, __uint_as_float(r16[j + 3]) * inv);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, Sm::kAlloc);
}

template <typename T, int D, int HC>
cudaError_t launch_tc(const PrefillParams &p, cudaStream_t st) {
  using Sm = TcSmem<D, HC>;
  auto k = prefill_attn_tc_kernel<T, D, HC>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::kBytes);
  if (e != cudaSuccess) return e;
  const int grid = p.nb * p.Hkv * (p.G / HC);
  return launch_pdl(k, grid, Sm::MT * 128, (size_t)Sm::kBytes, st, p);
}

template <typename T, int D>
cudaError_t launch_tc_g(const PrefillParams &p, cudaStream_t st) {
  return p.G == 2 ? launch_tc<T, D, 2>(p, st) : launch_tc<T, D, 4>(p, st);
}

}  // namespace

bool prefill_tc_supported(int G) { return G == 2 || G == 4 || G == 8; }

cudaError_t launch_prefill_attn_tc(const PrefillParams &p, int dtype, int d, cudaStream_t st) {
  if (dtype == 0) return d == 64 ? launch_tc_g<__half, 64>(p, st) : launch_tc_g<__half, 128>(p, st);
  return d == 64 ? launch_tc_g<__nv_bfloat16, 64>(p, st) : launch_tc_g<__nv_bfloat16, 128>(p, st);
}

}  // namespace spd
