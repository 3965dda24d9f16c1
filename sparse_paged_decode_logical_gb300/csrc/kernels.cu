// KV-cache write kernels (sm_103a).
//
//   pt_write      page-table entries from the host runtime's allocator
//   append        write new K/V rows (paged pool for dynamic heads, sink +
//                 ring for streaming heads) and fold them into the logical
//                 page's channel-wise key min/max ("LServe long-sequence LLM
//                 serving system", section 2.1, min-max pooling); used for
//                 bulk appends (prefill) -- the one-token append of a decode
//                 step is fused into the decode kernel; with fp8 storage the
//                 rows are written as E4M3 codes of value / scale
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "ptx.cuh"
#include "spd_internal.h"

namespace spd {
namespace {

// ---- element conversions ---------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<__half> {
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) {
    return __bfloat162float(x);
  }
};

template <typename T, int N>
__device__ __forceinline__ void load_row(const T *src, float (&dst)[N]) {
  // N consecutive 16-bit elements; N in {2, 4}: one 4- or 8-byte load
  if constexpr (N == 4) {
    uint2 raw = *reinterpret_cast<const uint2 *>(src);
    const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = Elem<T>::to_f(e[i]);
  } else {
    uint32_t raw = *reinterpret_cast<const uint32_t *>(src);
    const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
    for (int i = 0; i < 2; ++i) dst[i] = Elem<T>::to_f(e[i]);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void set_err(int *err, int code, int a, int b, int c) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}

// ---- page table ------------------------------------------------------------
__global__ void pt_write_kernel(const __grid_constant__ PtWriteParams p) {
  pdl_wait();
  pdl_launch_dependents();
  for (int i = threadIdx.x; i < p.n; i += blockDim.x) {
    const PtUpdate u = p.upd[i];
    p.page_table[(size_t)u.slot * p.max_pp + u.index] = u.phys;
  }
}

// ---- append + metadata -----------------------------------------------------
// Dynamic part: one CTA per (sequence, touched logical page, dynamic head);
// thread c owns channel c.  Streaming part: one CTA per (sequence, head).
// Storage element E: the input type T, or (kF8) one-byte E4M3 codes of
// value / scale, whose min/max compare by the code's sign-magnitude order.
template <typename T, bool kF8> struct Store;
template <typename T> struct Store<T, false> {
  using E = T;
  static __device__ __forceinline__ E put(T x, float) { return x; }
  static __device__ __forceinline__ float key(E e) { return Elem<T>::to_f(e); }
};
template <typename T> struct Store<T, true> {
  using E = uint8_t;
  static __device__ __forceinline__ E put(T x, float scale) {
    return (E)e4m3_code(Elem<T>::to_f(x), scale);
  }
  static __device__ __forceinline__ float key(E e) { return (float)e4m3_key(e); }
};

template <typename T, int D, bool kF8>
__global__ void __launch_bounds__(128) append_kernel(const __grid_constant__ AppendParams p) {
  using St = Store<T, kF8>;
  using E = typename St::E;
  pdl_wait();
  pdl_launch_dependents();
  const int c = threadIdx.x;
  const T *__restrict__ kin = static_cast<const T *>(p.k);
  const T *__restrict__ vin = static_cast<const T *>(p.v);
  const int n = p.n_tokens;
  if ((int)blockIdx.x < p.dyn_ctas) {
    int i = 0;
    while (i + 1 < p.n_seqs && p.seqs[i + 1].cta_off <= (int)blockIdx.x) ++i;
    const AppendSeq s = p.seqs[i];
    const int local = blockIdx.x - s.cta_off;
    const int hd = local % p.Hd;
    const int j = s.L_old / p.ell + local / p.Hd;  // logical page
    const int h = p.dyn_kv[hd];
    const float ks = kF8 ? p.k_scale[h] : 1.f, vs = kF8 ? p.v_scale[h] : 1.f;
    const int L_new = s.L_old + n;
    const int t0 = j * p.ell;
    const int t1 = min(t0 + p.ell, L_new);
    const int blk = t0 / p.P;
    if (blk >= p.max_pp) {
      if (c == 0) set_err(p.err, kDevBadPage, s.slot, j, blk);
      return;
    }
    const int phys = p.page_table[(size_t)s.slot * p.max_pp + blk];
    if (phys < 0 || phys >= p.num_phys) {
      if (c == 0) set_err(p.err, kDevBadPhys, s.slot, blk, phys);
      return;
    }
    const size_t page_base = ((size_t)phys * p.Hd + hd) * p.P;  // in rows
    E *__restrict__ kp = static_cast<E *>(p.k_pool);
    E *__restrict__ vp = static_cast<E *>(p.v_pool);
    E *__restrict__ meta = static_cast<E *>(p.meta) +
              (((size_t)phys * p.Hd + hd) * p.R + (j % p.R)) * 2 * D;
    if (c >= D) return;
    E bmin, bmax;
    float vmin, vmax;
    int t = max(t0, s.L_old);
    if (t0 < s.L_old) {  // the page already holds tokens: start from its metadata
      bmin = meta[c];
      bmax = meta[D + c];
    } else {
      bmin = bmax = St::put(kin[(((size_t)i * n + (t - s.L_old)) * p.Hkv + h) * D + c], ks);
    }
    vmin = St::key(bmin);
    vmax = St::key(bmax);
#pragma unroll 8
    for (; t < t1; ++t) {
      const size_t src = (((size_t)i * n + (t - s.L_old)) * p.Hkv + h) * D + c;
      const E kx = St::put(__ldg(kin + src), ks);
      const size_t dst = (page_base + (t % p.P)) * D + c;
      kp[dst] = kx;
      vp[dst] = St::put(__ldg(vin + src), vs);
      const float x = St::key(kx);
      if (x < vmin) { vmin = x; bmin = kx; }
      if (x > vmax) { vmax = x; bmax = kx; }
    }
    meta[c] = bmin;
    meta[D + c] = bmax;
  } else {
    const int b = blockIdx.x - p.dyn_ctas;
    const int i = b / p.Hs, hs = b % p.Hs;
    const int h = p.str_kv[hs];
    const float ks = kF8 ? p.k_scale[h] : 1.f, vs = kF8 ? p.v_scale[h] : 1.f;
    const AppendSeq s = p.seqs[i];
    const int L_new = s.L_old + n;
    const int SW = p.S + p.W;
    E *sk = static_cast<E *>(p.stream_k) + ((size_t)s.slot * p.Hs + hs) * SW * D;
    E *sv = static_cast<E *>(p.stream_v) + ((size_t)s.slot * p.Hs + hs) * SW * D;
    // positions that can still be read: sink t < S, window t >= L_new - W
    const int w0 = max(s.L_old, max(p.S, L_new - p.W));
    for (int t = s.L_old; t < L_new; ++t) {
      if (t >= p.S && t < w0) { t = w0 - 1; continue; }
      const int slot = t < p.S ? t : p.S + (t - p.S) % p.W;
      const size_t src = (((size_t)i * n + (t - s.L_old)) * p.Hkv + h) * D;
      for (int cc = c; cc < D; cc += blockDim.x) {
        sk[(size_t)slot * D + cc] = St::put(kin[src + cc], ks);
        sv[(size_t)slot * D + cc] = St::put(vin[src + cc], vs);
      }
    }
  }
}

}  // namespace

cudaError_t launch_pt_write(const PtWriteParams &p, cudaStream_t s, long long *n) {
  cudaError_t e = launch_pdl(pt_write_kernel, 1, 256, 0, s, p);
  *n += 1;
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_append(const AppendParams &p, int dtype, int d, cudaStream_t s,
                          long long *n) {
  const int grid = p.dyn_ctas + p.n_seqs * p.Hs;
  if (grid == 0) return cudaSuccess;
  *n += 1;
  cudaError_t e;
  if (p.kv_fp8) {  // (fp8 storage needs head_dim 128)
    if (d != 128) return cudaErrorInvalidValue;
    e = dtype == 0 ? launch_pdl(append_kernel<__half, 128, true>, grid, 128, 0, s, p)
                   : launch_pdl(append_kernel<__nv_bfloat16, 128, true>, grid, 128, 0, s, p);
  } else if (dtype == 0) {
    e = d == 64 ? launch_pdl(append_kernel<__half, 64, false>, grid, 128, 0, s, p)
                : launch_pdl(append_kernel<__half, 128, false>, grid, 128, 0, s, p);
  } else {
    e = d == 64 ? launch_pdl(append_kernel<__nv_bfloat16, 64, false>, grid, 128, 0, s, p)
                : launch_pdl(append_kernel<__nv_bfloat16, 128, false>, grid, 128, 0, s, p);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace spd
