// CUDA kernels for sparse paged decode attention (sm_103a).
//
//   pt_write      page-table entries from the host runtime's allocator
//   append        write new K/V rows (paged pool for dynamic heads, sink +
//                 ring for streaming heads) and fold them into the logical
//                 page's channel-wise key min/max ("LServe long-sequence LLM
//                 serving system", section 2.1, min-max pooling)
//   score         S(j) = max_h sum_c max(q_h[c] kmax_j[c], q_h[c] kmin_j[c])
//                 per logical page (query-aware selection, section 2.1)
//   topk          exact radix select of the K_sel - 1 best pages, ties to the
//                 lower index, plus the page holding the newest token
//   decode        split-K GQA decode over the unified work list (dynamic
//                 page chunks and streaming sink/window chunks), online
//                 softmax in fp32, partial (o, m, l) per split
//   combine       log-sum-exp merge of the split partials (the row max /
//                 row sum export of the Novita KV-sparsity article's modified
//                 FlashAttention, "attention mechanism modifications")
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

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
  for (int i = threadIdx.x; i < p.n; i += blockDim.x) {
    const PtUpdate u = p.upd[i];
    p.page_table[(size_t)u.slot * p.max_pp + u.index] = u.phys;
  }
}

// ---- append + metadata -----------------------------------------------------
// Dynamic part: one CTA per (sequence, touched logical page, dynamic head);
// thread c owns channel c.  Streaming part: one CTA per (sequence, head).
template <typename T, int D>
__global__ void __launch_bounds__(128) append_kernel(const __grid_constant__ AppendParams p) {
  const int c = threadIdx.x;
  const T *kin = static_cast<const T *>(p.k);
  const T *vin = static_cast<const T *>(p.v);
  const int n = p.n_tokens;
  if ((int)blockIdx.x < p.dyn_ctas) {
    int i = 0;
    while (i + 1 < p.n_seqs && p.seqs[i + 1].cta_off <= (int)blockIdx.x) ++i;
    const AppendSeq s = p.seqs[i];
    const int local = blockIdx.x - s.cta_off;
    const int hd = local % p.Hd;
    const int j = s.L_old / p.ell + local / p.Hd;  // logical page
    const int h = p.dyn_kv[hd];
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
    T *kp = static_cast<T *>(p.k_pool);
    T *vp = static_cast<T *>(p.v_pool);
    T *meta = static_cast<T *>(p.meta) +
              (((size_t)phys * p.Hd + hd) * p.R + (j % p.R)) * 2 * D;
    if (c >= D) return;
    T bmin, bmax;
    float vmin, vmax;
    int t = max(t0, s.L_old);
    if (t0 < s.L_old) {  // the page already holds tokens: start from its metadata
      bmin = meta[c];
      bmax = meta[D + c];
      vmin = Elem<T>::to_f(bmin);
      vmax = Elem<T>::to_f(bmax);
    } else {
      bmin = bmax = kin[(((size_t)i * n + (t - s.L_old)) * p.Hkv + h) * D + c];
      vmin = vmax = Elem<T>::to_f(bmin);
    }
    for (; t < t1; ++t) {
      const size_t src = (((size_t)i * n + (t - s.L_old)) * p.Hkv + h) * D + c;
      const T kx = kin[src];
      const size_t dst = (page_base + (t % p.P)) * D + c;
      kp[dst] = kx;
      vp[dst] = vin[src];
      const float x = Elem<T>::to_f(kx);
      if (x < vmin) { vmin = x; bmin = kx; }
      if (x > vmax) { vmax = x; bmax = kx; }
    }
    meta[c] = bmin;
    meta[D + c] = bmax;
  } else {
    const int b = blockIdx.x - p.dyn_ctas;
    const int i = b / p.Hs, hs = b % p.Hs;
    const int h = p.str_kv[hs];
    const AppendSeq s = p.seqs[i];
    const int L_new = s.L_old + n;
    const int SW = p.S + p.W;
    T *sk = static_cast<T *>(p.stream_k) + ((size_t)s.slot * p.Hs + hs) * SW * D;
    T *sv = static_cast<T *>(p.stream_v) + ((size_t)s.slot * p.Hs + hs) * SW * D;
    // positions that can still be read: sink t < S, window t >= L_new - W
    const int w0 = max(s.L_old, max(p.S, L_new - p.W));
    for (int t = s.L_old; t < L_new; ++t) {
      if (t >= p.S && t < w0) { t = w0 - 1; continue; }
      const int slot = t < p.S ? t : p.S + (t - p.S) % p.W;
      const size_t src = (((size_t)i * n + (t - s.L_old)) * p.Hkv + h) * D;
      for (int cc = c; cc < D; cc += blockDim.x) {
        sk[(size_t)slot * D + cc] = kin[src + cc];
        sv[(size_t)slot * D + cc] = vin[src + cc];
      }
    }
  }
}

// ---- page scoring ------------------------------------------------------------
// One CTA per (sequence, dynamic head, chunk of pages); one warp per page;
// lane owns D/32 consecutive channels.
template <typename T, int D, int G>
__global__ void __launch_bounds__(256) score_kernel(const __grid_constant__ SelectParams p) {
  constexpr int CPL = D / 32;
  int i = 0;
  while (i + 1 < p.n_seqs && p.seqs[i + 1].chunk_off <= (int)blockIdx.x) ++i;
  const SelectSeq s = p.seqs[i];
  const int local = blockIdx.x - s.chunk_off;
  const int hd = local / s.n_chunks;
  const int chunk = local % s.n_chunks;
  const int h = p.dyn_kv[hd];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T *qp = static_cast<const T *>(p.q) + ((size_t)s.qrow * p.Hq + h * G) * D;
  float q[G][CPL];
#pragma unroll
  for (int g = 0; g < G; ++g) load_row<T, CPL>(qp + g * D + lane * CPL, q[g]);
  const int j_end = min(s.nL - 1, (chunk + 1) * p.pages_per_chunk);
  float *out = p.scores + ((size_t)i * p.Hd + hd) * p.max_nL;
  const T *meta = static_cast<const T *>(p.meta);
  for (int j = chunk * p.pages_per_chunk + warp; j < j_end; j += 8) {
    const int blk = j / p.R;
    const int phys = p.page_table[(size_t)s.slot * p.max_pp + blk];
    if (phys < 0 || phys >= p.num_phys) {
      if (lane == 0) {
        set_err(p.err, kDevBadPhys, s.slot, blk, phys);
        out[j] = -CUDART_INF_F;
      }
      continue;
    }
    const T *row = meta + (((size_t)phys * p.Hd + hd) * p.R + (j % p.R)) * 2 * D;
    float mn[CPL], mx[CPL];
    load_row<T, CPL>(row + lane * CPL, mn);
    load_row<T, CPL>(row + D + lane * CPL, mx);
    float best = -CUDART_INF_F;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < CPL; ++e) acc += fmaxf(q[g][e] * mx[e], q[g][e] * mn[e]);
      acc = warp_sum(acc);
      best = g == 0 ? acc : fmaxf(best, acc);
    }
    if (lane == 0) out[j] = best;
  }
}

// ---- exact top-k ---------------------------------------------------------------
// Order-preserving map float -> uint32 (larger float, larger key).  -0 is
// folded onto +0 so that equal scores are equal keys; NaN maps to the lowest
// key.
__device__ __forceinline__ uint32_t score_key(float f) {
  if (f != f) return 0u;
  if (f == 0.f) f = 0.f;
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive scan of one int per thread over a 1024-thread block; *total gets
// the block sum.  `sh` holds 33 ints.
__device__ __forceinline__ int block_excl_scan(int v, int *sh, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;  // inclusive prefix of warp totals
    if (lane == 31) sh[32] = w;
  }
  __syncthreads();
  const int res = x - v + (warp > 0 ? sh[warp - 1] : 0);
  *total = sh[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(1024) topk_kernel(const __grid_constant__ SelectParams p) {
  __shared__ int hist[256];
  __shared__ int sh[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int i = blockIdx.x / p.Hd, hd = blockIdx.x % p.Hd;
  const SelectSeq s = p.seqs[i];
  int *out = p.selection + ((size_t)s.slot * p.Hd + hd) * p.ksel_max;
  const int tid = threadIdx.x;
  if (s.nL <= s.K_sel) {
    for (int j = tid; j < s.nL; j += blockDim.x) out[j] = j;
    return;
  }
  const int k = s.K_sel - 1;  // best pages besides the newest one
  const int n = s.nL - 1;     // candidate pages
  if (tid == 0) out[k] = s.nL - 1;
  if (k == 0) return;
  const float *sc = p.scores + ((size_t)i * p.Hd + hd) * p.max_nL;
  if (tid == 0) {
    s_prefix = 0;
    s_remaining = k;
  }
  uint32_t mask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int j = tid; j < n; j += blockDim.x) {
      const uint32_t u = score_key(sc[j]);
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 0xffu], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int rem = s_remaining, cum = 0, b = 255;
      for (; b > 0; --b) {
        if (cum + hist[b] >= rem) break;
        cum += hist[b];
      }
      s_remaining = rem - cum;
      s_prefix = prefix | ((uint32_t)b << shift);
    }
    mask |= 0xffu << shift;
    __syncthreads();
  }
  const uint32_t T = s_prefix;
  const int take_eq = s_remaining;  // keys equal to T to keep, lowest index first
  int eq_seen = 0, taken = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int j = base + tid;
    const uint32_t u = j < n ? score_key(sc[j]) : 0u;
    const int gt = j < n && u > T;
    const int eq = j < n && u == T;
    int tot_eq, tot_take;
    const int eq_rank = block_excl_scan(eq, sh, &tot_eq) + eq_seen;
    const int take = gt || (eq && eq_rank < take_eq);
    const int pos = block_excl_scan(take, sh, &tot_take) + taken;
    if (take && pos < k) out[pos] = j;
    eq_seen += tot_eq;
    taken += tot_take;
  }
  if (tid == 0 && taken != k) set_err(p.err, kDevTopkCount, s.slot, hd, taken);
}

// ---- split-K decode -------------------------------------------------------------
// One CTA (4 warps) per work item.  Lane owns CPL = D/32 consecutive channels;
// each warp runs its own online softmax over its share of the item's tokens;
// the four warps are merged through shared memory and the item's partial
// (unnormalised o, row max m in log2 units, row sum l) is written out.
template <typename T, int D, int G>
__global__ void __launch_bounds__(128) decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int CPL = D / 32;
  constexpr int NW = 4;
  __shared__ float sm_m[NW][G], sm_l[NW][G];
  __shared__ float sm_o[NW][G][D];
  const int item = blockIdx.x;
  int i = 0;
  while (i + 1 < p.n_seqs && p.seqs[i + 1].item_off <= item) ++i;
  const DecodeSeq s = p.seqs[i];
  int local = item - s.item_off;
  const bool dyn = local < p.Hd * s.ns_dyn;
  int sub, split;
  if (dyn) {
    sub = local / s.ns_dyn;
    split = local % s.ns_dyn;
  } else {
    local -= p.Hd * s.ns_dyn;
    sub = local / s.ns_str;
    split = local % s.ns_str;
  }
  const int h = dyn ? p.dyn_kv[sub] : p.str_kv[sub];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  float q[G][CPL];
  const T *qp = static_cast<const T *>(p.q) + ((size_t)i * p.Hq + h * G) * D;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    load_row<T, CPL>(qp + g * D + lane * CPL, q[g]);
#pragma unroll
    for (int e = 0; e < CPL; ++e) q[g][e] *= p.scale_log2;
  }
  float m[G], l[G], acc[G][CPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -CUDART_INF_F;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[g][e] = 0.f;
  }

  auto consume = [&](const T *krow, const T *vrow) {
    float kf[CPL], vf[CPL];
    load_row<T, CPL>(krow + lane * CPL, kf);
    load_row<T, CPL>(vrow + lane * CPL, vf);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float z = 0.f;
#pragma unroll
      for (int e = 0; e < CPL; ++e) z += q[g][e] * kf[e];
      z = warp_sum(z);
      const float mn = fmaxf(m[g], z);
      const float corr = exp2f(m[g] - mn);
      const float pz = exp2f(z - mn);
      l[g] = l[g] * corr + pz;
#pragma unroll
      for (int e = 0; e < CPL; ++e) acc[g][e] = acc[g][e] * corr + pz * vf[e];
      m[g] = mn;
    }
  };

  if (dyn) {
    const T *kp = static_cast<const T *>(p.k_pool);
    const T *vp = static_cast<const T *>(p.v_pool);
    const int *sel = p.selection + ((size_t)s.slot * p.Hd + sub) * p.ksel_max;
    const int n_att = s.sel_count + (((s.L + p.ell - 1) / p.ell) - s.nL0);
    const int p0 = split * s.pps, p1 = min(n_att, p0 + s.pps);
    for (int pi = p0; pi < p1; ++pi) {
      const int j = pi < s.sel_count ? sel[pi] : s.nL0 + (pi - s.sel_count);
      const int blk = j / p.R;
      if (j < 0 || blk >= p.max_pp) {
        if (threadIdx.x == 0) set_err(p.err, kDevBadSelection, s.slot, sub, j);
        continue;
      }
      const int phys = p.page_table[(size_t)s.slot * p.max_pp + blk];
      if (phys < 0 || phys >= p.num_phys) {
        if (threadIdx.x == 0) set_err(p.err, kDevBadPhys, s.slot, blk, phys);
        continue;
      }
      const size_t base = ((((size_t)phys * p.Hd + sub) * p.P) + (j % p.R) * p.ell) * D;
      const int nt = min(p.ell, s.L - j * p.ell);
      for (int r = warp; r < nt; r += NW) consume(kp + base + (size_t)r * D, vp + base + (size_t)r * D);
    }
  } else {
    const T *sk = static_cast<const T *>(p.stream_k) + ((size_t)s.slot * p.Hs + sub) * (p.S + p.W) * D;
    const T *sv = static_cast<const T *>(p.stream_v) + ((size_t)s.slot * p.Hs + sub) * (p.S + p.W) * D;
    const int n_tok = min(s.L, p.S + p.W);
    const bool all = s.L <= p.S + p.W;
    const int v0 = split * s.tps, v1 = min(n_tok, v0 + s.tps);
    for (int v = v0 + warp; v < v1; v += NW) {
      const int t = (all || v < p.S) ? v : s.L - p.W + (v - p.S);
      const int slot = t < p.S ? t : p.S + (t - p.S) % p.W;
      consume(sk + (size_t)slot * D, sv + (size_t)slot * D);
    }
  }

  // merge the warps
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      sm_m[warp][g] = m[g];
      sm_l[warp][g] = l[g];
    }
#pragma unroll
    for (int e = 0; e < CPL; ++e) sm_o[warp][g][lane * CPL + e] = acc[g][e];
  }
  __syncthreads();
  for (int x = threadIdx.x; x < G * D; x += blockDim.x) {
    const int g = x / D, c = x % D;
    float M = sm_m[0][g];
#pragma unroll
    for (int w = 1; w < NW; ++w) M = fmaxf(M, sm_m[w][g]);
    float o = 0.f, lsum = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = exp2f(sm_m[w][g] - M);
        o += f * sm_o[w][g][c];
        lsum += f * sm_l[w][g];
      }
    }
    p.part_o[((size_t)item * G + g) * D + c] = o;
    if (c == 0) p.part_ml[(size_t)item * G + g] = make_float2(M, lsum);
  }
}

// Combine: one CTA per (sequence, query head), thread c owns channel c.
template <int D, int G>
__global__ void __launch_bounds__(128) combine_kernel(const __grid_constant__ DecodeParams p) {
  const int i = blockIdx.x / p.Hq, hq = blockIdx.x % p.Hq;
  const int h = hq / G, g = hq % G;
  const DecodeSeq s = p.seqs[i];
  const int sub = p.kv_sub[h];
  int it0, ns;
  if (p.kv_kind[h] == 0) {
    it0 = s.item_off + sub * s.ns_dyn;
    ns = s.ns_dyn;
  } else {
    it0 = s.item_off + p.Hd * s.ns_dyn + sub * s.ns_str;
    ns = s.ns_str;
  }
  float M = -CUDART_INF_F;
  for (int k = 0; k < ns; ++k) M = fmaxf(M, p.part_ml[(size_t)(it0 + k) * G + g].x);
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float o = 0.f, lsum = 0.f;
    for (int k = 0; k < ns; ++k) {
      const float2 ml = p.part_ml[(size_t)(it0 + k) * G + g];
      if (ml.x == -CUDART_INF_F) continue;
      const float f = exp2f(ml.x - M);
      o += f * p.part_o[((size_t)(it0 + k) * G + g) * D + c];
      lsum += f * ml.y;
    }
    p.out[((size_t)i * p.Hq + hq) * D + c] = o / lsum;
  }
}

template <typename T, int D>
cudaError_t select_dispatch_g(const SelectParams &p, int G, cudaStream_t st) {
  if (p.score_ctas > 0) {
    switch (G) {
      case 1: score_kernel<T, D, 1><<<p.score_ctas, 256, 0, st>>>(p); break;
      case 2: score_kernel<T, D, 2><<<p.score_ctas, 256, 0, st>>>(p); break;
      case 4: score_kernel<T, D, 4><<<p.score_ctas, 256, 0, st>>>(p); break;
      case 8: score_kernel<T, D, 8><<<p.score_ctas, 256, 0, st>>>(p); break;
      default: return cudaErrorInvalidValue;
    }
  }
  topk_kernel<<<p.n_seqs * p.Hd, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename T, int D, int G>
cudaError_t decode_launch(const DecodeParams &p, cudaStream_t st) {
  decode_kernel<T, D, G><<<p.total_items, 128, 0, st>>>(p);
  combine_kernel<D, G><<<p.n_seqs * p.Hq, 128, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t decode_dispatch_g(const DecodeParams &p, int G, cudaStream_t st) {
  switch (G) {
    case 1: return decode_launch<T, D, 1>(p, st);
    case 2: return decode_launch<T, D, 2>(p, st);
    case 4: return decode_launch<T, D, 4>(p, st);
    case 8: return decode_launch<T, D, 8>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_pt_write(const PtWriteParams &p, cudaStream_t s) {
  pt_write_kernel<<<1, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams &p, int dtype, int d, cudaStream_t s) {
  const int grid = p.dyn_ctas + p.n_seqs * p.Hs;
  if (grid == 0) return cudaSuccess;
  if (dtype == 0) {
    if (d == 64) append_kernel<__half, 64><<<grid, 128, 0, s>>>(p);
    else append_kernel<__half, 128><<<grid, 128, 0, s>>>(p);
  } else {
    if (d == 64) append_kernel<__nv_bfloat16, 64><<<grid, 128, 0, s>>>(p);
    else append_kernel<__nv_bfloat16, 128><<<grid, 128, 0, s>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_select(const SelectParams &p, int dtype, int d, int G, cudaStream_t s) {
  if (p.n_seqs == 0 || p.Hd == 0) return cudaSuccess;
  if (dtype == 0)
    return d == 64 ? select_dispatch_g<__half, 64>(p, G, s) : select_dispatch_g<__half, 128>(p, G, s);
  return d == 64 ? select_dispatch_g<__nv_bfloat16, 64>(p, G, s)
                 : select_dispatch_g<__nv_bfloat16, 128>(p, G, s);
}

cudaError_t launch_decode(const DecodeParams &p, int dtype, int d, int G, cudaStream_t s) {
  if (p.n_seqs == 0) return cudaSuccess;
  if (dtype == 0)
    return d == 64 ? decode_dispatch_g<__half, 64>(p, G, s) : decode_dispatch_g<__half, 128>(p, G, s);
  return d == 64 ? decode_dispatch_g<__nv_bfloat16, 64>(p, G, s)
                 : decode_dispatch_g<__nv_bfloat16, 128>(p, G, s);
}

}  // namespace spd
