// Query-aware page selection for sm_103a ("LServe long-sequence LLM serving
// system", section 2.1 dynamic sparsity; section 3.2 reusable selector and
// dynamic budget).
//
// Score.  For a logical page j with channel-wise key bounds kmin <= kmax and
// a query head q,
//     s(j) = sum_c max(q_c kmax_c, q_c kmin_c) = sum_c (q+_c kmax_c + q-_c kmin_c)
// with q+ = max(q, 0), q- = min(q, 0): for q_c >= 0 the larger product is the
// one with kmax, for q_c < 0 the one with kmin.  So the score is a dot
// product of the page's 2d-long metadata row [kmin ; kmax] with [q- ; q+],
// and the G heads of a kv head make it a [pages x 2d] x [2d x G] contraction:
// mma.sync m16n8k16 with the pages as M, the heads (padded to 8) as N.  The
// products of 16-bit values are exact; the sum is fp32.  S(j) = max over the
// G heads.
//
// Fragments are loaded straight from global memory: the k order inside each
// pair of k-steps is permuted (both operands alike, which leaves the sum
// unchanged) so that every thread reads 16 contiguous bytes of a metadata
// row per load (8 with fp8 E4M3 metadata, widened exactly to fp16, q then
// narrowed to fp16 for fp16 products; the per-head key scale is positive and
// leaves the ranking unchanged).
//
// Top-k.  Each scoring CTA writes its pages' scores, then takes a ticket;
// the last CTA of a (sequence, head) runs an exact radix select for the
// K_sel - 1 highest scores among pages [0, nL-1) (ties to the lower page
// index, -0 folded onto +0), adds the newest page nL-1, and writes the set in
// ascending order.  No CTA ever waits for another.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "ptx.cuh"
#include "spd_internal.h"
#include "topk.cuh"

namespace spd {
namespace {

constexpr int kPagesPerWarp = 16;
constexpr int kPagesPerCta = kSelWarps * kPagesPerWarp;  // 128

template <typename T> struct IsBf { static constexpr bool v = false; };
template <> struct IsBf<__nv_bfloat16> { static constexpr bool v = true; };

// Strictly negative 16-bit float (sign set, magnitude nonzero; -0 counts as
// non-negative).  Same bit test for fp16 and bf16; written without branches.
template <typename T> struct Neg {
  static __device__ __forceinline__ bool neg(uint16_t b) {
    return ((b >> 15) & (uint32_t)((b & 0x7fffu) != 0u)) != 0u;
  }
};

__device__ __forceinline__ void set_err(int *err, int code, int a, int b, int c) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}


// Exclusive scan over the CTA (kSelThreads threads); *total = sum.
__device__ __forceinline__ int cta_excl_scan(int v, int *sh, int *total) {
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
    int w = lane < kSelWarps ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kSelWarps) sh[lane] = w;
    if (lane == kSelWarps - 1) sh[32] = w;
  }
  __syncthreads();
  const int res = x - v + (warp > 0 ? sh[warp - 1] : 0);
  *total = sh[32];
  __syncthreads();
  return res;
}

// Fallback for more candidates than shared memory holds: the same radix
// select, reading the keys from global memory in every pass.
__device__ int cta_topk_global(const float *sc, int n, int k, int *out) {
  __shared__ int ghist[256];
  __shared__ int gsh[33];
  __shared__ uint32_t g_prefix;
  __shared__ int g_remaining;
  const int tid = threadIdx.x;
  if (tid == 0) {
    g_prefix = 0;
    g_remaining = k;
  }
  uint32_t mask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    ghist[tid] = 0;
    __syncthreads();
    const uint32_t prefix = g_prefix;
    for (int j = tid; j < n; j += kSelThreads) {
      const uint32_t u = score_key(__ldcg(sc + j));
      if ((u & mask) == prefix) atomicAdd(&ghist[(u >> shift) & 0xffu], 1);
    }
    __syncthreads();
    const int b = 255 - tid;
    const int hb = ghist[b];
    int tot;
    const int above = cta_excl_scan(hb, gsh, &tot);
    const int rem = g_remaining;
    __syncthreads();
    if (above < rem && rem <= above + hb) {
      g_remaining = rem - above;
      g_prefix = prefix | ((uint32_t)b << shift);
    }
    mask |= 0xffu << shift;
    __syncthreads();
  }
  const uint32_t T = g_prefix;
  const int take_eq = g_remaining;
  int eq_seen = 0, taken = 0;
  for (int base = 0; base < n; base += kSelThreads) {
    const int j = base + tid;
    const uint32_t u = j < n ? score_key(__ldcg(sc + j)) : 0u;
    const int gt = j < n && u > T;
    const int eq = j < n && u == T;
    int tot_eq, tot_take;
    const int eq_rank = cta_excl_scan(eq, gsh, &tot_eq) + eq_seen;
    const int take = gt || (eq && eq_rank < take_eq);
    const int pos = cta_excl_scan(take, gsh, &tot_take) + taken;
    if (take && pos < k) out[pos] = j;
    eq_seen += tot_eq;
    taken += tot_take;
  }
  return taken;
}

// kF8: the metadata rows hold fp8 E4M3 codes, widened exactly to T as they load
template <typename T, int D, int G, bool kF8>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const __grid_constant__ SelectParams p) {
  __shared__ int s_last;
  // the group's [q- ; q+] rows (2D elements each), padded by 32 bytes so that a
  // warp's fragment loads meet at most two to a bank
  constexpr int QS = 2 * D + 16;
  __shared__ __align__(16) uint16_t q_s[G * QS];
  __shared__ uint32_t ks[kPagesPerCta];  // this CTA's score keys, for its bound
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int i = 0;
  while (i + 1 < p.n_seqs && p.seqs[i + 1].chunk_off <= (int)blockIdx.x) ++i;
  const SelectSeq s = p.seqs[i];
  const int local = blockIdx.x - s.chunk_off;
  const int per_head = max(1, s.n_chunks);
  const int hd = local / per_head;
  const int chunk = local % per_head;
  const int h = p.dyn_kv[hd];
  int *out = p.selection + ((size_t)s.slot * p.Hd + hd) * p.ksel_max;
  // Metadata and the page table are read before the wait for the previous
  // kernel on the stream only when the host knows that kernel cannot have
  // written this context's cache (p.early); q and every write come after it.
  const bool early = p.early && s.n_chunks != 0;
  if (threadIdx.x == 0 && s.n_chunks != 0)  // a hint: q is read only after the wait
    prefetch_l2_bulk(static_cast<const uint16_t *>(p.q) + ((size_t)s.qrow * p.Hq + h * G) * D,
                     G * D * 2);
  if (!early) {
    pdl_wait();
    pdl_launch_dependents();
  }
  if (s.n_chunks == 0) {
    // every page is kept (nL <= K_sel), or only the newest one (K_sel = 1)
    if (s.nL <= s.K_sel) {
      for (int j = tid; j < s.nL; j += kSelThreads) out[j] = j;
    } else if (tid == 0) {
      out[0] = s.nL - 1;
    }
    return;
  }
  const int n = s.nL - 1;  // candidate pages
  float *scores = p.scores + ((size_t)i * p.Hd + hd) * p.score_stride;
  constexpr int KSTEPS = 2 * D / 16;
  constexpr int PAIRS = KSTEPS / 2;
  const int g8 = lane >> 2, t4 = lane & 3;

  // ---- this warp's 16 pages: metadata rows straight into A fragments ----
  // k-step pair s2 covers metadata elements [32*s2, 32*s2 + 32); thread t4
  // of a k-step pair owns elements 32*s2 + 8*t4 + [0, 8): the first four are
  // its k indices {2t4, 2t4+1, 2t4+8, 2t4+9} of step 2*s2, the last four the
  // same k indices of step 2*s2+1.
  const int j0 = chunk * kPagesPerCta + warp * kPagesPerWarp;
  bool ok[2] = {false, false};
  uint4 ra[PAIRS], rb[PAIRS];
  if (j0 < n) {
    // a metadata row is 2D elements of 2 bytes, or of 1 byte (fp8)
    const uint8_t *meta = static_cast<const uint8_t *>(p.meta);
    constexpr int kRowBytes = 2 * D * (kF8 ? 1 : 2);
    const uint8_t *rowp[2] = {nullptr, nullptr};
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int j = j0 + g8 + 8 * hh;
      if (j < n) {
        const int blk = j / p.R;
        const int phys = p.page_table[(size_t)s.slot * p.max_pp + blk];
        if (phys < 0 || phys >= p.num_phys) {
          set_err(p.err, kDevBadPhys, s.slot, blk, phys);
        } else {
          ok[hh] = true;
          rowp[hh] = meta + (((size_t)phys * p.Hd + hd) * p.R + (j % p.R)) * kRowBytes;
        }
      }
    }
#pragma unroll
    for (int s2 = 0; s2 < PAIRS; ++s2) {
      if constexpr (kF8) {
        // the same 8 elements: 8 bytes, widened pair by pair
        const uint2 a8 = ok[0] ? __ldg(reinterpret_cast<const uint2 *>(rowp[0]) + 4 * s2 + t4)
                               : make_uint2(0, 0);
        const uint2 b8 = ok[1] ? __ldg(reinterpret_cast<const uint2 *>(rowp[1]) + 4 * s2 + t4)
                               : make_uint2(0, 0);
        ra[s2] = make_uint4(e4m3x2_to<__half>(a8.x), e4m3x2_to<__half>(a8.x >> 16), e4m3x2_to<__half>(a8.y),
                            e4m3x2_to<__half>(a8.y >> 16));
        rb[s2] = make_uint4(e4m3x2_to<__half>(b8.x), e4m3x2_to<__half>(b8.x >> 16), e4m3x2_to<__half>(b8.y),
                            e4m3x2_to<__half>(b8.y >> 16));
      } else {
        ra[s2] = ok[0] ? __ldg(reinterpret_cast<const uint4 *>(rowp[0]) + 4 * s2 + t4)
                       : make_uint4(0, 0, 0, 0);
        rb[s2] = ok[1] ? __ldg(reinterpret_cast<const uint4 *>(rowp[1]) + 4 * s2 + t4)
                       : make_uint4(0, 0, 0, 0);
      }
    }
  }
  if (early) {
    pdl_wait();
    pdl_launch_dependents();
  }

  // ---- B operand: [q- ; q+] over the 2D metadata elements, heads as columns ----
  uint32_t qb[KSTEPS][2];
  {
    // the group's G query rows: one coalesced 16-byte load per thread
    const uint4 *qg = reinterpret_cast<const uint4 *>(
        reinterpret_cast<const uint16_t *>(p.q) + ((size_t)s.qrow * p.Hq + h * G) * D);
    // staging: 8 elements of q per thread, split into q- (the kmin half of a
    // metadata row) and q+ (the kmax half)
    for (int x = tid; x < G * D / 8; x += kSelThreads) {
      const uint4 v = qg[x];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t neg[4], pos[4];
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const uint16_t lo = (uint16_t)(w[y] & 0xffffu), hi = (uint16_t)(w[y] >> 16);
        const bool nl = Neg<T>::neg(lo), nh = Neg<T>::neg(hi);
        neg[y] = (nl ? lo : 0u) | ((nh ? (uint32_t)hi : 0u) << 16);
        pos[y] = (nl ? 0u : lo) | ((nh ? 0u : (uint32_t)hi) << 16);
        if constexpr (kF8) {  // fp16 products with the widened fp8 metadata
          neg[y] = to_f16x2<T>(neg[y]);
          pos[y] = to_f16x2<T>(pos[y]);
        }
      }
      uint16_t *row = &q_s[(x / (D / 8)) * QS + (x % (D / 8)) * 8];
      *reinterpret_cast<uint4 *>(row) = make_uint4(neg[0], neg[1], neg[2], neg[3]);
      *reinterpret_cast<uint4 *>(row + D) = make_uint4(pos[0], pos[1], pos[2], pos[3]);
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      uint2 f = make_uint2(0u, 0u);
      if (g8 < G) {
        const int base = 32 * (kk >> 1) + 8 * t4 + 4 * (kk & 1);  // metadata element
        f = *reinterpret_cast<const uint2 *>(&q_s[g8 * QS + base]);
      }
      qb[kk][0] = f.x;
      qb[kk][1] = f.y;
    }
  }

  // ---- score 16 pages per warp ----
  if (j0 < n) {
    // two accumulators halve the chain of dependent MMAs
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s2 = 0; s2 < PAIRS; ++s2) {
      const uint32_t a0[4] = {ra[s2].x, rb[s2].x, ra[s2].y, rb[s2].y};
      mma_16816<(kF8 ? false : IsBf<T>::v)>(acc, a0, qb[2 * s2][0], qb[2 * s2][1]);
      const uint32_t a1[4] = {ra[s2].z, rb[s2].z, ra[s2].w, rb[s2].w};
      mma_16816<(kF8 ? false : IsBf<T>::v)>(acc2, a1, qb[2 * s2 + 1][0], qb[2 * s2 + 1][1]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] += acc2[e];
    // acc: [0],[1] page g8 heads 2t4, 2t4+1; [2],[3] page g8+8
    float s0 = -CUDART_INF_F, s1 = -CUDART_INF_F;
    if (2 * t4 < G) {
      s0 = acc[0];
      s1 = acc[2];
    }
    if (2 * t4 + 1 < G) {
      s0 = fmaxf(s0, acc[1]);
      s1 = fmaxf(s1, acc[3]);
    }
    s0 = fmaxf(s0, __shfl_xor_sync(0xffffffffu, s0, 1));
    s0 = fmaxf(s0, __shfl_xor_sync(0xffffffffu, s0, 2));
    s1 = fmaxf(s1, __shfl_xor_sync(0xffffffffu, s1, 1));
    s1 = fmaxf(s1, __shfl_xor_sync(0xffffffffu, s1, 2));
    if (t4 == 0) {
      if (ok[0]) scores[j0 + g8] = s0;
      if (ok[1]) scores[j0 + g8 + 8] = s1;
      ks[warp * kPagesPerWarp + g8] = ok[0] ? score_key(s0) : 0u;
      ks[warp * kPagesPerWarp + g8 + 8] = ok[1] ? score_key(s1) : 0u;
    }
  }

  // ---- this chunk's bound: its tau_m-th largest score key ----
  // A full chunk holds tau_m keys at or above it, and tau_m x full chunks is
  // at least the number of pages to choose, so the smallest bound over the
  // chunks is a key that every chosen page reaches.
  if (s.tau_m > 0) {
    __syncthreads();
    if (warp == 0) {
      uint32_t a[kPagesPerCta / 32];
#pragma unroll
      for (int x = 0; x < kPagesPerCta / 32; ++x) a[x] = ks[lane + 32 * x];
      uint32_t v = 0u;
      for (int it = 0; it < s.tau_m; ++it) {  // take the largest tau_m times
        uint32_t lm = a[0];
#pragma unroll
        for (int x = 1; x < kPagesPerCta / 32; ++x) lm = max(lm, a[x]);
        v = __reduce_max_sync(0xffffffffu, lm);
        const unsigned who = __ballot_sync(0xffffffffu, lm == v);
        if (lane == __ffs(who) - 1) {
          bool done = false;
#pragma unroll
          for (int x = 0; x < kPagesPerCta / 32; ++x)
            if (!done && a[x] == v) {
              a[x] = 0u;
              done = true;
            }
        }
      }
      if (lane == 0) {
        const bool full = (chunk + 1) * kPagesPerCta <= n;
        p.bounds[((size_t)i * p.Hd + hd) * p.bound_stride + chunk] = full ? v : 0xffffffffu;
      }
    }
  }

  if (p.score_only) return;  // the decode kernel of this step selects from the scores

  // ---- the last scoring CTA of this (sequence, head) selects ----
  __syncthreads();  // every score of this CTA precedes the release below
  if (tid == 0) {
    const int prev = atom_add_acq_rel_gpu(&p.tickets[i * p.Hd + hd], 1);
    s_last = prev == s.n_chunks - 1;
  }
  __syncthreads();  // ... and the acquire above precedes every read below
  if (!s_last) return;
  // the other CTAs wrote their scores through the generic proxy; the top-k's
  // bulk copy reads them through the async proxy
  asm volatile("fence.proxy.async.global;" ::: "memory");
  const int k = s.K_sel - 1;
  int got;
  if (n <= kMaxKeys) {
    __shared__ __align__(16) uint8_t topk_smem[kTopkSmemBytes];
    got = cta_topk(scores, n, k, p.bounds + ((size_t)i * p.Hd + hd) * p.bound_stride,
                   s.tau_m > 0 ? s.n_chunks : 0, out, p.err, carve_topk_smem(topk_smem));
  } else {
    got = cta_topk_global(scores, n, k, out);
  }
  if (tid == 0) {
    out[k] = s.nL - 1;
    if (got != k) set_err(p.err, kDevTopkCount, s.slot, hd, got);
    p.tickets[i * p.Hd + hd] = 0;
  }
}

template <typename T, int D, bool kF8>
cudaError_t launch_g(const SelectParams &p, int G, cudaStream_t st) {
  const int grid = p.score_ctas;
  cudaError_t e;
  switch (G) {
    case 1: e = launch_pdl(select_kernel<T, D, 1, kF8>, grid, kSelThreads, 0, st, p); break;
    case 2: e = launch_pdl(select_kernel<T, D, 2, kF8>, grid, kSelThreads, 0, st, p); break;
    case 4: e = launch_pdl(select_kernel<T, D, 4, kF8>, grid, kSelThreads, 0, st, p); break;
    case 8: e = launch_pdl(select_kernel<T, D, 8, kF8>, grid, kSelThreads, 0, st, p); break;
    default: return cudaErrorInvalidValue;
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int select_pages_per_cta() { return kPagesPerCta; }

cudaError_t launch_select_fused(const SelectParams &p, int dtype, int d, int G, cudaStream_t s,
                                long long *n) {
  if (p.n_seqs == 0 || p.Hd == 0 || p.score_ctas == 0) return cudaSuccess;
  *n += 1;
  if (p.kv_fp8) {  // (fp8 storage needs head_dim 128)
    if (d != 128) return cudaErrorInvalidValue;
    return dtype == 0 ? launch_g<__half, 128, true>(p, G, s)
                      : launch_g<__nv_bfloat16, 128, true>(p, G, s);
  }
  if (dtype == 0)
    return d == 64 ? launch_g<__half, 64, false>(p, G, s) : launch_g<__half, 128, false>(p, G, s);
  return d == 64 ? launch_g<__nv_bfloat16, 64, false>(p, G, s)
                 : launch_g<__nv_bfloat16, 128, false>(p, G, s);
}

}  // namespace spd
