// Block-sparse causal attention of a prompt on the 5th-generation tensor
// cores ("LServe long-sequence LLM serving system", section 3.1: exact
// attention on the chosen key blocks of every query block).
//
// One CTA per (query block b, kv head, group of HC query heads), HC = 2 or 4:
// its HC x 64 query rows are MT = HC / 2 matrices of 128 rows (two heads x
// the block's 64 tokens each).  The chosen key blocks (ascending) go in
// pairs; per pair:
//   S_m  = Q_m . K^T            one tcgen05.mma chain over both blocks, M 128 x
//                               N 128 x K d (N 64 for a lone last block),
//                               fp32 in tensor memory, block u in columns
//                               64 u ..; per block j of the pair:
//   softmax, one row per thread: its 64 logits from tensor memory, the
//        causal mask on the diagonal block (and keys past the prompt), an
//        online max and sum in fp32 (base 2), and P written back over S in
//        tensor memory as a 16-bit high part and the 16-bit rounding of the
//        rest (so P . V keeps about 16 bits of each weight);
//   O_m += (P_hi + P_lo)_m . V_j  tcgen05.mma with A = P from tensor memory,
//                               M 128 x N 64 (per 64 channels) x K 64 keys.
// The running max only moves when a row's block max exceeds it by more than
// 2^8 (log2 units), so O is rescaled rarely; weights then stay below 2^8,
// and the final O / l is the same quotient (every term of O and of l carries
// the same factor).
//
// Warp roles: warps 0 .. 4 MT - 1 run the softmax (matrix warp / 4, tensor
// memory lanes 32 (warp % 4) ..), warps 4 MT + m issue matrix m's MMAs (the
// whole warp runs the issue loop with warp-uniform operands, one elected lane
// issues; the tensor pipe interleaves the matrices' two independent chains),
// warp 5 MT loads Q once and K / V into a two-stage ring, a pair of blocks
// per stage, by TMA (4-D maps over [L][heads][d], 64 x 64 boxes, 128-byte
// swizzle).  One N 128 chain for S reads Q once per two blocks (an N 64 MMA
// with both operands in shared memory is bound by shared-memory bandwidth);
// P . V of a pair's first block runs while the softmax of its second runs;
// matrix 1 starts once matrix 0's first softmax is done, so the matrices'
// softmax phases and tensor work alternate.  Every wait is bounded: a CTA
// that gives up records the error, lets the other roles leave, waits
// (bounded) for its copies and MMAs in flight and frees its tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "prefill.h"
#include "ptx.cuh"
#include "spd_internal.h"

namespace spd {
namespace {

constexpr uint32_t kTcWait = 1u << 22;  // bounded mbarrier polls
constexpr float kRescaleAbove = 8.f;    // log2 growth of a row max that moves it

// Shared memory (offsets from a 1024-byte aligned base).  Every matrix is a
// stack of 64-column sub-tiles of rows x 128 bytes, 128-byte swizzled.
template <int D, int HC>
struct TcSmem {
  static constexpr int MT = HC / 2;                 // 128-row matrices of the CTA
  static constexpr int KB = D / 64;                 // 64-column sub-tiles of a row
  static constexpr int kStages = 2;                 // K / V ring, a pair of blocks per stage
  static constexpr int kStageBytes = KB * 16384;    // K (or V) of two 64-row blocks
  static constexpr int kQ = 0;                      // [MT][KB][128 x 128 B]
  static constexpr int kK = kQ + MT * KB * 16384;   // [stage][KB][block u][64 x 128 B]
  static constexpr int kV = kK + kStages * kStageBytes;  // [stage][block u][KB][64 x 128 B]
  static constexpr int kBars = kV + kStages * kStageBytes;
  // mbarriers: Q, K full, V full, K/V empty (per stage), S full (per matrix,
  // once per pair), P full (per matrix and block of the pair), O done (per
  // matrix and block), pair done (per matrix and pair), O final (per matrix,
  // once), drain.  A parity wait only tells apart phases one apart: every
  // waiter below is at most one completion behind the barrier, which is why
  // the end of O and the end of a pair have barriers of their own (O done
  // completes once per block: a wait for the second block of a pair, or for
  // the last block, could otherwise meet a phase two completions back).
  static constexpr int kBarQ = 0;
  static constexpr int kBarKF = 1;
  static constexpr int kBarVF = kBarKF + kStages;
  static constexpr int kBarKE = kBarVF + kStages;
  static constexpr int kBarSF = kBarKE + kStages;
  static constexpr int kBarPF = kBarSF + MT;
  static constexpr int kBarOD = kBarPF + 2 * MT;
  static constexpr int kBarOP = kBarOD + MT;
  static constexpr int kBarOF = kBarOP + MT;
  static constexpr int kBarDR = kBarOF + MT;  // per MMA warp
  // matrix 1 starts once matrix 0's first softmax is done (single use)
  static constexpr int kBarLag = kBarDR + MT;
  static constexpr int kNumBars = kBarLag + 1;
  static constexpr int kMisc = kBars + 8 * kNumBars;  // tmem base, fail flag
  static constexpr int kBytes = kMisc + 16 + 1024;    // + alignment slack
  // tensor-memory columns: S / P of matrix m, buffer u at 128 m + 64 u;
  // O_m at 128 MT + D m
  static constexpr int kCols = MT * (128 + D);
  static constexpr int kAlloc = kCols <= 256 ? 256 : 512;
  // warps: softmax 0 .. 4 MT - 1, MMA issue 4 MT .. 5 MT - 1 (one per
  // matrix), TMA 5 MT
  static constexpr int kMmaWarp = MT * 4, kLoadWarp = MT * 5;
  static constexpr int kThreads = (kLoadWarp + 1) * 32;
  static_assert(kBytes <= 232448, "shared memory");
  static_assert(kCols <= 512, "tensor memory");
};

__device__ __forceinline__ void pf_set_err(int *err, int code, int a, int b, int c) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}

// Bounded wait for the phase of `parity` to complete; gives up early once
// another role of the CTA has raised the fail flag.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *fail) {
  for (uint32_t i = 0; i < kTcWait; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *fail) return false;
  }
  *fail = 1;
  return false;
}

// A pair of softmax weights split into 16-bit high parts (packed) and the
// 16-bit rounding of what is left (packed), element 0 in the low half.
template <typename T> struct PSplit;
template <> struct PSplit<__nv_bfloat16> {
  static constexpr bool bf16 = true;
  static __device__ __forceinline__ void run(float2 pp, uint32_t &hi, uint32_t &lo) {
    // bf16 high parts by truncation (the top 16 bits of each fp32 pattern),
    // so p - hi is exact in fp32; the rest is rounded to bf16
    const uint32_t b0 = __float_as_uint(pp.x), b1 = __float_as_uint(pp.y);
    hi = __byte_perm(b0, b1, 0x7632);
    const float2 r = f2_sub(pp, make_float2(__uint_as_float(b0 & 0xffff0000u),
                                            __uint_as_float(b1 & 0xffff0000u)));
    const __nv_bfloat162 l = __floats2bfloat162_rn(r.x, r.y);
    lo = *reinterpret_cast<const uint32_t *>(&l);
  }
};

template <> struct PSplit<__half> {
  static constexpr bool bf16 = false;
  static __device__ __forceinline__ void run(float2 pp, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(pp.x, pp.y);
    const float2 r = f2_sub(pp, __half22float2(h));
    const __half2 l = __floats2half2_rn(r.x, r.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
  }
};

// Bounded wait that the fail flag does not cut short (copies and MMAs in
// flight before the CTA frees its memory).
__device__ __forceinline__ bool tc_drain(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kTcWait; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

template <typename T, int D, int HC>
__global__ void __launch_bounds__(TcSmem<D, HC>::kThreads, 1)
    prefill_attn_tc_kernel(const __grid_constant__ PrefillParams p) {
  using Sm = TcSmem<D, HC>;
  constexpr int MT = Sm::MT, KB = Sm::KB, S = Sm::kStages;
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Sm::kBars);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Sm::kMisc);
  volatile int *fail = reinterpret_cast<volatile int *>(smem + Sm::kMisc + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the heaviest query blocks (most causal key blocks) first
  const int b = p.nb - 1 - (int)(blockIdx.x % p.nb), rest = blockIdx.x / p.nb;
  const int hk = rest % p.Hkv, hg = rest / p.Hkv;
  const int t0 = b * kPrefillBlock;
  const int h0 = hk * p.G + hg * HC;  // the CTA's first query head

  if (warp == Sm::kMmaWarp) tmem_alloc(tmem_slot, Sm::kAlloc);  // (the first MMA warp)
  if (tid == Sm::kLoadWarp * 32) {
    for (int x = 0; x < Sm::kNumBars; ++x)
      mbar_init(&bars[x], (x >= Sm::kBarPF && x < Sm::kBarOD)   ? 4    // P: one per softmax warp
                          : (x >= Sm::kBarKE && x < Sm::kBarSF) ? MT   // K/V empty: one per MMA warp
                          : x == Sm::kBarLag                    ? 4    // matrix 0's softmax warps
                                                                : 1);
    *fail = 0;
    fence_mbar_init();
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);  // warp-uniform
  pdl_wait();  // the block lists come from the selection kernel
  pdl_launch_dependents();
  const int *list = p.lists + ((size_t)hk * p.nb + b) * p.KB;
  const int n = p.dense ? b + 1 : min(b + 1, p.kblocks);
  const int np = (n + 1) / 2;  // pairs of chosen blocks (the last may hold one)

  if (warp == Sm::kLoadWarp) {
    // ---- TMA: Q once, then K and V of every pair of chosen blocks through
    // the ring.  K of a pair lands as one 128-row operand per 64-column
    // sub-tile (block u's rows at 64 u), V block after block. ----
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(&bars[Sm::kBarQ], MT * KB * 16384);
      for (int mm = 0; mm < MT; ++mm)
        for (int kb = 0; kb < KB; ++kb)
          for (int hh = 0; hh < 2; ++hh)  // rows 0-63: head 2 mm, rows 64-127: head 2 mm + 1
            tma_load_4d(smem + Sm::kQ + (mm * KB + kb) * 16384 + hh * 8192, &p.tm_q, 0, kb,
                        h0 + 2 * mm + hh, t0, &bars[Sm::kBarQ]);
      for (int pp = 0; pp < np && ok; ++pp) {
        const int s = pp % S, nbk = min(2, n - 2 * pp);
        if (pp >= S && !(ok = tc_wait(&bars[Sm::kBarKE + s], ((pp / S) - 1) & 1, fail))) break;
        for (int u = 0; u < nbk; ++u) {
          const int i = list[2 * pp + u];
          if (i < 0 || i > b) {  // (the selection never yields one: record it and leave)
            pf_set_err(p.err, kDevBadSelection, hk, b, i);
            *fail = 1;
            ok = false;
          }
        }
        if (!ok) break;
        mbar_arrive_expect_tx(&bars[Sm::kBarKF + s], nbk * KB * 8192);
        for (int u = 0; u < nbk; ++u)
          for (int kb = 0; kb < KB; ++kb)
            tma_load_4d(smem + Sm::kK + s * Sm::kStageBytes + kb * 16384 + u * 8192, &p.tm_k, 0,
                        kb, hk, list[2 * pp + u] * kPrefillBlock, &bars[Sm::kBarKF + s]);
        mbar_arrive_expect_tx(&bars[Sm::kBarVF + s], nbk * KB * 8192);
        for (int u = 0; u < nbk; ++u)
          for (int kb = 0; kb < KB; ++kb)
            tma_load_4d(smem + Sm::kV + s * Sm::kStageBytes + (u * KB + kb) * 8192, &p.tm_v, 0,
                        kb, hk, list[2 * pp + u] * kPrefillBlock, &bars[Sm::kBarVF + s]);
        ++issued;
      }
      if (!ok) {  // the copies still in flight land before the CTA leaves
        tc_drain(&bars[Sm::kBarQ], 0);
        for (int pp = issued > S ? issued - S : 0; pp < issued; ++pp) {
          tc_drain(&bars[Sm::kBarKF + pp % S], (pp / S) & 1);
          tc_drain(&bars[Sm::kBarVF + pp % S], (pp / S) & 1);
        }
      }
    }
  } else if (warp >= Sm::kMmaWarp) {
    // ---- MMA issue for matrix m (the whole warp, one elected lane issuing):
    // S_m of a pair of blocks in one MMA (N = 128), then P_m . V block by
    // block as the softmax releases them ----
    const int m = warp - Sm::kMmaWarp;
    const bool bf = PSplit<T>::bf16;
    const uint32_t idesc_s2 = umma_idesc_f16(bf, 128, 128, 0, 0);  // Q . K^T, a pair
    const uint32_t idesc_s1 = umma_idesc_f16(bf, 128, 64, 0, 0);   // Q . K^T, a lone block
    const uint32_t idesc_o = umma_idesc_f16(bf, 128, 64, 0, 1);    // P . V: V MN-major
    // base descriptors; a byte offset o inside the region adds o / 16
    const uint64_t dq = umma_desc_sw128(smem_u32(smem + Sm::kQ + m * KB * 16384), 16, 1024);
    const uint64_t dk = umma_desc_sw128(smem_u32(smem + Sm::kK), 16, 1024);
    const uint64_t dv = umma_desc_sw128(smem_u32(smem + Sm::kV), 16, 1024);
    const uint32_t t_o = tmem + 128 * MT + D * m;
    // every lane waits; the warp goes on only if all saw the phase
    auto wwait = [&](uint64_t *bar, uint32_t parity) {
      return __all_sync(0xffffffffu, tc_wait(bar, parity, fail));
    };
    // S_m of pair pp = Q_m . K^T over its one or two blocks: block u's logits
    // in columns 64 u .. 64 u + 63 of the matrix's S / P region
    auto issue_s = [&](int pp) {
      const uint64_t kt = dk + (uint64_t)(((pp % S) * Sm::kStageBytes) >> 4);
      const uint32_t idesc = n - 2 * pp >= 2 ? idesc_s2 : idesc_s1;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = (uint64_t)((((kk >> 2)) * 16384 + (kk & 3) * 32) >> 4);
        umma_f16_warp(tmem + 128 * m, dq + off, kt + off, idesc, kk > 0);
      }
      umma_commit_warp(&bars[Sm::kBarSF + m]);
    };
    bool ok = wwait(&bars[Sm::kBarQ], 0) && wwait(&bars[Sm::kBarKF], 0);
    // the matrices start half a step apart: their softmax phases and their
    // MMAs then alternate instead of meeting (both follow the same K / V
    // stages, so in step they wait at the same time and the tensor pipe idles)
    if (m == 1 && ok) ok = wwait(&bars[Sm::kBarLag], 0);
    const bool any = ok;
    if (ok) {
      tc_fence_after();
      issue_s(0);
    }
    for (int pp = 0; pp < np && ok; ++pp) {
      const int s = pp % S, nbk = min(2, n - 2 * pp);
      if (!(ok = wwait(&bars[Sm::kBarVF + s], (pp / S) & 1))) break;
      for (int u = 0; u < nbk; ++u) {
        const int j = 2 * pp + u;
        if (!(ok = wwait(&bars[Sm::kBarPF + 2 * m + u], pp & 1))) break;
        tc_fence_after();
        const uint64_t vt = dv + (uint64_t)((s * Sm::kStageBytes + u * KB * 8192) >> 4);
        const uint32_t pa = tmem + 128 * m + 64 * u;
#pragma unroll
        for (int half = 0; half < KB; ++half)
#pragma unroll
          for (int part = 0; part < 2; ++part)  // P_hi, then P_lo
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_f16_ts_warp(t_o + 64 * half, pa + 32 * part + 8 * kk,
                               vt + (uint64_t)((half * 8192 + kk * 2048) >> 4), idesc_o,
                               j > 0 || part > 0 || kk > 0);
        umma_commit_warp(&bars[Sm::kBarOD + m]);
      }
      if (!ok) break;
      umma_commit_warp(&bars[Sm::kBarOP + m]);
      if (pp == np - 1) umma_commit_warp(&bars[Sm::kBarOF + m]);
      umma_commit_warp(&bars[Sm::kBarKE + s]);  // the stage is free once both warps' MMAs are done
      if (pp + 1 < np) {
        // the next pair's S overwrites this pair's P: both P . V done first
        const int p1 = pp + 1;
        if (!(ok = wwait(&bars[Sm::kBarKF + p1 % S], (p1 / S) & 1))) break;
        if (!(ok = wwait(&bars[Sm::kBarOP + m], pp & 1))) break;
        tc_fence_after();
        issue_s(p1);
      }
    }
    if (any) {  // every MMA of this warp done before the CTA frees its memory
      umma_commit_warp(&bars[Sm::kBarDR + m]);
      if (lane == 0) tc_drain(&bars[Sm::kBarDR + m], 0);
    }
  } else {
    // ---- softmax: one query row per thread ----
    const int m = warp >> 2, row = 32 * (warp & 3) + lane;
    const int h_row = h0 + 2 * m + (row >> 6), t_row = t0 + (row & 63);
    const uint32_t lanes = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t t_o = lanes + 128 * MT + D * m;
    const float sc = p.scale_log2;
    float m_run = -CUDART_INF_F, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int u = j & 1;  // block u of pair j / 2: S / P columns 64 u ..
      const uint32_t t_s = lanes + 128 * m + 64 * u;
      const int i = list[j];
      // (the pair's S: for its second block this phase has already completed)
      ok = tc_wait(&bars[Sm::kBarSF + m], (j >> 1) & 1, fail);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;  // the tensor-memory accesses are warp-wide
      tc_fence_after();
      uint32_t s[64];
      tmem_ld64_sync(t_s, s);
      if (i == b) {
        // the diagonal block: keys after the row's token, or past the prompt, drop out
        const int lim = min(row & 63, p.L - 1 - i * kPrefillBlock);
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c > lim) s[c] = 0xff800000u;  // -inf
      }
      float mq[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) mq[k] = __uint_as_float(s[k]);
#pragma unroll
      for (int c = 4; c < 64; c += 8)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mq[k] = fmax3f(mq[k], __uint_as_float(s[c + 2 * k]), __uint_as_float(s[c + 2 * k + 1]));
      const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * sc;
      const bool need = mx > m_run + kRescaleAbove;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mx : m_run;
        const float alpha = m_run == -CUDART_INF_F ? 0.f : exp2f(m_run - m_new);
        if (j > 0) {  // O_m follows the new max once P_m(j - 1) . V has landed
          ok = tc_wait(&bars[Sm::kBarOD + m], (j - 1) & 1, fail);
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32_sync(t_o + 32 * c, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(t_o + 32 * c, o);
          }
          tmem_wait_st();
        }
        l_run *= alpha;
        m_run = m_new;
      }
      // weights 2^(s sc - m) (masked keys: 2^-inf = 0), split into high and
      // low 16-bit parts, over S
      uint32_t hi[32], lo[32];
      const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-m_run, -m_run);
      float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float2 x =
            f2_fma(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), sc2, nm2);
        const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        ls[c & 1] = f2_add(ls[c & 1], pp);
        PSplit<T>::run(pp, hi[c], lo[c]);
      }
      l_run += (ls[0].x + ls[1].x) + (ls[0].y + ls[1].y);
      tmem_st32(t_s, hi);
      tmem_st32(t_s + 32, lo);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[Sm::kBarPF + 2 * m + u]);
      if (m == 0 && j == 0 && lane == 0) mbar_arrive(&bars[Sm::kBarLag]);
    }
    if (ok) {
      ok = tc_wait(&bars[Sm::kBarOF + m], 0, fail);
      if ((ok = __all_sync(0xffffffffu, ok))) {
        // ---- out = O / l (rows past the prompt store nothing) ----
        tc_fence_after();
        float *o = p.out + ((size_t)t_row * p.Hq + h_row) * D;
        const float inv = 1.f / l_run;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_sync(t_o + 32 * c, r);
          if (t_row < p.L) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4 *>(o + 32 * c + e) =
                  make_float4(__uint_as_float(r[e]) * inv, __uint_as_float(r[e + 1]) * inv,
                              __uint_as_float(r[e + 2]) * inv, __uint_as_float(r[e + 3]) * inv);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && *fail) pf_set_err(p.err, kDevTimeout, hk, b, 0);  // (a selection error stays)
  if (warp == Sm::kMmaWarp) tmem_dealloc(tmem, Sm::kAlloc);
}

template <typename T, int D, int HC>
cudaError_t launch_tc(const PrefillParams &p, cudaStream_t st) {
  using Sm = TcSmem<D, HC>;
  auto k = prefill_attn_tc_kernel<T, D, HC>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::kBytes);
  if (e != cudaSuccess) return e;
  const int grid = p.nb * p.Hkv * (p.G / HC);
  return launch_pdl(k, grid, Sm::kThreads, (size_t)Sm::kBytes, st, p);
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
