// Exact top-k of a row of page scores by one CTA of 256 threads ("LServe
// long-sequence LLM serving system", section 3.2: the query-aware selector
// keeps the pages of highest score under the token budget).  Used by the
// selection kernel and, on fused decode steps, by every dynamic-head CTA of
// the decode kernel.  Shared-memory buffers are passed in, so a caller can
// carve them from memory it uses for something else later.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"
#include "spd_internal.h"

namespace spd {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxKeys = kFusedMaxCandidates;  // candidate pages selected in shared memory
constexpr int kRankMax = 128;   // candidates finished by direct ranking
constexpr uint32_t kCopyWaitLimit = 1u << 24;
constexpr int kFusedMaxSel = kFusedMaxSelected;  // kept pages a fused decode step holds
constexpr int kFilterCap = 1024;  // candidates at or above a bound handled as a list

__device__ __forceinline__ void topk_set_err(int *err, int code, int a, int b, int c) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}

// Order-preserving unsigned key of a score: NaN lowest (0), -0 folded onto +0.
__device__ __forceinline__ uint32_t score_key(float f) {
  const uint32_t b = __float_as_uint(f), a = b & 0x7fffffffu;
  uint32_t key = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  key = a == 0u ? 0x80000000u : key;
  return a > 0x7f800000u ? 0u : key;
}

// Shared memory of one cta_topk call (pointers into the caller's memory).
struct TopkSmem {
  uint32_t *skey;     // [kMaxKeys], 16-byte aligned
  int *hist;          // [2][256]
  int *sh;            // [3][kSelWarps]
  uint32_t *mm;       // [2][kSelWarps]
  int *dec;           // [3]
  uint2 *cand;        // [kRankMax]
  int *ncand;         // [1]
  uint32_t *chosen;   // [kMaxKeys / 32]
  uint32_t *equal;    // [kMaxKeys / 32]
  uint32_t *ckey;     // [kFilterCap] keys of the candidates at or above a bound
  int *cidx;          // [kFilterCap] their page indices
  int *nfilt;         // [1]
  uint64_t *bar;      // [1], 8-byte aligned
};
// Bytes of a TopkSmem carved from one 16-byte aligned block.
constexpr int kTopkSmemBytes =
    kMaxKeys * 4 + 2 * 256 * 4 + 3 * kSelWarps * 4 + 2 * kSelWarps * 4 + 16 + kRankMax * 8 + 16 +
    2 * (kMaxKeys / 32) * 4 + 2 * kFilterCap * 4 + 16 + 16;
__device__ __forceinline__ TopkSmem carve_topk_smem(uint8_t *base) {
  TopkSmem m;
  uint8_t *p = base;
  m.skey = reinterpret_cast<uint32_t *>(p);  p += kMaxKeys * 4;
  m.hist = reinterpret_cast<int *>(p);       p += 2 * 256 * 4;
  m.sh = reinterpret_cast<int *>(p);         p += 3 * kSelWarps * 4;
  m.mm = reinterpret_cast<uint32_t *>(p);    p += 2 * kSelWarps * 4;
  m.dec = reinterpret_cast<int *>(p);        p += 16;
  m.cand = reinterpret_cast<uint2 *>(p);     p += kRankMax * 8;
  m.ncand = reinterpret_cast<int *>(p);      p += 16;
  m.chosen = reinterpret_cast<uint32_t *>(p); p += (kMaxKeys / 32) * 4;
  m.equal = reinterpret_cast<uint32_t *>(p); p += (kMaxKeys / 32) * 4;
  m.ckey = reinterpret_cast<uint32_t *>(p);  p += kFilterCap * 4;
  m.cidx = reinterpret_cast<int *>(p);       p += kFilterCap * 4;
  m.nfilt = reinterpret_cast<int *>(p);      p += 16;
  m.bar = reinterpret_cast<uint64_t *>(p);
  return m;
}


// Exclusive scan over the CTA, thread order; *total = the sum.  One barrier;
// `sh` must not be reused before the next barrier.
__device__ __forceinline__ int cta_scan1(int v, int *sh, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    x += lane >= o ? y : 0;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    const int t = sh[w];
    before += w < warp ? t : 0;
    tot += t;
  }
  *total = tot;
  return before + x - v;
}

// Exact selection of the k highest of C keys (k < C).  keys[e] belongs to
// page idx[e] (page e if idx is null); pages are < n.  Writes the chosen
// pages ascending to out[0..k) and returns the count.
//   1. The bits on which the largest and smallest key agree are shared by
//      every key: the search starts below them.
//   2. The k-th largest key T is narrowed 8 bits at a time: a 256-bin
//      histogram (shared-memory atomics) of the keys that match the bits
//      fixed so far, a CTA scan from the top bin down, and the bin where the
//      running count reaches k is fixed.
//   3. Once at most kRankMax keys still match, they are ranked directly
//      (greater key first, lower page first among equal keys); if every bit
//      is fixed with more matching keys, all equal T and the lowest pages are
//      taken.
//   4. The chosen pages are marked in a bitmap; a scan of its words' bit
//      counts writes them in ascending order.
// The loops are short and rolled: this runs on SMs whose instruction cache
// has not seen it.
__device__ int topk_core(const uint32_t *keys, const int *idx, int C, int n, int k, int *out,
                         const TopkSmem &m) {
  int(*hist)[256] = reinterpret_cast<int(*)[256]>(m.hist);
  int(*sh)[kSelWarps] = reinterpret_cast<int(*)[kSelWarps]>(m.sh);
  uint32_t(*mm)[kSelWarps] = reinterpret_cast<uint32_t(*)[kSelWarps]>(m.mm);
  int *dec = m.dec;
  uint2 *cand = m.cand;
  int &ncand = *m.ncand;
  uint32_t *chosen = m.chosen, *equal = m.equal;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = (n + 31) / 32;
  hist[0][tid] = 0;
  hist[1][tid] = 0;
  if (tid == 0) ncand = 0;
  if (idx)  // a list: bitmap words are set by atomics, so they start at zero
    for (int x = tid; x < nw; x += kSelThreads) chosen[x] = equal[x] = 0u;
  uint32_t kmax = 0u, kmin = 0xffffffffu;
  for (int e = tid; e < C; e += kSelThreads) {
    kmax = max(kmax, keys[e]);
    kmin = min(kmin, keys[e]);
  }
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  if (lane == 0) {
    mm[0][warp] = kmax;
    mm[1][warp] = kmin;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    kmax = max(kmax, mm[0][w]);
    kmin = min(kmin, mm[1][w]);
  }
  // `lo` low bits are unresolved; the bits above them equal `prefix` for T
  int lo = (kmax ^ kmin) ? 32 - __clz(kmax ^ kmin) : 0;
  uint32_t prefix = lo == 32 ? 0u : kmax & ~((1u << lo) - 1u);
  int remaining = k;  // keys still to take among those matching prefix
  int active = C;     // keys matching prefix
  for (int rnd = 0; lo > 0 && active > kRankMax; ++rnd) {
    const int w = min(8, lo);
    const int shift = lo - w;
    const uint32_t fmask = lo == 32 ? 0u : ~((1u << lo) - 1u);
    const uint32_t dmask = (1u << w) - 1u;
    int *hc = hist[rnd & 1];
#pragma unroll 4
    for (int e = tid; e < C; e += kSelThreads) {
      const uint32_t u = keys[e];
      if ((u & fmask) == prefix) atomicAdd(&hc[(u >> shift) & dmask], 1);
    }
    __syncthreads();
    // thread i takes bin 255 - i: the scan is then over bins from the top
    const int v = hc[255 - tid];
    hist[(rnd + 1) & 1][tid] = 0;  // the next round's bins (last read a round ago)
    int tot;
    const int excl = cta_scan1(v, sh[rnd & 1], &tot);
    if (excl < remaining && remaining <= excl + v) {  // exactly one thread
      dec[0] = 255 - tid;
      dec[1] = remaining - excl;
      dec[2] = v;
    }
    __syncthreads();
    prefix |= (uint32_t)dec[0] << shift;
    remaining = dec[1];
    active = dec[2];
    lo = shift;
  }
  const uint32_t fmask = lo == 32 ? 0u : ~((1u << lo) - 1u);
  const bool ranked = active <= kRankMax;
  if (!idx) {
    // warp w of pass r holds pages 256r + 32w + lane: its ballots are bitmap
    // word 8r + w (every word below the rounded-up n is written once)
    for (int j0 = 0; j0 < C; j0 += kSelThreads) {
      const int j = j0 + tid;
      const uint32_t u = j < C ? keys[j] : 0u;
      const uint32_t hb = u & fmask;
      const unsigned above = __ballot_sync(0xffffffffu, j < C && hb > prefix);
      const unsigned eq = __ballot_sync(0xffffffffu, j < C && hb == prefix);
      const int wd = (j0 >> 5) + warp;
      if (lane == 0) {
        chosen[wd] = above;
        equal[wd] = ranked ? 0u : eq;
      }
      if (ranked && eq) {
        int base = 0;
        if (lane == 0) base = atomicAdd(&ncand, __popc(eq));
        base = __shfl_sync(0xffffffffu, base, 0);
        if ((eq >> lane) & 1u) {
          const int e = base + __popc(eq & ((1u << lane) - 1u));
          if (e < kRankMax) cand[e] = make_uint2(u, (uint32_t)j);
        }
      }
    }
  } else {
    for (int e = tid; e < C; e += kSelThreads) {
      const uint32_t u = keys[e];
      const uint32_t hb = u & fmask;
      const int j = idx[e];
      if (hb > prefix) atomicOr(&chosen[j >> 5], 1u << (j & 31));
      if (hb == prefix) {
        if (ranked) {
          const int c = atomicAdd(&ncand, 1);
          if (c < kRankMax) cand[c] = make_uint2(u, (uint32_t)j);
        } else {
          atomicOr(&equal[j >> 5], 1u << (j & 31));
        }
      }
    }
  }
  __syncthreads();
  if (ranked) {
    if (tid < active) {
      const uint2 me = cand[tid];
      int rank = 0;
#pragma unroll 8
      for (int e = 0; e < active; ++e) {
        const uint2 o = cand[e];
        rank += (o.x > me.x) | ((o.x == me.x) & (o.y < me.y));
      }
      if (rank < remaining) atomicOr(&chosen[me.y >> 5], 1u << (me.y & 31u));
    }
  } else {
    int taken = 0;
    for (int w0 = 0; w0 < nw; w0 += kSelThreads) {
      const int wd = w0 + tid;
      uint32_t bits = wd < nw ? equal[wd] : 0u;
      int tot;
      int before = cta_scan1(__popc(bits), sh[2], &tot) + taken;
      uint32_t add = 0u;
      while (bits && before < remaining) {
        const uint32_t low = bits & (0u - bits);
        add |= low;
        bits ^= low;
        ++before;
      }
      if (add) chosen[wd] |= add;
      taken += tot;
      __syncthreads();
    }
  }
  __syncthreads();
  int written = 0;
  for (int w0 = 0; w0 < nw; w0 += kSelThreads) {
    const int wd = w0 + tid;
    uint32_t bits = wd < nw ? chosen[wd] : 0u;
    int tot;
    int pos = cta_scan1(__popc(bits), sh[(w0 / kSelThreads) & 1], &tot) + written;
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      if (pos < k) out[pos] = wd * 32 + b;
      ++pos;
    }
    written += tot;
  }
  return written;
}

// The smallest of `count` per-chunk bounds (0xffffffff: a chunk that gives
// none), the same in every thread; 0 (no bound) if no chunk gives one.
__device__ uint32_t min_chunk_bound(const uint32_t *b, int count, const TopkSmem &m) {
  uint32_t(*mm)[kSelWarps] = reinterpret_cast<uint32_t(*)[kSelWarps]>(m.mm);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t v = 0xffffffffu;
  for (int c = tid; c < count; c += kSelThreads) v = min(v, __ldcg(b + c));
  v = __reduce_min_sync(0xffffffffu, v);
  if (lane == 0) mm[0][warp] = v;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) v = min(v, mm[0][w]);
  __syncthreads();  // mm is reused by the caller
  return v == 0xffffffffu ? 0u : v;
}

// One bulk copy of n scores (16-byte aligned, readable up to n rounded up to
// 4 floats) into m.skey; while it is in flight, the smallest of `nb` chunk
// bounds (nb = 0: none) goes to *bound.  The same result in every thread:
// false if the copy did not land within the wait limit (the error word then
// says so).
__device__ bool load_scores(const float *sc, int n, int k, const uint32_t *bounds, int nb,
                            uint32_t *bound, int *err, const TopkSmem &m) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(m.bar, 1);
    fence_mbar_init();
    const uint32_t bytes = (uint32_t)((n * 4 + 15) & ~15);
    mbar_arrive_expect_tx(m.bar, bytes);
    bulk_load_1d(m.skey, sc, bytes, m.bar);
    *m.nfilt = 0;
  }
  // (its barriers also make the mbarrier's initialisation visible)
  *bound = nb > 0 ? min_chunk_bound(bounds, nb, m) : 0u;
  if (nb == 0) __syncthreads();
  const bool landed = mbar_wait(m.bar, 0, kCopyWaitLimit);
  if (__syncthreads_or(!landed)) {
    if (tid == 0) topk_set_err(err, kDevTimeout, -1, n, k);
    return false;
  }
  return true;
}

// Exact top-k of n scores (1 <= k < n <= kMaxKeys) into out[0..k), ascending;
// returns the count written.  The smallest of the nb chunk bounds (keys that
// at least k scores reach; nb = 0: none) bounds the candidates: every top-k
// key reaches it too, ties included, so only the scores at or above it are
// candidates.  Up to kFilterCap of them are selected as a list; more (or no
// bound) select over all n.
__device__ int cta_topk(const float *sc, int n, int k, const uint32_t *bounds, int nb, int *out,
                        int *err, const TopkSmem &m) {
  uint32_t bound = 0u;
  if (!load_scores(sc, n, k, bounds, nb, &bound, err, m)) return 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kSeg = kFilterCap / kSelWarps;  // candidates a warp may hold
  uint32_t *ck = m.ckey + warp * kSeg;
  int *ci = m.cidx + warp * kSeg;
  int cnt = 0;
  if (bound != 0u) {
    // warp w sees pages 256r + 32w + lane: it appends its candidates to its
    // own segment of the list (no atomics), keeping the count in registers.
    // A batch of keys is read into registers first, so the shared-memory
    // loads overlap and only the ballots and counts run in sequence.
    constexpr int kBatch = 8;
    for (int j0 = 0; j0 < n; j0 += kBatch * kSelThreads) {
      uint32_t key[kBatch];
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        const int j = j0 + r * kSelThreads + tid;
        key[r] = j < n ? score_key(__uint_as_float(m.skey[j])) : 0u;
      }
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        const int j = j0 + r * kSelThreads + tid;
        const bool c = j < n && key[r] >= bound;
        const unsigned cm = __ballot_sync(0xffffffffu, c);
        const int e = cnt + __popc(cm & ((1u << lane) - 1u));
        if (c && e < kSeg) {
          ck[e] = key[r];
          ci[e] = j;
        }
        cnt += __popc(cm);
      }
    }
    if (lane == 0) m.sh[warp] = cnt;
  }
  __syncthreads();
  int C = 0, before = 0;
  bool fits = bound != 0u;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    const int c = bound != 0u ? m.sh[w] : 0;
    fits = fits && c <= kSeg;
    before += w < warp ? c : 0;
    C += c;
  }
  fits = fits && C > k;
  __syncthreads();  // m.sh is reused by the scans below
  if (fits) {
    // pack the segments: warp w's run goes to [before, before + cnt) of the
    // second half of the score buffer (free once the candidates are out)
    uint32_t *pk = m.skey + kMaxKeys / 2;
    int *pi = reinterpret_cast<int *>(m.skey + kMaxKeys / 2 + kFilterCap);
    for (int e = lane; e < cnt; e += 32) {
      pk[before + e] = ck[e];
      pi[before + e] = ci[e];
    }
    __syncthreads();
    return topk_core(pk, pi, C, n, k, out, m);
  }
  for (int j = tid; j < n; j += kSelThreads) m.skey[j] = score_key(__uint_as_float(m.skey[j]));
  __syncthreads();
  return topk_core(m.skey, nullptr, n, n, k, out, m);
}

}  // namespace
}  // namespace spd
