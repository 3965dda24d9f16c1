// Split-K sparse decode attention for sm_103a ("LServe long-sequence LLM
// serving system", section 2.1: one unified kernel for streaming and dynamic
// heads; section 3.2: streaming heads read their recent tokens through
// shared memory).
//
// Work list.  A unit is (sequence, kv head).  Its attended tokens are cut
// into tiles of 16 rows:
//   dynamic head   the selected logical pages plus the pages created since the
//                  selection, each page ell/16 tiles (the newest page only as
//                  many as it holds tokens);
//   streaming head three runs of ring-buffer slots -- sink [0, min(S, L)),
//                  the window's slots up to the ring's end, and its wrapped
//                  remainder -- each run tiled from its start.
// A unit is split over nc clusters of CS CTAs (a thread-block cluster; CS and
// the CTAs' tile ranges are chosen by the host so the launch fills the GPU);
// a CTA ("item") takes a contiguous range of the unit's tiles.
//
// Data movement.  The CTA's tiles stream through a ring of kStages shared-
// memory stages: tile t lives in stage t mod kStages, filled by TMA tensor
// loads (one per tile of K and of V: boxes of 64 channels x 16 rows x the
// channel halves, 128-byte swizzle; one mbarrier per stage, its phase
// counting the stage's uses).  The first kStages tiles are
// requested at kernel start, the later ones are prefetched into L2 then, and
// the warp that finishes tile t refills its stage with tile t + kStages.
// Warps take tiles from a shared counter, so a CTA with more tiles than warps
// spreads the extra ones over whichever warps are free.  K/V bytes are read
// from HBM once.
//
// Math (per warp and tile, all G query heads of the kv head at once):
//   q.K^T   mma.sync m16n8k16, A = K tile rows (ldmatrix from the swizzled
//           tile), B = q^T in registers (heads padded to 8 columns), fp32
//           accumulate -- the products of 16-bit inputs are exact;
//   softmax online, in fp32, base 2 with log2(e)/sqrt(d) folded in;
//   P.V     mma.sync m16n8k16 as O^T = V^T P^T: A = V tile (ldmatrix.trans),
//           B = P^T with the 16 tokens as k and the heads as the 8 columns;
//           P is split into a 16-bit high part and the 16-bit rounding of
//           the rest, two mma each, so the weights carry ~2^-16 relative
//           error instead of 2^-9 (fp32 accumulate).
// Merge.  The 8 warps merge in shared memory into the CTA's (m, l, o).  The
// CTAs of a cluster then merge over distributed shared memory: every CTA
// pushes each channel slice of its (m, l, o) into the inbox of the CTA that
// owns that slice (remote shared-memory stores that count their bytes on the
// owner's inbox mbarrier), and once its inbox holds every rank's bytes each
// CTA combines its slice locally (a CTA leaves only after its own inbox is
// complete, so no peer is still storing into it; a second cluster phase
// remains only where CTAs read one another's global writes) -- the row max /
// row sum export
// of the Novita KV-sparsity article's modified FlashAttention ("attention
// mechanism modifications").  When a
// unit has several clusters (nc > 1), their results meet in global memory:
// the last cluster to finish (atomic ticket, no waiting) merges them.
//
// Fused append (decode step).  The CTA that owns a unit's newest token also
// appends it: the row is written to the pool / ring, patched into the
// staged tile, and folded into the logical page's key min/max.
//
// fp8 storage (kF8).  K/V rows are E4M3 codes of value / scale, one 128-byte
// row per token (head_dim 128): a tile of K or V is one 16 x 128-byte box
// (3-D map), the ring has 16 stages, and the tensor-core fragments are built
// from byte pairs (ldmatrix, byte permutes) widened in registers (keys to
// fp16, values to T).
//
// Files.  This header holds the kernel template and its launch helpers;
// decode.cu instantiates the plain kernel, decode_mass.cu the one that also
// exports the per-page attention mass, decode_fp8.cu the fp8-storage ones
// (separate translation units, built in parallel).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <type_traits>

#include "ptx.cuh"
#include "spd_internal.h"
#include "topk.cuh"

namespace spd {
namespace {

constexpr int kRows = 16;                  // rows per tile (one mma M tile)
constexpr int kWarps = 8;                  // 256 threads
constexpr int kThreads = kWarps * 32;
// Shared-memory stage ring.  Two launch shapes:
//   shared  12 stages of 16-bit tiles keep a CTA within half an SM, so a CTA
//           of the next launch stages its tiles beside it while it computes;
//           fp8 tiles are half the size, and 16 of them fit in the space the
//           selection buffers take anyway;
//   deep    (Deep, for launches whose tiles far exceed what two such rings
//           hold) 24 stages of 16-bit tiles, one CTA per SM: while the
//           eight warps each hold the stage they compute on, the others stay
//           in flight, and the ring keeps streaming at the HBM rate.
template <bool F8, bool Deep = false>
struct Ring {
  static constexpr int n = Deep ? 24 : (F8 ? 16 : 12);
};
constexpr int kMaxDesc = 256;              // tiles one CTA may take
constexpr uint32_t kWaitLimit = 1u << 24;  // bounded mbarrier polls

// A tile row is D elements of 2 bytes, or of 1 byte with fp8 storage (F8);
// it is stored as 128-byte "boxes" (64 16-bit channels or 128 fp8 ones).
template <int D, bool F8 = false>
struct Geo {
  static constexpr int kRowBytes = D * (F8 ? 1 : 2);
  static constexpr int kBoxes = kRowBytes / 128;             // 128-byte boxes per row
  static constexpr int kBoxBytes = kRows * 128;              // one box: 16 rows x 128 B
  static constexpr int kTileBytes = 2 * kBoxes * kBoxBytes;  // K boxes then V boxes
  static constexpr int kCPL = D / 32;                        // channels per lane (append)
};

template <int G>
struct GP {
  static constexpr int v = G < 4 ? 4 : G;  // padded head stride of the P buffer
};

struct TileDesc {
  int y, z;      // TMA coordinates (row, plane) of the tile's first row
  int n_valid;   // rows holding attended tokens (0: skip)
  int pad;
};

// Shared memory: a fixed region (stage barriers, tile descriptors, P and
// rescale buffers, per-warp and per-CTA row max / sum / output, flags), then
// the stages at a 1024-byte aligned offset.  After the tile loop the stage
// region holds the warp-merge buffer and later the global-merge buffers.
template <int D, int G, bool F8 = false, bool Deep = false>
struct Smem {
  static constexpr int kStages = Ring<F8, Deep>::n;
  static constexpr int kBars = 0;                                      // uint64 [kStages]
  static constexpr int kDesc = kBars + kStages * 8;                    // TileDesc [kMaxDesc]
  static constexpr int kP = kDesc + kMaxDesc * (int)sizeof(TileDesc);  // float [W][16][GP]
  static constexpr int kC = kP + kWarps * kRows * GP<G>::v * 4;        // float [W][GP]
  static constexpr int kML = kC + kWarps * GP<G>::v * 4;               // float [2][W][G]
  // inbox: what the cluster's CTAs send this CTA: M[16][G], L[16][G] and
  // O[CS ranks][G][D / CS + pad 4] (<= G * D + 64 floats for any CS <= 16)
  static constexpr int kInbox = (kML + 2 * kWarps * G * 4 + 15) / 16 * 16;
  static constexpr int kFlag = kInbox + (32 * G + G * D + 64) * 4;     // int [4 + kStages]
  static constexpr int kTopkBar = (kFlag + (4 + kStages) * 4 + 7) / 8 * 8;  // uint64
  static constexpr int kInboxBar = kTopkBar + 8;  // uint64: the inbox's bytes have landed
  static constexpr int kTiles = (kInboxBar + 8 + 1023) / 1024 * 1024;
  static constexpr int kStageRegion = kStages * Geo<D, F8>::kTileBytes;
  static constexpr int kMergeRegion = kWarps * G * (D + 4) * 4;        // o of every warp
  static constexpr int kCombineRegion = 256 * G * 12 + 64;             // (m, l), weights
  // before the tiles of a fused selection step: the top-k buffers, then the
  // unit's selected pages
  static constexpr int kTopkRegion = kTopkSmemBytes + kFusedMaxSel * 4;
  static constexpr int kPtCache = 2048;                  // page-table entries cached with it
  static constexpr int kPtCacheOff = kTopkRegion;        // bytes into the stage region
  static constexpr int kR1 = kStageRegion > kMergeRegion ? kStageRegion : kMergeRegion;
  static constexpr int kR2 = kCombineRegion > kTopkRegion + kPtCache * 4
                                 ? kCombineRegion
                                 : kTopkRegion + kPtCache * 4;
  static constexpr int kRegion = kR1 > kR2 ? kR1 : kR2;
  static constexpr int kAlloc = kTiles + kRegion + 1024;  // + alignment slack
  static_assert(kAlloc <= 232448, "more shared memory than a CTA may have");
};

template <typename T> struct IsBF16 { static constexpr bool v = false; };
template <> struct IsBF16<__nv_bfloat16> { static constexpr bool v = true; };

template <typename T>
__device__ __forceinline__ float tof(T x);
template <> __device__ __forceinline__ float tof(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float tof(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> struct Cvt;
template <> struct Cvt<__half> {
  static __device__ __forceinline__ __half from(float x) { return __float2half_rn(x); }
};
template <> struct Cvt<__nv_bfloat16> {
  static __device__ __forceinline__ __nv_bfloat16 from(float x) { return __float2bfloat16_rn(x); }
};

// Two weights (a in the low half) split into their 16-bit roundings (hi) and
// the 16-bit roundings of what is left (lo): the rest a - hi is exact in fp32.
template <typename T> struct Split2;
template <> struct Split2<__half> {
  static __device__ __forceinline__ void run(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 r = f2_sub(make_float2(a, b), __half22float2(h));
    const __half2 l = __floats2half2_rn(r.x, r.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
  }
};
template <> struct Split2<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 r = f2_sub(make_float2(a, b), __bfloat1622float2(h));
    const __nv_bfloat162 l = __floats2bfloat162_rn(r.x, r.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
  }
};

// A warp's running max of a head moves only when a tile's max exceeds it by
// more than this (log2 units), so the output accumulators are rescaled
// rarely; weights then stay below 2^8, and every merge pairs each (m, l, o)
// with its own m.  Launches that export the row max keep it exact (0).
constexpr float kStaleMax = 8.f;

__device__ __forceinline__ void set_err(int *err, int code, int a, int b, int c) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}

// Bounded wait until another warp of the CTA has counted more than `u` uses
// of a stage (its load for use u is issued).
__device__ __forceinline__ bool wait_issued(const int *count, int u, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (*reinterpret_cast<const volatile int *>(count) > u) return true;
  return false;
}

// Byte offset, inside a tile half (K or V), of channel `ch` of row `r`.
template <int D>
__device__ __forceinline__ uint32_t chan_off(int r, int ch) {
  return (uint32_t)((ch >> 6) * Geo<D>::kBoxBytes) + swz128(r, (ch & 63) >> 3) +
         (uint32_t)((ch & 7) * 2);
}

// Per-page attention mass of dynamic unit (launch sequence i, dynamic head
// sub) once its final max Mg[g] and sum Lg[g] (base 2) are known: every
// attended page's share of each head's softmax weight, from the (max, sum)
// pairs the tile loop stored per tile.  The page's tiles are consecutive
// (ell / 16 of them, the newest page's possibly fewer).  Work items
// x = g * max_pages + page, from x0 in steps of dx; pages past the attended
// ones get -1 and mass 0.
template <int G>
__device__ void write_page_mass(const TileDecodeParams &p, int i, int sub, const TileSeq &s,
                                int nL, int n_tiles, const float *Mg, const float *Lg, int x0,
                                int dx) {
  const int tpp = p.ell / kRows;
  const int n_att = s.sel_count + nL - s.nL0;
  const size_t urow = (size_t)i * p.Hd + sub;
  const float2 *part = p.page_part + urow * p.page_tile_cap * G;
  const int *sel = p.selection + ((size_t)s.slot * p.Hd + sub) * p.ksel_max;
  for (int x = x0; x < G * p.max_pages; x += dx) {
    const int g = x / p.max_pages, a = x - g * p.max_pages;
    float mass = 0.f;
    int j = -1;
    if (a < n_att) {
      j = a < s.sel_count ? sel[a] : s.nL0 + (a - s.sel_count);
      float acc = 0.f;
      for (int st = 0; st < tpp; ++st) {
        const int tau = a * tpp + st;
        if (tau >= n_tiles) break;
        const float2 pr = __ldcg(&part[(size_t)tau * G + g]);
        if (pr.y > 0.f) acc = fmaf(exp2f(pr.x - Mg[g]), pr.y, acc);
      }
      mass = acc / Lg[g];
    }
    p.page_mass[(urow * G + g) * p.max_pages + a] = mass;
    if (g == 0) p.pages[urow * p.max_pages + a] = j;
  }
}

// kMass: the per-page attention mass is exported (its own instance, so the
// plain kernel carries none of that work).  kF8: K/V are stored as fp8 E4M3
// codes of value / scale (head_dim 128): tiles are half the bytes, widened
// exactly on their way into the tensor-core fragments: keys to fp16 for fp16
// q.K products (q narrowed to fp16 once), values to T for the P.V products.
// kReuse: an instance for launches in which no unit selects its pages (the
// steps that reuse a stored selection), built without the fused top-k code so
// the code a launch runs once stays small.
template <typename T, int D, int G, bool kMass, bool kF8 = false, bool kDeep = false,
          bool kReuse = false>
__global__ void __launch_bounds__(kThreads) decode_tiles_kernel(const __grid_constant__ TileDecodeParams p) {
  static_assert(!kF8 || D == 128, "fp8 storage: one 128-byte row per token");
  // tensor-core element types.  q.K: T, or fp16 with fp8 storage (an E4M3
  // value widens to fp16 in one instruction; q is narrowed to fp16 once).
  // P.V: T; with fp8 storage fp16 (an E4M3 value widens to fp16 in one
  // instruction; the weights are at most 1, and their fp16 high and low parts
  // carry ~2^-22 of each, flushing only weights below 2^-24).
  constexpr bool kQkBf = kF8 ? false : IsBF16<T>::v;
  constexpr bool kPvBf = kF8 ? false : IsBF16<T>::v;
  using TP = typename std::conditional<kF8, __half, T>::type;  // P.V element type
  using Gm = Geo<D, kF8>;
  using Sm = Smem<D, G, kF8, kDeep>;
  constexpr int kStages = Sm::kStages;
  constexpr int CPL = Gm::kCPL;  // channels per lane of the fused append
  constexpr int GPAD = GP<G>::v;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *stages = smem + Sm::kTiles;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Sm::kBars);
  TileDesc *tdesc = reinterpret_cast<TileDesc *>(smem + Sm::kDesc);
  float *P_all = reinterpret_cast<float *>(smem + Sm::kP);
  float *m_w = reinterpret_cast<float *>(smem + Sm::kML);
  float *l_w = m_w + kWarps * G;
  float *in_M = reinterpret_cast<float *>(smem + Sm::kInbox);  // [rank][G]
  float *in_L = in_M + 16 * G;                                   // [rank][G]
  float *in_O = in_L + 16 * G;                                   // [rank][G][slice]
  int *s_flag = reinterpret_cast<int *>(smem + Sm::kFlag);  // [1] a wait gave up, [2] next tile
  int *s_iss = s_flag + 4;                                   // loads issued per stage

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // The inbox barrier counts the bytes the cluster's CTAs push into this
  // CTA's inbox: from each of CS ranks, its (M, L) and its O of this CTA's
  // channel slice for every head.  Set up before the cluster's start arrive,
  // so no rank stores into it before it exists.  (A launch of one-CTA
  // clusters is a plain grid, where the CTA fills its own inbox with plain
  // stores: the byte-counting remote stores need a cluster launch.)
  uint64_t *inbox_bar = reinterpret_cast<uint64_t *>(smem + Sm::kInboxBar);
  const bool remote = p.cluster > 1;
  if (tid == 0 && remote) {
    mbar_init(inbox_bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(inbox_bar, (uint32_t)(p.cluster * G * ((D / p.cluster) + 2) * 4));
  }
  cluster_arrive_relaxed();  // paired with the wait before the first remote store
  if (tid == 0) {
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_sk);
    prefetch_tmap(&p.tm_sv);
    s_flag[1] = 0;  // set if a bounded wait gives up
    s_flag[2] = kWarps;  // tiles 0..kWarps-1 go to warps 0..kWarps-1
  }
  const int item = blockIdx.x;
  int i = 0;
  while (i + 1 < p.n_seqs && p.seqs[i + 1].item_off <= item) ++i;
  const TileSeq s = p.seqs[i];
  int local = item - s.item_off;
  const bool dyn = local < p.Hd * s.ns_dyn;
  int sub, split, ns, tpi, unit_item0;
  if (dyn) {
    sub = local / s.ns_dyn;
    split = local % s.ns_dyn;
    ns = s.ns_dyn;
    tpi = s.tpi_dyn;
    unit_item0 = s.item_off + sub * s.ns_dyn;
  } else {
    local -= p.Hd * s.ns_dyn;
    sub = local / s.ns_str;
    split = local % s.ns_str;
    ns = s.ns_str;
    tpi = s.tpi_str;
    unit_item0 = s.item_off + p.Hd * s.ns_dyn + sub * s.ns_str;
  }
  const int CS = p.cluster;        // CTAs per cluster (units' item counts are multiples)
  const int rank = split % CS;     // == %cluster_ctarank: clusters start at multiples of CS
  const int ci = split / CS;       // cluster index within the unit
  const int nc = ns / CS;          // clusters of this unit
  const int h = dyn ? p.dyn_kv[sub] : p.str_kv[sub];
  const int L = s.L;

  // ---- unit geometry ----
  int n_tiles, nL = 0, n_att = 0, tpp = 0;
  int run_start[3] = {0, 0, 0}, run_len[3] = {0, 0, 0}, run_tiles[3] = {0, 0, 0};
  if (dyn) {
    nL = (L + p.ell - 1) / p.ell;
    n_att = s.sel_count + nL - s.nL0;
    tpp = p.ell / kRows;
    const int last_rows = (L - 1) % p.ell + 1;
    n_tiles = (n_att - 1) * tpp + (last_rows + kRows - 1) / kRows;
  } else {
    run_len[0] = min(p.S, L);
    if (L > p.S) {
      const int w0 = max(p.S, L - p.W);
      const int n_win = L - w0;
      const int a0 = (w0 - p.S) % p.W;
      run_start[1] = p.S + a0;
      run_len[1] = min(n_win, p.W - a0);
      run_start[2] = p.S;
      run_len[2] = n_win - run_len[1];
    }
    for (int r = 0; r < 3; ++r) run_tiles[r] = (run_len[r] + kRows - 1) / kRows;
    n_tiles = run_tiles[0] + run_tiles[1] + run_tiles[2];
  }
  const int tile0 = split * tpi;
  const int nt = min(kMaxDesc, max(0, min(n_tiles, tile0 + tpi) - tile0));
  const bool owns_newest = nt > 0 && tile0 + nt == n_tiles;
  const bool do_append = p.k_new != nullptr && owns_newest;
  // (a unit that selects its pages here reads this step's scores: never early)
  // this unit selects its pages here (never in a reuse instance: the host
  // launches one only when no unit of the launch selects)
  const bool selects = !kReuse && dyn && s.topk_n > 0;
  const bool early = ((p.early >> (dyn ? 0 : 1)) & 1) && !selects;
  // bit 2: the previous kernel is this context's own selection or page-table
  // kernel, which writes nothing a streaming unit reads; q is final once that
  // kernel runs (it waited for its own predecessor before releasing this one)
  const bool skip_wait = !dyn && ((p.early >> 2) & 1);
  if (tid == 0) {
    // q (and the new token) start their way into L2 now; they are read only
    // after the wait, and L2 is coherent, so this is a hint and nothing more
    prefetch_l2_bulk(static_cast<const uint16_t *>(p.q) + ((size_t)i * p.Hq + h * G) * D,
                     G * D * 2);
    if (do_append) {
      const size_t row = ((size_t)i * p.Hkv + h) * D;
      prefetch_l2_bulk(static_cast<const uint16_t *>(p.k_new) + row, D * 2);
      prefetch_l2_bulk(static_cast<const uint16_t *>(p.v_new) + row, D * 2);
    }
  }

  // Everything above used only the parameter block.  The KV cache (page
  // table, selection, pools) is read next: before the wait for the previous
  // kernel on the stream when the host knows that kernel cannot have written
  // the KV this unit reads (bit 0 of p.early for dynamic units, bit 1 for
  // streaming ones), after it otherwise.  q, the new token and every write
  // come after the wait.  Dependents are released only after the wait, so when
  // this kernel runs, every kernel before its immediate predecessor has
  // finished.
  // stage barriers: set up before any wait (the cluster-scope fence that
  // publishes them to the TMA unit stays off the path after it); they live
  // outside the stage region, and every use follows a CTA barrier below
  if (tid < kStages) {
    mbar_init(&bars[tid], 1);
    fence_mbar_init();
    s_iss[tid] = 0;
  }

  // A unit that selects its pages here follows this context's own selection
  // kernel, after the page-table flush had finished: the sequence's page
  // table is final, so it is copied to shared memory before the wait.
  int *pt_s = nullptr;
  if (selects && p.max_pp <= Sm::kPtCache) {
    pt_s = reinterpret_cast<int *>(stages + Sm::kPtCacheOff);
    const int *row = p.page_table + (size_t)s.slot * p.max_pp;
    for (int x = tid; x < p.max_pp; x += kThreads) pt_s[x] = row[x];
  }
  if (!early) {
    if (!skip_wait) pdl_wait();
    pdl_launch_dependents();
  }

  // ---- a fused selection step: this CTA selects the unit's pages ----
  // (every CTA of the unit computes the same selection from the same scores;
  // the stage region holds the work and the result until the tiles arrive)
  const int *sel_s = nullptr;
  if constexpr (kReuse) {
    if (dyn && s.topk_n > 0 && tid == 0) set_err(p.err, kDevBadSelection, s.slot, sub, -1);
  } else if (selects) {
    TopkSmem tm = carve_topk_smem(stages);
    tm.bar = reinterpret_cast<uint64_t *>(smem + Sm::kTopkBar);  // never repurposed
    int *list = reinterpret_cast<int *>(stages + kTopkSmemBytes);
    const int k = s.sel_count - 1;
    const float *scr = p.scores + ((size_t)s.topk_row * p.Hd + sub) * p.score_stride;
    const int got =
        cta_topk(scr, s.topk_n, k, p.bounds + ((size_t)s.topk_row * p.Hd + sub) * p.bound_stride,
                 s.topk_bounds, list, p.err, tm);
    __syncthreads();
    if (tid == 0) {
      list[k] = s.nL0 - 1;  // the newest page is always kept
      if (got != k) set_err(p.err, kDevTopkCount, s.slot, sub, got);
    }
    __syncthreads();
    if (split == 0) {  // one CTA of the unit stores it for the steps that reuse it
      int *gsel = const_cast<int *>(p.selection) + ((size_t)s.slot * p.Hd + sub) * p.ksel_max;
      for (int t = tid; t < s.sel_count; t += kThreads) gsel[t] = list[t];
    }
    sel_s = list;
  }

  // ---- tile descriptors (threads in parallel), stage barriers ----
  for (int t = tid; t < nt; t += kThreads) {
    const int tau = tile0 + t;
    TileDesc td{0, 0, 0, 0};
    if (dyn) {
      const int pi = tau / tpp, st = tau % tpp;
      const int *sel = sel_s ? sel_s : p.selection + ((size_t)s.slot * p.Hd + sub) * p.ksel_max;
      const int j = pi < s.sel_count ? sel[pi] : s.nL0 + (pi - s.sel_count);
      const int blk = j / p.R;
      if (j < 0 || j >= nL || blk >= p.max_pp) {
        set_err(p.err, kDevBadSelection, s.slot, sub, j);
      } else {
        const int phys = pt_s ? pt_s[blk] : p.page_table[(size_t)s.slot * p.max_pp + blk];
        if (phys < 0 || phys >= p.num_phys) {
          set_err(p.err, kDevBadPhys, s.slot, blk, phys);
        } else {
          td.y = (j % p.R) * p.ell + st * kRows;
          td.z = phys * p.Hd + sub;
          td.n_valid = min(kRows, L - (j * p.ell + st * kRows));
        }
      }
    } else {
      int r = 0, k = tau;
      while (r < 2 && k >= run_tiles[r]) k -= run_tiles[r++];
      td.y = ((s.slot * p.Hs + sub) * (p.S + p.W)) + run_start[r] + k * kRows;
      td.z = 0;
      td.n_valid = min(kRows, run_len[r] - k * kRows);
    }
    tdesc[t] = td;
  }
  __syncthreads();  // descriptors written; the stage barriers set up at the start

  const CUtensorMap *mk = dyn ? &p.tm_k : &p.tm_sk;
  const CUtensorMap *mv = dyn ? &p.tm_v : &p.tm_sv;
  // stage s: K boxes, then V boxes; tile t uses stage t % kStages, and its
  // use number t / kStages is the phase its waiter checks
  auto issue = [&](int t) {
    const int st = t % kStages;
    const TileDesc td = tdesc[t];
    atomicAdd(&s_iss[st], 1);
    if (td.n_valid <= 0) {  // nothing to load: complete the phase anyway
      mbar_arrive_expect_tx(&bars[st], 0);
      return;
    }
    uint8_t *kd = stages + st * Gm::kTileBytes;
    uint8_t *vd = kd + Gm::kBoxes * Gm::kBoxBytes;
    mbar_arrive_expect_tx(&bars[st], Gm::kTileBytes);
    // one copy per tile of K and one of V: the map's third dimension walks
    // the 64-channel halves, which land box after box (fp8: one 128-byte
    // box per row, a 3-D map)
    if constexpr (kF8) {
      tma_load_3d(kd, mk, 0, td.y, td.z, &bars[st]);
      tma_load_3d(vd, mv, 0, td.y, td.z, &bars[st]);
    } else {
      tma_load_4d(kd, mk, 0, td.y, 0, td.z, &bars[st]);
      tma_load_4d(vd, mv, 0, td.y, 0, td.z, &bars[st]);
    }
  };
  if (lane == 0) {
    // the stage region was read and written through the generic proxy (the
    // selection above): order that before the TMA writes
    if (sel_s) fence_proxy_async_smem();
    for (int t = warp; t < min(nt, kStages); t += kWarps) issue(t);
    // the later tiles start their way from HBM into L2 now; their stage
    // refills then read L2
    for (int t = kStages + warp; t < nt; t += kWarps) {
      const TileDesc td = tdesc[t];
      if (td.n_valid <= 0) continue;
      if constexpr (kF8) {
        tma_prefetch_l2_3d(mk, 0, td.y, td.z);
        tma_prefetch_l2_3d(mv, 0, td.y, td.z);
      } else {
        tma_prefetch_l2_4d(mk, 0, td.y, 0, td.z);
        tma_prefetch_l2_4d(mv, 0, td.y, 0, td.z);
      }
    }
  }

  if (early) {
    if (!skip_wait) pdl_wait();
    pdl_launch_dependents();
  }
  // every CTA of the cluster has started (its inbox barrier is set up): the
  // CTAs of a cluster start together, so this is off the merge's path
  cluster_wait();

  // ---- q^T fragments (B operand), heads padded to 8 columns ----
  const int g8 = lane >> 2, t4 = lane & 3;
  uint32_t qb[D / 16][2];
  {
    const uint32_t *qp = reinterpret_cast<const uint32_t *>(
        reinterpret_cast<const uint16_t *>(p.q) + ((size_t)i * p.Hq + h * G) * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      if (g8 < G) {
        if constexpr (kF8) {
          // k slots {2t4, 2t4+1 | 2t4+8, 2t4+9} of k-step kk are channels
          // 16kk + 4t4 + {0, 1 | 2, 3} (the order the fp8 K fragments use)
          qb[kk][0] = to_f16x2<T>(qp[(g8 * D + kk * 16 + 4 * t4) / 2]);
          qb[kk][1] = to_f16x2<T>(qp[(g8 * D + kk * 16 + 4 * t4 + 2) / 2]);
        } else {
          qb[kk][0] = qp[(g8 * D + kk * 16 + 2 * t4) / 2];
          qb[kk][1] = qp[(g8 * D + kk * 16 + 2 * t4 + 8) / 2];
        }
      } else {
        qb[kk][0] = qb[kk][1] = 0u;
      }
    }
  }

  // ---- per-warp online softmax over its tiles ----
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;  // heads 2t4, 2t4+1
  // O^T accumulators: m-tile m holds channels 16m + g8 (and + 8) x heads
  // 2t4, 2t4 + 1 -- the two heads whose running max this lane tracks
  constexpr int MT = D / 16;
  float oacc[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[m][e] = 0.f;
  float *Pw = P_all + warp * kRows * GPAD;
  // fp8: the stored keys are code * k_scale; the scale folds into the logits'
  const float sc = kF8 ? p.scale_log2 * p.k_scale[h] : p.scale_log2;
  const float stale = p.row_max ? 0.f : kStaleMax;

  for (int t = warp; t < nt;) {
    const TileDesc td = tdesc[t];
    const int st = t % kStages, u = t / kStages;  // stage and its use number
    uint8_t *kt = stages + st * Gm::kTileBytes;
    uint8_t *vt = kt + Gm::kBoxes * Gm::kBoxBytes;
    // Use u of the stage is loaded only after use u-1 was consumed, so the
    // barrier's parity identifies it once the load is known to be issued
    // (a wait on the parity alone could match use u-2).  Every tile is waited
    // for, empty ones too, so no copy is in flight when the loop ends.
    if (!wait_issued(&s_iss[st], u, kWaitLimit) || !mbar_wait(&bars[st], u & 1, kWaitLimit)) {
      if (lane == 0) {
        set_err(p.err, kDevTimeout, s.slot, h, t);
        s_flag[1] = 1;
      }
      break;
    }
    if (td.n_valid > 0) {
      const int nv = td.n_valid;

      if (kF8 && do_append && t == nt - 1) {
        // the newest token, row nv-1 of the unit's last tile, as E4M3 codes:
        // this lane's 4 channels are one 4-byte word of a 16-byte chunk
        const int r = nv - 1;
        const int cb = lane * CPL;
        const size_t src = ((size_t)i * p.Hkv + h) * D + cb;
        const T *kn = reinterpret_cast<const T *>(p.k_new) + src;
        const T *vn = reinterpret_cast<const T *>(p.v_new) + src;
        const float ksc = p.k_scale[h], vsc = p.v_scale[h];
        uint32_t kc = 0u, vc = 0u;
#pragma unroll
        for (int e = 0; e < CPL; ++e) {
          kc |= e4m3_code(tof(kn[e]), ksc) << (8 * e);
          vc |= e4m3_code(tof(vn[e]), vsc) << (8 * e);
        }
        const uint32_t off = (uint32_t)r * 128u + ((((uint32_t)cb >> 4) ^ (uint32_t)(r & 7)) << 4) +
                             (uint32_t)(cb & 15);
        *reinterpret_cast<uint32_t *>(kt + off) = kc;
        *reinterpret_cast<uint32_t *>(vt + off) = vc;
        const size_t grow = dyn ? ((size_t)td.z * p.P + td.y + r) * D + cb
                                : ((size_t)td.y + r) * D + cb;
        *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(dyn ? p.k_pool : p.stream_k) + grow) =
            kc;
        *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(dyn ? p.v_pool : p.stream_v) + grow) =
            vc;
        if (dyn) {
          const int j = nL - 1;
          uint8_t *mrow = static_cast<uint8_t *>(p.meta) +
                          ((size_t)td.z * p.R + (j % p.R)) * 2 * D + cb;
          const bool fresh = (L - 1) % p.ell == 0;
          uint32_t mn = kc, mx = kc;
          if (!fresh) {
            const uint32_t omin = *reinterpret_cast<const uint32_t *>(mrow);
            const uint32_t omax = *reinterpret_cast<const uint32_t *>(mrow + D);
            mn = mx = 0u;
#pragma unroll
            for (int e = 0; e < CPL; ++e) {
              const uint32_t x = (kc >> (8 * e)) & 0xffu;
              const uint32_t a = (omin >> (8 * e)) & 0xffu, b = (omax >> (8 * e)) & 0xffu;
              mn |= (e4m3_key(x) < e4m3_key(a) ? x : a) << (8 * e);
              mx |= (e4m3_key(x) > e4m3_key(b) ? x : b) << (8 * e);
            }
          }
          *reinterpret_cast<uint32_t *>(mrow) = mn;
          *reinterpret_cast<uint32_t *>(mrow + D) = mx;
        }
        __syncwarp();
      } else if (!kF8 && do_append && t == nt - 1) {
        // the newest token is row nv-1 of the unit's last tile
        const int r = nv - 1;
        const int cb = lane * CPL;
        const size_t src = ((size_t)i * p.Hkv + h) * D + cb;
        const uint16_t *kn = reinterpret_cast<const uint16_t *>(p.k_new) + src;
        const uint16_t *vn = reinterpret_cast<const uint16_t *>(p.v_new) + src;
        uint16_t kx[CPL], vx[CPL];
#pragma unroll
        for (int e = 0; e < CPL; ++e) {
          kx[e] = kn[e];
          vx[e] = vn[e];
        }
#pragma unroll
        for (int e = 0; e < CPL; ++e) {
          *reinterpret_cast<uint16_t *>(kt + chan_off<D>(r, cb + e)) = kx[e];
          *reinterpret_cast<uint16_t *>(vt + chan_off<D>(r, cb + e)) = vx[e];
        }
        size_t grow;
        uint16_t *kg, *vg;
        if (dyn) {
          grow = ((size_t)td.z * p.P + td.y + r) * D + cb;
          kg = static_cast<uint16_t *>(p.k_pool) + grow;
          vg = static_cast<uint16_t *>(p.v_pool) + grow;
        } else {
          grow = ((size_t)td.y + r) * D + cb;
          kg = static_cast<uint16_t *>(p.stream_k) + grow;
          vg = static_cast<uint16_t *>(p.stream_v) + grow;
        }
#pragma unroll
        for (int e = 0; e < CPL; ++e) {
          kg[e] = kx[e];
          vg[e] = vx[e];
        }
        if (dyn) {
          const int j = nL - 1;
          uint16_t *mrow = static_cast<uint16_t *>(p.meta) +
                           ((size_t)td.z * p.R + (j % p.R)) * 2 * D + cb;
          const bool fresh = (L - 1) % p.ell == 0;
#pragma unroll
          for (int e = 0; e < CPL; ++e) {
            uint16_t bmin = kx[e], bmax = kx[e];
            if (!fresh) {
              const uint16_t omin = mrow[e], omax = mrow[D + e];
              const float x = tof(*reinterpret_cast<const T *>(&kx[e]));
              bmin = x < tof(*reinterpret_cast<const T *>(&omin)) ? kx[e] : omin;
              bmax = x > tof(*reinterpret_cast<const T *>(&omax)) ? kx[e] : omax;
            }
            mrow[e] = bmin;
            mrow[D + e] = bmax;
          }
        }
        __syncwarp();
      }
      if (nv < kRows) {
        // rows past the tile's attended tokens: zero V so the unrolled P.V
        // below adds exactly 0 for them (their weights are 0 as well)
        for (int x = lane; x < (kRows - nv) * 8 * Gm::kBoxes; x += 32) {
          const int box = x / ((kRows - nv) * 8), rem = x % ((kRows - nv) * 8);
          const int r = nv + rem / 8, ch = rem % 8;
          *reinterpret_cast<uint4 *>(vt + box * Gm::kBoxBytes + r * 128 + ch * 16) =
              make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }

      // q.K^T for 16 rows x 8 (padded) heads
      // two accumulators (even and odd k-steps) halve the chain of dependent MMAs
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (kF8) {
        // ldmatrix of byte pairs: matrices (rows 0-7 | 8-15) x (16-channel
        // chunk 2k2 | 2k2+1); a lane gets channels 4t4..4t4+3 of rows g8 and
        // g8+8 -- the A fragment's k slots {2t4, 2t4+1} (low half) and
        // {2t4+8, 2t4+9} (high half) in the q fragments' channel order
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int chalf = lane >> 4;
        const uint32_t kbase = smem_u32(kt);
#pragma unroll
        for (int k2 = 0; k2 < D / 32; ++k2) {
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4(kbase + swz128(row, 2 * k2 + chalf), r0, r1, r2, r3);
          const uint32_t a0[4] = {e4m3x2_to<__half>(r0), e4m3x2_to<__half>(r1),
                                  e4m3x2_to<__half>(r0 >> 16), e4m3x2_to<__half>(r1 >> 16)};
          mma_16816<kQkBf>(acc, a0, qb[2 * k2][0], qb[2 * k2][1]);
          const uint32_t a1[4] = {e4m3x2_to<__half>(r2), e4m3x2_to<__half>(r3),
                                  e4m3x2_to<__half>(r2 >> 16), e4m3x2_to<__half>(r3 >> 16)};
          mma_16816<kQkBf>(acc2, a1, qb[2 * k2 + 1][0], qb[2 * k2 + 1][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] += acc2[e];
      } else {
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int chalf = lane >> 4;
        const uint32_t kbase = smem_u32(kt);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int box = kk >> 2;
          const int chunk = 2 * (kk & 3) + chalf;
          uint32_t a[4];
          ldmatrix_x4(kbase + box * Gm::kBoxBytes + swz128(row, chunk), a[0], a[1], a[2], a[3]);
          if (kk & 1)
            mma_16816<kQkBf>(acc2, a, qb[kk][0], qb[kk][1]);
          else
            mma_16816<kQkBf>(acc, a, qb[kk][0], qb[kk][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] += acc2[e];
      }
      // acc: [0] row g8 head 2t4, [1] row g8 head 2t4+1, [2] row g8+8 head 2t4, [3] row g8+8 head 2t4+1
      const bool v_lo = g8 < nv, v_hi = g8 + 8 < nv;
      const float z0 = v_lo ? acc[0] * sc : -CUDART_INF_F;
      const float z1 = v_lo ? acc[1] * sc : -CUDART_INF_F;
      const float z2 = v_hi ? acc[2] * sc : -CUDART_INF_F;
      const float z3 = v_hi ? acc[3] * sc : -CUDART_INF_F;
      float mx0 = fmaxf(z0, z2), mx1 = fmaxf(z1, z3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      // (m = -inf before the first tile: any finite tile max moves it)
      const float mn0 = mx0 > m0 + stale ? mx0 : m0, mn1 = mx1 > m1 + stale ? mx1 : m1;
      const bool moved = __any_sync(0xffffffffu, mn0 != m0 || mn1 != m1);
      const float c0 = ex2_approx(m0 - mn0), c1 = ex2_approx(m1 - mn1);
      const float p0 = ex2_approx(z0 - mn0), p1 = ex2_approx(z1 - mn1);
      const float p2 = ex2_approx(z2 - mn0), p3 = ex2_approx(z3 - mn1);
      l0 = l0 * c0 + p0 + p2;
      l1 = l1 * c1 + p1 + p3;
      m0 = mn0;
      m1 = mn1;
      const int h0 = 2 * t4, h1 = 2 * t4 + 1;
      if (kMass && dyn) {
        // the tile's share for the per-page mass: (running max, sum of
        // exp2(z - max) over its rows) per head
        float s0 = p0 + p2, s1 = p1 + p3;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          s0 += __shfl_xor_sync(0xffffffffu, s0, off);
          s1 += __shfl_xor_sync(0xffffffffu, s1, off);
        }
        if (g8 == 0) {
          float2 *pp = p.page_part +
                       (((size_t)i * p.Hd + sub) * p.page_tile_cap + tile0 + t) * G;
          if (h0 < G) pp[h0] = make_float2(mn0, s0);
          if (h1 < G) pp[h1] = make_float2(mn1, s1);
        }
      }
      if (h0 < G) {
        Pw[g8 * GPAD + h0] = p0;
        Pw[(g8 + 8) * GPAD + h0] = p2;
      }
      if (h1 < G) {
        Pw[g8 * GPAD + h1] = p1;
        Pw[(g8 + 8) * GPAD + h1] = p3;
      }
      __syncwarp();

      // P.V on tensor cores: rescale (when a max moved), then
      // O^T += V^T (P_hi + P_lo)^T
      if (moved) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          oacc[m][0] *= c0;
          oacc[m][1] *= c1;
          oacc[m][2] *= c0;
          oacc[m][3] *= c1;
        }
      }
      uint32_t bh0, bh1, bl0, bl1;  // B = P^T: k = tokens 2t4.. / 2t4+8.., n = head g8
      {
        float pv[4] = {0.f, 0.f, 0.f, 0.f};
        if (g8 < G) {
          pv[0] = Pw[(2 * t4) * GPAD + g8];
          pv[1] = Pw[(2 * t4 + 1) * GPAD + g8];
          pv[2] = Pw[(2 * t4 + 8) * GPAD + g8];
          pv[3] = Pw[(2 * t4 + 9) * GPAD + g8];
        }
        Split2<TP>::run(pv[0], pv[1], bh0, bl0);
        Split2<TP>::run(pv[2], pv[3], bh1, bl1);
      }
      if constexpr (kF8) {
        // A = V^T, transposed ldmatrix of byte pairs: matrices (tokens 0-7 |
        // 8-15) x (chunk 2m2 | 2m2+1); a lane gets tokens 2t4, 2t4+1 (+8) x
        // channels 2g8, 2g8+1.  Rows of the m-tile are channel 2g8 (m = g8)
        // and 2g8+1 (m = g8+8): a byte permute splits the word into them.
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int chalf = lane >> 4;
        const uint32_t vbase = smem_u32(vt);
#pragma unroll
        for (int m2 = 0; m2 < D / 32; ++m2) {
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4_trans(vbase + swz128(row, 2 * m2 + chalf), r0, r1, r2, r3);
          const uint32_t e0 = __byte_perm(r0, 0u, 0x3120), e1 = __byte_perm(r1, 0u, 0x3120);
          const uint32_t e2 = __byte_perm(r2, 0u, 0x3120), e3 = __byte_perm(r3, 0u, 0x3120);
          const uint32_t a0[4] = {e4m3x2_to<TP>(e0), e4m3x2_to<TP>(e0 >> 16), e4m3x2_to<TP>(e1),
                                  e4m3x2_to<TP>(e1 >> 16)};
          mma_16816<kPvBf>(oacc[2 * m2], a0, bh0, bh1);
          mma_16816<kPvBf>(oacc[2 * m2], a0, bl0, bl1);
          const uint32_t a1[4] = {e4m3x2_to<TP>(e2), e4m3x2_to<TP>(e2 >> 16), e4m3x2_to<TP>(e3),
                                  e4m3x2_to<TP>(e3 >> 16)};
          mma_16816<kPvBf>(oacc[2 * m2 + 1], a1, bh0, bh1);
          mma_16816<kPvBf>(oacc[2 * m2 + 1], a1, bl0, bl1);
        }
      } else {
        // A = V^T for m-tile m: matrix j of ldmatrix.x4.trans takes token rows
        // (lane & 7) + 8 * (j >> 1) and channel chunk 2m + (j & 1)
        const int j = lane >> 3;
        const int row = (lane & 7) + 8 * (j >> 1);
        const uint32_t vbase = smem_u32(vt);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const int box = m >> 2;
          const int chunk = 2 * (m & 3) + (j & 1);
          uint32_t a[4];
          ldmatrix_x4_trans(vbase + box * Gm::kBoxBytes + swz128(row, chunk), a[0], a[1], a[2],
                            a[3]);
          mma_16816<kPvBf>(oacc[m], a, bh0, bh1);
          mma_16816<kPvBf>(oacc[m], a, bl0, bl1);
        }
      }
      __syncwarp();
    } else if (kMass && dyn && lane < G) {
      p.page_part[(((size_t)i * p.Hd + sub) * p.page_tile_cap + tile0 + t) * G + lane] =
          make_float2(-CUDART_INF_F, 0.f);
    }
    // refill the stage with the tile kStages further on, then take the next tile
    if (t + kStages < nt) {
      fence_proxy_async_smem();  // the warp's reads of the stage precede the TMA write
      if (lane == 0) issue(t + kStages);
    }
    int nx = 0;
    if (lane == 0) nx = atomicAdd(&s_flag[2], 1);
    t = __shfl_sync(0xffffffffu, nx, 0);
  }

  // ---- merge the warps into this CTA's (M, L, O) ----
  // (fp8: the output scale is read now, its latency hidden by the merges)
  const float vsc = kF8 ? p.v_scale[h] : 1.f;
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  __syncthreads();  // every warp is done with its stage: reuse the region for o
  if (s_flag[1]) {
    // a wait gave up: give the last load issued to each stage one more
    // bounded wait before the stage region is reused
    if (lane == 0)
      for (int st = warp; st < kStages; st += kWarps)
        if (s_iss[st] > 0) mbar_wait(&bars[st], (s_iss[st] - 1) & 1, kWaitLimit);
    __syncthreads();
  }
  // [W][G][D + 4]: the 4 padding words per row put the heads of a lane
  // group's stores in different banks
  constexpr int OS = D + 4;
  float *o_w = reinterpret_cast<float *>(stages);
  if (g8 == 0) {
    if (2 * t4 < G) {
      m_w[warp * G + 2 * t4] = m0;
      l_w[warp * G + 2 * t4] = l0;
    }
    if (2 * t4 + 1 < G) {
      m_w[warp * G + 2 * t4 + 1] = m1;
      l_w[warp * G + 2 * t4 + 1] = l1;
    }
  }
  // channels contiguous per (warp, head): the push below reads 4 at a time
  // (fp8: rows g8 / g8+8 of m-tile m are channels 16m + 2g8 / + 1)
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const int ch = kF8 ? 16 * m + 2 * g8 : 16 * m + g8;
    const int ch2 = kF8 ? ch + 1 : ch + 8;
    if (2 * t4 < G) {
      o_w[(warp * G + 2 * t4) * OS + ch] = oacc[m][0];
      o_w[(warp * G + 2 * t4) * OS + ch2] = oacc[m][2];
    }
    if (2 * t4 + 1 < G) {
      o_w[(warp * G + 2 * t4 + 1) * OS + ch] = oacc[m][1];
      o_w[(warp * G + 2 * t4 + 1) * OS + ch2] = oacc[m][3];
    }
  }
  __syncthreads();
  // this CTA's (M, L, O), pushed straight into the inbox of the cluster CTA
  // that owns each channel slice (remote shared-memory stores)
  // CS, the slice and TPE below are powers of two: shifts and masks, not
  // run-time integer division
  const int lcs = __ffs(CS) - 1;
  const int slice = D >> lcs, lsl = __ffs(slice) - 1;
  const uint32_t aM = smem_u32(in_M), aL = smem_u32(in_L), aO = smem_u32(in_O);
  const uint32_t aB = smem_u32(inbox_bar);
  // a thread takes 4 adjacent channels of one head: the warp weights are
  // computed once for them, read and pushed 16 bytes at a time (a slice
  // holds a multiple of 4 channels, so the 4 share an owner)
  for (int x = tid; x < G * D / 4; x += kThreads) {
    const int g = x / (D / 4), c = 4 * (x % (D / 4));
    float M = m_w[g];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, m_w[w * G + g]);
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    float Ls = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = ex2_approx(m_w[w * G + g] - M);
        const float4 o = *reinterpret_cast<const float4 *>(&o_w[(w * G + g) * OS + c]);
        O.x = fmaf(f, o.x, O.x);
        O.y = fmaf(f, o.y, O.y);
        O.z = fmaf(f, o.z, O.z);
        O.w = fmaf(f, o.w, O.w);
        Ls = fmaf(f, l_w[w * G + g], Ls);
      }
    }
    const int owner = c >> lsl, cs_ = c & (slice - 1);
    // an owner's inbox row per sending rank is G * slice + 4 words: the
    // ranks of one element fall in different banks when it is read back
    const int io = rank * (G * slice + 4) + g * slice + cs_;
    if (remote) {
      const uint32_t rb = map_rank(aB, owner);
      st_async_v4_f32(map_rank(aO + 4 * io, owner), O, rb);
      if (cs_ == 0) {
        st_async_f32(map_rank(aM + 4 * (rank * G + g), owner), M, rb);
        st_async_f32(map_rank(aL + 4 * (rank * G + g), owner), Ls, rb);
      }
    } else {  // (rank 0 of one: its own inbox)
      *reinterpret_cast<float4 *>(&in_O[io]) = O;
      if (cs_ == 0) {
        in_M[g] = M;
        in_L[g] = Ls;
      }
    }
  }
  // A CTA leaves only once its inbox holds every rank's bytes, so no peer is
  // still storing into it.  A second cluster phase is needed only when the
  // cluster's CTAs read one another's global writes: the per-tile pairs of
  // the page-mass export (released here, acquired before they are read) and
  // the slices several clusters merge in global memory.
  const bool phase2 = kMass || nc > 1;  // (the same in every CTA of a cluster)
  if (phase2) {
    if constexpr (kMass)
      cluster_arrive_release();
    else
      cluster_arrive_relaxed();
  }

  // ---- merge the cluster: this CTA combines channels [rank*slice, +slice) ----
  // every rank's pushes into this CTA's inbox have landed
  if (!__syncthreads_and(!remote || mbar_wait(inbox_bar, 0, kWaitLimit))) {
    if (tid == 0) set_err(p.err, kDevTimeout, s.slot, h, -2);
    if (phase2) cluster_wait();
    return;
  }
  const int unit = i * p.Hkv + h;
  float *out = p.out + ((size_t)i * p.Hq + h * G) * D;
  const size_t cpart = (size_t)unit_item0 + (size_t)ci * CS;  // global slot of this cluster
  // one thread per output element of the slice.  Every rank's (m, l, o) is
  // loaded up front with no branch between the loads (independent loads,
  // then short max and sum chains: shorter than splitting the ranks over
  // lanes and reducing with shuffles).  A rank that attended nothing pushed
  // m = -inf, l = 0, o = 0 and ranks >= CS read as the same, so its weight
  // exp2(-inf - M) is 0 and adds exactly nothing.
  const int E = G * slice;
  for (int x = tid; x < E; x += kThreads) {
    const int g = x >> lsl, cl = x & (slice - 1), c = rank * slice + cl;
    float mr[16], lr[16], orr[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const bool in = r < CS;
      mr[r] = in ? in_M[r * G + g] : -CUDART_INF_F;
      lr[r] = in ? in_L[r * G + g] : 0.f;
      orr[r] = in ? in_O[r * (E + 4) + g * slice + cl] : 0.f;
    }
    float M = mr[0];
#pragma unroll
    for (int r = 1; r < 16; ++r) M = fmaxf(M, mr[r]);
    float O = 0.f, Ls = 0.f;
    if (M != -CUDART_INF_F) {
      // two chains each for the sums (even and odd ranks)
      float O1 = 0.f, L1 = 0.f;
#pragma unroll
      for (int r = 0; r < 16; r += 2) {
        const float f0 = ex2_approx(mr[r] - M), f1 = ex2_approx(mr[r + 1] - M);
        Ls = fmaf(f0, lr[r], Ls);
        O = fmaf(f0, orr[r], O);
        L1 = fmaf(f1, lr[r + 1], L1);
        O1 = fmaf(f1, orr[r + 1], O1);
      }
      O += O1;
      Ls += L1;
    }
    if (nc == 1) {
      // (fp8: the stored values are code * v_scale)
      out[g * D + c] = kF8 ? O / Ls * vsc : O / Ls;
      if (p.row_max && rank == 0 && cl == 0) {
        // the logits' max in natural units (M is base 2, scale folded in)
        // and the sum of exp(z - max) over the attended tokens
        const size_t hq = (size_t)i * p.Hq + h * G + g;
        p.row_max[hq] = M * 0.6931471805599453f;
        p.row_sum[hq] = Ls;
      }
    } else {
      p.part_o[(cpart * G + g) * D + c] = O;
      if (rank == 0 && cl == 0) p.part_ml[cpart * G + g] = make_float2(M, Ls);
    }
  }
  if (nc == 1) {
    if (kMass) cluster_wait();  // (acquire: the cluster's per-tile pairs)
    if (kMass && dyn) {
      // every CTA of the cluster stored its tiles' pairs before the cluster
      // barrier; the unit's final max and sum per head come from the inbox
      __syncthreads();  // (m_w, l_w are free: the push that read them is done)
      if (tid < G) {
        float M = -CUDART_INF_F, Ls = 0.f;
        for (int r = 0; r < CS; ++r) M = fmaxf(M, in_M[r * G + tid]);
        for (int r = 0; r < CS; ++r)
          if (in_M[r * G + tid] != -CUDART_INF_F)
            Ls = fmaf(exp2f(in_M[r * G + tid] - M), in_L[r * G + tid], Ls);
        m_w[tid] = M;
        l_w[tid] = Ls;
      }
      __syncthreads();
      write_page_mass<G>(p, i, sub, s, nL, n_tiles, m_w, l_w, rank * kThreads + tid,
                         CS * kThreads);
    }
    return;
  }
  cluster_wait();
  cluster_sync();  // every rank's slice is written before rank 0 releases it
  if (rank != 0) return;

  // ---- several clusters: the last one to finish merges their results ----
  if (tid == 0) {
    const int prev = atom_add_acq_rel_gpu(&p.tickets[unit], 1);
    *s_flag = prev == nc - 1;
  }
  __syncthreads();  // ... and the acquire above precedes every read below
  if (!*s_flag) return;
  // (1) every (m, l) pair into shared memory, (2) per-head max, weights and
  // row sum, (3) the weighted sum of the o partials, kU at a time.
  constexpr int kChunk = 256;                       // clusters per pass
  constexpr int OPT4 = (G * D / 4 + kThreads - 1) / kThreads;
  constexpr int kU = 8;
  float *Mh = m_w;                                  // [G]
  float *Lh = l_w;                                  // [G]
  float2 *mlk = reinterpret_cast<float2 *>(stages); // [kChunk][G]
  float *wk = reinterpret_cast<float *>(mlk + kChunk * G);  // [kChunk][G] + [G]
  float4 acc_o[OPT4];
#pragma unroll
  for (int j = 0; j < OPT4; ++j) acc_o[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid < G) {
    Mh[tid] = -CUDART_INF_F;
    Lh[tid] = 0.f;
  }
  for (int base = 0; base < nc; base += kChunk) {
    const int cnt = min(kChunk, nc - base);
    for (int x = tid; x < cnt * G; x += kThreads) {
      const int k = x / G, g = x % G;
      mlk[x] = __ldcg(&p.part_ml[((size_t)unit_item0 + (size_t)(base + k) * CS) * G + g]);
    }
    __syncthreads();
    if (tid < G) {
      const int g = tid;
      float M = Mh[g];
      for (int k = 0; k < cnt; ++k) M = fmaxf(M, mlk[k * G + g].x);
      const float resc = Mh[g] == -CUDART_INF_F ? 0.f : exp2f(Mh[g] - M);
      float Ls = Lh[g] * resc;
      for (int k = 0; k < cnt; ++k) {
        const float2 ml = mlk[k * G + g];
        const float w = ml.x == -CUDART_INF_F ? 0.f : exp2f(ml.x - M);
        wk[k * G + g] = w;
        Ls = fmaf(w, ml.y, Ls);
      }
      wk[kChunk * G + g] = resc;
      Mh[g] = M;
      Lh[g] = Ls;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < OPT4; ++j) {
      const int x4 = tid + kThreads * j;
      if (x4 < G * D / 4) {
        const float r = wk[kChunk * G + (4 * x4) / D];
        acc_o[j].x *= r;
        acc_o[j].y *= r;
        acc_o[j].z *= r;
        acc_o[j].w *= r;
      }
    }
    for (int k = 0; k < cnt; k += kU) {
      float4 v[kU][OPT4];
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int j = 0; j < OPT4; ++j) {
          const int x4 = tid + kThreads * j;
          const float4 *src = reinterpret_cast<const float4 *>(
              p.part_o + ((size_t)unit_item0 + (size_t)(base + k + u) * CS) * G * D);
          v[u][j] = (k + u < cnt && x4 < G * D / 4) ? __ldcg(src + x4)
                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int j = 0; j < OPT4; ++j) {
          const int x4 = tid + kThreads * j;
          if (k + u < cnt && x4 < G * D / 4) {
            const float w = wk[(k + u) * G + (4 * x4) / D];
            acc_o[j].x = fmaf(w, v[u][j].x, acc_o[j].x);
            acc_o[j].y = fmaf(w, v[u][j].y, acc_o[j].y);
            acc_o[j].z = fmaf(w, v[u][j].z, acc_o[j].z);
            acc_o[j].w = fmaf(w, v[u][j].w, acc_o[j].w);
          }
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < OPT4; ++j) {
    const int x4 = tid + kThreads * j;
    if (x4 < G * D / 4) {
      const float inv = vsc / Lh[(4 * x4) / D];
      reinterpret_cast<float4 *>(out)[x4] =
          make_float4(acc_o[j].x * inv, acc_o[j].y * inv, acc_o[j].z * inv, acc_o[j].w * inv);
    }
  }
  if (p.row_max && tid < G) {
    const size_t hq = (size_t)i * p.Hq + h * G + tid;
    p.row_max[hq] = Mh[tid] * 0.6931471805599453f;
    p.row_sum[hq] = Lh[tid];
  }
  // every cluster's pairs precede its ticket (cluster barrier, then the
  // acquire-release ticket): this CTA sees them all
  if (kMass && dyn)
    write_page_mass<G>(p, i, sub, s, nL, n_tiles, Mh, Lh, tid, kThreads);
  if (tid == 0) p.tickets[unit] = 0;
}


template <typename T, int D, int G, bool kMass, bool kF8 = false, bool kDeep = false,
          bool kReuse = false>
cudaError_t set_smem_attrs() {
  auto k = decode_tiles_kernel<T, D, G, kMass, kF8, kDeep, kReuse>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Smem<D, G, kF8, kDeep>::kAlloc);
  if (e != cudaSuccess) return e;
  (void)cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  (void)cudaGetLastError();
  return cudaSuccess;
}

template <typename T, int D, bool kMass>
cudaError_t set_smem_attrs_g() {
  cudaError_t e;
  if ((e = set_smem_attrs<T, D, 1, kMass>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs<T, D, 2, kMass>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs<T, D, 4, kMass>()) != cudaSuccess) return e;
  return set_smem_attrs<T, D, 8, kMass>();
}

template <bool kMass>
cudaError_t set_smem_attrs_all() {
  cudaError_t e;
  if ((e = set_smem_attrs_g<__half, 64, kMass>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs_g<__half, 128, kMass>()) != cudaSuccess) return e;
  if ((e = set_smem_attrs_g<__nv_bfloat16, 64, kMass>()) != cudaSuccess) return e;
  return set_smem_attrs_g<__nv_bfloat16, 128, kMass>();
}

template <typename T, int D, int G, bool kMass, bool kF8 = false, bool kDeep = false,
          bool kReuse = false>
cudaError_t launch_one(const TileDecodeParams &p, cudaStream_t st) {
  cudaError_t e = launch_pdl_cluster(decode_tiles_kernel<T, D, G, kMass, kF8, kDeep, kReuse>,
                                     p.total_items, kThreads,
                                     (size_t)Smem<D, G, kF8, kDeep>::kAlloc, p.cluster, st, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int D, bool kMass, bool kDeep = false, bool kReuse = false>
cudaError_t launch_g(const TileDecodeParams &p, int G, cudaStream_t st) {
  switch (G) {
    case 1: return launch_one<T, D, 1, kMass, false, kDeep, kReuse>(p, st);
    case 2: return launch_one<T, D, 2, kMass, false, kDeep, kReuse>(p, st);
    case 4: return launch_one<T, D, 4, kMass, false, kDeep, kReuse>(p, st);
    case 8: return launch_one<T, D, 8, kMass, false, kDeep, kReuse>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

template <bool kMass, bool kDeep = false, bool kReuse = false>
cudaError_t launch_variant(const TileDecodeParams &p, int dtype, int d, int G, cudaStream_t s) {
  if (dtype == 0)
    return d == 64 ? launch_g<__half, 64, kMass, kDeep, kReuse>(p, G, s)
                   : launch_g<__half, 128, kMass, kDeep, kReuse>(p, G, s);
  return d == 64 ? launch_g<__nv_bfloat16, 64, kMass, kDeep, kReuse>(p, G, s)
                 : launch_g<__nv_bfloat16, 128, kMass, kDeep, kReuse>(p, G, s);
}

}  // namespace
}  // namespace spd
