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
// A CTA (4 warps) takes up to 8 consecutive tiles of one unit (an "item").
//
// Data movement.  One thread issues every TMA tensor load of the item at
// kernel start (2-D boxes of 64 channels x 16 rows, 128-byte swizzle, one
// mbarrier per tile), so the whole item is in flight at once; K/V bytes are
// read from HBM exactly once.
//
// Math (per warp, per tile, all G query heads of the kv head at once):
//   q.K^T   mma.sync m16n8k16, A = K tile rows (ldmatrix from the swizzled
//           tile), B = q^T held in registers (heads padded to 8 columns),
//           fp32 accumulate -- the products of 16-bit inputs are exact;
//   softmax online, in fp32, base-2 with log2(e)/sqrt(d) folded in;
//   P.V     fp32 FMAs on CUDA cores (P stays fp32: no rounding of weights).
// Split combine.  Each item writes (o, m, l) for its unit; the last item of a
// unit to finish (atomic ticket, no waiting) merges them with a
// log-sum-exp rescale and writes the fp32 output -- the row max / row sum
// export of the Novita KV-sparsity article ("attention mechanism
// modifications").
//
// Fused append (decode step).  The CTA that owns a unit's newest token also
// appends it: the row is written to the pool / ring, patched into the
// staged tile, and folded into the logical page's key min/max.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "ptx.cuh"
#include "spd_internal.h"

namespace spd {
namespace {

constexpr int kRows = 16;          // rows per tile (one mma M tile)
constexpr int kMaxTiles = 8;       // tiles per item
constexpr int kWarps = 4;
constexpr uint32_t kWaitLimit = 1u << 24;  // bounded mbarrier polls

template <int D>
struct Geo {
  static constexpr int kBoxes = D / 64;                 // 64-channel boxes per row
  static constexpr int kBoxBytes = kRows * 128;         // one box: 16 rows x 128 B
  static constexpr int kTileBytes = 2 * kBoxes * kBoxBytes;  // K boxes then V boxes
  static constexpr int kCPL = D / 32;                   // channels per lane in P.V
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

// Shared memory: a small fixed region (barriers, tile descriptors, P and
// rescale buffers, per-warp row max / sum, flags), then the K/V tiles at a
// 1024-byte aligned offset.  The launch sizes the tile region for the largest
// item it holds, at least big enough for the warp-merge and combine buffers.
template <int D, int G>
struct Smem {
  static constexpr int kBars = 0;                                   // uint64 x kMaxTiles
  static constexpr int kDesc = kBars + kMaxTiles * 8;               // TileDesc x kMaxTiles
  static constexpr int kP = kDesc + kMaxTiles * (int)sizeof(TileDesc);  // float [W][16][GP]
  static constexpr int kC = kP + kWarps * kRows * GP<G>::v * 4;     // float [W][GP]
  static constexpr int kML = kC + kWarps * GP<G>::v * 4;            // float [2][W][G]
  static constexpr int kFlag = kML + 2 * kWarps * G * 4;            // int [4]
  static constexpr int kTiles = (kFlag + 16 + 1023) / 1024 * 1024;  // tiles start here
  // warp-merge buffer [W][G][D] floats, or the combine's (m, l) and weight
  // buffers for 256 items
  static constexpr int kMinTileRegion = (kWarps * G * D * 4 > 256 * G * 12 + 64)
                                            ? kWarps * G * D * 4
                                            : 256 * G * 12 + 64;
  static constexpr int bytes(int tiles) {
    return kTiles + (tiles * Geo<D>::kTileBytes > kMinTileRegion ? tiles * Geo<D>::kTileBytes
                                                                  : kMinTileRegion) +
           1024;  // alignment slack
  }
  static constexpr int kAlloc = bytes(kMaxTiles);
};

template <typename T> struct IsBF16 { static constexpr bool v = false; };
template <> struct IsBF16<__nv_bfloat16> { static constexpr bool v = true; };

template <typename T>
__device__ __forceinline__ float tof(T x);
template <> __device__ __forceinline__ float tof(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float tof(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ uint32_t pack2(uint16_t lo, uint16_t hi) {
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ void set_err(int *err, int code, int a, int b, int c) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}

// Byte offset, inside a tile half (K or V), of channel `ch` of row `r`.
template <int D>
__device__ __forceinline__ uint32_t chan_off(int r, int ch) {
  return (uint32_t)((ch >> 6) * Geo<D>::kBoxBytes) + swz128(r, (ch & 63) >> 3) +
         (uint32_t)((ch & 7) * 2);
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(128) decode_tiles_kernel(const __grid_constant__ TileDecodeParams p) {
  using Gm = Geo<D>;
  using Sm = Smem<D, G>;
  constexpr int CPL = Gm::kCPL;
  constexpr int GPAD = GP<G>::v;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *tiles = smem + Sm::kTiles;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Sm::kBars);
  TileDesc *tdesc = reinterpret_cast<TileDesc *>(smem + Sm::kDesc);
  float *P_all = reinterpret_cast<float *>(smem + Sm::kP);
  float *C_all = reinterpret_cast<float *>(smem + Sm::kC);
  float *m_w = reinterpret_cast<float *>(smem + Sm::kML);
  float *l_w = m_w + kWarps * G;
  int *s_flag = reinterpret_cast<int *>(smem + Sm::kFlag);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_sk);
    prefetch_tmap(&p.tm_sv);
    s_flag[1] = 0;  // set if a bounded wait gives up
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
  const int nt = max(0, min(n_tiles, tile0 + tpi) - tile0);
  const bool owns_newest = tile0 + nt == n_tiles;
  const bool do_append = p.k_new != nullptr && owns_newest;

  // Everything above used only the parameter block.  The KV cache (page
  // table, selection, pools) is read next: before the wait for the previous
  // kernel on the stream when the host knows that kernel cannot have written
  // this context's cache (p.early), after it otherwise.  q, the new token and
  // every write come after the wait.  Dependents are released only after the
  // wait, so when this kernel runs, every kernel before its immediate
  // predecessor has finished.
  if (!p.early) {
    pdl_wait();
    pdl_launch_dependents();
  }

  // ---- issue every TMA load of the item: thread t sets up tile t ----
  if (tid < nt) {
    const int t = tid;
    mbar_init(&bars[t], 1);
    fence_mbar_init();
    const CUtensorMap *mk = dyn ? &p.tm_k : &p.tm_sk;
    const CUtensorMap *mv = dyn ? &p.tm_v : &p.tm_sv;
    const int tau = tile0 + t;
    TileDesc td{0, 0, 0, 0};
    if (dyn) {
      const int pi = tau / tpp, st = tau % tpp;
      const int *sel = p.selection + ((size_t)s.slot * p.Hd + sub) * p.ksel_max;
      const int j = pi < s.sel_count ? sel[pi] : s.nL0 + (pi - s.sel_count);
      const int blk = j / p.R;
      if (j < 0 || j >= nL || blk >= p.max_pp) {
        set_err(p.err, kDevBadSelection, s.slot, sub, j);
      } else {
        const int phys = p.page_table[(size_t)s.slot * p.max_pp + blk];
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
    if (td.n_valid > 0) {
      uint8_t *kt = tiles + t * Gm::kTileBytes;
      uint8_t *vt = kt + Gm::kBoxes * Gm::kBoxBytes;
      mbar_arrive_expect_tx(&bars[t], Gm::kTileBytes);
      for (int b = 0; b < Gm::kBoxes; ++b) {
        tma_load_3d(kt + b * Gm::kBoxBytes, mk, b * 64, td.y, td.z, &bars[t]);
        tma_load_3d(vt + b * Gm::kBoxBytes, mv, b * 64, td.y, td.z, &bars[t]);
      }
    }
  }

  if (p.early) {
    pdl_wait();
    pdl_launch_dependents();
  }

  // ---- q^T fragments (B operand), heads padded to 8 columns ----
  const int g8 = lane >> 2, t4 = lane & 3;
  uint32_t qb[D / 16][2];
  {
    const uint16_t *qp = reinterpret_cast<const uint16_t *>(p.q) + ((size_t)i * p.Hq + h * G) * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      if (g8 < G) {
        const uint16_t *row = qp + g8 * D + kk * 16 + 2 * t4;
        qb[kk][0] = pack2(row[0], row[1]);
        qb[kk][1] = pack2(row[8], row[9]);
      } else {
        qb[kk][0] = qb[kk][1] = 0u;
      }
    }
  }
  __syncthreads();

  // ---- per-warp online softmax over its tiles ----
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;  // heads 2t4, 2t4+1
  float o[G][CPL];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < CPL; ++e) o[g][e] = 0.f;
  float *Pw = P_all + warp * kRows * GPAD;
  float *Cw = C_all + warp * GPAD;
  const float sc = p.scale_log2;

  for (int t = warp; t < nt; t += kWarps) {
    const TileDesc td = tdesc[t];
    if (td.n_valid <= 0) continue;
    if (!mbar_wait(&bars[t], 0, kWaitLimit)) {
      if (lane == 0) {
        set_err(p.err, kDevTimeout, s.slot, h, t);
        s_flag[1] = 1;
      }
      continue;
    }
    uint8_t *kt = tiles + t * Gm::kTileBytes;
    uint8_t *vt = kt + Gm::kBoxes * Gm::kBoxBytes;
    const int nv = td.n_valid;

    if (do_append && t == nt - 1) {
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
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int chalf = lane >> 4;
      const uint32_t kbase = smem_u32(kt);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int box = kk >> 2;
        const int chunk = 2 * (kk & 3) + chalf;
        uint32_t a[4];
        ldmatrix_x4(kbase + box * Gm::kBoxBytes + swz128(row, chunk), a[0], a[1], a[2], a[3]);
        mma_16816<IsBF16<T>::v>(acc, a, qb[kk][0], qb[kk][1]);
      }
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
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float c0 = exp2f(m0 - mn0), c1 = exp2f(m1 - mn1);
    const float p0 = exp2f(z0 - mn0), p1 = exp2f(z1 - mn1);
    const float p2 = exp2f(z2 - mn0), p3 = exp2f(z3 - mn1);
    l0 = l0 * c0 + p0 + p2;
    l1 = l1 * c1 + p1 + p3;
    m0 = mn0;
    m1 = mn1;
    const int h0 = 2 * t4, h1 = 2 * t4 + 1;
    if (h0 < G) {
      Pw[g8 * GPAD + h0] = p0;
      Pw[(g8 + 8) * GPAD + h0] = p2;
      if (g8 == 0) Cw[h0] = c0;
    }
    if (h1 < G) {
      Pw[g8 * GPAD + h1] = p1;
      Pw[(g8 + 8) * GPAD + h1] = p3;
      if (g8 == 0) Cw[h1] = c1;
    }
    __syncwarp();

    // P.V: lane owns channels [lane*CPL, lane*CPL + CPL) of every head
    {
      float cr[G];
#pragma unroll
      for (int g = 0; g < G; ++g) cr[g] = Cw[g];
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < CPL; ++e) o[g][e] *= cr[g];
      const int cb = lane * CPL;
      const uint32_t voff = (uint32_t)((cb >> 6) * Gm::kBoxBytes) + ((cb & 7) * 2);
      const int chunk = (cb & 63) >> 3;
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        float vf[CPL];
        const uint8_t *vp = vt + voff + swz128(r, chunk);
        if constexpr (CPL == 4) {
          const uint2 raw = *reinterpret_cast<const uint2 *>(vp);
          const T *e2 = reinterpret_cast<const T *>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) vf[e] = tof(e2[e]);
        } else {
          const uint32_t raw = *reinterpret_cast<const uint32_t *>(vp);
          const T *e2 = reinterpret_cast<const T *>(&raw);
#pragma unroll
          for (int e = 0; e < 2; ++e) vf[e] = tof(e2[e]);
        }
        float pr[GPAD];
        const float4 *prow = reinterpret_cast<const float4 *>(Pw + r * GPAD);
#pragma unroll
        for (int g4 = 0; g4 < GPAD / 4; ++g4) {
          const float4 x = prow[g4];
          pr[4 * g4] = x.x;
          pr[4 * g4 + 1] = x.y;
          pr[4 * g4 + 2] = x.z;
          pr[4 * g4 + 3] = x.w;
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < CPL; ++e) o[g][e] = fmaf(pr[g], vf[e], o[g][e]);
      }
    }
    __syncwarp();
  }

  // ---- merge the warps ----
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  __syncthreads();  // every warp is done with the tiles: reuse them for o
  if (s_flag[1]) {
    // a wait gave up: give the loads still in flight one more bounded wait
    // before their destination is reused
    if (tid == 0)
      for (int t = 0; t < nt; ++t)
        if (tdesc[t].n_valid > 0) mbar_wait(&bars[t], 0, kWaitLimit);
    __syncthreads();
  }
  float *o_w = reinterpret_cast<float *>(tiles);  // [W][G][D]
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
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < CPL; ++e) o_w[(warp * G + g) * D + lane * CPL + e] = o[g][e];
  __syncthreads();

  const int unit = i * p.Hkv + h;
  float *out = p.out + ((size_t)i * p.Hq + h * G) * D;
  for (int x = tid; x < G * D; x += blockDim.x) {
    const int g = x / D, c = x % D;
    float M = m_w[g];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, m_w[w * G + g]);
    float O = 0.f, Ls = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(m_w[w * G + g] - M);
        O += f * o_w[(w * G + g) * D + c];
        Ls += f * l_w[w * G + g];
      }
    }
    if (ns == 1) {
      out[x] = O / Ls;
    } else {
      p.part_o[((size_t)item * G + g) * D + c] = O;
      if (c == 0) p.part_ml[(size_t)item * G + g] = make_float2(M, Ls);
    }
  }
  if (ns == 1) return;

  // ---- last item of the unit merges the partials ----
  __syncthreads();  // every partial write of this CTA precedes the release below
  if (tid == 0) {
    const int prev = atom_add_acq_rel_gpu(&p.tickets[unit], 1);
    *s_flag = prev == ns - 1;
  }
  __syncthreads();  // ... and the acquire above precedes every read below
  if (!*s_flag) return;
  // Merge in three steps, each a single round of independent L2 loads:
  // (1) every (m, l) pair of the chunk into shared memory, (2) per-head max
  // M and weights 2^(m_k - M) with the weighted row sum (shared memory
  // only), (3) the weighted sum of the o partials, kU items per round.
  constexpr int kChunk = 256;                       // items per pass
  constexpr int OPT4 = (G * D / 4 + 127) / 128;     // float4 outputs per thread
  constexpr int kU = 16;                            // o-partial items in flight
  float *Mh = m_w;                                  // [G] (the warp buffers are free now)
  float *Lh = l_w;                                  // [G]
  float2 *mlk = reinterpret_cast<float2 *>(tiles);  // [kChunk][G] (m, l) of the chunk
  float *wk = reinterpret_cast<float *>(mlk + kChunk * G);  // [kChunk][G] weights
  const float2 *pml = p.part_ml + (size_t)unit_item0 * G;
  const float *po = p.part_o + (size_t)unit_item0 * G * D;
  float4 acc_o[OPT4];
#pragma unroll
  for (int j = 0; j < OPT4; ++j) acc_o[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid < G) {
    Mh[tid] = -CUDART_INF_F;
    Lh[tid] = 0.f;
  }
  for (int base = 0; base < ns; base += kChunk) {
    const int cnt = min(kChunk, ns - base);
    for (int x = tid; x < cnt * G; x += blockDim.x) mlk[x] = __ldcg(&pml[(size_t)base * G + x]);
    __syncthreads();
    // one thread per head: running max over the chunk, rescale what came before
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
      wk[kChunk * G + g] = resc;  // factor for the o accumulated so far
      Mh[g] = M;
      Lh[g] = Ls;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < OPT4; ++j) {
      const int x4 = tid + 128 * j;
      if (x4 < G * D / 4) {
        const float r = wk[kChunk * G + (4 * x4) / D];
        acc_o[j].x *= r;
        acc_o[j].y *= r;
        acc_o[j].z *= r;
        acc_o[j].w *= r;
      }
    }
    const float4 *pb = reinterpret_cast<const float4 *>(po + (size_t)base * G * D);
    for (int k = 0; k < cnt; k += kU) {
      float4 v[kU][OPT4];
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int j = 0; j < OPT4; ++j) {
          const int x4 = tid + 128 * j;
          v[u][j] = (k + u < cnt && x4 < G * D / 4)
                        ? __ldcg(pb + (size_t)(k + u) * (G * D / 4) + x4)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int j = 0; j < OPT4; ++j) {
          const int x4 = tid + 128 * j;
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
    const int x4 = tid + 128 * j;
    if (x4 < G * D / 4) {
      const float inv = 1.f / Lh[(4 * x4) / D];
      reinterpret_cast<float4 *>(out)[x4] =
          make_float4(acc_o[j].x * inv, acc_o[j].y * inv, acc_o[j].z * inv, acc_o[j].w * inv);
    }
  }
  if (tid == 0) p.tickets[unit] = 0;
}

template <typename T, int D, int G>
cudaError_t prep_one() {
  return cudaFuncSetAttribute(decode_tiles_kernel<T, D, G>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<D, G>::kAlloc);
}

template <typename T, int D>
cudaError_t prep_g() {
  cudaError_t e;
  if ((e = prep_one<T, D, 1>()) != cudaSuccess) return e;
  if ((e = prep_one<T, D, 2>()) != cudaSuccess) return e;
  if ((e = prep_one<T, D, 4>()) != cudaSuccess) return e;
  return prep_one<T, D, 8>();
}

template <typename T, int D, int G>
cudaError_t launch_one(const TileDecodeParams &p, cudaStream_t st) {
  int tiles = 1;
  for (int i = 0; i < p.n_seqs; ++i)
    tiles = max(tiles, max(p.seqs[i].ns_dyn ? p.seqs[i].tpi_dyn : 0,
                           p.seqs[i].ns_str ? p.seqs[i].tpi_str : 0));
  cudaError_t e = launch_pdl(decode_tiles_kernel<T, D, G>, p.total_items, 128,
                             (size_t)Smem<D, G>::bytes(min(tiles, kMaxTiles)), st, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_g(const TileDecodeParams &p, int G, cudaStream_t st) {
  switch (G) {
    case 1: return launch_one<T, D, 1>(p, st);
    case 2: return launch_one<T, D, 2>(p, st);
    case 4: return launch_one<T, D, 4>(p, st);
    case 8: return launch_one<T, D, 8>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t prepare_decode_kernels() {
  cudaError_t e;
  if ((e = prep_g<__half, 64>()) != cudaSuccess) return e;
  if ((e = prep_g<__half, 128>()) != cudaSuccess) return e;
  if ((e = prep_g<__nv_bfloat16, 64>()) != cudaSuccess) return e;
  return prep_g<__nv_bfloat16, 128>();
}

cudaError_t launch_decode_tiles(const TileDecodeParams &p, int dtype, int d, int G,
                                cudaStream_t s, long long *n) {
  if (p.n_seqs == 0 || p.total_items == 0) return cudaSuccess;
  *n += 1;
  if (dtype == 0) return d == 64 ? launch_g<__half, 64>(p, G, s) : launch_g<__half, 128>(p, G, s);
  return d == 64 ? launch_g<__nv_bfloat16, 64>(p, G, s) : launch_g<__nv_bfloat16, 128>(p, G, s);
}

}  // namespace spd
