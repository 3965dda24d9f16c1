// Host runtime of the sparse paged decode attention library: configuration
// checks, the fixed physical page pool with its free list, per-sequence
// tables (length, page list, step counter, selection bookkeeping), the
// split-K work partitioning and the C ABI declared in include/spd.h.
//
// Hierarchical paging follows "LServe long-sequence LLM serving system",
// section 2.2: a physical page of P tokens is the allocation unit and holds
// R = P / l consecutive logical pages of one sequence (the selection unit).
// The pool is fixed; an allocation that does not fit reports exhaustion and
// changes nothing (the free-list pager of "Long-context inference
// optimization for LLMs", section 3.4, raises on an empty list).
#include <algorithm>
#include <cfloat>
#include <cmath>
#include <mutex>
#include <unordered_map>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "spd.h"
#include "spd_internal.h"

using namespace spd;

namespace {

struct Seq {
  bool live = false;
  long long L = 0;
  long long counter = 0;   // decode steps taken (attention calls)
  bool has_sel = false;
  int nL0 = 0;             // logical pages when the selection was taken
  int sel_count = 0;       // pages kept at that selection
  int topk_pending = 0;    // candidates the next fused decode launch selects from (0: none)
  int topk_row = 0;        // their row in the score scratch
  int topk_bounds = 0;     // per-chunk score bounds written for them (0: none)
  std::vector<int> pages;  // physical page per P-token block
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

uint64_t splitmix64(uint64_t &s) {
  uint64_t z = (s += 0x9e3779b97f4a7c15ull);
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

struct Derived {
  int G = 0, Hd = 0, Hs = 0, R = 0, max_pp = 0, ksel_max = 0, max_nL = 0,
      seqs_per_launch = 0;
  int mass_pages = 0, mass_tiles = 0;  // per-page mass: attended pages / tiles per unit
  int kv_fp8 = 0;                       // K/V stored as E4M3 codes of value / scale
  float k_scale[kMaxKvHeads] = {}, v_scale[kMaxKvHeads] = {};
  unsigned char kv_kind[kMaxKvHeads] = {}, kv_sub[kMaxKvHeads] = {},
                dyn_kv[kMaxKvHeads] = {}, str_kv[kMaxKvHeads] = {};
  ScratchLayout sl{};
  spd_sizes sizes{};
};

// Validates cfg and fills the derived quantities; returns an error string or
// nullptr.
// Per-chunk score bounds a selection writes for each (sequence, head): one per
// scoring CTA, rows padded to 16 bytes.
int bound_stride_of(const Derived &d) {
  const int ppc = select_pages_per_cta();
  return (int)round_up((size_t)((d.max_nL + ppc - 1) / ppc), 4);
}

const char *derive(const spd_config *c, Derived *d) {
  if (!c) return "config is NULL";
  if (c->num_kv_heads < 1 || c->num_kv_heads > kMaxKvHeads)
    return "num_kv_heads must be in [1, 128]";
  if (c->num_q_heads < 1 || c->num_q_heads % c->num_kv_heads)
    return "num_q_heads must be a positive multiple of num_kv_heads";
  d->G = c->num_q_heads / c->num_kv_heads;
  if (d->G != 1 && d->G != 2 && d->G != 4 && d->G != 8)
    return "num_q_heads / num_kv_heads must be 1, 2, 4 or 8";
  if (c->head_dim != 64 && c->head_dim != 128) return "head_dim must be 64 or 128";
  if (c->dtype != SPD_F16 && c->dtype != SPD_BF16) return "dtype must be SPD_F16 or SPD_BF16";
  if (c->logical_page != 16 && c->logical_page != 32 && c->logical_page != 64)
    return "logical_page must be 16, 32 or 64";
  if (c->physical_page < c->logical_page || c->physical_page % c->logical_page ||
      c->physical_page > 4096)
    return "physical_page must be a multiple of logical_page, at most 4096";
  if (c->max_seqs < 1) return "max_seqs must be >= 1";
  if (c->max_context < 1 || c->max_context > (1 << 28)) return "max_context must be in [1, 2^28]";
  if (c->reuse_interval < 1) return "reuse_interval must be >= 1";
  if (c->kv_fp8 != 0 && c->kv_fp8 != 1) return "kv_fp8 must be 0 or 1";
  d->kv_fp8 = c->kv_fp8;
  if (d->kv_fp8 && c->head_dim != 128) return "fp8 KV storage needs head_dim 128";
  for (int h = 0; h < c->num_kv_heads; ++h) {
    d->k_scale[h] = d->kv_fp8 && c->k_scale ? c->k_scale[h] : 1.f;
    d->v_scale[h] = d->kv_fp8 && c->v_scale ? c->v_scale[h] : 1.f;
    if (!(d->k_scale[h] > 0.f && d->k_scale[h] <= FLT_MAX) ||
        !(d->v_scale[h] > 0.f && d->v_scale[h] <= FLT_MAX))
      return "k_scale and v_scale must be positive and finite";
  }
  d->Hd = d->Hs = 0;
  for (int h = 0; h < c->num_kv_heads; ++h) {
    const bool str = c->kv_head_is_streaming && c->kv_head_is_streaming[h];
    d->kv_kind[h] = str ? 1 : 0;
    if (str) {
      d->kv_sub[h] = (unsigned char)d->Hs;
      d->str_kv[d->Hs++] = (unsigned char)h;
    } else {
      d->kv_sub[h] = (unsigned char)d->Hd;
      d->dyn_kv[d->Hd++] = (unsigned char)h;
    }
  }
  if (d->Hs > 0 && (c->sink < 0 || c->window < 1 || (long long)c->sink + c->window > (1 << 24)))
    return "streaming heads need sink >= 0 and window >= 1";
  if (d->Hd > 0 && c->num_physical_pages < 1) return "num_physical_pages must be >= 1";
  if (c->num_physical_pages < 0) return "num_physical_pages must be >= 0";
  d->R = c->physical_page / c->logical_page;
  d->max_pp = (c->max_context + c->physical_page - 1) / c->physical_page;
  d->max_nL = (c->max_context + c->logical_page - 1) / c->logical_page;
  long long budget = c->token_budget > 0 ? c->token_budget
                                         : std::min<long long>(4096, c->max_context / 32);
  // pages kept never exceed the pages a sequence can have
  d->ksel_max = (int)std::min<long long>(std::max<long long>(1, budget / c->logical_page),
                                         d->max_nL);
  d->seqs_per_launch = std::min(c->max_seqs, kSeqsPerLaunch);
  // one unit (sequence, kv head) must fit in one launch's work items
  const long long unit_cap = (long long)kMaxItems * kMaxTilesPerItem * kTileRows / 2;
  if (d->Hs > 0 && (long long)c->sink + c->window > unit_cap) return "sink + window too large";
  if ((long long)d->ksel_max * c->logical_page > unit_cap) return "token budget too large";
  if (d->Hs > 0 && (long long)c->max_seqs * d->Hs * (c->sink + c->window) >= (1LL << 31))
    return "streaming buffers exceed 2^31 rows";

  const size_t e = d->kv_fp8 ? 1 : 2, dim = (size_t)c->head_dim;
  const int S = d->Hs ? c->sink : 0, W = d->Hs ? c->window : 0;
  spd_sizes &z = d->sizes;
  z.k_pool = z.v_pool = (size_t)c->num_physical_pages * d->Hd * c->physical_page * dim * e;
  z.meta = (size_t)c->num_physical_pages * d->Hd * d->R * 2 * dim * e;
  z.stream_k = z.stream_v = (size_t)c->max_seqs * d->Hs * (size_t)(S + W) * dim * e;
  z.page_table = d->Hd ? (size_t)c->max_seqs * d->max_pp * 4 : 0;
  z.selection = d->Hd ? (size_t)c->max_seqs * d->Hd * d->ksel_max * 4 : 0;
  ScratchLayout &sl = d->sl;
  size_t off = kScratchHeader;
  sl.tickets_dec = off;
  off = round_up(off + (size_t)d->seqs_per_launch * c->num_kv_heads * 4, 256);
  sl.tickets_sel = off;
  off = round_up(off + (size_t)d->seqs_per_launch * d->Hd * 4, 256);
  sl.bounds = off;
  off = round_up(off + (size_t)d->seqs_per_launch * d->Hd * bound_stride_of(*d) * 4, 256);
  sl.part_ml = off;
  off = round_up(off + (size_t)kMaxItems * d->G * 8, 256);
  sl.part_o = off;
  off = round_up(off + (size_t)kMaxItems * d->G * dim * 4, 256);
  sl.scores = off;
  off = round_up(off + (size_t)d->seqs_per_launch * d->Hd * round_up((size_t)d->max_nL, 4) * 4, 256);
  d->mass_pages = std::min(d->ksel_max + kMassExtraPages, d->max_nL);
  d->mass_tiles = d->mass_pages * (c->logical_page / kTileRows);
  sl.page_part = off;
  off = round_up(off + (size_t)d->seqs_per_launch * d->Hd * d->mass_tiles * d->G * 8, 256);
  sl.total = off;
  z.scratch = off;
  return nullptr;
}

}  // namespace

struct spd_ctx {
  spd_config cfg{};
  std::vector<unsigned char> streaming;
  Derived dv;
  spd_buffers buf{};
  std::vector<int> free_pages;  // back() is handed out next
  std::vector<Seq> seqs;
  std::vector<PtUpdate> pending_pt;
  bool device_ready = false;
  int device = 0;
  int num_sms = 152;
  long long launches = 0;  // kernels enqueued by this context
  bool early_staging = false;
  CUtensorMap tm_k{}, tm_v{}, tm_sk{}, tm_sv{};
  std::string err;

  spd_status fail(spd_status s, const char *fmt, ...) {
    char b[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(b, sizeof b, fmt, ap);
    va_end(ap);
    err = b;
    return s;
  }
  int *err_word() { return reinterpret_cast<int *>(buf.scratch); }
  char *scratch(size_t off) { return static_cast<char *>(buf.scratch) + off; }
};

namespace {

// Stream -> the context whose kernel this library enqueued last on it, and
// which kernel.  A kernel may read its own KV cache before the previous kernel
// on the stream has finished only when that kernel cannot have written what
// it reads: a kernel of another context (or other code) writes nothing of
// this cache; this context's selection kernel writes only the selection, and
// its page-table flush only the page table, neither of which a streaming
// head reads.
enum LaunchKind { kKindOther = 0, kKindSelect = 1, kKindPageTable = 2 };
struct LastLaunch {
  const spd_ctx *ctx;
  LaunchKind kind;
};
std::mutex g_last_mu;
std::unordered_map<cudaStream_t, LastLaunch> g_last_launcher;

bool previous_launcher_is(const spd_ctx *c, cudaStream_t st, LaunchKind *kind = nullptr) {
  std::lock_guard<std::mutex> lock(g_last_mu);
  auto it = g_last_launcher.find(st);
  const bool mine = it != g_last_launcher.end() && it->second.ctx == c;
  if (kind) *kind = mine ? it->second.kind : kKindOther;
  return mine;
}

void note_launcher(const spd_ctx *c, cudaStream_t st, LaunchKind kind = kKindOther) {
  std::lock_guard<std::mutex> lock(g_last_mu);
  g_last_launcher[st] = LastLaunch{c, kind};
}

void forget_launcher(const spd_ctx *c) {
  std::lock_guard<std::mutex> lock(g_last_mu);
  for (auto it = g_last_launcher.begin(); it != g_last_launcher.end();)
    it = it->second.ctx == c ? g_last_launcher.erase(it) : std::next(it);
}

spd_status cuda_fail(spd_ctx *c, cudaError_t e, const char *what) {
  return c->fail(SPD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// TMA descriptors over the paged pool and the streaming buffers: tiled maps
// whose box is a 16-row tile of a whole row (128-byte swizzle).
spd_status encode_map(spd_ctx *c, CUtensorMap *m, void *base, uint64_t rows_per_plane,
                      uint64_t planes) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return c->fail(SPD_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const uint64_t d = (uint64_t)c->cfg.head_dim;
  if (c->dv.kv_fp8) {
    // fp8 rows are 128 bytes (head_dim 128): {channels, rows, planes}, one
    // box of 16 rows x 128 bytes per tile of K or of V, swizzled
    cuuint64_t dims[3] = {d, rows_per_plane, planes};
    cuuint64_t strides[2] = {d, rows_per_plane * d};
    cuuint32_t box[3] = {(cuuint32_t)d, (cuuint32_t)kTileRows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return c->fail(SPD_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return SPD_OK;
  }
  // {64 channels, rows, channel halves, planes}: one box is a 16-row tile of
  // every channel, laid out in shared memory half after half (each half 16
  // rows of 128 bytes, swizzled), i.e. one copy per tile of K or of V
  cuuint64_t dims[4] = {64, rows_per_plane, d / 64, planes};
  cuuint64_t strides[3] = {d * 2, 128, rows_per_plane * d * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)kTileRows, (cuuint32_t)(d / 64), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(m,
                      c->cfg.dtype == SPD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return c->fail(SPD_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return SPD_OK;
}

spd_status make_tensor_maps(spd_ctx *c) {
  const Derived &dv = c->dv;
  spd_status r;
  if (dv.Hd > 0) {
    const uint64_t planes = (uint64_t)c->cfg.num_physical_pages * dv.Hd;
    if ((r = encode_map(c, &c->tm_k, c->buf.k_pool, c->cfg.physical_page, planes)) != SPD_OK) return r;
    if ((r = encode_map(c, &c->tm_v, c->buf.v_pool, c->cfg.physical_page, planes)) != SPD_OK) return r;
  }
  if (dv.Hs > 0) {
    const uint64_t rows = (uint64_t)c->cfg.max_seqs * dv.Hs * (c->cfg.sink + c->cfg.window);
    if ((r = encode_map(c, &c->tm_sk, c->buf.stream_k, rows, 1)) != SPD_OK) return r;
    if ((r = encode_map(c, &c->tm_sv, c->buf.stream_v, rows, 1)) != SPD_OK) return r;
  }
  return SPD_OK;
}

// The set-up of ensure_device, with the buffers' device current.
spd_status ensure_device_current(spd_ctx *c, cudaStream_t st) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c->device) == cudaSuccess &&
      sms > 0)
    c->num_sms = sms;
  cudaError_t e;
  if ((e = prepare_decode_kernels()) != cudaSuccess) return cuda_fail(c, e, "kernel attributes");
  spd_status r = make_tensor_maps(c);
  if (r != SPD_OK) return r;
  e = cudaMemsetAsync(c->buf.scratch, 0, c->dv.sl.part_ml, st);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaMemsetAsync(scratch header)");
  return SPD_OK;
}

// First GPU-side call: find the device that owns the buffers, learn its SM
// count, set the kernels' attributes and zero the scratch header (error word)
// and ticket counters.  The caller's current device is left as it was.
spd_status ensure_device(spd_ctx *c, cudaStream_t st) {
  if (c->device_ready) return SPD_OK;
  cudaPointerAttributes a{};
  cudaError_t e = cudaPointerGetAttributes(&a, c->buf.scratch);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaPointerGetAttributes(scratch)");
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
    return c->fail(SPD_ERR_INVALID_ARG, "scratch is not device memory");
  c->device = a.device;
  // kernel attributes are per device: set them with the buffers' device
  // current, then give the caller back the device it had
  int prev = -1;
  const bool had = cudaGetDevice(&prev) == cudaSuccess;
  if (!had || prev != c->device)
    if ((e = cudaSetDevice(c->device)) != cudaSuccess) return cuda_fail(c, e, "cudaSetDevice");
  spd_status r = ensure_device_current(c, st);
  if (had && prev != c->device) {
    const cudaError_t e2 = cudaSetDevice(prev);
    if (r == SPD_OK && e2 != cudaSuccess) return cuda_fail(c, e2, "cudaSetDevice(restore)");
  }
  if (r == SPD_OK) c->device_ready = true;
  return r;
}

spd_status check_seqs(spd_ctx *c, const int *ids, int n) {
  if (!ids || n < 1) return c->fail(SPD_ERR_INVALID_ARG, "seq_ids must list at least one sequence");
  for (int i = 0; i < n; ++i) {
    const int s = ids[i];
    if (s < 0 || s >= (int)c->seqs.size() || !c->seqs[s].live)
      return c->fail(SPD_ERR_BAD_SEQ, "sequence %d is not live", s);
    for (int j = 0; j < i; ++j)
      if (ids[j] == s) return c->fail(SPD_ERR_BAD_SEQ, "sequence %d listed twice", s);
  }
  return SPD_OK;
}

long long pages_needed(const spd_ctx *c, const Seq &s, long long n_tokens) {
  if (c->dv.Hd == 0) return 0;
  const long long P = c->cfg.physical_page;
  const long long need = (s.L + n_tokens + P - 1) / P;
  return std::max<long long>(0, need - (long long)s.pages.size());
}

void take_pages(spd_ctx *c, int slot, long long n_tokens) {
  Seq &s = c->seqs[slot];
  long long k = pages_needed(c, s, n_tokens);
  for (; k > 0; --k) {
    const int phys = c->free_pages.back();
    c->free_pages.pop_back();
    c->pending_pt.push_back(PtUpdate{slot, (int)s.pages.size(), phys});
    s.pages.push_back(phys);
  }
}

spd_status flush_page_table(spd_ctx *c, cudaStream_t st) {
  size_t i = 0;
  while (i < c->pending_pt.size()) {
    PtWriteParams p{};
    p.page_table = static_cast<int *>(c->buf.page_table);
    p.max_pp = c->dv.max_pp;
    p.n = (int)std::min<size_t>(kPtUpdPerLaunch, c->pending_pt.size() - i);
    for (int k = 0; k < p.n; ++k) p.upd[k] = c->pending_pt[i + k];
    cudaError_t e = launch_pt_write(p, st, &c->launches);
    if (e != cudaSuccess) return cuda_fail(c, e, "pt_write launch");
    note_launcher(c, st, kKindPageTable);
    i += p.n;
  }
  c->pending_pt.clear();
  return SPD_OK;
}

int nL_of(long long L, int ell) { return (int)((L + ell - 1) / ell); }

int budget_pages(const spd_ctx *c, long long L) {
  long long budget = c->cfg.token_budget > 0 ? c->cfg.token_budget
                                             : std::min<long long>(4096, L / 32);
  return (int)std::max<long long>(1, budget / c->cfg.logical_page);
}

spd_status append_impl(spd_ctx *c, const int *ids, int n, int n_tokens, const void *k,
                       const void *v, cudaStream_t st) {
  spd_status r = ensure_device(c, st);
  if (r != SPD_OK) return r;
  for (int i = 0; i < n; ++i) take_pages(c, ids[i], n_tokens);
  if ((r = flush_page_table(c, st)) != SPD_OK) return r;
  const Derived &dv = c->dv;
  const size_t row = (size_t)c->cfg.num_kv_heads * c->cfg.head_dim * 2;  // bytes per token
  for (int b = 0; b < n; b += dv.seqs_per_launch) {
    AppendParams p{};
    p.n_seqs = std::min(dv.seqs_per_launch, n - b);
    p.k = static_cast<const char *>(k) + (size_t)b * n_tokens * row;
    p.v = static_cast<const char *>(v) + (size_t)b * n_tokens * row;
    p.k_pool = c->buf.k_pool;
    p.v_pool = c->buf.v_pool;
    p.meta = c->buf.meta;
    p.stream_k = c->buf.stream_k;
    p.stream_v = c->buf.stream_v;
    p.page_table = static_cast<const int *>(c->buf.page_table);
    p.err = c->err_word();
    p.n_tokens = n_tokens;
    p.Hkv = c->cfg.num_kv_heads;
    p.Hd = dv.Hd;
    p.Hs = dv.Hs;
    p.ell = c->cfg.logical_page;
    p.P = c->cfg.physical_page;
    p.R = dv.R;
    p.max_pp = dv.max_pp;
    p.S = dv.Hs ? c->cfg.sink : 0;
    p.W = dv.Hs ? c->cfg.window : 0;
    p.num_phys = c->cfg.num_physical_pages;
    p.kv_fp8 = dv.kv_fp8;
    memcpy(p.k_scale, dv.k_scale, sizeof p.k_scale);
    memcpy(p.v_scale, dv.v_scale, sizeof p.v_scale);
    memcpy(p.dyn_kv, dv.dyn_kv, sizeof p.dyn_kv);
    memcpy(p.str_kv, dv.str_kv, sizeof p.str_kv);
    long long ctas = 0;
    for (int i = 0; i < p.n_seqs; ++i) {
      const Seq &s = c->seqs[ids[b + i]];
      p.seqs[i].slot = ids[b + i];
      p.seqs[i].L_old = (int)s.L;
      p.seqs[i].cta_off = (int)ctas;
      const long long j0 = s.L / p.ell, j1 = (s.L + n_tokens + p.ell - 1) / p.ell;
      ctas += (j1 - j0) * dv.Hd;
    }
    if (ctas > 0x7fffffffLL - p.n_seqs * dv.Hs)
      return c->fail(SPD_ERR_CAPACITY, "append too large for one launch");
    p.dyn_ctas = (int)ctas;
    cudaError_t e = launch_append(p, c->cfg.dtype, c->cfg.head_dim, st, &c->launches);
    if (e != cudaSuccess) return cuda_fail(c, e, "append launch");
    note_launcher(c, st);
  }
  for (int i = 0; i < n; ++i) c->seqs[ids[i]].L += n_tokens;
  return SPD_OK;
}

// score_only: the decode kernel launched next (attention_impl with
// fused_topk) selects the pages from the scores this launch writes; used when
// every due sequence fits one selection launch and the kernel's shared-memory
// limits (candidates, kept pages), otherwise the selection kernel selects.
spd_status select_impl(spd_ctx *c, const void *q, const int *ids, int n, bool force,
                       cudaStream_t st, bool score_only = false) {
  const Derived &dv = c->dv;
  std::vector<int> due;  // positions in the call
  for (int i = 0; i < n; ++i) {
    Seq &s = c->seqs[ids[i]];
    s.topk_pending = 0;
    if (force || s.counter % c->cfg.reuse_interval == 0) due.push_back(i);
  }
  if (due.empty()) return SPD_OK;
  if (score_only) {
    score_only = (int)due.size() <= dv.seqs_per_launch;
    for (int pos : due) {
      const Seq &s = c->seqs[ids[pos]];
      const int nL = nL_of(s.L, c->cfg.logical_page);
      if (nL - 1 > kFusedMaxCandidates || budget_pages(c, s.L) > kFusedMaxSelected)
        score_only = false;
    }
  }
  if (dv.Hd > 0) {
    spd_status r = ensure_device(c, st);
    if (r != SPD_OK) return r;
    const int ppc = select_pages_per_cta();
    for (size_t b = 0; b < due.size(); b += dv.seqs_per_launch) {
      SelectParams p{};
      p.n_seqs = (int)std::min<size_t>(dv.seqs_per_launch, due.size() - b);
      p.q = q;
      p.meta = c->buf.meta;
      p.page_table = static_cast<const int *>(c->buf.page_table);
      p.selection = static_cast<int *>(c->buf.selection);
      p.scores = reinterpret_cast<float *>(c->scratch(dv.sl.scores));
      p.tickets = reinterpret_cast<int *>(c->scratch(dv.sl.tickets_sel));
      p.bounds = reinterpret_cast<uint32_t *>(c->scratch(dv.sl.bounds));
      p.bound_stride = bound_stride_of(dv);
      p.err = c->err_word();
      p.Hq = c->cfg.num_q_heads;
      p.Hd = dv.Hd;
      p.ell = c->cfg.logical_page;
      p.R = dv.R;
      p.max_pp = dv.max_pp;
      p.ksel_max = dv.ksel_max;
      p.score_stride = (int)round_up((size_t)dv.max_nL, 4);  // 16-byte aligned rows
      p.pages_per_chunk = ppc;
      p.kv_fp8 = dv.kv_fp8;
      p.num_phys = c->cfg.num_physical_pages;
      memcpy(p.dyn_kv, dv.dyn_kv, sizeof p.dyn_kv);
      int off = 0;
      for (int i = 0; i < p.n_seqs; ++i) {
        const int pos = due[b + i];
        const Seq &s = c->seqs[ids[pos]];
        SelectSeq &d = p.seqs[i];
        d.slot = ids[pos];
        d.qrow = pos;
        d.nL = nL_of(s.L, p.ell);
        d.K_sel = budget_pages(c, s.L);
        d.chunk_off = off;
        d.n_chunks = (d.nL > d.K_sel && d.K_sel > 1) ? (d.nL - 1 + ppc - 1) / ppc : 0;
        // bound from each full chunk's tau_m-th key, when a few per chunk suffice
        const int n_full = (d.nL - 1) / ppc;
        const int tau_m = n_full > 0 ? (d.K_sel - 1 + n_full - 1) / n_full : 0;
        d.tau_m = d.n_chunks > 0 && tau_m <= kMaxBoundRank ? tau_m : 0;
        off += std::max(1, d.n_chunks) * dv.Hd;
      }
      p.score_ctas = off;
      p.score_only = score_only ? 1 : 0;
      if (score_only)
        for (int i = 0; i < p.n_seqs; ++i) {
          Seq &s = c->seqs[ids[due[b + i]]];
          s.topk_pending = p.seqs[i].n_chunks > 0 ? p.seqs[i].nL - 1 : 0;
          s.topk_row = i;
          s.topk_bounds = p.seqs[i].tau_m > 0 ? p.seqs[i].n_chunks : 0;
        }
      p.early = c->early_staging && !previous_launcher_is(c, st) ? 1 : 0;
      cudaError_t e = launch_select_fused(p, c->cfg.dtype, c->cfg.head_dim, dv.G, st, &c->launches);
      if (e != cudaSuccess) return cuda_fail(c, e, "select launch");
      note_launcher(c, st, kKindSelect);
    }
  }
  for (int pos : due) {
    Seq &s = c->seqs[ids[pos]];
    const int nL = nL_of(s.L, c->cfg.logical_page);
    s.nL0 = nL;
    s.sel_count = std::min(nL, budget_pages(c, s.L));
    s.has_sel = true;
  }
  return SPD_OK;
}

// Tiles of 16 rows a unit (sequence, kv head) attends to.
int unit_tiles_dyn(const spd_ctx *c, const Seq &s) {
  const int ell = c->cfg.logical_page;
  const int n_att = s.sel_count + nL_of(s.L, ell) - s.nL0;
  const int last_rows = (int)((s.L - 1) % ell) + 1;
  return (n_att - 1) * (ell / kTileRows) + (last_rows + kTileRows - 1) / kTileRows;
}

int unit_tiles_str(const spd_ctx *c, const Seq &s) {
  const long long S = c->cfg.sink, W = c->cfg.window, L = s.L;
  long long n0 = std::min(S, L), n1 = 0, n2 = 0;
  if (L > S) {
    const long long w0 = std::max(S, L - W), n_win = L - w0, a0 = (w0 - S) % W;
    n1 = std::min(n_win, W - a0);
    n2 = n_win - n1;
  }
  auto t = [](long long n) { return (int)((n + kTileRows - 1) / kTileRows); };
  return t(n0) + t(n1) + t(n2);
}

// Split policy.  Every unit (sequence, kv head) gets nc clusters of CS CTAs;
// CS, the same for the whole launch, is the largest power of two (up to the
// size the kernel can be co-scheduled with) that keeps units x CS within one
// CTA per SM.  Tiles are then spread evenly over the unit's CTAs.
//
// Launch shape.  The shared shape (two CTAs per SM: this launch's and the
// next one's, which stages its tiles early) is planned first.  Its nc is 1
// while a unit's tiles fit kPreferTiles per CTA (merging several clusters
// goes through global memory and costs more than the longer tile loop),
// else the unit's share of the launch's tiles over CS CTAs (rounded).  When
// that plan needs more CTAs than SMs (some SMs would run two CTAs of the
// launch) or merges clusters in global memory, and the launch holds more
// than kDeepTilesPerSm tiles per SM, the deep-ring shape (one CTA per SM, 24
// stages) is planned instead when allow_deep: the SMs are shared out in
// proportion to the tiles, one cluster per unit first and then, cluster by
// cluster, to the (sequence, head kind) whose units hold the most tiles per
// CTA, never more CTAs than SMs.  Either way a CTA takes at most
// decode_max_tiles_per_cta() tiles.
constexpr int kPreferTiles = 24;
constexpr int kDeepTilesPerSm = 16;

int plan_tiles(const spd_ctx *c, TileDecodeParams &p, const int *ids, int n, bool allow_deep) {
  const Derived &dv = c->dv;
  long long total = 0;
  for (int i = 0; i < n; ++i) {
    const Seq &s = c->seqs[ids[i]];
    if (dv.Hd) total += (long long)dv.Hd * unit_tiles_dyn(c, s);
    if (dv.Hs) total += (long long)dv.Hs * unit_tiles_str(c, s);
  }
  const long long units = (long long)n * (dv.Hd + dv.Hs);
  const int max_tiles = decode_max_tiles_per_cta();
  auto fill = [&](int i, int ns_dyn, int ns_str, int *items) {
    const Seq &s = c->seqs[ids[i]];
    TileSeq &d = p.seqs[i];
    d.slot = ids[i];
    d.L = (int)s.L;
    d.nL0 = s.nL0;
    d.sel_count = s.sel_count;
    d.item_off = *items;
    d.ns_dyn = dv.Hd ? ns_dyn : 0;
    d.ns_str = dv.Hs ? ns_str : 0;
    d.tpi_dyn = dv.Hd ? std::max(1, (unit_tiles_dyn(c, s) + ns_dyn - 1) / ns_dyn) : 1;
    d.tpi_str = dv.Hs ? std::max(1, (unit_tiles_str(c, s) + ns_str - 1) / ns_str) : 1;
    *items += dv.Hd * d.ns_dyn + dv.Hs * d.ns_str;
  };

  int cs = 1;
  const int cs_max = decode_max_cluster(c->cfg.dtype, c->cfg.head_dim, dv.G);
  while (cs * 2 <= cs_max && units * cs * 2 <= c->num_sms) cs *= 2;
  const long long tpc = std::max<long long>(1, (total + c->num_sms - 1) / c->num_sms);
  bool merges = false;  // some unit has several clusters
  auto split = [&](int nt) {
    long long nc = nt <= (long long)cs * kPreferTiles
                       ? 1
                       : std::max<long long>(1, (nt + cs * tpc / 2) / (cs * tpc));  // rounded
    nc = std::max<long long>(nc, (nt + (long long)cs * max_tiles - 1) / ((long long)cs * max_tiles));
    merges = merges || nc > 1;
    return (int)(nc * cs);
  };
  int items = 0;
  for (int i = 0; i < n; ++i) {
    const Seq &s = c->seqs[ids[i]];
    fill(i, dv.Hd ? split(unit_tiles_dyn(c, s)) : 0, dv.Hs ? split(unit_tiles_str(c, s)) : 0,
         &items);
  }
  p.cluster = cs;
  p.total_items = items;
  p.deep = 0;
  if (!allow_deep || (items <= c->num_sms && !merges) ||
      total <= (long long)c->num_sms * kDeepTilesPerSm)
    return items;
  {
    int cs = 1;
    const int cs_max = decode_max_cluster(c->cfg.dtype, c->cfg.head_dim, dv.G, true);
    while (cs * 2 <= cs_max && units * cs * 2 <= c->num_sms) cs *= 2;
    if (units * cs <= c->num_sms) {
      // groups: (sequence, head kind); a step gives each unit of a group one
      // more cluster
      struct Grp {
        int seq, kind, units, ns;
        long long nt;
      };
      std::vector<Grp> gs;
      for (int i = 0; i < n; ++i) {
        const Seq &s = c->seqs[ids[i]];
        if (dv.Hd) gs.push_back(Grp{i, 0, dv.Hd, cs, unit_tiles_dyn(c, s)});
        if (dv.Hs) gs.push_back(Grp{i, 1, dv.Hs, cs, unit_tiles_str(c, s)});
      }
      long long free_ctas = c->num_sms - units * cs;
      auto load = [](const Grp &g) { return (double)g.nt / g.ns; };
      auto cmp = [&](int a, int b) { return load(gs[a]) < load(gs[b]); };
      std::vector<int> heap(gs.size());
      for (size_t k = 0; k < gs.size(); ++k) heap[k] = (int)k;
      std::make_heap(heap.begin(), heap.end(), cmp);
      while (!heap.empty()) {
        std::pop_heap(heap.begin(), heap.end(), cmp);
        Grp &g = gs[heap.back()];
        const long long cost = (long long)g.units * cs;
        if (cost > free_ctas || g.ns + cs > g.nt) {
          heap.pop_back();  // no room for this group's next cluster
          continue;
        }
        g.ns += cs;
        free_ctas -= cost;
        std::push_heap(heap.begin(), heap.end(), cmp);
      }
      bool ok = true;
      for (const Grp &g : gs) ok = ok && (g.nt + g.ns - 1) / g.ns <= max_tiles;
      if (ok) {
        int items = 0;
        std::vector<int> nsd(n, cs), nss(n, cs);
        for (const Grp &g : gs) (g.kind ? nss : nsd)[g.seq] = g.ns;
        for (int i = 0; i < n; ++i) fill(i, nsd[i], nss[i], &items);
        p.cluster = cs;
        p.total_items = items;
        p.deep = 1;
        return items;
      }
    }
  }

  // (the deep plan did not fit: the shared one again)
  return plan_tiles(c, p, ids, n, false);
}

// The deep-ring shape serves the plain 16-bit kernel (no per-page mass
// export, no fp8 storage).
bool deep_allowed(const spd_ctx *c, bool mass) { return !c->dv.kv_fp8 && !mass; }

// The sequences [b, b + m) of a call that one decode launch takes: as many as
// fit one parameter block and max_items, halving until they do (down to one
// sequence).  Leaves p planned for them and returns m.
int next_batch(const spd_ctx *c, TileDecodeParams &p, const int *ids, int b, int n,
               int max_items, bool allow_deep) {
  int m = std::min(c->dv.seqs_per_launch, n - b);
  while (plan_tiles(c, p, ids + b, m, allow_deep) > max_items && m > 1) m = (m + 1) / 2;
  return m;
}

// Plans every launch of an attention call without enqueuing anything; fails
// with SPD_ERR_CAPACITY if a launch would need more than max_items items
// (a single sequence whose split items alone exceed it).
spd_status check_capacity(spd_ctx *c, const int *ids, int n, int max_items, bool allow_deep) {
  static thread_local TileDecodeParams p;
  for (int b = 0; b < n;) {
    const int m = next_batch(c, p, ids, b, n, max_items, allow_deep);
    if (p.total_items > max_items)
      return c->fail(SPD_ERR_CAPACITY, "sequence %d needs %d split items, the library-owned "
                     "scratch holds %d", ids[b], p.total_items, max_items);
    b += m;
  }
  return SPD_OK;
}

// `scr` (optional) replaces the context's scratch for the split partials and
// tickets; a launch then holds at most scr->max_items items.
// fused_topk: the selection launched just before wrote only scores for the
// sequences marked topk_pending; this launch selects their pages.
// Optional exports of an attention call: the softmax row max / row sum and the
// per-page attention mass of the dynamic heads.
struct StatsOut {
  float *row_max = nullptr, *row_sum = nullptr;
  int *pages = nullptr;
  float *page_mass = nullptr;
  int max_pages = 0;
};

spd_status attention_impl(spd_ctx *c, const void *q, const int *ids, int n, float *out,
                          const void *k_new, const void *v_new, cudaStream_t st,
                          const DecodeScratch *scr = nullptr, bool fused_topk = false,
                          const StatsOut &so = StatsOut()) {
  spd_status r = ensure_device(c, st);
  if (r != SPD_OK) return r;
  const Derived &dv = c->dv;
  const size_t qrow = (size_t)c->cfg.num_q_heads * c->cfg.head_dim;
  const size_t kvrow = (size_t)c->cfg.num_kv_heads * c->cfg.head_dim;
  const int max_items = scr ? scr->max_items : kMaxItems;
  const bool allow_deep = deep_allowed(c, so.page_mass != nullptr && dv.Hd > 0);
  // a bounded scratch: every launch is planned before the first is enqueued
  if (scr && (r = check_capacity(c, ids, n, max_items, allow_deep)) != SPD_OK) return r;
  int b = 0;
  while (b < n) {
    static thread_local TileDecodeParams p;
    const int m = next_batch(c, p, ids, b, n, max_items, allow_deep);
    p.n_seqs = m;
    p.tm_k = c->tm_k;
    p.tm_v = c->tm_v;
    p.tm_sk = c->tm_sk;
    p.tm_sv = c->tm_sv;
    p.q = static_cast<const char *>(q) + (size_t)b * qrow * 2;
    p.k_new = k_new ? static_cast<const char *>(k_new) + (size_t)b * kvrow * 2 : nullptr;
    p.v_new = v_new ? static_cast<const char *>(v_new) + (size_t)b * kvrow * 2 : nullptr;
    p.out = out + (size_t)b * qrow;
    p.row_max = so.row_max ? so.row_max + (size_t)b * c->cfg.num_q_heads : nullptr;
    p.row_sum = so.row_sum ? so.row_sum + (size_t)b * c->cfg.num_q_heads : nullptr;
    const bool mass = so.page_mass != nullptr && dv.Hd > 0;
    p.page_part = mass ? reinterpret_cast<float2 *>(c->scratch(dv.sl.page_part)) : nullptr;
    p.page_tile_cap = dv.mass_tiles;
    p.pages = mass ? so.pages + (size_t)b * dv.Hd * so.max_pages : nullptr;
    p.page_mass = mass ? so.page_mass + (size_t)b * dv.Hd * dv.G * so.max_pages : nullptr;
    p.max_pages = so.max_pages;
    p.k_pool = c->buf.k_pool;
    p.v_pool = c->buf.v_pool;
    p.meta = c->buf.meta;
    p.stream_k = c->buf.stream_k;
    p.stream_v = c->buf.stream_v;
    p.page_table = static_cast<const int *>(c->buf.page_table);
    p.selection = static_cast<const int *>(c->buf.selection);
    p.part_o = scr ? scr->part_o : reinterpret_cast<float *>(c->scratch(dv.sl.part_o));
    p.part_ml = scr ? scr->part_ml : reinterpret_cast<float2 *>(c->scratch(dv.sl.part_ml));
    p.tickets = scr ? scr->tickets : reinterpret_cast<int *>(c->scratch(dv.sl.tickets_dec));
    p.err = c->err_word();
    p.scores = reinterpret_cast<const float *>(c->scratch(dv.sl.scores));
    p.score_stride = (int)round_up((size_t)dv.max_nL, 4);
    p.bounds = reinterpret_cast<const uint32_t *>(c->scratch(dv.sl.bounds));
    p.bound_stride = bound_stride_of(dv);
    for (int i = 0; i < m; ++i) {
      const Seq &s = c->seqs[ids[b + i]];
      p.seqs[i].topk_n = fused_topk ? s.topk_pending : 0;
      p.seqs[i].topk_row = s.topk_row;
      p.seqs[i].topk_bounds = fused_topk ? s.topk_bounds : 0;
    }
    p.Hq = c->cfg.num_q_heads;
    p.Hkv = c->cfg.num_kv_heads;
    p.Hd = dv.Hd;
    p.Hs = dv.Hs;
    p.ell = c->cfg.logical_page;
    p.P = c->cfg.physical_page;
    p.R = dv.R;
    p.max_pp = dv.max_pp;
    p.ksel_max = dv.ksel_max;
    p.S = dv.Hs ? c->cfg.sink : 0;
    p.W = dv.Hs ? c->cfg.window : 0;
    p.num_phys = c->cfg.num_physical_pages;
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->cfg.head_dim));
    p.kv_fp8 = dv.kv_fp8;
    memcpy(p.k_scale, dv.k_scale, sizeof p.k_scale);
    memcpy(p.v_scale, dv.v_scale, sizeof p.v_scale);
    memcpy(p.dyn_kv, dv.dyn_kv, sizeof p.dyn_kv);
    memcpy(p.str_kv, dv.str_kv, sizeof p.str_kv);
    // bit 0: dynamic units may stage before the wait, bit 1: streaming units;
    // bit 2: streaming units need not wait at all (the previous kernel is this
    // context's selection or page-table flush, which q and the streaming
    // buffers do not depend on)
    LaunchKind prev = kKindOther;
    if (!c->early_staging) p.early = 0;
    else if (!previous_launcher_is(c, st, &prev)) p.early = 3;
    else p.early = (prev == kKindSelect || prev == kKindPageTable) ? 2 | 4 : 0;
    cudaError_t e = launch_decode_tiles(p, c->cfg.dtype, c->cfg.head_dim, dv.G, st, &c->launches);
    if (e != cudaSuccess) return cuda_fail(c, e, "decode launch");
    note_launcher(c, st);
    b += m;
  }
  for (int i = 0; i < n; ++i) {
    c->seqs[ids[i]].counter += 1;
    c->seqs[ids[i]].topk_pending = 0;
  }
  return SPD_OK;
}

// will_append: the call appends one token first (so the length will be >= 1)
// and selects the sequences that are due before attending.
spd_status check_attend_state(spd_ctx *c, const int *ids, int n, bool will_append) {
  const bool will_select = will_append;
  for (int i = 0; i < n; ++i) {
    const Seq &s = c->seqs[ids[i]];
    if (s.L < 1 && !will_append)
      return c->fail(SPD_ERR_STATE, "sequence %d has no tokens", ids[i]);
    const bool due = s.counter % c->cfg.reuse_interval == 0;
    if (c->dv.Hd > 0 && !s.has_sel && !(will_select && due))
      return c->fail(SPD_ERR_STATE, "sequence %d has no page selection yet", ids[i]);
  }
  return SPD_OK;
}

}  // namespace

namespace spd {

spd_status check_attention_call(spd_ctx *c, const void *q, const int *ids, int n,
                                const float *out) {
  if (!q || !out || !aligned16(q) || !aligned16(out))
    return c->fail(SPD_ERR_INVALID_ARG, "q and out must be 16-byte aligned pointers");
  spd_status r = check_seqs(c, ids, n);
  if (r != SPD_OK) return r;
  return check_attend_state(c, ids, n, false);
}

spd_status check_attention_capacity(spd_ctx *c, const int *ids, int n, int max_items) {
  return check_capacity(c, ids, n, max_items, deep_allowed(c, false));
}

spd_status bind_device(spd_ctx *c, cudaStream_t st, int *device) {
  spd_status r = ensure_device(c, st);
  if (r == SPD_OK) *device = c->device;
  return r;
}

spd_status attention_with_scratch(spd_ctx *c, const void *q, const int *ids, int n, float *out,
                                  cudaStream_t st, const DecodeScratch &scratch) {
  return attention_impl(c, q, ids, n, out, nullptr, nullptr, st, &scratch);
}

spd_status fail_message(spd_ctx *c, spd_status s, const char *msg) {
  return c->fail(s, "%s", msg);
}

}  // namespace spd

extern "C" {

spd_status spd_query_sizes(const spd_config *cfg, spd_sizes *out) {
  if (!out) return SPD_ERR_INVALID_ARG;
  Derived d;
  if (derive(cfg, &d)) return SPD_ERR_INVALID_ARG;
  *out = d.sizes;
  return SPD_OK;
}

spd_status spd_create(const spd_config *cfg, const spd_buffers *bufs, spd_ctx **out) {
  if (!out || !bufs) return SPD_ERR_INVALID_ARG;
  *out = nullptr;
  Derived d;
  if (derive(cfg, &d)) return SPD_ERR_INVALID_ARG;
  const void *ptrs[8] = {bufs->k_pool, bufs->v_pool, bufs->meta, bufs->stream_k,
                         bufs->stream_v, bufs->page_table, bufs->selection, bufs->scratch};
  const size_t sizes[8] = {d.sizes.k_pool, d.sizes.v_pool, d.sizes.meta, d.sizes.stream_k,
                           d.sizes.stream_v, d.sizes.page_table, d.sizes.selection,
                           d.sizes.scratch};
  for (int i = 0; i < 8; ++i) {
    if (sizes[i] && !ptrs[i]) return SPD_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ptrs[i]) % 256) return SPD_ERR_INVALID_ARG;
  }
  spd_ctx *c = new (std::nothrow) spd_ctx();
  if (!c) return SPD_ERR_INVALID_ARG;
  c->cfg = *cfg;
  c->dv = d;
  if (cfg->kv_head_is_streaming)
    c->streaming.assign(cfg->kv_head_is_streaming, cfg->kv_head_is_streaming + cfg->num_kv_heads);
  c->cfg.kv_head_is_streaming = c->streaming.empty() ? nullptr : c->streaming.data();
  c->cfg.k_scale = c->cfg.v_scale = nullptr;  // copied into c->dv
  c->buf = *bufs;
  const int N = d.Hd ? cfg->num_physical_pages : 0;
  c->free_pages.resize(N);
  for (int i = 0; i < N; ++i) c->free_pages[i] = N - 1 - i;  // page 0 first
  if (cfg->free_list_seed) {
    uint64_t st = cfg->free_list_seed;
    for (int i = N - 1; i > 0; --i) {
      const int j = (int)(splitmix64(st) % (uint64_t)(i + 1));
      std::swap(c->free_pages[i], c->free_pages[j]);
    }
  }
  c->seqs.resize(cfg->max_seqs);
  *out = c;
  return SPD_OK;
}

void spd_destroy(spd_ctx *ctx) {
  if (ctx) forget_launcher(ctx);
  delete ctx;
}

spd_status spd_seq_create(spd_ctx *c, int *seq_id_out) {
  if (!c || !seq_id_out) return SPD_ERR_INVALID_ARG;
  for (int i = 0; i < (int)c->seqs.size(); ++i)
    if (!c->seqs[i].live) {
      c->seqs[i] = Seq();
      c->seqs[i].live = true;
      *seq_id_out = i;
      return SPD_OK;
    }
  return c->fail(SPD_ERR_CAPACITY, "all %d sequence slots are live", (int)c->seqs.size());
}

spd_status spd_seq_free(spd_ctx *c, int seq_id) {
  if (!c) return SPD_ERR_INVALID_ARG;
  if (seq_id < 0 || seq_id >= (int)c->seqs.size() || !c->seqs[seq_id].live)
    return c->fail(SPD_ERR_BAD_SEQ, "sequence %d is not live", seq_id);
  Seq &s = c->seqs[seq_id];
  for (auto it = s.pages.rbegin(); it != s.pages.rend(); ++it) c->free_pages.push_back(*it);
  // drop queued page-table writes of this sequence (its pages are free again)
  c->pending_pt.erase(std::remove_if(c->pending_pt.begin(), c->pending_pt.end(),
                                     [&](const PtUpdate &u) { return u.slot == seq_id; }),
                      c->pending_pt.end());
  s = Seq();
  return SPD_OK;
}

spd_status spd_seq_reserve(spd_ctx *c, int seq_id, int n_tokens) {
  if (!c || n_tokens < 0) return SPD_ERR_INVALID_ARG;
  spd_status r = check_seqs(c, &seq_id, 1);
  if (r != SPD_OK) return r;
  const Seq &s = c->seqs[seq_id];
  if (s.L + n_tokens > c->cfg.max_context)
    return c->fail(SPD_ERR_CAPACITY, "sequence %d: %lld + %d tokens exceed max_context %d", seq_id,
                   s.L, n_tokens, c->cfg.max_context);
  const long long need = pages_needed(c, s, n_tokens);
  if (need > (long long)c->free_pages.size())
    return c->fail(SPD_ERR_NO_PAGES, "need %lld physical pages, %zu free", need,
                   c->free_pages.size());
  take_pages(c, seq_id, n_tokens);
  return SPD_OK;
}

spd_status spd_seq_info(spd_ctx *c, int seq_id, long long *length, long long *step_counter,
                        int *pages_at_selection, int *pages_kept) {
  if (!c) return SPD_ERR_INVALID_ARG;
  spd_status r = check_seqs(c, &seq_id, 1);
  if (r != SPD_OK) return r;
  const Seq &s = c->seqs[seq_id];
  if (length) *length = s.L;
  if (step_counter) *step_counter = s.counter;
  if (pages_at_selection) *pages_at_selection = s.has_sel ? s.nL0 : 0;
  if (pages_kept) *pages_kept = s.has_sel ? s.sel_count : 0;
  return SPD_OK;
}

spd_status spd_get_page_table(spd_ctx *c, int seq_id, int *phys_host, int cap, int *n_host) {
  if (!c || !n_host) return SPD_ERR_INVALID_ARG;
  spd_status r = check_seqs(c, &seq_id, 1);
  if (r != SPD_OK) return r;
  const Seq &s = c->seqs[seq_id];
  *n_host = (int)s.pages.size();
  if (phys_host)
    for (int i = 0; i < std::min(cap, (int)s.pages.size()); ++i) phys_host[i] = s.pages[i];
  return SPD_OK;
}

spd_status spd_free_pages(spd_ctx *c, int *n_free) {
  if (!c || !n_free) return SPD_ERR_INVALID_ARG;
  *n_free = (int)c->free_pages.size();
  return SPD_OK;
}

static spd_status check_append(spd_ctx *c, const int *ids, int n, int n_tokens, const void *k,
                               const void *v) {
  if (n_tokens < 1 || !k || !v) return c->fail(SPD_ERR_INVALID_ARG, "n_tokens >= 1 and k, v required");
  if (!aligned16(k) || !aligned16(v)) return c->fail(SPD_ERR_INVALID_ARG, "k, v must be 16-byte aligned");
  spd_status r = check_seqs(c, ids, n);
  if (r != SPD_OK) return r;
  long long need = 0;
  for (int i = 0; i < n; ++i) {
    const Seq &s = c->seqs[ids[i]];
    if (s.L + n_tokens > c->cfg.max_context)
      return c->fail(SPD_ERR_CAPACITY, "sequence %d: %lld + %d tokens exceed max_context %d",
                     ids[i], s.L, n_tokens, c->cfg.max_context);
    need += pages_needed(c, s, n_tokens);
  }
  if (need > (long long)c->free_pages.size())
    return c->fail(SPD_ERR_NO_PAGES, "need %lld physical pages, %zu free", need,
                   c->free_pages.size());
  return SPD_OK;
}

spd_status spd_kv_append(spd_ctx *c, const int *seq_ids, int n_seqs, int n_tokens, const void *k,
                         const void *v, spd_stream stream) {
  if (!c) return SPD_ERR_INVALID_ARG;
  spd_status r = check_append(c, seq_ids, n_seqs, n_tokens, k, v);
  if (r != SPD_OK) return r;
  return append_impl(c, seq_ids, n_seqs, n_tokens, k, v, (cudaStream_t)stream);
}

spd_status spd_select_pages(spd_ctx *c, const void *q, const int *seq_ids, int n_seqs, int force,
                            spd_stream stream) {
  if (!c) return SPD_ERR_INVALID_ARG;
  if (!q || !aligned16(q)) return c->fail(SPD_ERR_INVALID_ARG, "q must be a 16-byte aligned pointer");
  spd_status r = check_seqs(c, seq_ids, n_seqs);
  if (r != SPD_OK) return r;
  for (int i = 0; i < n_seqs; ++i)
    if (c->seqs[seq_ids[i]].L < 1)
      return c->fail(SPD_ERR_STATE, "sequence %d has no tokens", seq_ids[i]);
  return select_impl(c, q, seq_ids, n_seqs, force != 0, (cudaStream_t)stream);
}

spd_status spd_sparse_decode_attention(spd_ctx *c, const void *q, const int *seq_ids, int n_seqs,
                                       float *out, spd_stream stream) {
  if (!c) return SPD_ERR_INVALID_ARG;
  if (!q || !out || !aligned16(q) || !aligned16(out))
    return c->fail(SPD_ERR_INVALID_ARG, "q and out must be 16-byte aligned pointers");
  spd_status r = check_seqs(c, seq_ids, n_seqs);
  if (r != SPD_OK) return r;
  if ((r = check_attend_state(c, seq_ids, n_seqs, false)) != SPD_OK) return r;
  return attention_impl(c, q, seq_ids, n_seqs, out, nullptr, nullptr, (cudaStream_t)stream);
}

spd_status spd_sparse_decode_attention_stats(spd_ctx *c, const void *q, const int *seq_ids,
                                             int n_seqs, float *out, float *row_max,
                                             float *row_sum, spd_stream stream) {
  if (!c) return SPD_ERR_INVALID_ARG;
  if (!row_max || !row_sum || !aligned4(row_max) || !aligned4(row_sum))
    return c->fail(SPD_ERR_INVALID_ARG, "row_max and row_sum must be 4-byte aligned pointers");
  spd_status r = check_attention_call(c, q, seq_ids, n_seqs, out);
  if (r != SPD_OK) return r;
  StatsOut so;
  so.row_max = row_max;
  so.row_sum = row_sum;
  return attention_impl(c, q, seq_ids, n_seqs, out, nullptr, nullptr, (cudaStream_t)stream,
                        nullptr, false, so);
}

spd_status spd_sparse_decode_attention_page_mass(spd_ctx *c, const void *q, const int *seq_ids,
                                                 int n_seqs, float *out, float *row_max,
                                                 float *row_sum, int *pages, float *page_mass,
                                                 int max_pages, spd_stream stream) {
  if (!c) return SPD_ERR_INVALID_ARG;
  if ((row_max == nullptr) != (row_sum == nullptr) ||
      (row_max && (!aligned4(row_max) || !aligned4(row_sum))))
    return c->fail(SPD_ERR_INVALID_ARG,
                   "row_max and row_sum must both be NULL or both 4-byte aligned pointers");
  const Derived &dv = c->dv;
  if (dv.Hd > 0 && (!pages || !page_mass || !aligned4(pages) || !aligned4(page_mass)))
    return c->fail(SPD_ERR_INVALID_ARG, "pages and page_mass must be 4-byte aligned pointers");
  if (dv.Hd > 0 && max_pages < 1) return c->fail(SPD_ERR_INVALID_ARG, "max_pages must be >= 1");
  spd_status r = check_attention_call(c, q, seq_ids, n_seqs, out);
  if (r != SPD_OK) return r;
  if (dv.Hd > 0) {
    for (int i = 0; i < n_seqs; ++i) {
      const Seq &s = c->seqs[seq_ids[i]];
      const int n_att = s.sel_count + nL_of(s.L, c->cfg.logical_page) - s.nL0;
      if (n_att > max_pages)
        return c->fail(SPD_ERR_CAPACITY, "sequence %d attends %d pages per dynamic head, "
                       "max_pages is %d", seq_ids[i], n_att, max_pages);
      if (n_att > dv.mass_pages)
        return c->fail(SPD_ERR_CAPACITY, "sequence %d attends %d pages per dynamic head; the "
                       "per-page mass covers at most %d (select its pages again)", seq_ids[i],
                       n_att, dv.mass_pages);
    }
  }
  StatsOut so;
  so.row_max = row_max;
  so.row_sum = row_sum;
  so.pages = pages;
  so.page_mass = page_mass;
  so.max_pages = max_pages;
  return attention_impl(c, q, seq_ids, n_seqs, out, nullptr, nullptr, (cudaStream_t)stream,
                        nullptr, false, so);
}

spd_status spd_decode_step(spd_ctx *c, const void *q, const void *k, const void *v,
                           const int *seq_ids, int n_seqs, float *out, spd_stream stream) {
  if (!c) return SPD_ERR_INVALID_ARG;
  if (!q || !out || !aligned16(q) || !aligned16(out))
    return c->fail(SPD_ERR_INVALID_ARG, "q and out must be 16-byte aligned pointers");
  spd_status r = check_append(c, seq_ids, n_seqs, 1, k, v);
  if (r != SPD_OK) return r;
  if ((r = check_attend_state(c, seq_ids, n_seqs, true)) != SPD_OK) return r;
  cudaStream_t st = (cudaStream_t)stream;
  if ((r = ensure_device(c, st)) != SPD_OK) return r;
  // pages for the new token, then the token itself is appended by the decode
  // kernel (after this step's selection, which never reads it: the page
  // holding it is always kept)
  for (int i = 0; i < n_seqs; ++i) take_pages(c, seq_ids[i], 1);
  if ((r = flush_page_table(c, st)) != SPD_OK) return r;
  for (int i = 0; i < n_seqs; ++i) c->seqs[seq_ids[i]].L += 1;
  if ((r = select_impl(c, q, seq_ids, n_seqs, false, st, /*score_only=*/true)) != SPD_OK) return r;
  return attention_impl(c, q, seq_ids, n_seqs, out, k, v, st, nullptr, /*fused_topk=*/true);
}

spd_status spd_get_selection(spd_ctx *c, int seq_id, int kv_head, int *idx_host, int cap,
                             int *count_host, spd_stream stream) {
  if (!c || !count_host) return SPD_ERR_INVALID_ARG;
  spd_status r = check_seqs(c, &seq_id, 1);
  if (r != SPD_OK) return r;
  if (kv_head < 0 || kv_head >= c->cfg.num_kv_heads || c->dv.kv_kind[kv_head] != 0)
    return c->fail(SPD_ERR_INVALID_ARG, "kv head %d is not a dynamic head", kv_head);
  const Seq &s = c->seqs[seq_id];
  if (!s.has_sel) return c->fail(SPD_ERR_STATE, "sequence %d has no selection", seq_id);
  *count_host = s.sel_count;
  if (!idx_host) return SPD_OK;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaStreamSynchronize");
  const int *src = static_cast<const int *>(c->buf.selection) +
                   ((size_t)seq_id * c->dv.Hd + c->dv.kv_sub[kv_head]) * c->dv.ksel_max;
  e = cudaMemcpy(idx_host, src, sizeof(int) * std::min(cap, s.sel_count), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaMemcpy(selection)");
  return SPD_OK;
}

spd_status spd_check_status(spd_ctx *c, spd_stream stream) {
  if (!c) return SPD_ERR_INVALID_ARG;
  if (!c->device_ready) return SPD_OK;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaStreamSynchronize");
  int w[4] = {0, 0, 0, 0};
  e = cudaMemcpy(w, c->buf.scratch, sizeof w, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaMemcpy(error word)");
  if (w[0] == 0) return SPD_OK;
  cudaMemset(c->buf.scratch, 0, sizeof w);
  return c->fail(SPD_ERR_DEVICE_CHECK, "device check %d (details %d %d %d)", w[0], w[1], w[2], w[3]);
}

const char *spd_status_string(spd_status s) {
  switch (s) {
    case SPD_OK: return "ok";
    case SPD_ERR_INVALID_ARG: return "invalid argument";
    case SPD_ERR_NO_PAGES: return "no free physical pages";
    case SPD_ERR_BAD_SEQ: return "bad sequence id";
    case SPD_ERR_CAPACITY: return "capacity exceeded";
    case SPD_ERR_CUDA: return "CUDA error";
    case SPD_ERR_DEVICE_CHECK: return "device bounds check failed";
    case SPD_ERR_STATE: return "call out of order";
  }
  return "unknown status";
}

const char *spd_last_error(spd_ctx *c) { return c ? c->err.c_str() : ""; }

spd_status spd_set_early_kv_staging(spd_ctx *c, int enable) {
  if (!c) return SPD_ERR_INVALID_ARG;
  c->early_staging = enable != 0;
  return SPD_OK;
}

spd_status spd_launch_count(spd_ctx *c, long long *n) {
  if (!c || !n) return SPD_ERR_INVALID_ARG;
  *n = c->launches;
  return SPD_OK;
}

}  // extern "C"
