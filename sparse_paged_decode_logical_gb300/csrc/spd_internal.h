// Internal interface between the host runtime (spd_runtime.cpp) and the CUDA
// kernels.  Every per-call quantity travels in a parameter block passed by
// value, so a launch needs no host staging buffer and can be captured into a
// CUDA graph as is.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "spd.h"

namespace spd {

constexpr int kSeqsPerLaunch = 64;    // sequences described per parameter block
constexpr int kMaxItems = 4096;       // split-K work items per decode launch
constexpr int kMaxKvHeads = 128;
constexpr int kPtUpdPerLaunch = 240;  // page-table entries per pt_write launch
constexpr int kScratchHeader = 256;   // bytes: device error word and info

// Device error word layout (int32 at scratch + 0): 0 = ok, else a code below;
// scratch + 4 .. + 16 hold details of the first violation.
enum DevErr : int {
  kDevOk = 0,
  kDevBadPhys = 1,      // page table entry outside the pool
  kDevBadPage = 2,      // logical page beyond the page table row
  kDevBadSelection = 3, // selection entry out of range
  kDevTopkCount = 4,    // top-k produced a count different from K_sel
  kDevTimeout = 5,      // a bounded mbarrier wait gave up
};

struct ScratchLayout {
  size_t tickets_dec;  // int [kSeqsPerLaunch * Hkv]
  size_t tickets_sel;  // int [kSeqsPerLaunch * Hd]
  size_t bounds;       // uint32 [kSeqsPerLaunch * Hd * bound_stride] per-chunk score bounds
  size_t part_ml;      // float2 [kMaxItems * G]   (row max in log2 units, sum)
  size_t part_o;       // float  [kMaxItems * G * d]
  size_t scores;       // float  [kSeqsPerLaunch * Hd * score_stride]
  size_t page_part;    // float2 [kSeqsPerLaunch * Hd * mass_tiles * G] per-tile (max, sum)
  size_t total;
};

// ---- kv append + metadata ------------------------------------------------
struct AppendSeq {
  int slot;      // sequence slot (row of the page table / stream buffers)
  int L_old;     // length before this append
  int cta_off;   // first dynamic CTA of this sequence
};

struct AppendParams {
  const void *k, *v;           // [n_seqs][n_tokens][Hkv][d]
  void *k_pool, *v_pool, *meta, *stream_k, *stream_v;
  const int *page_table;
  int *err;
  int n_seqs, n_tokens, Hkv, Hd, Hs, ell, P, R, max_pp, S, W, num_phys;
  int dyn_ctas;                // sum over seqs of touched logical pages * Hd
  int kv_fp8;                  // store fp8 E4M3 codes of value / scale
  float k_scale[kMaxKvHeads], v_scale[kMaxKvHeads];
  unsigned char dyn_kv[kMaxKvHeads];  // dynamic index -> kv head
  unsigned char str_kv[kMaxKvHeads];  // streaming index -> kv head
  AppendSeq seqs[kSeqsPerLaunch];
};

struct PtUpdate {
  int slot, index, phys;
};
struct PtWriteParams {
  int *page_table;
  int max_pp, n;
  PtUpdate upd[kPtUpdPerLaunch];
};

// ---- page selection --------------------------------------------------------
struct SelectSeq {
  int slot;
  int qrow;       // row of this sequence in the call's q array
  int nL;         // logical pages at selection time
  int K_sel;      // pages to keep
  int chunk_off;  // first CTA of this sequence
  int n_chunks;   // scoring CTAs per dynamic head (0: nothing to score, one CTA
                  // writes the trivial selection)
  int tau_m;      // > 0: each full chunk publishes its tau_m-th largest score key
                  // (tau_m x full chunks >= the pages to choose), 0: none
};

struct SelectParams {
  const void *q;        // [n_seqs][Hq][d]
  const void *meta;
  const int *page_table;
  int *selection;       // [max_seqs][Hd][ksel_max]
  float *scores;        // [kSeqsPerLaunch][Hd][score_stride], rows 16-byte aligned
  int *tickets;         // [kSeqsPerLaunch][Hd], zero between launches
  uint32_t *bounds;     // [kSeqsPerLaunch][Hd][bound_stride]
  int bound_stride;
  int *err;
  int n_seqs, Hq, Hd, ell, R, max_pp, ksel_max, score_stride, pages_per_chunk,
      num_phys;
  int score_ctas;       // total scoring CTAs
  int score_only;       // 1: write the scores and stop (the decode kernel selects)
  int early;            // 1: read metadata before waiting for the previous kernel
  int kv_fp8;           // metadata rows are fp8 E4M3 codes (one byte each)
  unsigned char dyn_kv[kMaxKvHeads];
  SelectSeq seqs[kSeqsPerLaunch];
};

// ---- split-K decode over 16-row tiles (decode.cu) ---------------------------
struct TileSeq {
  int slot, L;
  int nL0;        // logical pages when the selection was taken
  int sel_count;  // pages in the stored selection
  int item_off;   // first work item of this sequence
  int ns_dyn;     // items (CTAs) per dynamic head: clusters x cluster size
  int ns_str;     // items (CTAs) per streaming head
  int tpi_dyn;    // tiles per dynamic item
  int tpi_str;    // tiles per streaming item
  int topk_n;     // > 0: this launch selects the pages itself, from topk_n candidate
                  // scores in row topk_row of `scores` (sel_count - 1 of them plus
                  // the newest page), and stores the selection
  int topk_row;
  int topk_bounds;  // per-chunk score bounds to read for it (0: none)
};

struct TileDecodeParams {
  CUtensorMap tm_k, tm_v;    // pool:      dims {d, P, Nphys*Hd}, box {64, 16, 1}
  CUtensorMap tm_sk, tm_sv;  // streaming: dims {d, max_seqs*Hs*(S+W), 1}, box {64, 16, 1}
  const void *q;             // [n_seqs][Hq][d]
  const void *k_new, *v_new; // [n_seqs][Hkv][d] for a fused append, else null
  float *out;                // [n_seqs][Hq][d]
  float *row_max, *row_sum;  // [n_seqs][Hq] softmax statistics, or null
  // per-page attention mass of the dynamic units (all null when not asked for)
  float2 *page_part;         // [n_seqs][Hd][page_tile_cap][G] each tile's (max, sum), base 2
  int page_tile_cap;
  int *pages;                // [n_seqs][Hd][max_pages] attended logical pages, -1 after
  float *page_mass;          // [n_seqs][Hd][G][max_pages] softmax weight per attended page
  int max_pages;
  void *k_pool, *v_pool, *meta, *stream_k, *stream_v;
  const int *page_table, *selection;
  float *part_o;
  float2 *part_ml;
  int *tickets;
  int *err;
  const float *scores;       // [kSeqsPerLaunch][Hd][score_stride] page scores (fused steps)
  int score_stride;
  const uint32_t *bounds;    // [kSeqsPerLaunch][Hd][bound_stride] their per-chunk bounds
  int bound_stride;
  int n_seqs, Hq, Hkv, Hd, Hs, ell, P, R, max_pp, ksel_max, S, W, num_phys;
  int total_items;
  int cluster;        // CTAs per thread-block cluster; every unit's item count is a multiple
  int deep;           // the deep-ring launch shape (one CTA per SM, 24 stages)
  int early;          // stage K/V tiles before waiting for the previous kernel:
                      // bit 0 dynamic units, bit 1 streaming units; bit 2:
                      // streaming units do not wait at all
  float scale_log2;
  int kv_fp8;                // K/V stored as fp8 E4M3 codes of value / scale
  float k_scale[kMaxKvHeads], v_scale[kMaxKvHeads];  // per kv head (fp8 only)
  unsigned char dyn_kv[kMaxKvHeads];
  unsigned char str_kv[kMaxKvHeads];
  TileSeq seqs[kSeqsPerLaunch];
};

// kernel parameter blocks are passed by value: at most 32764 bytes
static_assert(sizeof(TileDecodeParams) <= 32764, "decode parameter block too large");

// A fused decode step (selection inside the decode kernel) holds at most this
// many candidate scores and kept pages in shared memory; larger ones use the
// selection kernel's own top-k.
constexpr int kFusedMaxCandidates = 8192;
constexpr int kFusedMaxSelected = 4096;
// A selection bounds its candidates from each scoring chunk's m-th largest
// score only while m (pages to choose / full chunks) is at most this.
constexpr int kMaxBoundRank = 8;

constexpr int kTileRows = 16;
constexpr int kMaxTilesPerItem = 8;
// The per-page attention mass covers a selection's pages plus this many
// logical pages created after it was taken.
constexpr int kMassExtraPages = 64;

cudaError_t prepare_decode_kernels();
cudaError_t prepare_decode_mass_kernels();  // called by prepare_decode_kernels()
cudaError_t launch_decode_tiles_mass(const TileDecodeParams &p, int dtype, int d, int G,
                                     cudaStream_t s);
cudaError_t prepare_decode_reuse_kernels();  // called by prepare_decode_kernels()
// the plain 16-bit decode for launches in which no unit selects its pages
cudaError_t launch_decode_tiles_reuse(const TileDecodeParams &p, int dtype, int d, int G,
                                      cudaStream_t s);
cudaError_t prepare_decode_fp8_kernels();  // called by prepare_decode_kernels()
cudaError_t launch_decode_tiles_fp8(const TileDecodeParams &p, int dtype, int G,
                                    cudaStream_t s);
// after prepare_decode_kernels(); deep: the deep-ring launch shape
int decode_max_cluster(int dtype, int d, int G, bool deep = false);
int decode_max_tiles_per_cta();
int decode_ring_stages(bool deep);  // 16-bit tiles the ring of a launch shape holds
cudaError_t launch_decode_tiles(const TileDecodeParams &p, int dtype, int d, int G,
                                cudaStream_t s, long long *launches);

// Temporaries of a decode launch (split partials and the per-unit tickets)
// supplied from outside the context's scratch buffer.
struct DecodeScratch {
  float *part_o;   // [max_items][G][d]
  float2 *part_ml; // [max_items][G]
  int *tickets;    // [kSeqsPerLaunch][Hkv], zero before the launch
  int max_items;   // split items one launch may use
};

// Runtime hooks (spd_runtime.cpp) for entry points defined in other files.
spd_status check_attention_call(spd_ctx *c, const void *q, const int *ids, int n,
                                const float *out);
spd_status bind_device(spd_ctx *c, cudaStream_t st, int *device);
// SPD_ERR_CAPACITY (with nothing enqueued) if some launch of the call would
// need more than max_items split items.
spd_status check_attention_capacity(spd_ctx *c, const int *ids, int n, int max_items);
spd_status attention_with_scratch(spd_ctx *c, const void *q, const int *ids, int n, float *out,
                                  cudaStream_t st, const DecodeScratch &scratch);
spd_status fail_message(spd_ctx *c, spd_status s, const char *msg);

// Launchers.  dtype: 0 fp16, 1 bf16.  Return cudaGetLastError() and add the
// number of kernels enqueued to *launches.
cudaError_t launch_pt_write(const PtWriteParams &p, cudaStream_t s, long long *launches);
cudaError_t launch_append(const AppendParams &p, int dtype, int d, cudaStream_t s,
                          long long *launches);
int select_pages_per_cta();
cudaError_t launch_select_fused(const SelectParams &p, int dtype, int d, int G, cudaStream_t s,
                                long long *launches);

}  // namespace spd
