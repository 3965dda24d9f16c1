// spd_sparse_decode_attention_static: the split-K decode attention launch of
// spd_sparse_decode_attention, with its temporaries (split partials and the
// per-unit tickets of the fused combine) kept in a fixed, library-owned
// device array instead of the context's scratch buffer.
//
// Who needs it: callers that cannot allocate device memory when they run
// attention -- code executing while a CUDA stream is being captured (device
// allocation is not allowed there), integrations whose device memory plan is
// fixed at start-up and forbids later allocation, and plugins embedded in a
// host framework that owns every device allocation.  This entry point calls
// no cudaMalloc, cudaFree or allocating library routine.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// the library holds it (4,292,608 bytes) until the process exits.  Host code
// may not hand its name to a kernel -- on the host the name is only a
// stand-in for the symbol -- so its device address is fetched once per device
// with cudaGetSymbolAddress, with that device current, on the first call on
// that device (make that first call before any stream capture), and then
// passed to the kernel as a pointer.
//
// Every call shares the array and the array keeps the last call's contents:
// the tickets are cleared at the start of each call (they must start at
// zero); the partials are always written before they are read.  Calls whose
// work overlaps on the GPU (two streams, two contexts at once) race on the
// array; issue them in order on one stream.
#include <mutex>

#include "spd_internal.h"

namespace {

constexpr int kStaticItems = 1024;   // split items per launch (<= 256 tiles of 16 rows each)
constexpr int kStaticMaxG = 8;       // query heads per kv head
constexpr int kStaticMaxD = 128;     // head_dim
constexpr size_t kTicketBytes = (size_t)spd::kSeqsPerLaunch * spd::kMaxKvHeads * sizeof(int);
constexpr size_t kMlBytes = (size_t)kStaticItems * kStaticMaxG * sizeof(float2);
constexpr size_t kOBytes = (size_t)kStaticItems * kStaticMaxG * kStaticMaxD * sizeof(float);
constexpr size_t kStaticBytes = kTicketBytes + kMlBytes + kOBytes;  // 4,292,608
static_assert(kStaticBytes == 4292608, "documented size");
static_assert(kTicketBytes % 256 == 0 && kMlBytes % 256 == 0, "sub-arrays stay aligned");

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices] = {};

}  // namespace

// Library-owned decode temporaries: [tickets | (m, l) partials | o partials].
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticBytes];

extern "C" spd_status spd_sparse_decode_attention_static(spd_ctx *ctx, const void *q,
                                                         const int *seq_ids, int n_seqs,
                                                         float *out, spd_stream stream) {
  if (!ctx) return SPD_ERR_INVALID_ARG;
  spd_status r = spd::check_attention_call(ctx, q, seq_ids, n_seqs, out);
  if (r != SPD_OK) return r;
  cudaStream_t st = (cudaStream_t)stream;
  int dev = -1;
  if ((r = spd::bind_device(ctx, st, &dev)) != SPD_OK) return r;
  if (dev < 0 || dev >= kMaxDevices)
    return spd::fail_message(ctx, SPD_ERR_CUDA, "device index beyond the static scratch table");
  void *base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
      // set-up, once per device, with that device current; the caller's
      // current device is restored afterwards, on success and on failure
      int cur = -1;
      const bool had = cudaGetDevice(&cur) == cudaSuccess;
      if (!had || cur != dev) {
        if (cudaSetDevice(dev) != cudaSuccess)
          return spd::fail_message(ctx, SPD_ERR_CUDA, "cudaSetDevice failed");
      }
      void *p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
      const bool restored = !(had && cur != dev) || cudaSetDevice(cur) == cudaSuccess;
      if (e != cudaSuccess || !p)
        return spd::fail_message(ctx, SPD_ERR_CUDA, "cudaGetSymbolAddress(static scratch) failed");
      if (!restored)
        return spd::fail_message(ctx, SPD_ERR_CUDA, "cudaSetDevice(restore) failed");
      g_scratch_addr[dev] = p;
    }
    base = g_scratch_addr[dev];
  }
  // every launch of the call is planned against the array's capacity before
  // anything (the ticket clear included) is enqueued
  if ((r = spd::check_attention_capacity(ctx, seq_ids, n_seqs, kStaticItems)) != SPD_OK) return r;
  // the per-unit tickets must start at zero
  cudaError_t e = cudaMemsetAsync(base, 0, kTicketBytes, st);
  if (e != cudaSuccess) return spd::fail_message(ctx, SPD_ERR_CUDA, "cudaMemsetAsync(tickets) failed");
  unsigned char *b = static_cast<unsigned char *>(base);
  spd::DecodeScratch s;
  s.tickets = reinterpret_cast<int *>(b);
  s.part_ml = reinterpret_cast<float2 *>(b + kTicketBytes);
  s.part_o = reinterpret_cast<float *>(b + kTicketBytes + kMlBytes);
  s.max_items = kStaticItems;
  return spd::attention_with_scratch(ctx, q, seq_ids, n_seqs, out, st, s);
}
