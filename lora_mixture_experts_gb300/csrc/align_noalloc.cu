// moe_lora_align_noalloc: the align step for callers that cannot hand the
// library a workspace.
//
// Some callers have no way to obtain device memory for scratch: code that
// runs while a stream is being captured into a CUDA graph (where a
// cudaMalloc would break or invalidate the capture), plug-ins and hooks
// that are handed tensors but no allocator, and serving processes that have
// reserved all device memory for their own pool up front.  This entry point
// takes the same inputs and outputs as moe_lora_align but keeps its scratch
// in a fixed array that lives in the library's own device memory, so it
// allocates nothing.
//
// Costs and limits of that choice:
//  * every GPU that loads the library holds kNoallocScratchBytes (4 MiB) of
//    device memory for it until the process exits;
//  * sizes whose align scratch exceeds that are rejected with
//    MOELORA_ERR_WORKSPACE;
//  * all calls share the one array, so two calls whose work overlaps on the
//    GPU (different streams, no ordering between them) race and may both
//    produce wrong results; order them on one stream;
//  * the first call on each device (and again after the device's context
//    was destroyed and created anew) looks up the array's device address
//    with cudaGetSymbolAddress; make that first call outside any stream
//    capture.
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "align.cuh"

namespace moelora {
namespace {

constexpr size_t kNoallocScratchBytes = 4u << 20;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code `g_noalloc_scratch` names a host-side
// stand-in, not device memory: only the address looked up below may be
// passed to kernels.
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

// Cached device address of the array, per device, with the id of the
// context it was looked up in.  A context torn down and made again (for
// instance after cudaDeviceReset) reloads the library's module and moves the
// array, so a cached address is used only while the current context's id is
// the one it was found in.
struct CachedAddr {
  unsigned long long ctx_id;
  void* ptr;
};
std::mutex g_addr_mu;
CachedAddr g_addr[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The driver's cuCtxGetCurrent and cuCtxGetId, looked up once through the
// runtime (the library links only the runtime).
bool context_id_fns(CtxGetCurrentFn& get_current, CtxGetIdFn& get_id) {
  static CtxGetCurrentFn cur = nullptr;
  static CtxGetIdFn idf = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      idf = reinterpret_cast<CtxGetIdFn>(p);
  }
  get_current = cur;
  get_id = idf;
  return cur && idf;
}

// Id of the current context, 0 if there is none yet or it cannot be read.
unsigned long long current_context_id(CtxGetCurrentFn get_current, CtxGetIdFn get_id) {
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device, looked up with
// cudaGetSymbolAddress (with that device current) on the first call in each
// context.  nullptr on failure.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  CtxGetCurrentFn get_current;
  CtxGetIdFn get_id;
  std::lock_guard<std::mutex> lk(g_addr_mu);
  if (!context_id_fns(get_current, get_id)) return nullptr;
  const unsigned long long id = current_context_id(get_current, get_id);
  if (id != 0 && g_addr[dev].ptr && g_addr[dev].ctx_id == id) return g_addr[dev].ptr;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
  // (the lookup makes the device's primary context current if it was not)
  const unsigned long long id_now = current_context_id(get_current, get_id);
  g_addr[dev] = {id_now, ptr};
  return ptr;
}

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace
}  // namespace moelora

using namespace moelora;

extern "C" int moe_lora_align_noalloc(const moelora_dims* d, const int32_t* topk_ids,
                                      const int32_t* lora_ids, int32_t block_m,
                                      int32_t* sorted_ids, int32_t* blk_expert, int32_t* seg_off,
                                      int32_t* num_post_pad, moelora_stream_t stream_) {
  if (!d || d->T < 0 || d->k < 1 || d->E < 1 || d->L < 0 || block_m < 1 || block_m > 1024)
    return MOELORA_ERR_INVALID_ARG;
  if (d->E > kMaxExperts || static_cast<long long>(d->E) * (d->L + 1) > kMaxBins)
    return MOELORA_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->T) * d->k >= (1ll << 30)) return MOELORA_ERR_UNSUPPORTED;
  if ((d->T > 0 && (!topk_ids || !lora_ids)) || !sorted_ids || !blk_expert || !seg_off ||
      !num_post_pad)
    return MOELORA_ERR_INVALID_ARG;

  // scratch layout: header | per-chunk histograms | bin of each entry |
  // rank of each entry | bin starts
  const int n = d->T * d->k;
  const int nbins = d->E * (d->L + 1);
  const int nchunks = (n + kAlignChunk - 1) / kAlignChunk;
  const size_t off_hist = round256(sizeof(WsHeader));
  const size_t off_bin = off_hist + round256(static_cast<size_t>(nchunks) * nbins * 4);
  const size_t off_rank = off_bin + round256(static_cast<size_t>(n) * 4);
  const size_t off_start = off_rank + round256(static_cast<size_t>(n) * 4);
  const size_t total = off_start + round256(static_cast<size_t>(nbins) * 4);
  if (total > kNoallocScratchBytes) return MOELORA_ERR_WORKSPACE;

  uint8_t* base = static_cast<uint8_t*>(scratch_address());
  if (!base) return MOELORA_ERR_CUDA;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  AlignArgs a;
  std::memset(&a, 0, sizeof(a));
  a.topk_ids = topk_ids;
  a.lora_ids = lora_ids;
  a.T = d->T;
  a.k = d->k;
  a.E = d->E;
  a.L = d->L;
  a.n = n;
  a.nbins = nbins;
  a.nchunks = nchunks;
  a.block_m = block_m;
  a.Pmax = n + d->E * (block_m - 1);
  a.hdr = reinterpret_cast<WsHeader*>(base);
  a.chunk_hist = reinterpret_cast<int*>(base + off_hist);
  a.bin_of = reinterpret_cast<int*>(base + off_bin);
  a.rank_of = reinterpret_cast<int*>(base + off_rank);
  a.bin_start = reinterpret_cast<int*>(base + off_start);
  a.sorted_ids = sorted_ids;
  a.blk_expert = blk_expert;
  a.seg_off = seg_off;
  a.num_post_pad = num_post_pad;

  // the error word must start at zero; every other scratch word is written
  // before it is read within the call
  if (cudaMemsetAsync(&a.hdr->err, 0, sizeof(int), stream) != cudaSuccess) return MOELORA_ERR_CUDA;
  if (launch_align_hist(a, stream, false) != cudaSuccess) return MOELORA_ERR_CUDA;
  if (launch_align_scan(a, stream, nchunks > 0) != cudaSuccess) return MOELORA_ERR_CUDA;
  if (launch_align_scatter(a, stream, true) != cudaSuccess) return MOELORA_ERR_CUDA;
  return MOELORA_OK;
}
