// noalloc.cu -- moe_align_sort_noalloc: the expert sort with its scratch in a static device array.
//
// Some callers cannot allocate device memory at the point where they need the sort: a serving
// engine that hands all device memory to its own pool at start-up and forbids any later
// cudaMalloc (an allocation there would synchronise the device and fragment the pool), or a
// plugin entry point whose host framework passes only input and output buffers and offers no
// workspace.  For them this entry point runs the chunked form of the sort (three kernels over
// 256-route chunks, the form moe_align_sort uses above 8192 routes), whose per-chunk expert
// histograms and status word live in `g_sort_scratch` below, a
// file-scope device array that every GPU loading the library holds until the process exits.
//
// Set-up: the first call on a device (with that device current) looks up the array's device
// address with cudaGetSymbolAddress and caches it per device; make that first call before any
// stream capture.  No call allocates: the library calls no cudaMalloc, cudaFree or allocating
// library routine here.  All calls share the one array and it keeps the last call's contents:
// each call clears the status word (the only part that must start at zero; every histogram
// slot is written before it is read) and calls that overlap on the GPU race on the array.
#include <mutex>

#include "common.cuh"

namespace gb300moe {

namespace {

// Per-chunk histograms: at most kNoAllocHistInts int32 (256 KiB), i.e.
// ceil(T*top_k / 256) * E <= 65536; the status word sits in the first 256 bytes.
constexpr int kNoAllocHistInts = 65536;
constexpr int kNoAllocHeaderInts = 64;

static __device__ __align__(256) int32_t g_sort_scratch[kNoAllocHeaderInts + kNoAllocHistInts];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_sort_scratch on the current device (looked up once per device).
cudaError_t scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_sort_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

}  // namespace gb300moe

using namespace gb300moe;

extern "C" moe_status_t moe_align_sort_noalloc(const moe_problem_t* p, int32_t block_m,
                                               const int32_t* topk_ids, int32_t* counts,
                                               int32_t* offsets, int32_t* sorted_ids,
                                               int32_t* tile_expert, int32_t* inv_route,
                                               int32_t* status_out, void* stream) {
  // The same checks as moe_align_sort: sizes, top_k <= 32, E <= 1024 and a shard
  // (ep_local_offset, ep_num_local) inside [0, E), so the local expert count is at most 1024.
  const moe_status_t st = check_problem(p);
  if (st != MOE_OK) return st;
  if (block_m <= 0 || block_m > 1024) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || !sorted_ids || !inv_route) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && !topk_ids) return MOE_ERR_INVALID_ARG;
  const moe_problem_t Pl = local_view(*p);  // ids index the local experts of a shard
  const int64_t P = (int64_t)p->T * p->top_k;
  const int64_t n_chunks = (P + 255) / 256;
  if (n_chunks * Pl.E > kNoAllocHistInts) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  int* status = reinterpret_cast<int*>(scratch);
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  const int64_t cap = P + (int64_t)p->E * (block_m - 1);
  if (launch_align_sort_chunked(Pl, block_m, topk_ids, counts, offsets, sorted_ids, cap,
                                tile_expert, inv_route, scratch + kNoAllocHeaderInts, status, s,
                                false, nullptr, nullptr, kTileRows, nullptr, nullptr,
                                kTileRows) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (status_out &&
      cudaMemcpyAsync(status_out, status, sizeof(int), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
