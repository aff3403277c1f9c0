// moe_permute_amax_noalloc: the routing / permutation / amax pass with its
// chunk-histogram scratch held in a fixed array that the library itself
// carries in device memory, for callers that cannot allocate device memory.
//
// Such callers are, for example, a plugin run by another inference runtime
// that owns every byte of device memory and hands the plugin only its input
// and output buffers and a stream, or a serving loop that must not call
// cudaMalloc on its critical path because the call can synchronise the whole
// device.  This entry point computes exactly what moe_permute_amax computes,
// with the same kernels, but takes no workspace argument.
//
// The array is a file-scope device variable of MOE_PERMUTE_NOALLOC_SCRATCH_BYTES
// (4 MiB): every GPU on which the library is loaded keeps it until the process
// exits.  Host code cannot use the array's name as a device address, so every
// call looks the address up on the current device with cudaGetSymbolAddress
// (a table lookup once the device code is loaded).  The address is not kept
// between calls: after a cudaDeviceReset the device code is loaded again and
// the array may sit elsewhere, and a kept address would then point at freed
// memory.  The first call on a device may load the library's device code on
// that device, so make it before any stream capture begins.
//
// Every call shares the one array.  Calls whose work overlaps on the GPU (two
// streams, or two host threads, at the same time) race on it and produce
// wrong results: the caller serialises them.  Nothing in the array needs to
// start at zero: the routing kernel writes every histogram entry that the
// later kernels of the same call read.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

static __device__ __align__(256) int32_t g_permute_noalloc_hist[MOE_PERMUTE_NOALLOC_SCRATCH_BYTES / 4];

namespace {

std::mutex g_noalloc_mu;
int g_noalloc_dev_ok[64];  // per device ordinal: 0 unknown, 1 compute capability 10.3, -1 other

// Device address of the scratch array on the current device.  The device
// check is cached per ordinal (a reset does not change it); the address is
// looked up on every call.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MOE_ERR_DEVICE;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_dev_ok[dev] == 0) {
      int maj = 0, min = 0;
      if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
      g_noalloc_dev_ok[dev] = (maj == 10 && min == 3) ? 1 : -1;
    }
    if (g_noalloc_dev_ok[dev] < 0) return MOE_ERR_DEVICE;
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_noalloc_hist);
  if (e != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  *out = p;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_permute_amax_noalloc(const float* logits, const int32_t* ext_ids, const float* ext_w,
                                        const uint16_t* x, int T, int E, int k, int d, int32_t* topk_ids,
                                        float* topk_w, int32_t* counts, int32_t* offsets, int32_t* row_to_token,
                                        int32_t* token_slot_row, float* amax_tok, float* amax_row, int* status,
                                        void* stream) {
  if (T < 0 || E < 1 || E > 1024) return MOE_ERR_SHAPE;
  const size_t need = moe_permute_workspace_bytes(T, E);
  if (need > (size_t)MOE_PERMUTE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  void* ws = nullptr;
  const int rc = noalloc_scratch(&ws);
  if (rc != MOE_OK) return rc;
  return moe_permute_amax(logits, ext_ids, ext_w, x, T, E, k, d, topk_ids, topk_w, counts, offsets, row_to_token,
                          token_slot_row, amax_tok, amax_row, ws, (size_t)MOE_PERMUTE_NOALLOC_SCRATCH_BYTES, status,
                          stream);
}
