// mtpsd_indexer_topk_noalloc: the indexer + top-k call for callers that
// cannot allocate device memory.  Its scratch (the score matrix) lives in a
// file-scope static __device__ array of MTPSD_NOALLOC_SCRATCH_BYTES that every
// GPU loading this library holds until the process exits.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mtpsd {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MTPSD_NOALLOC_SCRATCH_BYTES];

// Device address of the array, looked up once per device (host code must not
// use the symbol itself: on the host it is only a stand-in, not a device
// address).
constexpr int kMaxDevices = 128;
static void* g_scratch_addr[kMaxDevices];
static std::mutex g_scratch_mu;

static int noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("indexer_topk_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
    return MTPSD_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("indexer_topk_noalloc: device ordinal %d not supported", dev);
    return MTPSD_EUNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      set_error("indexer_topk_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
      return MTPSD_ECUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MTPSD_OK;
}

}  // namespace mtpsd

using namespace mtpsd;

extern "C" int mtpsd_indexer_topk_noalloc(const mtpsd_indexer_args* args, void* stream) {
  if (!args) {
    set_error("indexer_topk_noalloc: null args");
    return MTPSD_EINVAL;
  }
  // with a caller score buffer only the work plan and the top-k candidate lists live in the scratch
  size_t need = args->scores ? mtpsd_indexer_topk_aux_bytes(args->B, args->R, args->max_visible, args->topk)
                             : mtpsd_indexer_topk_workspace_size(args->B, args->R, args->max_visible, args->topk);
  if (need > (size_t)MTPSD_NOALLOC_SCRATCH_BYTES) {
    set_error("indexer_topk_noalloc: this call needs %zu bytes of scratch but the static maximum is %zu bytes "
              "(R * mtpsd_scores_ld(max_visible) * 4 plus the plan and top-k lists, or only those when "
              "args->scores is given); pass args->scores or use mtpsd_indexer_topk with a workspace",
              need, (size_t)MTPSD_NOALLOC_SCRATCH_BYTES);
    return MTPSD_EWORKSPACE;
  }
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  // Nothing in the scratch has to start at zero: every score a row reads is
  // written by the same call first.
  mtpsd_indexer_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = MTPSD_NOALLOC_SCRATCH_BYTES;
  return mtpsd_indexer_topk(&a, stream);
}
