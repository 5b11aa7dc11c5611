// FP8 lightning-indexer score GEMM on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA).  Placeholder until the kernel lands: the generic
// CUDA-core kernel serves every shape.
#include "common.cuh"
#include "internal.h"

namespace mtpsd {

bool indexer_tc_supported(const IndexerPlan& p) {
  (void)p;
  return false;
}

int launch_indexer_scores_tc(const IndexerPlan& p, cudaStream_t st) {
  (void)p; (void)st;
  set_error("indexer: tensor-core kernel not built");
  return MTPSD_EUNSUPPORTED;
}

}  // namespace mtpsd
