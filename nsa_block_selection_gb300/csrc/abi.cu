// Library-wide entry points of the C ABI: status strings, version, and the
// device status check that covers every kernel's bounded waits.

#include <cuda_runtime.h>

#include "nsa_sel_attn.h"
#include "status.cuh"

namespace nsa {
int topk_read_and_clear_status(unsigned int* value);  // top-k block selection (topk_blocks.cu)
}  // namespace nsa

extern "C" {

const char* nsa_status_string(int status) {
  switch (status) {
    case NSA_OK: return "ok";
    case NSA_ERR_NULL: return "null pointer";
    case NSA_ERR_SHAPE: return "invalid shape";
    case NSA_ERR_BLOCK_SIZE: return "block_size must be 32 or 64";
    case NSA_ERR_HEAD_DIM: return "head dim D must be 64 or 128";
    case NSA_ERR_GROUPS:
      return "H must be a multiple of G, with H/G <= 8 or a multiple of 8";
    case NSA_ERR_ALIGN: return "misaligned pointer";
    case NSA_ERR_LAUNCH: return "CUDA launch failed";
    case NSA_ERR_TIMEOUT: return "device wait timed out";
    case NSA_ERR_WORKSPACE: return "workspace too small";
    case NSA_ERR_SCRATCH:
      return "problem needs more scratch than the fixed buffer of the no-allocation entry point";
    case NSA_ERR_DTYPE:
      return "unsupported dtype: Q/K/V fp16 or bf16; O fp32 or the type of Q/K/V";
    case NSA_ERR_BOUNDS:
      return "a debug-build bounds check failed (library built with NSA_DEBUG_BOUNDS)";
    default: return "unknown status";
  }
}

int nsa_version(void) { return 200; }

int nsa_sync_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return NSA_ERR_LAUNCH;
  unsigned int fwd = 0u, bwd = 0u, swa = 0u, shr = 0u, prb = 0u, tpk = 0u;
  if (nsa::fwd_read_and_clear_status(&fwd) != NSA_OK) return NSA_ERR_LAUNCH;
  if (nsa::bwd_read_and_clear_status(&bwd) != NSA_OK) return NSA_ERR_LAUNCH;
  if (nsa::swa_read_and_clear_status(&swa) != NSA_OK) return NSA_ERR_LAUNCH;
  if (nsa::shared_read_and_clear_status(&shr) != NSA_OK) return NSA_ERR_LAUNCH;
  if (nsa::probe_read_and_clear_status(&prb) != NSA_OK) return NSA_ERR_LAUNCH;
  if (nsa::topk_read_and_clear_status(&tpk) != NSA_OK) return NSA_ERR_LAUNCH;
  const unsigned int all = fwd | bwd | swa | shr | prb | tpk;
  if (all & 2u) return NSA_ERR_BOUNDS;
  return all ? NSA_ERR_TIMEOUT : NSA_OK;
}

}  // extern "C"
