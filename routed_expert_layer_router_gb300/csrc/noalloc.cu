// noalloc.cu - moe_expert_ffn_noalloc: the decode expert FFN for callers that
// cannot allocate device memory.
//
// The decode FFN needs scratch between its two kernels: the SiLU(gate)*up
// activations h of every route (T*k*I floats) and of the shared expert (T*Is
// floats).  moe_expert_ffn takes that scratch from the caller's workspace.
// This variant instead uses one fixed array in the library's own device
// memory, so the call itself allocates nothing (no cudaMalloc, no cudaFree, no
// allocating library routine).  Every GPU that loads the library holds the
// array (kNoAllocScratchBytes) until the process exits.
#include "common.cuh"

// 8 MiB of fp32 scratch (MOE_NOALLOC_SCRATCH_BYTES in moe.h): enough for
// (T*k*I + T*Is) * 4 + 256 bytes, e.g. 64 tokens with top-8 and
// I = Is = 2048 (4.6 MiB), or one token of any supported width.
constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the real address is
// asked for with cudaGetSymbolAddress, with the device current.  It is asked
// on every call (after the first it costs a driver lookup, no allocation),
// so a device reset or another context never leaves a stale address behind.
moe_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  *out = p;
  return MOE_OK;
}
}  // namespace

namespace moe {
// Loads the array's module on the current device.  CUDA loads a module
// lazily, on the first use of something in it, and loading it reserves the
// array's device memory; the library's set-up (the first expcache_create,
// moe_layer_create or FFN call of the process) calls this, so that on that
// device the first moe_expert_ffn_noalloc allocates nothing either.
moe_status noalloc_setup() {
  void* p = nullptr;
  return scratch_address(&p);
}
}  // namespace moe

namespace moe {
size_t decode_workspace_bytes(int T, int I, int k, int Is);
}

MOE_API moe_status moe_expert_ffn_noalloc(const moe_ffn_args* a, void* stream) {
  if (!a) return MOE_ERR_INVALID_ARG;
  if (a->mode != MOE_MODE_DECODE) return MOE_ERR_UNSUPPORTED;
  if (a->T < 0 || a->I <= 0 || a->k <= 0 || a->Is < 0) return MOE_ERR_INVALID_ARG;
  if (moe::decode_workspace_bytes(a->T, a->I, a->k, a->Is) > kNoAllocScratchBytes)
    return MOE_ERR_UNSUPPORTED;  // larger than the fixed scratch: use moe_expert_ffn
  void* scratch = nullptr;
  moe_status st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  moe_ffn_args b = *a;
  b.workspace = scratch;
  b.workspace_bytes = kNoAllocScratchBytes;
  return moe_expert_ffn(&b, stream);
}
