// common.cuh - small device helpers shared by the library's kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

constexpr int kSMs = 152;  // GB300: 2 dies x 76 SMs

// ---- sticky device status: first error wins --------------------------------
__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}

// ---- expert-cache lookup of one layer (K-lookup), run on its own or as the
// tail of K-perm ----------------------------------------------------------------
struct LookupArgs {
  const int32_t* table;  // the layer's row of the slot table, nullptr: no lookup
  int slot_lo, slot_hi, n_cache, n_stage;
  int32_t *src_slot, *act_list, *n_act, *miss_ids, *n_miss;
  // optional (small-route path): per act_list position a, meta[2a] = {expert,
  // slot, first route position, routes}, meta[2a+1] = its gscale row (fp32
  // bits), so that the FFN's CTAs read one record instead of a chain of loads
  int4* meta;
  const float* gscale;
};

// ---- record layout (see moe.h) ---------------------------------------------
// values per block scale: NVFP4 16 (E4M3), MXFP4 32 (E8M0)
__host__ __device__ __forceinline__ int fmt_block(int fmt) { return fmt == MOE_FMT_MXFP4 ? 32 : 16; }

struct RecordLayout {
  uint64_t gate_codes, up_codes, down_codes;
  uint64_t gate_scales, up_scales, down_scales;
  uint64_t bytes;
  __host__ __device__ RecordLayout(int H, int I, int fmt) {
    uint64_t gu = (uint64_t)I * H / 2;
    gate_codes = 0;
    up_codes = gu;
    down_codes = 2 * gu;
    uint64_t sgu = (uint64_t)I * H / (uint64_t)fmt_block(fmt);
    gate_scales = 3 * gu;
    up_scales = gate_scales + sgu;
    down_scales = up_scales + sgu;
    bytes = down_scales + sgu;
  }
};

// byte offset of the 512-byte atom (row tile rt = r/128, k group kg = kb/4)
__host__ __device__ __forceinline__ uint64_t atom_offset(int rt, int kg, int KB) {
  return ((uint64_t)rt * (uint64_t)(KB / 4) + (uint64_t)kg) * 512u;
}

// ---- numeric helpers --------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// two E2M1 codes (one byte, element 2j in the low nibble) -> two floats
__device__ __forceinline__ void e2m1x4_to_f16x2x2(uint32_t w16, uint32_t& lo, uint32_t& hi) {
  // w16: bits 0..15 hold two bytes = four codes
  asm("{\n .reg .b8 a, b, c, d;\n mov.b32 {a, b, c, d}, %2;\n"
      " cvt.rn.f16x2.e2m1x2 %0, a;\n cvt.rn.f16x2.e2m1x2 %1, b;\n}"
      : "=r"(lo), "=r"(hi) : "r"(w16));
}

__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t h[4]) {
  asm("{\n .reg .b8 a, b, c, d;\n mov.b32 {a, b, c, d}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, a;\n cvt.rn.f16x2.e2m1x2 %1, b;\n"
      " cvt.rn.f16x2.e2m1x2 %2, c;\n cvt.rn.f16x2.e2m1x2 %3, d;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
}

// two E4M3 bytes (bits 0..15) -> f16x2 (exact)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w16) {
  uint32_t r;
  asm("{\n .reg .b16 a;\n cvt.u16.u32 a, %1;\n cvt.rn.f16x2.e4m3x2 %0, a;\n}" : "=r"(r) : "r"(w16));
  return r;
}

// E8M0 byte (MX scale) -> its value 2^(b - 127); 0xFF is NaN
__device__ __forceinline__ float e8m0_value(uint32_t b) {
  uint32_t u = b << 23;                      // 2^(b - 127) for b in [1, 254]
  u = b == 0u ? 0x00400000u : u;             // 2^-127 (an fp32 subnormal)
  u = b == 0xFFu ? 0x7FC00000u : u;          // NaN
  return __uint_as_float(u);
}

__device__ __forceinline__ float f16_lo(uint32_t h2) {
  float f;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.f32.f16 %0, l;\n}" : "=f"(f) : "r"(h2));
  return f;
}
__device__ __forceinline__ float f16_hi(uint32_t h2) {
  float f;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n cvt.f32.f16 %0, h;\n}" : "=f"(f) : "r"(h2));
  return f;
}

// streaming 128-bit load that does not allocate in L1
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// ---- programmatic dependent launch ------------------------------------------
// A kernel launched with launch_pdl() may start while the previous kernel on
// its stream is still running (in streams and in captured CUDA graphs, where
// it measured faster too).  pdl_wait() blocks until that kernel has
// completed and its writes are visible; pdl_launch_dependents() lets the next
// kernel start launching.  Every kernel launched with launch_pdl() calls
// pdl_wait() before it touches memory that an earlier kernel writes or reads,
// and triggers only after that wait, so each launch can run ahead of at most
// the one kernel before it.  Both are no-ops after a normal launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// What the layer's own sequence lets the decode FFN do beyond moe_expert_ffn:
// start the shared-expert gate/up units before the routing is complete (the
// kernel before it neither reads nor writes their buffer), and write y in
// the down kernel (comb_ctl: H/128 zeroed tile counters; only when that
// launch is the last FFN launch of the forward).
struct DecodeFuse {
  void (*mark)(void*);  // called after each kernel launch (timing hook), or nullptr
  void* mark_ctx;
  const int4* act_meta;  // LookupArgs::meta of this forward, or nullptr
  bool shared_early;
  bool shared_gu_done;  // the shared expert's h is already in the workspace (one token)
  unsigned int* comb_ctl;
  const int32_t* inv;
  uint16_t* y;
  // the layer's control words for the one-launch decode FFN (zero before a
  // launch, left zero by it): ticket, done, shared h ready, pad, then one
  // h-ready count per act position (up to 1024); nullptr: two launches
  unsigned int* ffn_ctl;
  // the misses' records are gathered by the FFN itself (one staging group):
  // the cache and layer, the lookup's miss list, and the adaptive policy's
  // destination slots (nullptr: staging slot i mod n_stage)
  const expcache* g_cache;
  int g_layer;
  const int32_t* g_miss_ids;
  const int32_t* g_n_miss;
  const int32_t* g_dst_slots;
  // prefill: clear y_acc in the token quantisation; write y from the shared
  // expert's down GEMM (the call's last writer of y_acc), or nullptr
  bool pf_zero_y;
  uint16_t* pf_y;
  // two-launch decode FFN: 2 x 1024 counts (zero before a launch, left zero)
  // with which the down kernel's routed units start as soon as their expert's
  // h is written; nullptr: the down kernel waits for the gate/up kernel
  unsigned int* h_counts;
};

// the gather fields of one layer's records (cache.cu)
struct GatherArgs {
  const uint8_t* host;
  const int64_t* host_index;
  uint64_t host_records;
  int n_cache, n_stage, slot_lo, slot_hi;
};
void cache_gather_args(const expcache* c, int layer, GatherArgs* out);

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ((KArgs)args)...);
}

}  // namespace moe

// host-side error plumbing
#define MOE_CHECK_LAUNCH()                                          \
  do {                                                              \
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;     \
  } while (0)
