// Shared device helpers of the sm_103a sparse-reduction library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include <utility>

#include "sparcml.h"

namespace sparcml {

// Programmatic dependent launch. Kernels are launched with programmatic
// stream serialisation, so a kernel's grid may be set up while the previous
// kernel of the stream drains; every kernel's first statement waits for the
// previous grid to complete and its memory to be visible (a no-op when a
// kernel was launched without the attribute), so no kernel touches memory
// before its predecessor is done. No kernel triggers early: a dependent grid
// starts only once every block of the previous one has exited.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // a failure is recorded as the runtime's last error, read by launch_status()
  (void)cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// A named NVTX range over a C-ABI call: profilers (ncu --nvtx, nsys) group
// the call's kernels under the entry point's name. Free when no tool is
// attached (NVTX v3 is header-only).
struct ApiRange {
  explicit ApiRange(const char* name) { nvtxRangePushA(name); }
  ~ApiRange() { nvtxRangePop(); }
  ApiRange(const ApiRange&) = delete;
  ApiRange& operator=(const ApiRange&) = delete;
};

// Count of kernels launched by the library (see sparcml_launch_count).
void note_launches(uint64_t n);

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device; the runtime call is made once per (device, kernel, size).
bool ensure_smem(const void* func, size_t bytes);

// Workspace header: the status word at byte 0, the fault-injection word at
// byte kInjectOffset (written by sparcml_set_fault_injection, kept across
// calls). The word arms the injection only when it holds kInjectArmed, a
// pattern that a workspace left uninitialised is very unlikely to contain.
constexpr size_t kInjectOffset = 32;
constexpr uint8_t kInjectByte = 0xa5;
constexpr uint32_t kInjectArmed = 0xa5a5a5a5u;
// Polls of a bounded wait, normally and while a fault is injected (then a
// wait that nothing will end gives up within milliseconds).
constexpr uint32_t kSpinLimit = 1u << 21;
constexpr uint32_t kInjectSpinLimit = 1u << 12;

// Whether a fault is injected through this workspace word (nullptr: none).
__device__ __forceinline__ bool injected(const uint32_t* inject) {
  return inject != nullptr && *reinterpret_cast<const volatile uint32_t*>(inject) == kInjectArmed;
}

// Record the first device-side error in a status word (never traps).
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Magnitude key: IEEE bit pattern of |x|, ordered like |x| for non-NaN x.
__device__ __forceinline__ uint32_t mag_key(float x) {
  return __float_as_uint(x) & 0x7fffffffu;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive prefix over the warp of a small per-lane count c (0 <= c < 8),
// in lane order, from three ballots.
__device__ __forceinline__ uint32_t warp_excl_small(uint32_t c, uint32_t* total) {
  const uint32_t b0 = __ballot_sync(0xffffffffu, c & 1u);
  const uint32_t b1 = __ballot_sync(0xffffffffu, c & 2u);
  const uint32_t b2 = __ballot_sync(0xffffffffu, c & 4u);
  const uint32_t lt = lanemask_lt();
  *total = __popc(b0) + 2u * __popc(b1) + 4u * __popc(b2);
  return __popc(b0 & lt) + 2u * __popc(b1 & lt) + 4u * __popc(b2 & lt);
}

__device__ __forceinline__ uint32_t warp_incl_sum(uint32_t v) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, v, d);
    if (lane_id() >= (uint32_t)d) v += t;
  }
  return v;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Block-wide exclusive scan of one uint32 per thread. `scratch` holds at
// least 33 words of shared memory. Returns the exclusive prefix; *total gets
// the block sum. Contains two __syncthreads().
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch,
                                                    uint32_t* total) {
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t nwarps = (blockDim.x + 31) >> 5;
  const uint32_t incl = warp_incl_sum(v);
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < nwarps ? scratch[lane] : 0u;
    const uint32_t wi = warp_incl_sum(w);
    scratch[lane] = wi - w;
    if (lane == 31) scratch[32] = wi;
  }
  __syncthreads();
  *total = scratch[32];
  return scratch[warp] + incl - v;
}

// Histogram increment with warp aggregation: lanes that hit the same bin
// in one step add once, which keeps skewed key distributions from
// serialising on one shared-memory word.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
  const uint32_t am = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const uint32_t peers = __match_any_sync(am, bin);
  const uint32_t leader = __ffs(peers) - 1;
  if (lane_id() == leader) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

// SplitMix64 (Steele, Lea and Flood, OOPSLA 2014): the output for state x.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9e3779b97f4a7c15ull;
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

// L2 eviction-priority hints (PTX createpolicy / .L2::cache_hint). Data that
// a later kernel of the same step reads back (candidates, streams) is stored
// evict-last so the multi-GB streaming pass does not flush it from L2.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void st_keep(uint32_t* ptr, uint32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(ptr), "r"(v), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st_keep(float* ptr, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(pol)
               : "memory");
}

// Asynchronous 4-byte global -> shared copy (no register round trip).
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gmem) : "memory");
}
// 16-byte form: both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Read-only global loads that skip L1 allocation: data read exactly once.
__device__ __forceinline__ uint32_t ld_stream(const uint32_t* ptr) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(ptr));
  return v;
}
__device__ __forceinline__ float ld_stream(const float* ptr) {
  float v;
  asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
  return v;
}
__device__ __forceinline__ uint4 ld_stream(const uint4* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? SPARCML_OK : SPARCML_ERR_CUDA;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace sparcml
