// 4-bit stochastic quantisation of stream values and its inverse, sm_103a.
//
// "SparCML: High-Performance Sparse Communication for Machine Learning",
// §2.2 (quantisation Q is an element-wise stochastic operator whose noise
// has zero mean) and §6 (QSGD: buckets of entries quantised independently,
// packed low-precision items plus one full-precision scale per bucket; 2-,
// 4- and 8-bit outputs). This file provides the 4-bit form: sign bit plus a
// 3-bit level in 0..7 of the bucket's max |v|.
//
// One warp per bucket: a warp max-reduction gives the scale, then each lane
// encodes pairs of entries into one byte (even entry in the low nibble).
// The rounding draw for an entry is SplitMix64 keyed by (seed, node, index),
// so it does not depend on which thread or launch handles the entry.

#include <algorithm>

#include "common.cuh"

namespace sparcml {
namespace {

constexpr uint32_t kQuantThreads = 256;

__device__ __forceinline__ uint32_t encode4(float v, uint32_t i, float scale, uint64_t node_mix) {
  uint32_t level = 0;
  if (scale > 0.0f) {
    const float r = __fmul_rn(__fdiv_rn(fabsf(v), scale), 7.0f);
    const float f = floorf(r);
    const float frac = __fsub_rn(r, f);
    const uint64_t h = splitmix64(node_mix ^ (uint64_t)i);
    const float u = __fmul_rn((float)(uint32_t)(h >> 40), 1.0f / 16777216.0f);
    level = (uint32_t)f + (u < frac ? 1u : 0u);
    level = min(level, 7u);
  }
  return (v < 0.0f ? 8u : 0u) | level;
}

__global__ void __launch_bounds__(kQuantThreads)
quantize4_kernel(const uint32_t* __restrict__ idx, const float* __restrict__ val,
                 const uint32_t* __restrict__ nnz, int32_t P, uint64_t cap, uint32_t bucket,
                 uint32_t nbk, uint64_t seed, uint8_t* __restrict__ codes,
                 float* __restrict__ scales, uint64_t code_stride, uint64_t scale_stride,
                 int32_t* status) {
  const uint64_t gw = (uint64_t)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5);
  if (gw >= (uint64_t)P * nbk) return;  // warp-uniform
  const uint32_t p = (uint32_t)(gw / nbk), b = (uint32_t)(gw % nbk);
  const uint32_t lane = lane_id();
  uint64_t n = nnz[p];
  if (n > cap) {
    if (lane == 0 && b == 0) set_status(status, SPARCML_ERR_CAPACITY);
    n = cap;
  }
  const uint64_t b0 = (uint64_t)b * bucket;
  if (b0 >= n) return;
  const uint64_t b1 = min(b0 + bucket, n);
  const float* vp = val + (uint64_t)p * cap;
  const uint32_t* ip = idx + (uint64_t)p * cap;
  float m = 0.0f;
  for (uint64_t j = b0 + lane; j < b1; j += 32) m = fmaxf(m, fabsf(vp[j]));
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  if (lane == 0) scales[(uint64_t)p * scale_stride + b] = m;
  const uint64_t node_mix = splitmix64(splitmix64(seed) ^ (uint64_t)p);
  uint8_t* cp = codes + (uint64_t)p * code_stride;
  for (uint64_t j = b0 + 2 * lane; j < b1; j += 64) {
    const uint32_t c0 = encode4(vp[j], ip[j], m, node_mix);
    const uint32_t c1 = j + 1 < b1 ? encode4(vp[j + 1], ip[j + 1], m, node_mix) : 0u;
    cp[j >> 1] = (uint8_t)(c0 | (c1 << 4));
  }
}

__device__ __forceinline__ float decode4(uint32_t code, float scale) {
  const uint32_t level = code & 7u;
  if (level == 0) return 0.0f;
  const float v = __fmul_rn(__fdiv_rn((float)level, 7.0f), scale);
  return (code & 8u) ? -v : v;
}

__global__ void __launch_bounds__(kQuantThreads)
dequantize4_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                   const uint32_t* __restrict__ nnz, int32_t P, uint64_t cap, uint32_t bucket,
                   uint64_t code_stride, uint64_t scale_stride, float* __restrict__ out,
                   int32_t* status) {
  const uint64_t total = (uint64_t)P * code_stride;
  for (uint64_t q = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total;
       q += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t p = (uint32_t)(q / code_stride);
    const uint64_t j = (q % code_stride) * 2;
    uint64_t n = nnz[p];
    if (n > cap) {
      if (j == 0) set_status(status, SPARCML_ERR_CAPACITY);
      n = cap;
    }
    if (j >= n) continue;
    const uint8_t byte = codes[q];
    const float* sp = scales + (uint64_t)p * scale_stride;
    float* op = out + (uint64_t)p * cap;
    op[j] = decode4(byte & 15u, sp[j / bucket]);
    if (j + 1 < n) op[j + 1] = decode4(byte >> 4, sp[(j + 1) / bucket]);
  }
}

}  // namespace
}  // namespace sparcml

using namespace sparcml;

extern "C" int sparcml_quantize4(const uint32_t* idx, const float* val, const uint32_t* nnz,
                                 int32_t P, uint64_t cap, uint32_t bucket, uint64_t seed,
                                 uint8_t* codes, float* scales, int32_t* status, void* stream) {
  if (!idx || !val || !nnz || !codes || !scales || P < 1 || P > 65535 || cap < 1 ||
      cap > 0xffffffffull || bucket < 2 || (bucket & 1))
    return SPARCML_ERR_INVALID_ARG;
  const uint64_t nbk = (cap + bucket - 1) / bucket;
  const uint64_t warps = (uint64_t)P * nbk;
  const uint64_t blocks = (warps + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
  if (nbk > 0xffffffffull || blocks > 0x7fffffffull) return SPARCML_ERR_INVALID_ARG;
  quantize4_kernel<<<(unsigned)blocks, kQuantThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      idx, val, nnz, P, cap, bucket, (uint32_t)nbk, seed, codes, scales, (cap + 1) / 2, nbk,
      status);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  note_launches(1);
  return SPARCML_OK;
}

extern "C" int sparcml_dequantize4(const uint8_t* codes, const float* scales, const uint32_t* nnz,
                                   int32_t P, uint64_t cap, uint32_t bucket, float* val_out,
                                   int32_t* status, void* stream) {
  if (!codes || !scales || !nnz || !val_out || P < 1 || P > 65535 || cap < 1 ||
      cap > 0xffffffffull || bucket < 2 || (bucket & 1))
    return SPARCML_ERR_INVALID_ARG;
  const uint64_t code_stride = (cap + 1) / 2;
  const uint64_t total = (uint64_t)P * code_stride;
  const uint64_t blocks = std::min<uint64_t>((total + kQuantThreads - 1) / kQuantThreads, 152u * 32u);
  dequantize4_kernel<<<(unsigned)blocks, kQuantThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      codes, scales, nnz, P, cap, bucket, code_stride, (cap + bucket - 1) / bucket, val_out,
      status);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  note_launches(1);
  return SPARCML_OK;
}
