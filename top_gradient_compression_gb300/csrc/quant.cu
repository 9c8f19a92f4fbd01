// b-bit (2, 4, 8) stochastic quantisation of stream values or dense rows and
// its inverse, sm_103a.
//
// "SparCML: High-Performance Sparse Communication for Machine Learning",
// §2.2 (quantisation Q is an element-wise stochastic operator whose noise
// has zero mean) and §6 (QSGD: buckets of entries quantised independently,
// packed low-precision items plus one full-precision scale per bucket; 2-,
// 4- and 8-bit outputs). Code: sign bit plus a (b-1)-bit level in 0..s,
// s = 2^(b-1) - 1 (1, 7, 127), of the bucket's max |v|; 8/b codes per byte,
// the earliest entry in the lowest bits.
//
// Two passes: one warp per bucket takes the scale (a warp max-reduction),
// then one thread per 32-bit word of codes encodes its 4 * 8/b entries.
// The rounding draw for an entry is SplitMix64 keyed by (seed, node, index),
// so it does not depend on which thread or launch handles the entry.

#include <algorithm>

#include "common.cuh"

namespace sparcml {
namespace {

constexpr uint32_t kQuantThreads = 256;

// level / s as the correctly rounded fp32 quotient: selects on constant
// quotients for s = 7, the level itself for s = 1, an IEEE division else.
template <int BITS>
__device__ __forceinline__ float level_over_s(uint32_t level) {
  if constexpr (BITS == 2) {
    return (float)level;
  } else if constexpr (BITS == 4) {
    const float lo = (level & 2u) ? ((level & 1u) ? 3.0f / 7.0f : 2.0f / 7.0f)
                                  : ((level & 1u) ? 1.0f / 7.0f : 0.0f);
    const float hi = (level & 2u) ? ((level & 1u) ? 7.0f / 7.0f : 6.0f / 7.0f)
                                  : ((level & 1u) ? 5.0f / 7.0f : 4.0f / 7.0f);
    return (level & 4u) ? hi : lo;
  } else {
    return __fdiv_rn((float)level, 127.0f);
  }
}

template <int BITS>
__device__ __forceinline__ float decode(uint32_t code, float scale) {
  constexpr uint32_t kS = (1u << (BITS - 1)) - 1u;
  const uint32_t level = code & kS;
  if (level == 0) return 0.0f;
  const float v = __fmul_rn(level_over_s<BITS>(level), scale);
  return (code >> (BITS - 1)) ? -v : v;
}

// Code of v: sign << (BITS-1) | level, level = floor(r) rounded up with
// probability frac(r), r = (|v| / scale) * s, the draw keyed by the index.
template <int BITS>
__device__ __forceinline__ uint32_t encode(float v, uint64_t index, float scale,
                                           uint64_t node_mix) {
  constexpr uint32_t kS = (1u << (BITS - 1)) - 1u;
  uint32_t level = 0;
  if (scale > 0.0f) {
    const float r = __fmul_rn(__fdiv_rn(fabsf(v), scale), (float)kS);
    const float f = floorf(r);
    const float frac = __fsub_rn(r, f);
    const uint64_t h = splitmix64(node_mix ^ index);
    const float u = __fmul_rn((float)(uint32_t)(h >> 40), 1.0f / 16777216.0f);
    level = (uint32_t)f + (u < frac ? 1u : 0u);
    level = min(level, kS);
  }
  return (v < 0.0f ? 1u << (BITS - 1) : 0u) | level;
}

// Pass 1, one warp per bucket: scale = max |v| over the bucket.
__global__ void __launch_bounds__(kQuantThreads)
quantize_scale_kernel(const float* __restrict__ val, const uint32_t* __restrict__ nnz, int32_t P,
                      uint64_t cap, uint32_t bucket, uint32_t nbk, float* __restrict__ scales,
                      uint64_t scale_stride, int32_t* status) {
  griddep_wait();
  const uint64_t gw = (uint64_t)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5);
  if (gw >= (uint64_t)P * nbk) return;  // warp-uniform
  const uint32_t p = (uint32_t)(gw / nbk), b = (uint32_t)(gw % nbk);
  const uint32_t lane = lane_id();
  uint64_t n = nnz ? (uint64_t)nnz[p] : cap;
  if (n > cap) {
    if (lane == 0 && b == 0) set_status(status, SPARCML_ERR_CAPACITY);
    n = cap;
  }
  const uint64_t b0 = (uint64_t)b * bucket;
  if (b0 >= n) return;
  const uint64_t b1 = min(b0 + bucket, n);
  const float* vp = val + (uint64_t)p * cap;
  float m = 0.0f;
  for (uint64_t j = b0 + lane; j < b1; j += 32) m = fmaxf(m, fabsf(vp[j]));
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  if (lane == 0) scales[(uint64_t)p * scale_stride + b] = m;
}

// Pass 1 for aligned rows and buckets of 128 * VPL entries: each lane issues
// its VPL float4 loads together (a latency chain of one load, not 32).
template <int VPL>
__global__ void __launch_bounds__(kQuantThreads)
quantize_scale_vec_kernel(const float* __restrict__ val, const uint32_t* __restrict__ nnz,
                          int32_t P, uint64_t cap, uint32_t nbk, float* __restrict__ scales,
                          uint64_t scale_stride, int32_t* status) {
  griddep_wait();
  constexpr uint32_t kBucket = 128 * VPL;
  const uint64_t gw = (uint64_t)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5);
  if (gw >= (uint64_t)P * nbk) return;  // warp-uniform
  const uint32_t p = (uint32_t)(gw / nbk), b = (uint32_t)(gw % nbk);
  const uint32_t lane = lane_id();
  uint64_t n = nnz ? (uint64_t)nnz[p] : cap;
  if (n > cap) {
    if (lane == 0 && b == 0) set_status(status, SPARCML_ERR_CAPACITY);
    n = cap;
  }
  const uint64_t b0 = (uint64_t)b * kBucket;
  if (b0 >= n) return;
  const uint64_t b1 = min(b0 + kBucket, n);
  const float4* vp = reinterpret_cast<const float4*>(val + (uint64_t)p * cap + b0);
  float4 v[VPL];
#pragma unroll
  for (int k = 0; k < VPL; ++k) {
    const uint64_t j = b0 + 4ull * (lane + 32u * k);
    v[k] = j < b1 ? vp[lane + 32 * k] : make_float4(0.f, 0.f, 0.f, 0.f);  // inside the row
  }
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < VPL; ++k) {
    const uint64_t j = b0 + 4ull * (lane + 32u * k);
    // entries past the row's end (the float4 holding its last entry) do not count
    const float e[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (j + t < b1) m = fmaxf(m, fabsf(e[t]));
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  if (lane == 0) scales[(uint64_t)p * scale_stride + b] = m;
}

// Pass 2, one thread per 32-bit word of codes: four bytes, each 8/BITS entries
// of one bucket (a bucket is a whole number of bytes), encoded against the
// bucket's scale; the word is stored whole when all four bytes hold entries.
// idx == nullptr: dense rows (the position is the rounding key); nnz ==
// nullptr: full rows.
template <int BITS>
__global__ void __launch_bounds__(kQuantThreads)
quantize_encode_kernel(const uint32_t* __restrict__ idx, const float* __restrict__ val,
                       const uint32_t* __restrict__ nnz, uint64_t cap, uint32_t bucket_shift,
                       uint32_t bucket, uint64_t seed, uint8_t* __restrict__ codes,
                       const float* __restrict__ scales, float* __restrict__ err_out,
                       uint32_t code_stride, uint64_t scale_stride) {
  griddep_wait();
  constexpr uint32_t kPer = 8 / BITS;
  const uint32_t p = blockIdx.y;  // grid: (code words of a row, node)
  __shared__ uint64_t mix;        // the node's part of the draw key, once per CTA
  if (threadIdx.x == 0) mix = splitmix64(splitmix64(seed) ^ (uint64_t)p);
  __syncthreads();
  const uint64_t node_mix = mix;
  const uint32_t n = nnz ? (uint32_t)min((uint64_t)nnz[p], cap) : (uint32_t)cap;
  const uint64_t row = (uint64_t)p * cap;
  const float* sp = scales + (uint64_t)p * scale_stride;
  uint8_t* cp = codes + (uint64_t)p * code_stride;
  const bool aligned = (reinterpret_cast<uintptr_t>(cp) & 3) == 0;
  // 128-bit loads of a word's entries: rows 16-byte aligned, power-of-two
  // buckets, no error output
  const bool vrow = aligned && err_out == nullptr && bucket_shift < 32 &&
                    ((reinterpret_cast<uintptr_t>(val + row) |
                      (idx ? reinterpret_cast<uintptr_t>(idx + row) : 0)) & 15) == 0;
  constexpr uint32_t kE = 4 * kPer;  // entries of one word of codes
  const uint32_t nwords = (code_stride + 3) / 4;
  // each thread: one 32-bit word of codes (4 bytes, 4 * kPer entries)
  for (uint32_t w = blockIdx.x * blockDim.x + threadIdx.x; w < nwords;
       w += gridDim.x * blockDim.x) {
    const uint32_t q0 = 4 * w;
    if (q0 * kPer >= n) break;  // bytes past the row's entries stay untouched
    const uint32_t j0 = q0 * kPer;  // a multiple of 4
    if (vrow && q0 + 4 <= code_stride && j0 + kE <= n &&
        (j0 >> bucket_shift) == ((j0 + kE - 1) >> bucket_shift)) {
      // The word's entries all lie in the row and in one bucket: one scale,
      // 128-bit loads, no per-entry checks; the same codes as below.
      const float m = sp[j0 >> bucket_shift];
      float v[kE];
      uint32_t key[kE];
#pragma unroll
      for (uint32_t i = 0; i < kE / 4; ++i) {
        const float4 f = *reinterpret_cast<const float4*>(val + row + j0 + 4 * i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
        if (idx) {
          const uint4 q = *reinterpret_cast<const uint4*>(idx + row + j0 + 4 * i);
          key[4 * i] = q.x;
          key[4 * i + 1] = q.y;
          key[4 * i + 2] = q.z;
          key[4 * i + 3] = q.w;
        } else {
#pragma unroll
          for (uint32_t c = 0; c < 4; ++c) key[4 * i + c] = j0 + 4 * i + c;
        }
      }
      uint32_t word = 0;
#pragma unroll
      for (uint32_t e = 0; e < kE; ++e)
        word |= encode<BITS>(v[e], (uint64_t)key[e], m, node_mix) << (e * BITS);
      *reinterpret_cast<uint32_t*>(cp + q0) = word;
      continue;
    }
    uint32_t word = 0;
#pragma unroll
    for (uint32_t b = 0; b < 4; ++b) {
      const uint32_t j0 = (q0 + b) * kPer;
      if (q0 + b < code_stride && j0 < n) {
        const float m = sp[bucket_shift < 32 ? j0 >> bucket_shift : j0 / bucket];
        uint32_t byte = 0;
#pragma unroll
        for (uint32_t k = 0; k < kPer; ++k) {
          const uint32_t j = j0 + k;
          if (j < n) {
            const float v = val[row + j];
            const uint32_t c = encode<BITS>(v, idx ? (uint64_t)idx[row + j] : (uint64_t)j, m, node_mix);
            byte |= c << (k * BITS);
            if (err_out) err_out[row + j] = __fsub_rn(v, decode<BITS>(c, m));
          }
        }
        word |= byte << (8 * b);
      }
    }
    if (aligned && q0 + 4 <= code_stride && (q0 + 3) * kPer < n) {
      *reinterpret_cast<uint32_t*>(cp + q0) = word;  // all four bytes hold entries
    } else {
#pragma unroll
      for (uint32_t b = 0; b < 4; ++b)
        if (q0 + b < code_stride && (q0 + b) * kPer < n) cp[q0 + b] = (uint8_t)(word >> (8 * b));
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kQuantThreads)
dequantize_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                  const uint32_t* __restrict__ nnz, int32_t P, uint64_t cap, uint32_t bucket,
                  uint64_t code_stride, uint64_t scale_stride, float* __restrict__ out,
                  int32_t* status) {
  griddep_wait();
  constexpr uint32_t kPer = 8 / BITS;
  const uint64_t total = (uint64_t)P * code_stride;
  for (uint64_t q = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total;
       q += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t p = (uint32_t)(q / code_stride);
    const uint64_t j0 = (q % code_stride) * kPer;
    uint64_t n = nnz ? (uint64_t)nnz[p] : cap;
    if (n > cap) {
      if (j0 == 0) set_status(status, SPARCML_ERR_CAPACITY);
      n = cap;
    }
    if (j0 >= n) continue;
    const uint32_t byte = codes[q];
    const float* sp = scales + (uint64_t)p * scale_stride;
    float* op = out + (uint64_t)p * cap;
#pragma unroll
    for (uint32_t k = 0; k < kPer; ++k) {
      const uint64_t j = j0 + k;
      if (j < n) op[j] = decode<BITS>((byte >> (k * BITS)) & ((1u << BITS) - 1u), sp[j / bucket]);
    }
  }
}

bool valid_width(uint32_t bits, uint32_t bucket) {
  if (bits != 2 && bits != 4 && bits != 8) return false;
  return bucket >= 1 && bucket % (8 / bits) == 0;
}

int launch_quantize(const uint32_t* idx, const float* val, const uint32_t* nnz, int32_t P,
                    uint64_t cap, uint32_t bucket, uint32_t bits, uint64_t seed, uint8_t* codes,
                    float* scales, float* err_out, int32_t* status, void* stream) {
  if (!val || !codes || !scales || P < 1 || P > 65535 || cap < 1 || cap > 0xffffffffull ||
      !valid_width(bits, bucket))
    return SPARCML_ERR_INVALID_ARG;
  const uint64_t nbk = (cap + bucket - 1) / bucket;
  const uint64_t warps = (uint64_t)P * nbk;
  const uint64_t blocks = (warps + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
  if (nbk > 0xffffffffull || blocks > 0x7fffffffull) return SPARCML_ERR_INVALID_ARG;
  const uint64_t per = 8 / bits, code_stride = (cap + per - 1) / per;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool vec = (bucket == 512 || bucket == 1024) && cap % 4 == 0 &&
                   (reinterpret_cast<uintptr_t>(val) & 15) == 0;
  if (vec && bucket == 512)
    launch_pdl(quantize_scale_vec_kernel<4>, (unsigned)blocks, kQuantThreads, 0, s, val, nnz, P,
               cap, (uint32_t)nbk, scales, nbk, status);
  else if (vec)
    launch_pdl(quantize_scale_vec_kernel<8>, (unsigned)blocks, kQuantThreads, 0, s, val, nnz, P,
               cap, (uint32_t)nbk, scales, nbk, status);
  else
    launch_pdl(quantize_scale_kernel, (unsigned)blocks, kQuantThreads, 0, s, val, nnz, P, cap,
               bucket, (uint32_t)nbk, scales, nbk, status);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  const uint32_t shift = (bucket & (bucket - 1)) == 0 ? (uint32_t)__builtin_ctz(bucket) : 32u;
  const uint64_t code_words = (code_stride + 3) / 4;
  const dim3 eg((unsigned)std::min<uint64_t>((code_words + kQuantThreads - 1) / kQuantThreads,
                                             std::max<uint64_t>(1, 152u * 64u / (uint64_t)P)),
                (unsigned)P);
  const uint32_t cs = (uint32_t)code_stride;
  if (bits == 2)
    launch_pdl(quantize_encode_kernel<2>, eg, kQuantThreads, 0, s, idx, val, nnz, cap, shift,
               bucket, seed, codes, scales, err_out, cs, nbk);
  else if (bits == 4)
    launch_pdl(quantize_encode_kernel<4>, eg, kQuantThreads, 0, s, idx, val, nnz, cap, shift,
               bucket, seed, codes, scales, err_out, cs, nbk);
  else
    launch_pdl(quantize_encode_kernel<8>, eg, kQuantThreads, 0, s, idx, val, nnz, cap, shift,
               bucket, seed, codes, scales, err_out, cs, nbk);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  note_launches(2);
  return SPARCML_OK;
}

int launch_dequantize(const uint8_t* codes, const float* scales, const uint32_t* nnz,
                      int32_t P, uint64_t cap, uint32_t bucket, uint32_t bits, float* val_out,
                      int32_t* status, void* stream) {
  if (!codes || !scales || !val_out || P < 1 || P > 65535 || cap < 1 ||
      cap > 0xffffffffull || !valid_width(bits, bucket))
    return SPARCML_ERR_INVALID_ARG;
  const uint64_t per = 8 / bits, code_stride = (cap + per - 1) / per;
  const uint64_t total = (uint64_t)P * code_stride;
  const unsigned blocks =
      (unsigned)std::min<uint64_t>((total + kQuantThreads - 1) / kQuantThreads, 152u * 32u);
  const uint64_t scale_stride = (cap + bucket - 1) / bucket;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (bits == 2)
    launch_pdl(dequantize_kernel<2>, blocks, kQuantThreads, 0, s, codes, scales, nnz, P, cap,
               bucket, code_stride, scale_stride, val_out, status);
  else if (bits == 4)
    launch_pdl(dequantize_kernel<4>, blocks, kQuantThreads, 0, s, codes, scales, nnz, P, cap,
               bucket, code_stride, scale_stride, val_out, status);
  else
    launch_pdl(dequantize_kernel<8>, blocks, kQuantThreads, 0, s, codes, scales, nnz, P, cap,
               bucket, code_stride, scale_stride, val_out, status);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  note_launches(1);
  return SPARCML_OK;
}

}  // namespace
}  // namespace sparcml

using namespace sparcml;

extern "C" int sparcml_quantize4(const uint32_t* idx, const float* val, const uint32_t* nnz,
                                 int32_t P, uint64_t cap, uint32_t bucket, uint64_t seed,
                                 uint8_t* codes, float* scales, int32_t* status, void* stream) {
  const ApiRange nvtx_range(__func__);
  if (!idx || !nnz || bucket < 2 || (bucket & 1)) return SPARCML_ERR_INVALID_ARG;
  return launch_quantize(idx, val, nnz, P, cap, bucket, 4, seed, codes, scales, nullptr, status,
                         stream);
}

extern "C" int sparcml_dequantize4(const uint8_t* codes, const float* scales, const uint32_t* nnz,
                                   int32_t P, uint64_t cap, uint32_t bucket, float* val_out,
                                   int32_t* status, void* stream) {
  const ApiRange nvtx_range(__func__);
  if (!nnz || bucket < 2 || (bucket & 1)) return SPARCML_ERR_INVALID_ARG;
  return launch_dequantize(codes, scales, nnz, P, cap, bucket, 4, val_out, status, stream);
}

extern "C" int sparcml_quantize(const uint32_t* idx, const float* val, const uint32_t* nnz,
                                int32_t P, uint64_t cap, uint32_t bucket, uint32_t bits,
                                uint64_t seed, uint8_t* codes, float* scales, float* err_out,
                                int32_t* status, void* stream) {
  const ApiRange nvtx_range(__func__);
  return launch_quantize(idx, val, nnz, P, cap, bucket, bits, seed, codes, scales, err_out,
                         status, stream);
}

extern "C" int sparcml_dequantize(const uint8_t* codes, const float* scales, const uint32_t* nnz,
                                  int32_t P, uint64_t cap, uint32_t bucket, uint32_t bits,
                                  float* val_out, int32_t* status, void* stream) {
  const ApiRange nvtx_range(__func__);
  return launch_dequantize(codes, scales, nnz, P, cap, bucket, bits, val_out, status, stream);
}
