// Pack, densify, status and launch bookkeeping of the sm_103a library.
//
// "SparCML: High-Performance Sparse Communication for Machine Learning",
// §5.1: data moves as sparse streams of index-value pairs and switches to
// a dense representation when that is cheaper. Pack turns a naturally sparse
// dense vector into a stream (threshold selection); densify is the reverse.

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"

namespace sparcml {
namespace {

std::atomic<uint64_t> g_launches{0};

constexpr uint32_t kPackChunk = 8192;
constexpr uint32_t kPackThreads = 256;
constexpr uint32_t kPackRounds = kPackChunk / (kPackThreads * 4);

// Count (WRITE = false) or write (WRITE = true) the entries |x| > thr of one
// chunk, in index order. Warp w owns chunk entries [1024 w, 1024 (w + 1)).
template <bool WRITE>
__global__ void __launch_bounds__(kPackThreads)
pack_chunk_kernel(const float* __restrict__ x, uint64_t N, uint32_t nchunk, float thr,
                  uint32_t* __restrict__ chunk_cnt, const uint32_t* __restrict__ chunk_off,
                  uint32_t* __restrict__ out_idx, float* __restrict__ out_val, uint64_t cap) {
  griddep_wait();
  __shared__ uint32_t warp_tot[kPackThreads / 32];
  const uint32_t p = blockIdx.x / nchunk, c = blockIdx.x % nchunk;
  const uint64_t start = (uint64_t)c * kPackChunk;
  const uint32_t nn = (uint32_t)min((uint64_t)kPackChunk, N - start);
  const float* xp = x + (uint64_t)p * N + start;
  const bool aligned = (reinterpret_cast<uintptr_t>(xp) & 15) == 0;
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  uint32_t mask = 0;
#pragma unroll
  for (uint32_t t = 0; t < kPackRounds; ++t) {
    const uint32_t e0 = 4 * (warp * (kPackRounds * 32) + t * 32 + lane);
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (aligned && e0 + 4 <= nn) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(xp + e0));
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q)
        if (e0 + q < nn) v[q] = xp[e0 + q];
    }
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q)
      if (e0 + q < nn && fabsf(v[q]) > thr) mask |= 1u << (4 * t + q);
  }
  const uint32_t wsum = warp_sum(__popc(mask));
  if (!WRITE) {
    if (lane == 0) warp_tot[warp] = wsum;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t s = 0;
      for (uint32_t w = 0; w < kPackThreads / 32; ++w) s += warp_tot[w];
      chunk_cnt[blockIdx.x] = s;
    }
    return;
  }
  if (lane == 0) warp_tot[warp] = wsum;
  __syncthreads();
  uint64_t run = chunk_off[blockIdx.x];
  for (uint32_t w = 0; w < warp; ++w) run += warp_tot[w];
  if (wsum == 0) return;
  const uint64_t base = (uint64_t)p * cap;
#pragma unroll
  for (uint32_t t = 0; t < kPackRounds; ++t) {
    const uint32_t bits = (mask >> (4 * t)) & 15u;
    uint32_t tot;
    uint64_t pos = run + warp_excl_small(__popc(bits), &tot);
    run += tot;
    const uint32_t e0 = 4 * (warp * (kPackRounds * 32) + t * 32 + lane);
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q)
      if (bits & (1u << q)) {
        if (pos < cap) {
          out_idx[base + pos] = (uint32_t)(start + e0 + q);
          out_val[base + pos] = xp[e0 + q];
        }
        ++pos;
      }
  }
}

// Exclusive scan of one node's chunk counts; nnz = min(total, cap).
__global__ void __launch_bounds__(1024)
pack_scan_kernel(const uint32_t* __restrict__ chunk_cnt, uint32_t nchunk,
                 uint32_t* __restrict__ chunk_off, uint32_t* __restrict__ out_nnz, uint64_t cap,
                 int32_t* status) {
  griddep_wait();
  __shared__ uint32_t scratch[34];
  const uint32_t p = blockIdx.x;
  const uint32_t* cc = chunk_cnt + (uint64_t)p * nchunk;
  uint32_t* co = chunk_off + (uint64_t)p * nchunk;
  uint64_t run = 0;
  for (uint32_t c0 = 0; c0 < nchunk; c0 += blockDim.x) {
    const uint32_t c = c0 + threadIdx.x;
    const uint32_t v = c < nchunk ? cc[c] : 0u;
    uint32_t tot;
    const uint32_t ex = block_excl_scan(v, scratch, &tot);
    if (c < nchunk) co[c] = (uint32_t)min(run + ex, (uint64_t)0xffffffffu);
    run += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    out_nnz[p] = (uint32_t)min(run, cap);
    if (run > cap) set_status(status, SPARCML_ERR_CAPACITY);
  }
}

__global__ void densify_zero_kernel(float* __restrict__ dense, uint64_t total) {
  griddep_wait();
  const bool vec = (reinterpret_cast<uintptr_t>(dense) & 15) == 0;
  const uint64_t nv = vec ? total / 4 : 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride)
    reinterpret_cast<float4*>(dense)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (uint64_t i = nv * 4 + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += stride)
    dense[i] = 0.0f;
}

__global__ void densify_scatter_kernel(const uint32_t* __restrict__ idx,
                                       const float* __restrict__ val,
                                       const uint32_t* __restrict__ nnz, int32_t P, uint64_t cap,
                                       uint64_t N, float* __restrict__ dense, int32_t* status) {
  griddep_wait();
  const uint64_t total = (uint64_t)P * cap;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t e = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
    const uint32_t p = (uint32_t)(e / cap);
    const uint64_t j = e % cap;
    const uint64_t n = min((uint64_t)nnz[p], cap);
    if (j >= n) continue;
    const uint32_t i = idx[e];
    if (i < N)
      dense[(uint64_t)p * N + i] = val[e];
    else
      set_status(status, SPARCML_ERR_BAD_STREAM);
  }
}

size_t pack_chunk_array_bytes(int32_t P, uint64_t N) {
  return align_up(4 * (size_t)P * ((N + kPackChunk - 1) / kPackChunk), 256);
}

}  // namespace

void note_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

bool ensure_smem(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = done[{dev, func}];
  if (have >= bytes) return true;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess)
    return false;
  have = bytes;
  return true;
}

}  // namespace sparcml

using namespace sparcml;

extern "C" const char* sparcml_status_string(int status) {
  switch (status) {
    case SPARCML_OK: return "SPARCML_OK";
    case SPARCML_ERR_INVALID_ARG: return "SPARCML_ERR_INVALID_ARG";
    case SPARCML_ERR_WORKSPACE: return "SPARCML_ERR_WORKSPACE";
    case SPARCML_ERR_CAPACITY: return "SPARCML_ERR_CAPACITY";
    case SPARCML_ERR_BAD_STREAM: return "SPARCML_ERR_BAD_STREAM";
    case SPARCML_ERR_NONFINITE: return "SPARCML_ERR_NONFINITE";
    case SPARCML_ERR_TIMEOUT: return "SPARCML_ERR_TIMEOUT";
    case SPARCML_ERR_CUDA: return "SPARCML_ERR_CUDA";
    default: return "SPARCML_ERR_UNKNOWN";
  }
}

extern "C" uint64_t sparcml_launch_count(void) {
  return g_launches.load(std::memory_order_relaxed);
}

extern "C" int sparcml_get_status(void* status_word, void* stream) {
  if (!status_word) return SPARCML_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPARCML_ERR_CUDA;
  int32_t h = 0;
  if (cudaMemcpy(&h, status_word, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPARCML_ERR_CUDA;
  if (h != 0 && cudaMemset(status_word, 0, sizeof h) != cudaSuccess) return SPARCML_ERR_CUDA;
  return h;
}

extern "C" int sparcml_set_fault_injection(void* ws, int32_t mode, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 || mode < 0 ||
      mode > SPARCML_INJECT_WITHHOLD_FIRST)
    return SPARCML_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(static_cast<char*>(ws) + kInjectOffset, mode ? kInjectByte : 0, 4, s) !=
      cudaSuccess)
    return SPARCML_ERR_CUDA;
  return SPARCML_OK;
}

extern "C" size_t sparcml_pack_workspace_size(int32_t P, uint64_t N) {
  if (P < 1 || P > 65535 || N < 1 || N > 0xffffffffull) return 0;
  return 256 + 2 * pack_chunk_array_bytes(P, N);
}

extern "C" int sparcml_pack(const float* x, int32_t P, uint64_t N, float thr, uint32_t* out_idx,
                            float* out_val, uint32_t* out_nnz, uint64_t cap, void* ws,
                            size_t ws_bytes, void* stream) {
  const ApiRange nvtx_range(__func__);
  if (!x || !out_idx || !out_val || !out_nnz || !ws || P < 1 || P > 65535 || N < 1 ||
      N > 0xffffffffull || !(thr >= 0.0f) || cap > 0xffffffffull)
    return SPARCML_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return SPARCML_ERR_INVALID_ARG;
  if (ws_bytes < sparcml_pack_workspace_size(P, N)) return SPARCML_ERR_WORKSPACE;
  const uint64_t nchunk = (N + kPackChunk - 1) / kPackChunk;
  if ((uint64_t)P * nchunk > 0x7fffffffull) return SPARCML_ERR_INVALID_ARG;
  char* w = static_cast<char*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  uint32_t* chunk_cnt = reinterpret_cast<uint32_t*>(w + 256);
  uint32_t* chunk_off = reinterpret_cast<uint32_t*>(w + 256 + pack_chunk_array_bytes(P, N));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned grid = (unsigned)((uint64_t)P * nchunk);
  launch_pdl(pack_chunk_kernel<false>, grid, kPackThreads, 0, s, x, N, (uint32_t)nchunk, thr,
             chunk_cnt, nullptr, nullptr, nullptr, cap);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  launch_pdl(pack_scan_kernel, (unsigned)P, 1024, 0, s, chunk_cnt, (uint32_t)nchunk, chunk_off,
             out_nnz, cap, status);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  launch_pdl(pack_chunk_kernel<true>, grid, kPackThreads, 0, s, x, N, (uint32_t)nchunk, thr,
             chunk_cnt, chunk_off, out_idx, out_val, cap);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  note_launches(3);
  return SPARCML_OK;
}

// Checked mode for inputs: any NaN or +-inf in x[0 .. n) records
// SPARCML_ERR_NONFINITE. Grid-stride over 16-byte quads of the aligned part
// (the unaligned head and the tail entry by entry); one vote per warp.
__global__ void __launch_bounds__(256) check_finite_kernel(const float* __restrict__ x,
                                                           uint64_t n, uint64_t head,
                                                           int32_t* status) {
  griddep_wait();
  const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  bool bad = false;
  auto nonfinite = [](float v) { return (__float_as_uint(v) & 0x7f800000u) == 0x7f800000u; };
  for (uint64_t i = tid; i < head; i += stride) bad |= nonfinite(x[i]);
  const uint64_t nq = (n - head) / 4;
  const float4* q4 = reinterpret_cast<const float4*>(x + head);
  for (uint64_t i = tid; i < nq; i += stride) {
    const float4 v = q4[i];
    bad |= nonfinite(v.x) | nonfinite(v.y) | nonfinite(v.z) | nonfinite(v.w);
  }
  for (uint64_t i = head + 4 * nq + tid; i < n; i += stride) bad |= nonfinite(x[i]);
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31u) == 0)
    set_status(status, SPARCML_ERR_NONFINITE);
}

extern "C" int sparcml_check_finite(const float* x, uint64_t n, int32_t* status, void* stream) {
  const ApiRange nvtx_range(__func__);
  if (!status || (n > 0 && !x)) return SPARCML_ERR_INVALID_ARG;
  if (n == 0) return SPARCML_OK;
  // entries before the first 16-byte boundary (x is at least 4-byte aligned)
  const uint64_t mis = (reinterpret_cast<uintptr_t>(x) & 15u) / 4u;
  const uint64_t head = std::min<uint64_t>(n, mis ? 4 - mis : 0);
  const unsigned grid = (unsigned)std::min<uint64_t>((n / 4 + 255) / 256 + 1, 152u * 8u);
  launch_pdl(check_finite_kernel, grid, 256, 0, static_cast<cudaStream_t>(stream), x, n, head,
             status);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  note_launches(1);
  return SPARCML_OK;
}

extern "C" int sparcml_densify(const uint32_t* idx, const float* val, const uint32_t* nnz,
                               int32_t P, uint64_t cap, uint64_t N, float* dense, int32_t* status,
                               void* stream) {
  const ApiRange nvtx_range(__func__);
  if (!idx || !val || !nnz || !dense || P < 1 || P > 65535 || N < 1 || N > 0xffffffffull)
    return SPARCML_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t total = (uint64_t)P * N;
  const unsigned zgrid = (unsigned)std::min<uint64_t>((total / 4 + 255) / 256 + 1, 152u * 16u);
  launch_pdl(densify_zero_kernel, zgrid, 256, 0, s, dense, total);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  note_launches(1);
  if (cap == 0) return SPARCML_OK;
  const uint64_t entries = (uint64_t)P * cap;
  const unsigned sgrid = (unsigned)std::min<uint64_t>((entries + 255) / 256, 152u * 16u);
  launch_pdl(densify_scatter_kernel, sgrid, 256, 0, s, idx, val, nnz, P, cap, N, dense, status);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  note_launches(1);
  return SPARCML_OK;
}
