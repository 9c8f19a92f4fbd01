// Static sparse allreduce by recursive doubling (SSAR), emulated on one GPU,
// sm_103a.
//
// "SparCML: High-Performance Sparse Communication for Machine Learning",
// §5.3.1: in log2(P) stages every node combines its sparse partial result
// with the one of node i XOR 2^s; fully overlapping indices keep the
// intermediate results at k items, disjoint ones grow them at every stage.
// Here the P nodes share one HBM, so both partners' identical results are
// kept once: stage s holds P / 2^(s+1) partial results. Combining the lower
// group's partial result A with the upper group's B is the two-stream sum
// reduce: (+0.0f + a) + b for an index in both, +0.0f + v otherwise. The
// result stays sparse at every stage (static sparse).
//
// One stage is two kernels over all of its pairs at once, with work
// proportional to the entries, not to N:
//   ssar_partition_kernel  merge-path splits of every pair's merged sequence
//                          into chunks of kChunk positions (one warp per
//                          split, 33-ary search on the sorted streams);
//   ssar_merge_kernel      one CTA per chunk: both sub-ranges staged in
//                          shared memory, each thread merges its positions
//                          (equal indices from A and B combine), then the
//                          chunk's offset comes from a decoupled look-back
//                          along its pair's chunks and the merged entries are
//                          written in index order.

#include <algorithm>

#include "common.cuh"

namespace sparcml {
namespace {

constexpr uint32_t kChunk = 2048;        // merged positions per CTA
constexpr uint32_t kMergeThreads = 256;  // kChunk / kMergeThreads positions per thread
constexpr uint32_t kPerThread = kChunk / kMergeThreads;
constexpr unsigned long long kAggFlag = 1ull << 62;
constexpr unsigned long long kIncFlag = 2ull << 62;

struct Pair {
  const uint32_t* a_idx;
  const float* a_val;
  const uint32_t* b_idx;
  const float* b_val;
  uint32_t na, nb;
};

struct StageArgs {
  const uint32_t* in_idx;  // [2G][cap_in]
  const float* in_val;
  const uint32_t* in_nnz;  // [2G]
  uint64_t cap_in;
  uint32_t G;
  uint32_t chunks;          // chunk slots per pair (capacity bound)
  uint32_t N;
  uint32_t* out_idx;        // [G][cap_out]
  float* out_val;
  uint32_t* out_nnz;        // [G]
  uint64_t cap_out;
  uint32_t* split;          // [G][chunks + 1] A-count at each chunk boundary (B = d - A, adjusted)
  uint32_t* split_b;        // [G][chunks + 1]
  unsigned long long* state;  // [G][chunks] look-back words
  uint32_t* ticket;
  unsigned long long* fill;   // stage fill-in (may be null)
  int32_t* status;
  const uint32_t* inject;    // the workspace's fault-injection word
  bool validate;            // stage 0: check the caller's streams
};

__device__ __forceinline__ Pair pair_of(const StageArgs& s, uint32_t g) {
  Pair q;
  const uint64_t ra = (uint64_t)(2 * g) * s.cap_in, rb = ra + s.cap_in;
  q.a_idx = s.in_idx + ra;
  q.a_val = s.in_val + ra;
  q.b_idx = s.in_idx + rb;
  q.b_val = s.in_val + rb;
  q.na = (uint32_t)min((uint64_t)s.in_nnz[2 * g], s.cap_in);
  q.nb = (uint32_t)min((uint64_t)s.in_nnz[2 * g + 1], s.cap_in);
  return q;
}

// Merge-path split at diagonal d (A-first on equal keys): the number i of A
// entries among the first d merged positions, i.e. the first i in
// [max(0, d - nb), min(d, na)] with !(A[i] <= B[d - 1 - i]). Then a pair of
// equal keys cut by the split (A[i-1] == B[d-i]) is kept whole on the left:
// the B side moves one past it. Warp-cooperative 33-ary search; all lanes
// return (i, j).
__device__ void merge_split(const uint32_t* A, uint32_t na, const uint32_t* B, uint32_t nb,
                            uint32_t d, uint32_t* oi, uint32_t* oj) {
  const uint32_t lane = lane_id();
  uint32_t lo = d > nb ? d - nb : 0u, hi = min(d, na);  // answer in [lo, hi]
  while (hi - lo > 32) {
    const uint32_t span = hi - lo;
    const uint32_t pos = lo + (uint32_t)((uint64_t)span * (lane + 1) / 33);
    const bool take = A[pos] <= B[d - 1 - pos];  // A[pos] goes before B[d-1-pos]
    const uint32_t c = __popc(__ballot_sync(0xffffffffu, take));
    const uint32_t nlo = c ? lo + (uint32_t)((uint64_t)span * c / 33) + 1 : lo;
    const uint32_t nhi = c < 32 ? lo + (uint32_t)((uint64_t)span * (c + 1) / 33) : hi;
    lo = nlo;
    hi = nhi;
  }
  const uint32_t pos = lo + lane;
  const bool take = pos < hi && A[pos] <= B[d - 1 - pos];
  const uint32_t i = lo + __popc(__ballot_sync(0xffffffffu, take));
  uint32_t j = d - i;
  if (i > 0 && j < nb && A[i - 1] == B[j]) ++j;
  *oi = i;
  *oj = j;
}

// One warp per (pair, boundary c in 0..chunks): split at min(c * kChunk, na + nb).
__global__ void __launch_bounds__(256) ssar_partition_kernel(StageArgs s) {
  griddep_wait();
  const uint64_t w = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint64_t per = (uint64_t)s.chunks + 1;
  if (w >= (uint64_t)s.G * per) return;  // warp-uniform
  const uint32_t g = (uint32_t)(w / per), c = (uint32_t)(w % per);
  const Pair q = pair_of(s, g);
  const uint32_t total = q.na + q.nb;
  const uint32_t d = (uint32_t)min((uint64_t)c * kChunk, (uint64_t)total);
  uint32_t i, j;
  merge_split(q.a_idx, q.na, q.b_idx, q.nb, d, &i, &j);
  if (lane_id() == 0) {
    s.split[(uint64_t)g * per + c] = i;
    s.split_b[(uint64_t)g * per + c] = j;
  }
}

// Look-back along a pair's chunks (warp 0 of the CTA): returns the exclusive
// offset and publishes the inclusive one. Bounded waits.
__device__ uint32_t chunk_lookback(const StageArgs& s, uint64_t slot0, uint32_t c, uint32_t count) {
  const uint32_t lane = lane_id();
  unsigned long long* st = s.state + slot0;
  // an injected fault: each pair's first chunk withholds its flag and every
  // wait gives up early (SPARCML_ERR_TIMEOUT)
  const bool inject = injected(s.inject);
  const uint32_t limit = inject ? kInjectSpinLimit : kSpinLimit;
  if (c == 0) {
    if (lane == 0 && !inject) atomicExch(&st[0], kIncFlag | count);
    return 0;
  }
  if (lane == 0) atomicExch(&st[c], kAggFlag | count);
  uint32_t excl = 0;
  int64_t base = (int64_t)c - 1;
  uint32_t spins = 0, backoff = 32;
  while (true) {
    const int64_t j = base - (int64_t)lane;
    const unsigned long long v =
        j >= 0 ? *reinterpret_cast<volatile unsigned long long*>(&st[j]) : (2ull << 62);
    const unsigned long long flag = v & (3ull << 62);
    const uint32_t inc = __ballot_sync(0xffffffffu, flag == kIncFlag);
    const uint32_t notready = __ballot_sync(0xffffffffu, flag == 0);
    const uint32_t upto = inc ? (uint32_t)(__ffs(inc) - 1) : 31u;
    const uint32_t need = upto == 31 ? 0xffffffffu : ((2u << upto) - 1u);
    if (notready & need) {
      if (++spins > limit) {
        if (lane == 0) set_status(s.status, SPARCML_ERR_TIMEOUT);
        break;
      }
      __nanosleep(backoff);
      backoff = min(backoff * 2, 1024u);
      continue;
    }
    excl += warp_sum(lane <= upto ? (uint32_t)v : 0u);
    if (inc) break;
    base -= 32;
  }
  if (lane == 0) atomicExch(&st[c], kIncFlag | (excl + count));
  return excl;
}

// Stages entries [off, off + len) of a stage's input (idx and val buffers of
// `total` entries) into shared memory, 16 bytes at a time from the 16-byte
// boundary at or below `off` when both buffers are 16-byte aligned (`vec`);
// a quad that would pass the buffers' end is copied entry by entry. Returns
// the position in shared memory of entry `off`. Asynchronous: the caller
// waits for the copies.
__device__ __forceinline__ uint32_t stage_range(uint32_t* sdst_i, float* sdst_v, const uint32_t* gi,
                                                const float* gv, uint64_t off, uint32_t len,
                                                uint64_t total, bool vec) {
  if (!vec) {
    for (uint32_t x = threadIdx.x; x < len; x += blockDim.x) {
      cp_async4(&sdst_i[x], gi + off + x);
      cp_async4(&sdst_v[x], gv + off + x);
    }
    return 0;
  }
  const uint32_t head = (uint32_t)(off & 3);
  const uint64_t q0 = off - head;
  const uint32_t nq = (head + len + 3) / 4;
  for (uint32_t k = threadIdx.x; k < nq; k += blockDim.x) {
    const uint64_t e = q0 + 4ull * k;
    if (e + 4 <= total) {
      cp_async16(&sdst_i[4 * k], gi + e);
      cp_async16(&sdst_v[4 * k], gv + e);
    } else {
      for (uint32_t u = 0; u < 4; ++u)
        if (e + u < total) {
          cp_async4(&sdst_i[4 * k + u], gi + e + u);
          cp_async4(&sdst_v[4 * k + u], gv + e + u);
        }
    }
  }
  return head;
}

__global__ void __launch_bounds__(kMergeThreads) ssar_merge_kernel(StageArgs s) {
  griddep_wait();
  // a range of at most kChunk + 1 entries, staged from the 16-byte boundary
  // at or below its start (up to 3 entries before it, 3 after)
  __shared__ __align__(16) uint32_t sa_idx[kChunk + 8], sb_idx[kChunk + 8];
  __shared__ __align__(16) float sa_val[kChunk + 8], sb_val[kChunk + 8];
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t bc[2];
  const uint32_t t = threadIdx.x;
  if (t == 0) bc[0] = atomicAdd(s.ticket, 1u);
  __syncthreads();
  const uint32_t ticket = bc[0];
  const uint32_t g = ticket / s.chunks, c = ticket % s.chunks;  // pair-major order
  if (g >= s.G) return;
  const Pair q = pair_of(s, g);
  const uint32_t total = q.na + q.nb;
  if ((uint64_t)c * kChunk >= total && !(c == 0 && total == 0)) return;  // past this pair's end
  const uint64_t per = (uint64_t)s.chunks + 1;
  const uint32_t i0 = s.split[(uint64_t)g * per + c], i1 = s.split[(uint64_t)g * per + c + 1];
  const uint32_t j0 = s.split_b[(uint64_t)g * per + c], j1 = s.split_b[(uint64_t)g * per + c + 1];
  const uint32_t la = i1 > i0 ? min(i1 - i0, kChunk + 1) : 0u;  // bounds kept for bad streams
  const uint32_t lb = j1 > j0 ? min(j1 - j0, kChunk + 1) : 0u;
  // stage both sub-ranges with asynchronous copies: every load in flight at once
  const uint64_t in_total = 2ull * s.G * s.cap_in;  // entries of the stage's input buffers
  const bool vec = ((reinterpret_cast<uintptr_t>(s.in_idx) | reinterpret_cast<uintptr_t>(s.in_val)) &
                    15) == 0;
  const uint32_t ha = stage_range(sa_idx, sa_val, s.in_idx, s.in_val,
                                  (uint64_t)(2 * g) * s.cap_in + i0, la, in_total, vec);
  const uint32_t hb = stage_range(sb_idx, sb_val, s.in_idx, s.in_val,
                                  (uint64_t)(2 * g + 1) * s.cap_in + j0, lb, in_total, vec);
  cp_async_wait_all();
  __syncthreads();
  const uint32_t* A_idx = sa_idx + ha;  // A_idx[x] = entry i0 + x of A
  const float* A_val = sa_val + ha;
  const uint32_t* B_idx = sb_idx + hb;
  const float* B_val = sb_val + hb;
  if (s.validate) {  // strictly ascending streams with indices < N
    for (uint32_t x = t; x < la; x += blockDim.x) {
      const uint32_t prev = x > 0 ? A_idx[x - 1] : (i0 > 0 ? q.a_idx[i0 - 1] : 0u);
      if (A_idx[x] >= s.N || ((x > 0 || i0 > 0) && A_idx[x] <= prev))
        set_status(s.status, SPARCML_ERR_BAD_STREAM);
    }
    for (uint32_t x = t; x < lb; x += blockDim.x) {
      const uint32_t prev = x > 0 ? B_idx[x - 1] : (j0 > 0 ? q.b_idx[j0 - 1] : 0u);
      if (B_idx[x] >= s.N || ((x > 0 || j0 > 0) && B_idx[x] <= prev))
        set_status(s.status, SPARCML_ERR_BAD_STREAM);
    }
  }
  // This thread's positions: local diagonals [t * kPerThread, ...) of la + lb.
  const uint32_t L = la + lb;
  auto local_split = [&](uint32_t d, uint32_t* oa, uint32_t* ob) {
    uint32_t lo = d > lb ? d - lb : 0u, hi = min(d, la);
    while (lo < hi) {
      const uint32_t mid = (lo + hi) >> 1;
      if (A_idx[mid] <= B_idx[d - 1 - mid]) lo = mid + 1; else hi = mid;
    }
    uint32_t b = d - lo;
    if (lo > 0 && b < lb && A_idx[lo - 1] == B_idx[b]) ++b;
    *oa = lo;
    *ob = b;
  };
  uint32_t a0, b0, a1, b1;
  local_split(min(t * kPerThread, L), &a0, &b0);
  local_split(min((t + 1) * kPerThread, L), &a1, &b1);
  if (b0 > b1) b0 = b1;  // a tie moved the start past a short range
  // One walk over the thread's positions (at most kPerThread + 1 entries: a
  // pair of equal keys kept whole can add one), its entries held in registers
  // (the loop is unrolled, so every index is static).
  uint32_t okey[kPerThread + 1];
  float oval[kPerThread + 1];
  uint32_t n = 0;
  {
    uint32_t ia = a0, ib = b0;
#pragma unroll
    for (uint32_t u = 0; u <= kPerThread; ++u) {
      okey[u] = 0;
      oval[u] = 0.0f;
      if (ia < a1 || ib < b1) {  // once false, false for the rest of the walk
        if (ib >= b1 || (ia < a1 && A_idx[ia] < B_idx[ib])) {
          okey[u] = A_idx[ia];
          oval[u] = __fadd_rn(0.0f, A_val[ia]);
          ++ia;
        } else if (ia >= a1 || B_idx[ib] < A_idx[ia]) {
          okey[u] = B_idx[ib];
          oval[u] = __fadd_rn(0.0f, B_val[ib]);
          ++ib;
        } else {  // the same index in A and B: (+0 + a) + b
          okey[u] = A_idx[ia];
          oval[u] = __fadd_rn(__fadd_rn(0.0f, A_val[ia]), B_val[ib]);
          ++ia;
          ++ib;
        }
        n = u + 1;
      }
    }
  }
  uint32_t count;
  const uint32_t ex = block_excl_scan(n, scratch, &count);  // its barriers end every walk
  if (t < 32) {
    const uint32_t excl = chunk_lookback(s, (uint64_t)g * s.chunks, c, count);
    if (t == 0) bc[1] = excl;
  }
  // The chunk's merged entries, in order, into the (now free) A staging
  // arrays, then out with consecutive threads on consecutive positions.
  // count <= la + lb <= kChunk + 2 fits them.
#pragma unroll
  for (uint32_t u = 0; u <= kPerThread; ++u) {
    if (u < n && ex + u < kChunk + 2) {
      sa_idx[ex + u] = okey[u];
      sa_val[ex + u] = oval[u];
    }
  }
  __syncthreads();
  const uint64_t pos0 = bc[1];
  const uint64_t base = (uint64_t)g * s.cap_out;
  const uint32_t cnt = min(count, kChunk + 2);
  for (uint32_t x = t; x < cnt; x += blockDim.x) {
    if (pos0 + x < s.cap_out) {
      s.out_idx[base + pos0 + x] = sa_idx[x];
      s.out_val[base + pos0 + x] = sa_val[x];
    } else {
      set_status(s.status, SPARCML_ERR_CAPACITY);
    }
  }
  const bool last = (uint64_t)(c + 1) * kChunk >= total;
  if (t == 0 && last) {
    const uint32_t u = bc[1] + count;
    s.out_nnz[g] = u;
    if (s.fill) atomicAdd(s.fill, (unsigned long long)u);
  }
}

struct SsarLayout {
  size_t ticket, state, split, split_b, buf_idx[2], buf_val[2], nnz[2], total;
  uint32_t chunks0;
};

// Stage s (0-based) of P nodes with per-node capacity cap: 2G = P >> s input
// streams of capacity cap << s (bounded by N), outputs of twice that.
uint64_t stage_cap(uint64_t cap, uint64_t N, int s) { return std::min<uint64_t>(N, cap << s); }

SsarLayout ssar_layout(int32_t P, uint64_t cap, uint64_t N) {
  SsarLayout l;
  // chunk slots per pair at stage 0 bound every stage: pairs halve while a
  // pair's merged length at most doubles
  const uint64_t chunks = (2 * cap + kChunk - 1) / kChunk + 1;
  const uint64_t G = (uint64_t)P / 2;
  l.chunks0 = (uint32_t)chunks;
  l.ticket = 64;
  l.state = 256;
  l.split = align_up(l.state + 8 * G * chunks, 256);
  l.split_b = align_up(l.split + 4 * G * (chunks + 1), 256);
  size_t off = align_up(l.split_b + 4 * G * (chunks + 1), 256);
  const uint64_t entries = (uint64_t)P * std::min<uint64_t>(cap, N);  // any stage's outputs
  for (int b = 0; b < 2; ++b) {
    l.buf_idx[b] = off;
    off = align_up(off + 4 * entries, 256);
    l.buf_val[b] = off;
    off = align_up(off + 4 * entries, 256);
    l.nnz[b] = off;
    off = align_up(off + 4 * G, 256);
  }
  l.total = off;
  return l;
}

}  // namespace
}  // namespace sparcml

using namespace sparcml;

extern "C" size_t sparcml_ssar_workspace_size(int32_t P, uint64_t cap, uint64_t N) {
  if (P < 2 || (P & (P - 1)) != 0 || P > 65536 || cap < 1 || cap > 0x7fffffffull || N < 1 ||
      N > 0xffffffffull)
    return 0;
  return ssar_layout(P, cap, N).total;
}

extern "C" int sparcml_ssar_allreduce_traced(const uint32_t* idx, const float* val,
                                             const uint32_t* nnz, int32_t P, uint64_t cap,
                                             uint64_t N, uint32_t* out_idx, float* out_val,
                                             uint64_t out_cap, uint32_t* out_nnz,
                                             unsigned long long* stage_nnz, void* ws,
                                             size_t ws_bytes, void* stream,
                                             void* const* events) {
  const ApiRange nvtx_range(__func__);
  if (!idx || !val || !nnz || !out_idx || !out_val || !out_nnz || !ws)
    return SPARCML_ERR_INVALID_ARG;
  if (P < 2 || (P & (P - 1)) != 0 || P > 65536 || cap < 1 || cap > 0x7fffffffull || N < 1 ||
      N > 0xffffffffull)
    return SPARCML_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return SPARCML_ERR_INVALID_ARG;
  const SsarLayout l = ssar_layout(P, cap, N);
  if (ws_bytes < l.total) return SPARCML_ERR_WORKSPACE;
  if (out_cap < std::min<uint64_t>(N, (uint64_t)P * cap)) return SPARCML_ERR_CAPACITY;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  int stages = 0;
  while ((1 << stages) < P) ++stages;
  if (stage_nnz &&
      cudaMemsetAsync(stage_nnz, 0, sizeof(unsigned long long) * stages, s) != cudaSuccess)
    return SPARCML_ERR_CUDA;
  const uint32_t* in_idx = idx;
  const float* in_val = val;
  const uint32_t* in_nnz = nnz;
  uint64_t cap_in = cap;
  for (int st = 0; st < stages; ++st) {
    if (events && events[st]) cudaEventRecord(static_cast<cudaEvent_t>(events[st]), s);
    const uint32_t G = (uint32_t)(P >> (st + 1));
    const bool last = st == stages - 1;
    const uint64_t cap_out = last ? out_cap : stage_cap(cap, N, st + 1);
    StageArgs a = {};
    a.in_idx = in_idx;
    a.in_val = in_val;
    a.in_nnz = in_nnz;
    a.cap_in = cap_in;
    a.G = G;
    a.chunks = (uint32_t)((2 * cap_in + kChunk - 1) / kChunk + 1);
    a.N = (uint32_t)N;
    a.out_idx = last ? out_idx : reinterpret_cast<uint32_t*>(w + l.buf_idx[st & 1]);
    a.out_val = last ? out_val : reinterpret_cast<float*>(w + l.buf_val[st & 1]);
    a.out_nnz = last ? out_nnz : reinterpret_cast<uint32_t*>(w + l.nnz[st & 1]);
    a.cap_out = cap_out;
    a.split = reinterpret_cast<uint32_t*>(w + l.split);
    a.split_b = reinterpret_cast<uint32_t*>(w + l.split_b);
    a.state = reinterpret_cast<unsigned long long*>(w + l.state);
    a.ticket = reinterpret_cast<uint32_t*>(w + l.ticket);
    a.fill = stage_nnz ? stage_nnz + st : nullptr;
    a.status = reinterpret_cast<int32_t*>(w);
    a.inject = reinterpret_cast<const uint32_t*>(w + kInjectOffset);
    a.validate = st == 0;
    if ((uint64_t)G * a.chunks > (uint64_t)P / 2 * l.chunks0) return SPARCML_ERR_WORKSPACE;
    // the ticket and this stage's look-back words start at zero
    if (cudaMemsetAsync(w + l.ticket, 0, l.split - l.ticket, s) != cudaSuccess)
      return SPARCML_ERR_CUDA;
    const uint64_t warps = (uint64_t)G * (a.chunks + 1);
    launch_pdl(ssar_partition_kernel, (unsigned)((warps * 32 + 255) / 256), 256, 0, s, a);
    launch_pdl(ssar_merge_kernel, (unsigned)((uint64_t)G * a.chunks), kMergeThreads, 0, s, a);
    if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
    note_launches(2);
    in_idx = a.out_idx;
    in_val = a.out_val;
    in_nnz = a.out_nnz;
    cap_in = cap_out;
  }
  if (events && events[stages]) cudaEventRecord(static_cast<cudaEvent_t>(events[stages]), s);
  return SPARCML_OK;
}

extern "C" int sparcml_ssar_allreduce(const uint32_t* idx, const float* val, const uint32_t* nnz,
                                      int32_t P, uint64_t cap, uint64_t N, uint32_t* out_idx,
                                      float* out_val, uint64_t out_cap, uint32_t* out_nnz,
                                      unsigned long long* stage_nnz, void* ws, size_t ws_bytes,
                                      void* stream) {
  return sparcml_ssar_allreduce_traced(idx, val, nnz, P, cap, N, out_idx, out_val, out_cap,
                                       out_nnz, stage_nnz, ws, ws_bytes, stream, nullptr);
}
