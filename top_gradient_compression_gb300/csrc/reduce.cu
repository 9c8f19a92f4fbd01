// Sparse sum-reduction of P streams with the adaptive dense switch, sm_103a.
//
// "SparCML: High-Performance Sparse Communication for Machine Learning",
// §5.2 (allreduce of sparse vectors with a coordinate-wise associative op
// that has a neutral element: fp32 sum with neutral +0.0, and max, min,
// bitwise or), §5.3.2 (the split phase routes index ranges to owners: here
// a warp or CTA owns each tile of the index space), §5.1 / §5.3.3 (switch to
// a dense representation once fill-in passes the threshold delta), App. B
// (the result size is the size of the union of the contributed index sets).
//
// No sort and no floating-point atomics: the index space is cut into tiles,
// each tile is reduced by one owner (a warp or a CTA) that adds its nodes'
// entries in ascending node order, so every result is bit-exact. The host
// picks the tiling from P, cap and N (no device read):
//
//  warp tiles (P <= 64, P * cap >= N / 16): a streaming split pass
//      (reduce_split_quad_kernel / reduce_split_stream_kernel) finds where
//      every node's entries enter every 1,024-index tile and validates the
//      streams; one warp per tile (reduce_mini_quad_kernel with 16-byte
//      quads, or reduce_mini_kernel) sums into a shared accumulator.
//      P * cap >= N / 4: dense-first (slice + bitmap + union size, then
//      reduce_mini_compact_kernel if the result is sparse after all);
//      otherwise sparse-first with a decoupled look-back per CTA group
//      (Merrill and Garland, 2016) and reduce_fixup_kernel if the union
//      crosses the dense threshold after all.
//  compact-accumulator CTA tiles (P * cap < N / 4 when P > 64, or
//      P * cap < N / 16): reduce_split_kernel (33-ary search per (tile,
//      node)), reduce_sparse_tile_kernel (tiles of 8,192..131,072 indices,
//      bitmap + prefix-popcount slots, look-back), fix-up.
//  staged CTA tiles (P > 64 with P * cap >= N / 4, or P > 1,024):
//      reduce_dense_tile_kernel (8,192-index tiles, per-node items through a
//      cp.async ring), dense-first with reduce_finalize_kernel and
//      reduce_compact_kernel, or look-back + fix-up.
//
// Tiles past the sparse capacity floor(N * num / den) write dense slices;
// a dense result holds the operation's neutral element (+0.0f for the sum)
// where no node has the index. The same kernels serve max, min and bitwise
// or (sparcml_sparse_reduce_op) and 2/4/8-bit values decoded on load.
//
// Every wait on a predecessor is bounded; on expiry the kernel records
// SPARCML_ERR_TIMEOUT and carries on, so a bad input can never hang the GPU.

#include <algorithm>

#include "common.cuh"

namespace sparcml {
namespace {

constexpr uint32_t kTile = 8192;  // indices per tile
constexpr uint32_t kWords = kTile / 32;
constexpr uint32_t kReduceThreads = 256;
constexpr uint32_t kUnroll = 8;
constexpr int32_t kMaxReduceP = 4096;
constexpr unsigned long long kFlagAgg = 1ull << 62;
constexpr unsigned long long kFlagInc = 2ull << 62;

struct ReduceArgs {
  const uint32_t* idx;
  const float* val;
  const uint8_t* codes;
  const float* scales;
  const uint32_t* nnz;
  uint64_t cap;
  uint64_t code_stride;
  uint64_t scale_stride;
  uint32_t bucket;
  uint32_t bucket_shift;  // log2(bucket) when a power of two, else 32
  uint32_t bits;          // width of the quantised codes: 2, 4 or 8
  int32_t op;             // kOpSum, kOpMax, kOpMin or kOpOr
  int32_t P;
  uint32_t N;
  uint32_t ntiles;
  uint32_t tile_w;      // indices per tile: kTile (dense regime) or a wider power of two
  uint32_t cap_sparse;  // floor(N * num / den): largest sparse result
  uint32_t* out_idx;
  float* out_val;
  float* out_dense;
  uint32_t* out_nnz;
  int32_t* out_is_dense;
  uint32_t* ticket;
  unsigned long long* tile_state;
  uint2* tile_info;  // (offset, count | dense << 31)
  const uint32_t* split;  // [(ntiles + 1) * P] node sub-range starts per tile
  uint32_t* tile_bm;      // dense-first mode: [ntiles][kWords] presence bits per tile
  uint32_t* u_total;      // warp-tile mode: union size, summed by atomics
  uint32_t hot_thr;       // dense-first warp tiles with more entries go to the hot kernel
  uint32_t* hot_cnt;      // dense-first warp tiles: tiles left to reduce_hot_tile_kernel
  uint32_t* hot;          // [ntiles] their ids
  int32_t* status;
  const uint32_t* inject;  // the workspace's fault-injection word (or nullptr)
};

__device__ __forceinline__ uint32_t lower_bound_u32(const uint32_t* a, uint32_t n, uint32_t x) {
  uint32_t lo = 0, hi = n;
  while (lo < hi) {
    const uint32_t mid = lo + ((hi - lo) >> 1);
    if (a[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// The reduction (§5.2: any coordinate-wise associative operation with a
// neutral element): a stream stands for the vector holding the neutral
// element at unlisted indices; an index's result folds its nodes' values in
// ascending node order starting from the neutral element.
enum : int32_t { kOpSum = 0, kOpMax = 1, kOpMin = 2, kOpOr = 3 };

__device__ __forceinline__ float op_neutral(int32_t op) {
  return op == kOpMax ? -INFINITY : op == kOpMin ? INFINITY : 0.0f;
}

// The fold of one value into a partial result. max/min take the new value
// only when it is strictly greater / smaller (ties keep the lower node's); or
// works on the fp32 bit patterns. op is the same for the whole launch.
__device__ __forceinline__ float op_fold(int32_t op, float acc, float v) {
  if (op == kOpSum) return __fadd_rn(acc, v);
  if (op == kOpMax) return v > acc ? v : acc;
  if (op == kOpMin) return v < acc ? v : acc;
  return __uint_as_float(__float_as_uint(acc) | __float_as_uint(v));
}

// level / 7 for a 4-bit level 1..7: the correctly rounded fp32 quotient (the
// constant expressions are IEEE divisions, as __fdiv_rn would give), picked by
// selects on the level's bits rather than an indexed table, which lanes with
// different levels would serialise on.
__device__ __forceinline__ float level_over_7(uint32_t level) {
  const float lo = (level & 2u) ? ((level & 1u) ? 3.0f / 7.0f : 2.0f / 7.0f)
                                : ((level & 1u) ? 1.0f / 7.0f : 0.0f);
  const float hi = (level & 2u) ? ((level & 1u) ? 7.0f / 7.0f : 6.0f / 7.0f)
                                : ((level & 1u) ? 5.0f / 7.0f : 4.0f / 7.0f);
  return (level & 4u) ? hi : lo;
}

// Value of entry j of node p: fp32 as stored, or decoded from its b-bit code
// (sign bit over a level of s = 2^(b-1) - 1; v = +-(level / s) * scale).
template <bool Q4>
__device__ __forceinline__ float load_value(const ReduceArgs& a, uint32_t p, uint32_t j) {
  if constexpr (!Q4) {
    return a.val[(uint64_t)p * a.cap + j];
  } else {
    // a.bits is the same for the whole launch: a uniform branch
    uint32_t code, level;
    float q;
    const uint8_t* cp = a.codes + (uint64_t)p * a.code_stride;
    if (a.bits == 4) {
      const uint8_t byte = cp[j >> 1];
      code = (j & 1) ? (byte >> 4) : (byte & 15u);
      level = code & 7u;
      q = level_over_7(level);
    } else if (a.bits == 8) {
      code = cp[j];
      level = code & 127u;
      q = __fdiv_rn((float)level, 127.0f);
    } else {
      code = (cp[j >> 2] >> ((j & 3) * 2)) & 3u;
      level = code & 1u;
      q = (float)level;
    }
    // The scale is read whatever the level (j < cap keeps it inside the
    // node's ceil(cap / bucket) scales), so its load does not wait for the
    // code's; a zero level then gives +0.0f by a select.
    const uint32_t b = a.bucket_shift < 32 ? j >> a.bucket_shift : j / a.bucket;
    const float scale = a.scales[(uint64_t)p * a.scale_stride + b];
    const float v = __fmul_rn(q, scale);
    return level == 0 ? 0.0f : (code >> (a.bits - 1)) ? -v : v;
  }
}

// Decoupled look-back (Merrill and Garland, 2016), one warp wide: the tile
// publishes its count, then reads the states of the 32 nearest predecessors
// at once and sums back to the nearest inclusive prefix; it publishes its own
// inclusive prefix and leaves its exclusive offset in *out. Every wait is
// bounded (SPARCML_ERR_TIMEOUT, then it carries on). Called by the whole
// CTA; only warp 0 works.
__device__ void tile_lookback(const ReduceArgs& a, uint32_t tile, uint32_t count, uint32_t* out) {
  const uint32_t t = threadIdx.x, lane = lane_id();
  if (t >= 32) return;
  unsigned long long* st = a.tile_state;
  uint32_t excl = 0;
  // an injected fault: the chain's first tile withholds its flag and every
  // wait gives up early (SPARCML_ERR_TIMEOUT)
  const bool inject = injected(a.inject);
  const uint32_t limit = inject ? kInjectSpinLimit : kSpinLimit;
  if (tile == 0) {
    if (t == 0 && !inject) atomicExch(&st[0], kFlagInc | count);
  } else {
    if (t == 0) atomicExch(&st[tile], kFlagAgg | count);
    int64_t base = (int64_t)tile - 1;
    uint32_t spins = 0, backoff = 32;
    while (true) {
      const int64_t j = base - (int64_t)lane;
      const unsigned long long sv =
          j >= 0 ? *reinterpret_cast<volatile unsigned long long*>(&st[j]) : (2ull << 62);
      const unsigned long long flag = sv & (3ull << 62);
      const uint32_t inc = __ballot_sync(0xffffffffu, flag == kFlagInc);
      const uint32_t notready = __ballot_sync(0xffffffffu, flag == 0);
      const uint32_t upto = inc ? (uint32_t)(__ffs(inc) - 1) : 31u;  // lanes 0..upto count
      const uint32_t need = upto == 31 ? 0xffffffffu : ((2u << upto) - 1u);
      if (notready & need) {
        if (++spins > limit) {
          if (t == 0) set_status(a.status, SPARCML_ERR_TIMEOUT);
          break;
        }
        __nanosleep(backoff);
        backoff = min(backoff * 2, 1024u);
        continue;
      }
      excl += warp_sum(lane <= upto ? (uint32_t)sv : 0u);
      if (inc) break;
      base -= 32;
    }
    if (t == 0) atomicExch(&st[tile], kFlagInc | (excl + count));
  }
  if (t == 0) *out = excl;
}

// Where each node's entries for tile t start: split[t * P + p] =
// lower_bound(idx_p, t * kTile) for t < ntiles and lower_bound(idx_p, N) for
// t = ntiles. One warp per (tile boundary, node): each round probes 32
// evenly spaced entries and keeps the bracket, narrowing the range 33-fold
// per memory round trip instead of 2-fold.
__global__ void __launch_bounds__(256)
reduce_split_kernel(const uint32_t* __restrict__ idx, const uint32_t* __restrict__ nnz,
                    int32_t P, uint64_t cap, uint32_t N, uint32_t ntiles, uint32_t tile_w,
                    uint32_t* __restrict__ split) {
  griddep_wait();
  const uint64_t w = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (w >= (uint64_t)(ntiles + 1) * P) return;  // warp-uniform
  const uint32_t lane = lane_id();
  const uint32_t t = (uint32_t)(w / P), p = (uint32_t)(w % P);
  const uint32_t n = (uint32_t)min((uint64_t)nnz[p], cap);
  const uint32_t x = t == ntiles ? N : t * tile_w;
  const uint32_t* a = idx + (uint64_t)p * cap;
  uint32_t lo = 0, hi = n;  // the answer lies in [lo, hi]
  while (hi - lo > 32) {
    const uint32_t span = hi - lo;
    const uint32_t pos = lo + (uint32_t)((uint64_t)span * (lane + 1) / 33);
    const uint32_t c = __popc(__ballot_sync(0xffffffffu, a[pos] < x));
    const uint32_t nlo = c ? lo + (uint32_t)((uint64_t)span * c / 33) + 1 : lo;
    const uint32_t nhi = c < 32 ? lo + (uint32_t)((uint64_t)span * (c + 1) / 33) : hi;
    lo = nlo;
    hi = nhi;
  }
  const uint32_t pos = lo + lane;
  const uint32_t c = __popc(__ballot_sync(0xffffffffu, pos < hi && a[pos] < x));
  if (lane == 0) split[w] = lo + c;
}

// TABLE: node sub-ranges come from reduce_split_kernel's table; otherwise the
// CTA binary-searches them itself (no table in the scratch).
template <bool Q4, bool TABLE = false>
__global__ void __launch_bounds__(kReduceThreads)
reduce_tile_kernel(ReduceArgs a) {
  griddep_wait();
  extern __shared__ __align__(16) uint32_t dyn[];
  float* acc = reinterpret_cast<float*>(dyn);
  uint32_t* bm = dyn + kTile;
  uint32_t* lo = bm + kWords;  // [P] first entry of each node in this tile
  uint32_t* pre = lo + a.P;    // [P + 1] exclusive prefix of the nodes' entry counts
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t bc[4];
  const uint32_t t = threadIdx.x;

  if (t == 0) {
    bc[0] = atomicAdd(a.ticket, 1u);
    bc[1] = 0;
  }
  const float e = op_neutral(a.op);  // +0.0f for the sum
  for (uint32_t w = t; w < kTile / 4; w += blockDim.x)
    reinterpret_cast<float4*>(acc)[w] = make_float4(e, e, e, e);
  for (uint32_t w = t; w < kWords; w += blockDim.x) bm[w] = 0;
  __syncthreads();
  const uint32_t tile = bc[0];
  const uint32_t tile_lo = tile * kTile;
  const uint32_t tile_n = min(kTile, a.N - tile_lo);
  const bool last = tile == a.ntiles - 1;

  // Each node's sub-range [lo, hi) of entries with tile_lo <= idx < tile_lo + tile_n.
  for (int32_t p = t; p < a.P; p += blockDim.x) {
    uint32_t n = a.nnz[p];
    if (n > a.cap) {
      set_status(a.status, SPARCML_ERR_CAPACITY);
      n = (uint32_t)a.cap;
    }
    uint32_t l, h;
    if constexpr (TABLE) {
      l = a.split[(uint64_t)tile * a.P + p];
      h = a.split[(uint64_t)(tile + 1) * a.P + p];
    } else {
      const uint32_t* ip = a.idx + (uint64_t)p * a.cap;
      l = lower_bound_u32(ip, n, tile_lo);
      h = lower_bound_u32(ip, n, tile_lo + tile_n);
    }
    if (last && h < n) set_status(a.status, SPARCML_ERR_BAD_STREAM);  // idx >= N
    if (h < l) {
      set_status(a.status, SPARCML_ERR_BAD_STREAM);
      h = l;
    }
    lo[p] = l;
    pre[p] = h - l;
    atomicMax(&bc[1], n);  // U >= max nnz: dense for certain if above the cap
  }
  __syncthreads();
  uint32_t E = 0;  // entries of the tile, all nodes
  for (int32_t base = 0; base < a.P; base += blockDim.x) {
    const int32_t p = base + (int32_t)t;
    const uint32_t c = p < a.P ? pre[p] : 0u;
    uint32_t tot;
    const uint32_t ex = block_excl_scan(c, scratch, &tot);
    if (p < a.P) pre[p] = E + ex;
    E += tot;
    __syncthreads();
  }
  if (t == 0) pre[a.P] = E;
  __syncthreads();
  const bool dense_certain = bc[1] > a.cap_sparse;

  // Node of flattened entry v: the largest p with pre[p] <= v.
  auto node_of = [&](uint32_t v) {
    uint32_t l = 0, h = (uint32_t)a.P;  // pre[l] <= v < pre[h]
    while (h - l > 1) {
      const uint32_t m = (l + h) >> 1;
      if (pre[m] <= v) l = m; else h = m;
    }
    return l;
  };

  // Accumulate. Entries are taken in node-major order, kUnroll * blockDim at
  // a time (all loads in flight together); the adds of one batch then run
  // node by node, a barrier after each node that has entries in the batch,
  // so every index sees its nodes in ascending order.
  const uint32_t lane = lane_id();
  const uint32_t batch = blockDim.x * kUnroll;
  for (uint32_t c0 = 0; c0 < E; c0 += batch) {
    uint32_t iv[kUnroll], pv[kUnroll];
    float vv[kUnroll];
#pragma unroll
    for (uint32_t u = 0; u < kUnroll; ++u) {
      const uint32_t v = c0 + u * blockDim.x + t;
      iv[u] = 0;
      vv[u] = 0.0f;
      pv[u] = 0xffffffffu;
      if (v < E) {
        const uint32_t p = node_of(v);
        const uint32_t j = lo[p] + (v - pre[p]);
        iv[u] = a.idx[(uint64_t)p * a.cap + j];
        vv[u] = load_value<Q4>(a, p, j);
        pv[u] = p;
      }
    }
#pragma unroll
    for (uint32_t u = 0; u < kUnroll; ++u) {
      const uint32_t v = c0 + u * blockDim.x + t;
      // Strictly ascending check against entry j - 1 of the same node: the
      // previous lane holds it unless this is a warp's or a node's first entry.
      uint32_t prev = __shfl_up_sync(0xffffffffu, iv[u], 1);
      if (v < E) {
        const uint32_t p = pv[u];
        const uint32_t j = lo[p] + (v - pre[p]);
        if ((lane == 0 || v == pre[p]) && j > 0) prev = a.idx[(uint64_t)p * a.cap + j - 1];
        if (!((j == 0 || prev < iv[u]) && iv[u] - tile_lo < tile_n)) {
          set_status(a.status, SPARCML_ERR_BAD_STREAM);
          pv[u] = 0xffffffffu;  // skip it
        }
      }
    }
    const uint32_t c1 = min(c0 + batch, E);
    const uint32_t p_first = node_of(c0), p_last = node_of(c1 - 1);
    for (uint32_t p = p_first; p <= p_last; ++p) {
      if (pre[p + 1] == pre[p]) continue;  // no entries: no barrier needed
#pragma unroll
      for (uint32_t u = 0; u < kUnroll; ++u) {
        if (pv[u] == p) {
          const uint32_t off = iv[u] - tile_lo;
          acc[off] = __fadd_rn(acc[off], vv[u]);
          atomicOr(&bm[off >> 5], 1u << (off & 31));
        }
      }
      __syncthreads();
    }
  }

  // Union count of the tile.
  uint32_t c = 0;
  for (uint32_t w = t; w < kWords; w += blockDim.x) c += __popc(bm[w]);
  uint32_t count;
  block_excl_scan(c, scratch, &count);

  // Decoupled look-back for the tile's exclusive offset.
  tile_lookback(a, tile, count, &bc[2]);
  __syncthreads();
  const uint32_t excl = bc[2];
  const uint32_t incl = excl + count;
  const bool dense = dense_certain || incl > a.cap_sparse;

  if (dense) {
    float* od = a.out_dense + tile_lo;
    const bool vec = (reinterpret_cast<uintptr_t>(od) & 15) == 0;
    const uint32_t nv = vec ? tile_n / 4 : 0;
    for (uint32_t w = t; w < nv; w += blockDim.x)
      reinterpret_cast<float4*>(od)[w] = reinterpret_cast<const float4*>(acc)[w];
    for (uint32_t x = nv * 4 + t; x < tile_n; x += blockDim.x) od[x] = acc[x];
  } else {
    // Ascending compaction: one bitmap word per thread, prefix of popcounts.
    const uint32_t word = t < kWords ? bm[t] : 0u;
    uint32_t tot;
    uint32_t pos = excl + block_excl_scan(__popc(word), scratch, &tot);
    uint32_t bits = word;
    while (bits) {
      const uint32_t b = __ffs(bits) - 1;
      bits &= bits - 1;
      const uint32_t off = t * 32 + b;
      a.out_idx[pos] = tile_lo + off;
      a.out_val[pos] = acc[off];
      ++pos;
    }
  }
  if (t == 0) {
    a.tile_info[tile] = make_uint2(excl, count | (dense ? 0x80000000u : 0u));
    if (last) {
      *a.out_nnz = incl;
      *a.out_is_dense = dense ? 1 : 0;
    }
  }
}

// Dense regime: tiles of kTile indices with a dense fp32 shared accumulator.
// The tile's entries are taken node by node in work items of at most
// kStageEntries, copied global -> shared with cp.async through a kStages-deep
// ring, so the next items' loads are in flight while this one is added. A
// barrier after each item keeps ascending node order (and frees its stage).
// DENSE_FIRST (chosen when P * cap >= N, so the result is almost surely
// dense): the tile writes its dense slice and its count straight away, with
// no look-back; reduce_finalize_kernel and reduce_compact_kernel produce U,
// the dense flag and, if the result is sparse after all, the sparse output.
constexpr uint32_t kStages = 4;
constexpr uint32_t kStageEntries = 1024;
constexpr uint32_t kNoPrev = 0xffffffffu;

template <bool Q4, bool DENSE_FIRST, bool ANY>
__global__ void __launch_bounds__(kReduceThreads)
reduce_dense_tile_kernel(ReduceArgs a) {
  griddep_wait();
  extern __shared__ __align__(16) uint32_t dyn[];
  const int32_t kop = ANY ? a.op : kOpSum;  // sum-only launches fold the branch away
  float* acc = reinterpret_cast<float*>(dyn);                       // [kTile]
  uint32_t* bm = dyn + kTile;                                        // [kWords]
  uint32_t* sidx = bm + kWords;                                      // [kStages][kStageEntries]
  float* sval = reinterpret_cast<float*>(sidx + kStages * kStageEntries);
  uint32_t* lo = reinterpret_cast<uint32_t*>(sval + kStages * kStageEntries);  // [P]
  uint32_t* hi = lo + a.P;                                           // [P]
  uint32_t* ipre = hi + a.P;                                         // [P + 1] items per node, prefix
  __shared__ uint32_t sprev[kStages];
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t bc[4];
  const uint32_t t = threadIdx.x;

  if (t == 0) {
    bc[0] = atomicAdd(a.ticket, 1u);
    bc[1] = 0;
  }
  const float e = op_neutral(kop);  // +0.0f for the sum
  for (uint32_t w = t; w < kTile / 4; w += blockDim.x)
    reinterpret_cast<float4*>(acc)[w] = make_float4(e, e, e, e);
  for (uint32_t w = t; w < kWords; w += blockDim.x) bm[w] = 0;
  __syncthreads();
  const uint32_t tile = bc[0];
  const uint32_t tile_lo = tile * kTile;
  const uint32_t tile_n = min(kTile, a.N - tile_lo);
  const bool last = tile == a.ntiles - 1;
  for (int32_t p = t; p < a.P; p += blockDim.x) {
    uint32_t n = a.nnz[p];
    if (n > a.cap) {
      set_status(a.status, SPARCML_ERR_CAPACITY);
      n = (uint32_t)a.cap;
    }
    const uint32_t l = a.split[(uint64_t)tile * a.P + p];
    uint32_t h = a.split[(uint64_t)(tile + 1) * a.P + p];
    if (last && h < n) set_status(a.status, SPARCML_ERR_BAD_STREAM);  // idx >= N
    if (h < l) {
      set_status(a.status, SPARCML_ERR_BAD_STREAM);
      h = l;
    }
    lo[p] = l;
    hi[p] = h;
    ipre[p] = (h - l + kStageEntries - 1) / kStageEntries;
    atomicMax(&bc[1], n);
  }
  __syncthreads();
  uint32_t n_items = 0;
  for (int32_t base = 0; base < a.P; base += blockDim.x) {
    const int32_t p = base + (int32_t)t;
    const uint32_t c = p < a.P ? ipre[p] : 0u;
    uint32_t tot;
    const uint32_t ex = block_excl_scan(c, scratch, &tot);
    if (p < a.P) ipre[p] = n_items + ex;
    n_items += tot;
    __syncthreads();
  }
  if (t == 0) ipre[a.P] = n_items;
  __syncthreads();
  const bool dense_certain = bc[1] > a.cap_sparse;

  // work item i -> node p and entries [j0, j1) of that node's stream
  auto item = [&](uint32_t i, uint32_t* p, uint32_t* j0, uint32_t* j1) {
    uint32_t l = 0, h = (uint32_t)a.P;  // ipre[l] <= i < ipre[h]
    while (h - l > 1) {
      const uint32_t m = (l + h) >> 1;
      if (ipre[m] <= i) l = m; else h = m;
    }
    *p = l;
    *j0 = lo[l] + (i - ipre[l]) * kStageEntries;
    *j1 = min(*j0 + kStageEntries, hi[l]);
  };
  auto issue = [&](uint32_t i) {
    if (i < n_items) {
      uint32_t p, j0, j1;
      item(i, &p, &j0, &j1);
      const uint32_t st = i % kStages;
      const uint32_t* ip = a.idx + (uint64_t)p * a.cap;
      for (uint32_t j = j0 + t; j < j1; j += blockDim.x) {
        cp_async4(sidx + st * kStageEntries + (j - j0), ip + j);
        if constexpr (!Q4) cp_async4(sval + st * kStageEntries + (j - j0), a.val + (uint64_t)p * a.cap + j);
      }
      if (t == 0) {
        if (j0 > 0) cp_async4(&sprev[st], ip + j0 - 1);
        else sprev[st] = kNoPrev;
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  for (uint32_t i = 0; i + 1 < kStages; ++i) issue(i);
  for (uint32_t i = 0; i < n_items; ++i) {
    issue(i + kStages - 1);  // refills the stage item i - 1 used
    asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 1) : "memory");
    __syncthreads();
    uint32_t p, j0, j1;
    item(i, &p, &j0, &j1);
    const uint32_t st = i % kStages;
    const uint32_t* si = sidx + st * kStageEntries;
    for (uint32_t j = j0 + t; j < j1; j += blockDim.x) {
      const uint32_t e = j - j0;
      const uint32_t iv = si[e];
      const uint32_t prev = e > 0 ? si[e - 1] : sprev[st];
      const uint32_t off = iv - tile_lo;
      if ((j == 0 || (prev != kNoPrev && prev < iv)) && off < tile_n) {
        float v;
        if constexpr (Q4) v = load_value<Q4>(a, p, j);
        else v = sval[st * kStageEntries + e];
        acc[off] = op_fold(kop, acc[off], v);
        atomicOr(&bm[off >> 5], 1u << (off & 31));
      } else {
        set_status(a.status, SPARCML_ERR_BAD_STREAM);
      }
    }
    __syncthreads();  // ascending node order; the stage may be refilled
  }
  asm volatile("cp.async.wait_all;" ::: "memory");

  uint32_t c = 0;
  for (uint32_t w = t; w < kWords; w += blockDim.x) c += __popc(bm[w]);
  uint32_t count;
  block_excl_scan(c, scratch, &count);
  if constexpr (DENSE_FIRST) {
    float* od = a.out_dense + tile_lo;
    const bool vec = (reinterpret_cast<uintptr_t>(od) & 15) == 0;
    const uint32_t nv = vec ? tile_n / 4 : 0;
    for (uint32_t w = t; w < nv; w += blockDim.x)
      reinterpret_cast<float4*>(od)[w] = reinterpret_cast<const float4*>(acc)[w];
    for (uint32_t x = nv * 4 + t; x < tile_n; x += blockDim.x) od[x] = acc[x];
    uint32_t* tb = a.tile_bm + (uint64_t)tile * kWords;
    for (uint32_t w = t; w < kWords; w += blockDim.x) tb[w] = bm[w];
    if (t == 0) a.tile_info[tile] = make_uint2(0, count);
    (void)dense_certain;
    return;
  }
  tile_lookback(a, tile, count, &bc[2]);
  __syncthreads();
  const uint32_t excl = bc[2];
  const uint32_t incl = excl + count;
  const bool dense = dense_certain || incl > a.cap_sparse;
  if (dense) {
    float* od = a.out_dense + tile_lo;
    const bool vec = (reinterpret_cast<uintptr_t>(od) & 15) == 0;
    const uint32_t nv = vec ? tile_n / 4 : 0;
    for (uint32_t w = t; w < nv; w += blockDim.x)
      reinterpret_cast<float4*>(od)[w] = reinterpret_cast<const float4*>(acc)[w];
    for (uint32_t x = nv * 4 + t; x < tile_n; x += blockDim.x) od[x] = acc[x];
  } else {
    const uint32_t word = t < kWords ? bm[t] : 0u;
    uint32_t tot;
    uint32_t pos = excl + block_excl_scan(__popc(word), scratch, &tot);
    uint32_t bits = word;
    while (bits) {
      const uint32_t b = __ffs(bits) - 1;
      bits &= bits - 1;
      const uint32_t off = t * 32 + b;
      a.out_idx[pos] = tile_lo + off;
      a.out_val[pos] = acc[off];
      ++pos;
    }
  }
  if (t == 0) {
    a.tile_info[tile] = make_uint2(excl, count | (dense ? 0x80000000u : 0u));
    if (last) {
      *a.out_nnz = incl;
      *a.out_is_dense = dense ? 1 : 0;
    }
  }
}

// Heavy coverage (P <= kMiniMaxP, P * cap >= N / 4): one warp per mini-tile
// of kMini indices, no block barrier and no shared-memory staging. The
// warp's entries of the mini-tile are numbered in ascending node order
// ("positions"); lane l takes positions l, l + 32, ... so one round of 32
// positions covers one node, or a few at node changes. A round loads its
// indices and values straight into registers (kMiniRounds rounds in
// flight), then adds them into the warp's shared accumulator; rounds, and the
// nodes within a round, are applied in order, so every index is summed in
// ascending node order. The streams were validated by the split pass; here
// every access is only kept in bounds. Output: the dense slice, the presence
// bitmap and the union size (reduce_mini_compact_kernel finishes).
constexpr uint32_t kMini = 1024;
constexpr uint32_t kMiniShift = 10;
constexpr uint32_t kMiniWords = kMini / 32;
constexpr uint32_t kMiniRounds = 6;
constexpr int32_t kMiniMaxP = 64;
constexpr uint32_t kMiniWarps = 4;  // mini-tiles per CTA
// Dense-first warp tiles with more entries than max(kHot, kHotRatio x the
// average tile) (a skewed, Zipf-like head) are left to reduce_hot_tile_kernel,
// which spreads one over a CTA.
constexpr uint32_t kHot = 1024;
constexpr uint32_t kHotRatio = 2;
constexpr uint32_t kHotThreads = 512;
constexpr uint32_t kHotAhead = 8;  // nodes whose loads are in flight at once
constexpr uint64_t kHotGrid = 4 * 152;  // CTAs of the hot launch: the GPU's 152 SMs, 4 each
// per-warp region, a multiple of 16 bytes: acc is accessed as uint4
constexpr uint32_t kAccWords = kMini;
constexpr uint32_t kMiniWarpWords = (kAccWords + 3 * kMiniMaxP + 1 + 31) / 32 * 32;
static_assert(kMiniWarpWords % 4 == 0, "uint4 access to each warp's accumulator");
// The scalar warp tile's per-warp region sized for the launch's P (the
// accumulator, lo[P] and cpre[P + 1], a multiple of 4 words): at P = 16 ten
// CTAs fit an SM's shared memory, against nine at the largest P.
__host__ __device__ __forceinline__ uint32_t mini_warp_words(int32_t P) {
  return kAccWords + ((2u * (uint32_t)P + 1u + 3u) & ~3u);
}
constexpr uint32_t kAbsent = 0xffffffffu;

// Split table of the warp tiles by one streaming pass over every node's
// indices (grid: x over entries, y = node): entry j of node p is the first of
// node p at or past every tile boundary between its predecessor's and its own
// (boundary t is t * kMini, and N for t = ntiles); the closing run (entry
// nnz, boundaries past the last index) is written by warp 0 of CTA x = 0.
// Validates the streams on the way: strictly ascending, every index < N.
__device__ __forceinline__ uint32_t mini_tiles_at_or_below(uint32_t v, uint32_t N, uint32_t ntiles) {
  return v >= N ? ntiles + 1 : (v >> kMiniShift) + 1;
}

// Write split[t][p] = j for t in [t0, t1): short runs by the lane itself,
// long ones (sparse nodes) by the whole warp. Called by all 32 lanes.
__device__ __forceinline__ void split_fill(uint32_t* split, int32_t P, uint32_t p, uint32_t t0,
                                           uint32_t t1, uint32_t j) {
  const bool wide = t1 - t0 > 4;
  if (!wide)
    for (uint32_t t = t0; t < t1; ++t) split[(uint64_t)t * P + p] = j;
  uint32_t todo = __ballot_sync(0xffffffffu, wide);
  while (todo) {
    const uint32_t src = __ffs(todo) - 1;
    todo &= todo - 1;
    const uint32_t a0 = __shfl_sync(0xffffffffu, t0, src);
    const uint32_t a1 = __shfl_sync(0xffffffffu, t1, src);
    const uint32_t jj = __shfl_sync(0xffffffffu, j, src);
    for (uint32_t t = a0 + lane_id(); t < a1; t += 32) split[(uint64_t)t * P + p] = jj;
  }
}

__device__ __forceinline__ void split_close(const uint32_t* row, uint32_t n, int32_t P, uint32_t p,
                                            uint32_t N, uint32_t ntiles, uint32_t* split) {
  if (blockIdx.x != 0 || threadIdx.x >= 32) return;  // warp-uniform
  const uint32_t t0 = n > 0 ? mini_tiles_at_or_below(row[n - 1], N, ntiles) : 0u;
  for (uint32_t t = t0 + lane_id(); t <= ntiles; t += 32) split[(uint64_t)t * P + p] = n;
}

constexpr uint32_t kSplitBatch = 8;  // scalar pass: entries per thread, loaded together
constexpr uint32_t kSplitQuads = 4;  // vector pass: 16-byte quads per thread

// Scalar pass: any alignment.
__global__ void __launch_bounds__(256)
reduce_split_stream_kernel(const uint32_t* __restrict__ idx, const uint32_t* __restrict__ nnz,
                           int32_t P, uint64_t cap, uint32_t N, uint32_t ntiles,
                           uint32_t* __restrict__ split, int32_t* status) {
  griddep_wait();
  const uint32_t p = blockIdx.y, lane = lane_id();
  uint32_t n = nnz[p];
  if (n > cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, SPARCML_ERR_CAPACITY);
    n = (uint32_t)cap;
  }
  const uint32_t* row = idx + (uint64_t)p * cap;
  split_close(row, n, P, p, N, ntiles, split);
  const uint64_t span = (uint64_t)blockDim.x * kSplitBatch;
  bool bad = false;
  for (uint64_t j0 = (uint64_t)blockIdx.x * span; j0 < n; j0 += (uint64_t)gridDim.x * span) {
    // batch u covers entries j0 + u * blockDim + threadIdx.x: coalesced per u
    uint32_t cur[kSplitBatch], before[kSplitBatch];
#pragma unroll
    for (uint32_t u = 0; u < kSplitBatch; ++u) {
      const uint64_t j = j0 + (uint64_t)u * blockDim.x + threadIdx.x;
      cur[u] = j < n ? ld_stream(row + j) : 0u;
      before[u] = (lane == 0 && j > 0 && j < n) ? row[j - 1] : 0u;
    }
#pragma unroll
    for (uint32_t u = 0; u < kSplitBatch; ++u) {
      const uint64_t j = j0 + (uint64_t)u * blockDim.x + threadIdx.x;
      uint32_t prev = __shfl_up_sync(0xffffffffu, cur[u], 1);
      if (lane == 0) prev = before[u];
      const bool entry = j < n, head = j == 0;
      bad |= entry && (cur[u] >= N || (!head && cur[u] <= prev));
      // no boundary between prev and cur: the common case, nothing to write
      const bool inner =
          !entry || (!head && cur[u] < N && (cur[u] >> kMiniShift) == (prev >> kMiniShift));
      if (__all_sync(0xffffffffu, inner)) continue;
      uint32_t t0 = 0, t1 = 0;
      if (!inner) {
        t0 = head ? 0u : mini_tiles_at_or_below(prev, N, ntiles);
        t1 = max(t0, mini_tiles_at_or_below(cur[u], N, ntiles));  // a step down writes nothing
      }
      split_fill(split, P, p, t0, t1, (uint32_t)j);
    }
  }
  if (bad) set_status(status, SPARCML_ERR_BAD_STREAM);
}

// Vector pass: idx 16-byte aligned and P * cap a multiple of 4, so every
// 16-byte quad that overlaps a row lies inside the buffer. Quad k of node p
// holds entries j = 4k - lead .. 4k - lead + 3 (lead = (p * cap) mod 4); a
// quad whose four entries are valid and stay in one tile needs four compares.
__global__ void __launch_bounds__(256)
reduce_split_quad_kernel(const uint32_t* __restrict__ idx, const uint32_t* __restrict__ nnz,
                         int32_t P, uint64_t cap, uint32_t N, uint32_t ntiles,
                         uint32_t* __restrict__ split, int32_t* status) {
  griddep_wait();
  const uint32_t p = blockIdx.y, lane = lane_id();
  uint32_t n = nnz[p];
  if (n > cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, SPARCML_ERR_CAPACITY);
    n = (uint32_t)cap;
  }
  const uint64_t e0 = (uint64_t)p * cap;
  const uint32_t lead = (uint32_t)(e0 & 3u);
  const uint32_t* row = idx + e0;
  const uint4* quads = reinterpret_cast<const uint4*>(idx + (e0 - lead));
  // 32-bit positions: the host sends rows of at most 2^31 entries here
  const uint32_t nq = (lead + n + 3) / 4;
  split_close(row, n, P, p, N, ntiles, split);
  const uint32_t span = blockDim.x * kSplitQuads;
  bool bad = false;
  for (uint32_t k0 = blockIdx.x * span; k0 < nq; k0 += gridDim.x * span) {
    uint4 v[kSplitQuads];
    uint32_t before[kSplitQuads];
    // every quad of this span holds four entries of the row (CTA-uniform):
    // no per-quad range checks and no partial quads
    const bool interior = 4 * (uint64_t)k0 > lead && 4 * ((uint64_t)k0 + span) <= (uint64_t)lead + n;
    if (interior) {
#pragma unroll
      for (uint32_t u = 0; u < kSplitQuads; ++u) {
        const uint32_t k = k0 + u * blockDim.x + threadIdx.x;
        v[u] = ld_stream(quads + k);
        before[u] = lane == 0 ? row[4 * k - lead - 1] : 0u;
      }
#pragma unroll
      for (uint32_t u = 0; u < kSplitQuads; ++u) {
        const uint32_t k = k0 + u * blockDim.x + threadIdx.x;
        uint32_t prev = __shfl_up_sync(0xffffffffu, v[u].w, 1);
        if (lane == 0) prev = before[u];
        const uint4 q = v[u];
        const uint32_t jf = 4 * k - lead;
        const bool ok = prev < q.x && q.x < q.y && q.y < q.z && q.z < q.w && q.w < N;
        bad |= !ok;
        // tiles whose boundary falls in (prev, q.w]: none for most quads
        const uint32_t t0 = ok ? (prev >> kMiniShift) + 1 : 0u;
        const uint32_t t1 = ok ? (q.w >> kMiniShift) + 1 : 0u;
        const bool wide = t1 - t0 > 4;
        if (!wide) {
          for (uint32_t t = t0; t < t1; ++t) {
            const uint32_t b = t << kMiniShift;
            split[(uint64_t)t * P + p] = jf + (q.x < b) + (q.y < b) + (q.z < b);
          }
        }
        uint32_t todo = __ballot_sync(0xffffffffu, wide);
        while (todo) {
          const uint32_t src = __ffs(todo) - 1;
          todo &= todo - 1;
          const uint32_t a0 = __shfl_sync(0xffffffffu, t0, src);
          const uint32_t a1 = __shfl_sync(0xffffffffu, t1, src);
          const uint32_t sj = __shfl_sync(0xffffffffu, jf, src);
          const uint32_t sx = __shfl_sync(0xffffffffu, q.x, src);
          const uint32_t sy = __shfl_sync(0xffffffffu, q.y, src);
          const uint32_t sz = __shfl_sync(0xffffffffu, q.z, src);
          for (uint32_t t = a0 + lane; t < a1; t += 32) {
            const uint32_t b = t << kMiniShift;
            split[(uint64_t)t * P + p] = sj + (sx < b) + (sy < b) + (sz < b);
          }
        }
      }
      continue;
    }
#pragma unroll
    for (uint32_t u = 0; u < kSplitQuads; ++u) {
      const uint32_t k = k0 + u * blockDim.x + threadIdx.x;
      v[u] = k < nq ? ld_stream(quads + k) : make_uint4(0, 0, 0, 0);
      // entry before the quad: row[4k - lead - 1], inside the buffer when 4k > lead
      before[u] = (lane == 0 && k < nq && 4 * k > lead) ? row[4 * k - lead - 1] : 0u;
    }
#pragma unroll
    for (uint32_t u = 0; u < kSplitQuads; ++u) {
      const uint32_t k = k0 + u * blockDim.x + threadIdx.x;
      uint32_t prev = __shfl_up_sync(0xffffffffu, v[u].w, 1);
      if (lane == 0) prev = before[u];
      const uint4 q = v[u];
      const uint32_t jq = 4 * k;  // j + lead of the quad's first entry
      const bool live = k < nq;
      const bool full = live && jq > lead && n >= 4 && jq - lead <= n - 4;
      const uint32_t jf = jq - lead;
      // A full quad of a valid stream crosses the boundaries t * kMini for t
      // in [t0, t1), all in (prev, q.w]; the first entry at or past one is
      // found by three compares. A bad quad writes nothing (flagged).
      uint32_t t0 = 0, t1 = 0;
      if (full) {
        const bool ok = prev < q.x && q.x < q.y && q.y < q.z && q.z < q.w && q.w < N;
        bad |= !ok;
        if (ok) {
          t0 = (prev >> kMiniShift) + 1;
          t1 = (q.w >> kMiniShift) + 1;
        }
      }
      const bool wide = t1 - t0 > 4;
      if (!wide) {
        for (uint32_t t = t0; t < t1; ++t) {
          const uint32_t b = t << kMiniShift;
          split[(uint64_t)t * P + p] = jf + (q.x < b) + (q.y < b) + (q.z < b);
        }
      }
      uint32_t todo = __ballot_sync(0xffffffffu, wide);
      while (todo) {
        const uint32_t src = __ffs(todo) - 1;
        todo &= todo - 1;
        const uint32_t a0 = __shfl_sync(0xffffffffu, t0, src);
        const uint32_t a1 = __shfl_sync(0xffffffffu, t1, src);
        const uint32_t sj = __shfl_sync(0xffffffffu, jf, src);
        const uint32_t sx = __shfl_sync(0xffffffffu, q.x, src);
        const uint32_t sy = __shfl_sync(0xffffffffu, q.y, src);
        const uint32_t sz = __shfl_sync(0xffffffffu, q.z, src);
        for (uint32_t t = a0 + lane; t < a1; t += 32) {
          const uint32_t b = t << kMiniShift;
          split[(uint64_t)t * P + p] = sj + (sx < b) + (sy < b) + (sz < b);
        }
      }
      // quads cut by the row's ends: entry by entry
      const bool part = live && !full;
      if (!__any_sync(0xffffffffu, part)) continue;
      const uint32_t e[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (uint32_t i = 0; i < 4; ++i) {
        const uint32_t jj = jq + i;  // j + lead
        const bool ent = part && jj >= lead && jj - lead < n;
        const uint32_t j = jj - lead;
        const uint32_t pv = i == 0 ? prev : e[i - 1];
        uint32_t s0 = 0, s1 = 0;
        if (ent) {
          bad |= e[i] >= N || (j > 0 && e[i] <= pv);
          s0 = j > 0 ? mini_tiles_at_or_below(pv, N, ntiles) : 0u;
          s1 = max(s0, mini_tiles_at_or_below(e[i], N, ntiles));
        }
        split_fill(split, P, p, s0, s1, j);
      }
    }
  }
  if (bad) set_status(status, SPARCML_ERR_BAD_STREAM);
}

// Decoupled look-back for one warp's tile (the calling warp, all 32 lanes):
// publish the count, sum predecessors back to the nearest inclusive prefix,
// publish the inclusive prefix, return the exclusive offset. Tiles are
// claimed in ticket order, so every tile waited on is already running. Each
// wait is bounded (SPARCML_ERR_TIMEOUT, then it carries on).
__device__ uint32_t warp_lookback(const ReduceArgs& a, uint32_t tile, uint32_t count) {
  const uint32_t lane = lane_id();
  unsigned long long* st = a.tile_state;
  const bool inject = injected(a.inject);
  const uint32_t limit = inject ? kInjectSpinLimit : kSpinLimit;
  if (tile == 0) {
    if (lane == 0 && !inject) atomicExch(&st[0], kFlagInc | count);
    return 0;
  }
  if (lane == 0) atomicExch(&st[tile], kFlagAgg | count);
  uint32_t excl = 0;
  int64_t base = (int64_t)tile - 1;
  uint32_t spins = 0, backoff = 32;
  while (true) {
    const int64_t j = base - (int64_t)lane;
    const unsigned long long sv =
        j >= 0 ? *reinterpret_cast<volatile unsigned long long*>(&st[j]) : (2ull << 62);
    const unsigned long long flag = sv & (3ull << 62);
    const uint32_t inc = __ballot_sync(0xffffffffu, flag == kFlagInc);
    const uint32_t notready = __ballot_sync(0xffffffffu, flag == 0);
    const uint32_t upto = inc ? (uint32_t)(__ffs(inc) - 1) : 31u;  // lanes 0..upto count
    const uint32_t need = upto == 31 ? 0xffffffffu : ((2u << upto) - 1u);
    if (notready & need) {
      if (++spins > limit) {
        if (lane == 0) set_status(a.status, SPARCML_ERR_TIMEOUT);
        break;
      }
      __nanosleep(backoff);
      backoff = min(backoff * 2, 1024u);
      continue;
    }
    excl += warp_sum(lane <= upto ? (uint32_t)sv : 0u);
    if (inc) break;
    base -= 32;
  }
  if (lane == 0) atomicExch(&st[tile], kFlagInc | (excl + count));
  return excl;
}

// Warp tile epilogue, sparse-first: the CTA's kMiniWarps tiles take one
// offset by look-back (their counts summed), each tile its share in tile
// order. While the running union stays within cap_sparse a tile emits its
// present indices ascending (each lane the indices of its bitmap word), past
// it the dense slice. tile_info records which, for the fix-up pass; the last
// tile writes U. Called by every warp of the CTA (inactive ones add nothing).
// Presence word of lane i (indices 32i..32i+31 of the tile) from an
// accumulator that marks absent indices with kAbsent: 32 ballots.
__device__ __forceinline__ uint32_t presence_word(const uint32_t* acc) {
  const uint32_t lane = lane_id();
  uint32_t word = 0;
#pragma unroll 8
  for (uint32_t i = 0; i < kMiniWords; ++i) {
    const uint32_t b = __ballot_sync(0xffffffffu, acc[i * 32 + lane] != kAbsent);
    if (lane == i) word = b;
  }
  return word;
}

// `word`: the lane's presence word (0 for a tile past the end). `stage`
// (optional, kMini / 2 entries of the warp's own shared memory): a sparse
// tile of at most that many entries stages its offsets in order there and
// is written 32 consecutive entries at a time; otherwise each lane writes
// its word's entries.
__device__ __forceinline__ void mini_epilogue_lookback(const ReduceArgs& a, uint32_t m,
                                                       const uint32_t* acc, bool active,
                                                       uint32_t* sh /* [kMiniWarps + 1] */,
                                                       uint32_t word,
                                                       uint16_t* stage = nullptr) {
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t wincl = warp_incl_sum(__popc(word));
  const uint32_t count = __shfl_sync(0xffffffffu, wincl, 31);
  if (lane == 0) sh[warp] = count;
  __syncthreads();
  if (warp == 0) {
    const uint32_t total = warp_sum(lane < kMiniWarps ? sh[lane] : 0u);
    const uint32_t gexcl = warp_lookback(a, m / kMiniWarps, total);
    __syncwarp();
    if (lane == 0) sh[kMiniWarps] = gexcl;
  }
  __syncthreads();
  if (!active) return;
  uint32_t excl = sh[kMiniWarps];
  for (uint32_t w = 0; w < warp; ++w) excl += sh[w];
  const uint32_t tile_lo = m * kMini;
  const uint32_t tile_n = min(kMini, a.N - tile_lo);
  const uint32_t incl = excl + count;
  const bool dense = incl > a.cap_sparse;
  if (dense) {
    float* od = a.out_dense + tile_lo;
    for (uint32_t x = lane; x < tile_n; x += 32)
      od[x] = acc[x] == kAbsent ? op_neutral(a.op) : __uint_as_float(acc[x]);
  } else if (stage != nullptr && count <= kMini / 2) {  // warp-uniform
    uint32_t pos = wincl - __popc(word);
    uint32_t bits = word;
    while (bits) {
      stage[pos++] = (uint16_t)(lane * 32 + (__ffs(bits) - 1));
      bits &= bits - 1;
    }
    __syncwarp();
    for (uint32_t o = lane; o < count; o += 32) {
      const uint32_t x = stage[o];
      a.out_idx[excl + o] = tile_lo + x;
      a.out_val[excl + o] = __uint_as_float(acc[x]);
    }
  } else {
    uint32_t pos = excl + wincl - __popc(word);  // entries before word `lane`
    uint32_t bits = word;
    while (bits) {
      const uint32_t x = lane * 32 + (__ffs(bits) - 1);
      bits &= bits - 1;
      a.out_idx[pos] = tile_lo + x;
      a.out_val[pos] = __uint_as_float(acc[x]);
      ++pos;
    }
  }
  if (lane == 0) {
    a.tile_info[m] = make_uint2(excl, count | (dense ? 0x80000000u : 0u));
    if (m == a.ntiles - 1) {
      *a.out_nnz = incl;
      *a.out_is_dense = dense ? 1 : 0;
    }
  }
}

// Warp tile epilogue: presence bitmap (absent = kAbsent), dense slice with
// absent indices as +0.0f, and the tile's count added to the union size.
// `word`: the lane's presence word (indices 32 lane .. 32 lane + 31).
__device__ __forceinline__ void mini_epilogue(const ReduceArgs& a, uint32_t m, const uint32_t* acc,
                                              uint32_t word) {
  const uint32_t lane = lane_id();
  const uint32_t tile_lo = m * kMini;
  const uint32_t tile_n = min(kMini, a.N - tile_lo);
  const uint32_t count = warp_sum(__popc(word));
  float* od = a.out_dense + tile_lo;
  const float e = op_neutral(a.op);
  auto fix = [e](uint32_t b) { return b == kAbsent ? e : __uint_as_float(b); };
  if (tile_n == kMini && (reinterpret_cast<uintptr_t>(od) & 15) == 0) {
#pragma unroll
    for (uint32_t i = 0; i < kMini / 128; ++i) {
      const uint4 q = reinterpret_cast<const uint4*>(acc)[i * 32 + lane];
      reinterpret_cast<float4*>(od)[i * 32 + lane] = make_float4(fix(q.x), fix(q.y), fix(q.z), fix(q.w));
    }
  } else {
    for (uint32_t x = lane; x < tile_n; x += 32) od[x] = fix(acc[x]);
  }
  a.tile_bm[(uint64_t)m * kMiniWords + lane] = word;
  if (lane == 0 && count) atomicAdd(a.u_total, count);
}

// LB: sparse-first output with look-back, the CTA's group of tiles claimed by
// ticket (so every group waited on is already running); else dense-first
// (slice, bitmap and union size; the tile is the warp's grid position).
__device__ __forceinline__ uint32_t mini_tile_of_warp(const ReduceArgs& a, bool lb, uint32_t* sh) {
  if (!lb) return blockIdx.x * kMiniWarps + (threadIdx.x >> 5);
  if (threadIdx.x == 0) sh[0] = atomicAdd(a.ticket, 1u);
  __syncthreads();
  const uint32_t m = sh[0] * kMiniWarps + (threadIdx.x >> 5);
  __syncthreads();  // sh is reused by the epilogue
  return m;
}

// The entries of one node-major run of positions [0, total) into a warp's
// accumulator (absent = kAbsent): position x is entry lo[p] + (x - cpre[p]) of
// node p, cpre being the nodes' exclusive prefix. Each lane walks its
// positions x = lane, lane + 32, ...: it finds its node again only when x
// leaves the current node's range, and otherwise steps its entry pointers by
// 32. kMiniRounds rounds of loads are in flight at once. A round is applied
// at once when its indices are distinct (one node, or no index shared by two
// nodes); otherwise its nodes are applied one at a time, in order, so every
// index sees its nodes in ascending order.
// The signed 4-bit levels: lut[c] = +-(c & 7) / 7, negative when c & 8.
__device__ __forceinline__ void init_level_table(float* lut) {
  if (threadIdx.x < 16) {
    const float q = level_over_7(threadIdx.x & 7u);
    lut[threadIdx.x] = (threadIdx.x & 8u) ? -q : q;
  }
}

// load_value<true> with the 4-bit level read from the table above: one shared
// load in place of the selects, and the same bits (under round-to-nearest a
// product with the sign moved into a factor is the negated product).
__device__ __forceinline__ float load_value_lut(const ReduceArgs& a, uint32_t p, uint32_t j,
                                                const float* lut) {
  if (a.bits != 4) return load_value<true>(a, p, j);  // uniform branch
  const uint8_t byte = a.codes[(uint64_t)p * a.code_stride + (j >> 1)];
  const uint32_t b = a.bucket_shift < 32 ? j >> a.bucket_shift : j / a.bucket;
  const float scale = a.scales[(uint64_t)p * a.scale_stride + b];  // not behind the code
  const uint32_t code = (j & 1) ? (byte >> 4) : (byte & 15u);
  const float v = __fmul_rn(lut[code], scale);
  return (code & 7u) == 0 ? 0.0f : v;
}

template <bool Q4>
__device__ __forceinline__ void mini_accumulate(const ReduceArgs& a, int32_t kop, uint32_t* acc,
                                                uint32_t tile_lo, uint32_t tile_n,
                                                const uint32_t* lo, const uint32_t* cpre,
                                                uint32_t total, float e, const float* lut,
                                                uint8_t* tag /* [kMini] */,
                                                uint32_t* bm /* [kMiniWords] presence bits */) {
  const uint32_t lane = lane_id();
  // Position x of the tile's flattened entries belongs to the largest node q
  // with cpre[q] <= x (an empty node starts where its successor does, so the
  // search passes over it): a binary search per position, independent from
  // round to round, so a round's loads need not wait for the previous round's.
  const uint32_t P = (uint32_t)a.P;
  const uint32_t step0 = P > 1 ? 1u << (31 - __clz(P - 1)) : 0u;
  for (uint32_t r0 = 0; r0 < total; r0 += 32 * kMiniRounds) {
    uint32_t ix[kMiniRounds], pn[kMiniRounds];
    float vx[kMiniRounds];
#pragma unroll
    for (uint32_t u = 0; u < kMiniRounds; ++u) {
      const uint32_t x = r0 + 32 * u + lane;
      pn[u] = kMiniMaxP;  // no entry
      ix[u] = 0;
      vx[u] = 0.0f;
      if (x < total) {
        uint32_t q = 0;
        for (uint32_t st = step0; st; st >>= 1)
          if (q + st < P && cpre[q + st] <= x) q += st;
        const uint32_t j = lo[q] + (x - cpre[q]);
        pn[u] = q;
        ix[u] = ld_stream(a.idx + (uint64_t)q * a.cap + j);
        if constexpr (Q4) vx[u] = load_value_lut(a, q, j, lut);
        else vx[u] = ld_stream(a.val + (uint64_t)q * a.cap + j);
      }
    }
#pragma unroll
    for (uint32_t u = 0; u < kMiniRounds; ++u) {
      // live lanes are a prefix: lane 0 is live in every non-empty round
      const uint32_t first = __shfl_sync(0xffffffffu, pn[u], 0);
      if (first == kMiniMaxP) break;  // warp-uniform: later rounds are empty too
      const bool live = pn[u] != kMiniMaxP;
      const uint32_t off = ix[u] - tile_lo;
      const bool mine = live && off < tile_n;
      bool at_once = __all_sync(0xffffffffu, pn[u] == first || !live);  // one node: distinct
      if (!at_once) {
        // Several nodes: at once unless an index repeats in the round. Every
        // lane with an entry writes its id at its index and reads it back; a
        // repeat leaves some lane reading another's id. (The tags need no
        // clearing: a round reads only what it wrote.)
        if (mine) tag[off] = (uint8_t)lane;
        __syncwarp();
        at_once = !__any_sync(0xffffffffu, mine && tag[off] != lane);
      }
      if (mine) atomicOr(&bm[off >> 5], 1u << (off & 31));
      if (at_once) {
        if (mine) {
          const uint32_t old = acc[off];
          acc[off] = __float_as_uint(op_fold(kop, old == kAbsent ? e : __uint_as_float(old), vx[u]));
        }
      } else {
        const uint32_t last = __reduce_max_sync(0xffffffffu, live ? pn[u] : 0u);
        for (uint32_t q = first; q <= last; ++q) {  // node changes: one node at a time
          if (mine && pn[u] == q) {
            const uint32_t old = acc[off];
            acc[off] =
                __float_as_uint(op_fold(kop, old == kAbsent ? e : __uint_as_float(old), vx[u]));
          }
          __syncwarp();
        }
      }
      __syncwarp();
    }
  }
}

template <bool Q4, bool LB, bool ANY>
__global__ void __launch_bounds__(kMiniWarps * 32)
reduce_mini_kernel(ReduceArgs a) {
  griddep_wait();
  extern __shared__ __align__(16) uint32_t dyn[];
  const int32_t kop = ANY ? a.op : kOpSum;  // sum-only launches fold the branch away
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  __shared__ uint32_t sh[kMiniWarps + 1];
  __shared__ float lut[16];
  // repeat tags while folding; then the staged offsets of a sparse tile
  __shared__ __align__(16) uint8_t tags[kMiniWarps][kMini];
  __shared__ uint32_t bmw[kMiniWarps][kMiniWords];  // presence bits, set as entries are folded
  __shared__ uint32_t tk;                            // the CTA's ticket (sparse-first)
  // Sparse-first: the CTA's group of tiles is claimed by ticket (so every
  // group waited on is already running); the ticket is in flight while the
  // level table and the accumulators are initialised. Dense-first: the tile
  // is the warp's grid position.
  uint32_t ticket = 0;
  if (LB && threadIdx.x == 0) ticket = atomicAdd(a.ticket, 1u);
  if constexpr (Q4) init_level_table(lut);
  uint32_t* acc = dyn + warp * mini_warp_words(a.P);  // [kMini] float bits
  uint32_t* lo = acc + kAccWords;                      // [P] first entry in the tile
  uint32_t* cpre = lo + a.P;                           // [P + 1] first position
  // Absent indices hold kAbsent, a NaN that neither the sum (the GPU's NaN
  // results are 0x7fffffff) nor max/min (a NaN value never replaces the
  // partial result) ever leaves there: presence needs no bitmap. Bitwise or
  // can produce any pattern and is not run here.
#pragma unroll
  for (uint32_t i = 0; i < kMini / 128; ++i)
    reinterpret_cast<uint4*>(acc)[i * 32 + lane] = make_uint4(kAbsent, kAbsent, kAbsent, kAbsent);
  bmw[warp][lane] = 0;
  if (LB && threadIdx.x == 0) tk = ticket;
  if (LB || Q4) __syncthreads();
  const uint32_t m = (LB ? tk : blockIdx.x) * kMiniWarps + warp;
  if constexpr (!LB) {
    if (m >= a.ntiles) return;  // warp-uniform
  }
  const bool active = m < a.ntiles;
  const uint32_t tile_lo = m * kMini;
  const uint32_t tile_n = min(kMini, a.N - tile_lo);
  const float e = op_neutral(kop);
  uint32_t c[2] = {0, 0};
#pragma unroll
  for (uint32_t q = 0; q < 2; ++q) {
    const int32_t p = (int32_t)(lane + 32 * q);
    if (active && p < a.P) {  // a tile past the end (last CTA group) has no entries
      const uint32_t n = (uint32_t)min((uint64_t)a.nnz[p], a.cap);
      const uint32_t l = min(a.split[(uint64_t)m * a.P + p], n);
      const uint32_t h = min(a.split[(uint64_t)(m + 1) * a.P + p], n);
      lo[p] = l;
      c[q] = h > l ? h - l : 0u;
    }
  }
  {
    const uint32_t i0 = warp_incl_sum(c[0]), t0 = __shfl_sync(0xffffffffu, i0, 31);
    const uint32_t i1 = warp_incl_sum(c[1]);
    if (lane < (uint32_t)a.P) cpre[lane] = i0 - c[0];
    if (lane + 32 < (uint32_t)a.P) cpre[lane + 32] = t0 + i1 - c[1];
    if (lane == 31) cpre[a.P] = t0 + i1;
  }
  __syncwarp();
  const uint32_t total = cpre[a.P];
  if constexpr (!LB) {
    if (total > a.hot_thr) {  // warp-uniform: a Zipf-like head, for a whole CTA later
      if (lane == 0) a.hot[atomicAdd(a.hot_cnt, 1u)] = m;
      return;
    }
  }
  mini_accumulate<Q4>(a, kop, acc, tile_lo, tile_n, lo, cpre, total, e, lut, tags[warp],
                      bmw[warp]);
  __syncwarp();
  if constexpr (LB)
    mini_epilogue_lookback(a, m, acc, active, sh, bmw[warp][lane],
                           reinterpret_cast<uint16_t*>(tags[warp]));
  else mini_epilogue(a, m, acc, bmw[warp][lane]);
}

// Vector form of the warp tile (fp32 values, idx and val 16-byte aligned):
// each node's entries of the tile are read as the 16-byte quads of the
// buffer that hold them, so a lane takes 4 entries per round with two
// 128-bit loads. The first and last quad of a node are masked to the node's
// range; a quad that would run past the end of the buffer is read entry by
// entry. A round of 32 quads spans a few nodes: their entries are added one
// node at a time, in ascending order.
constexpr uint32_t kQuadRounds = 4;

template <bool LB, bool ANY>
__global__ void __launch_bounds__(kMiniWarps * 32)
reduce_mini_quad_kernel(ReduceArgs a) {
  griddep_wait();
  extern __shared__ __align__(16) uint32_t dyn[];
  const int32_t kop = ANY ? a.op : kOpSum;  // sum-only launches fold the branch away
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  __shared__ uint32_t sh[kMiniWarps + 1];
  const uint32_t m = mini_tile_of_warp(a, LB, sh);
  if constexpr (!LB) {
    if (m >= a.ntiles) return;  // warp-uniform
  }
  const bool active = m < a.ntiles;
  uint32_t* acc = dyn + warp * kMiniWarpWords;        // [kMini] float bits
  uint32_t* lo = acc + kAccWords;                      // [P] first entry in the tile
  uint32_t* qpre = lo + kMiniMaxP;                     // [P + 1] first quad position
  uint32_t* hi = qpre + kMiniMaxP + 1;                 // [P] end entry in the tile
  const uint32_t tile_lo = m * kMini;
  const uint32_t tile_n = min(kMini, a.N - tile_lo);
  const float e = op_neutral(kop);
#pragma unroll
  for (uint32_t i = 0; i < kMini / 128; ++i)
    reinterpret_cast<uint4*>(acc)[i * 32 + lane] = make_uint4(kAbsent, kAbsent, kAbsent, kAbsent);
  uint32_t c[2] = {0, 0};
#pragma unroll
  for (uint32_t q = 0; q < 2; ++q) {
    const int32_t p = (int32_t)(lane + 32 * q);
    if (active && p < a.P) {  // a tile past the end (last CTA group) has no entries
      const uint32_t n = (uint32_t)min((uint64_t)a.nnz[p], a.cap);
      const uint32_t l = min(a.split[(uint64_t)m * a.P + p], n);
      const uint32_t h = min(a.split[(uint64_t)(m + 1) * a.P + p], n);
      lo[p] = l;
      hi[p] = h;
      if (h > l) {  // quads of the buffer holding entries [row + l, row + h)
        const uint64_t row = (uint64_t)p * a.cap;
        c[q] = (uint32_t)(((row + h + 3) >> 2) - ((row + l) >> 2));
      }
    }
  }
  {
    const uint32_t i0 = warp_incl_sum(c[0]), t0 = __shfl_sync(0xffffffffu, i0, 31);
    const uint32_t i1 = warp_incl_sum(c[1]);
    if (lane < (uint32_t)a.P) qpre[lane] = i0 - c[0];
    if (lane + 32 < (uint32_t)a.P) qpre[lane + 32] = t0 + i1 - c[1];
    if (lane == 31) qpre[a.P] = t0 + i1;
  }
  __syncwarp();
  const uint32_t total = qpre[a.P];
  if constexpr (!LB) {
    if (total > a.hot_thr / 4) {  // warp-uniform (quads): a Zipf-like head, for a CTA later
      if (lane == 0) a.hot[atomicAdd(a.hot_cnt, 1u)] = m;
      return;
    }
  }
  const uint64_t buf_end = (uint64_t)a.P * a.cap;  // entries in the buffer
  const uint4* idx4 = reinterpret_cast<const uint4*>(a.idx);
  const float4* val4 = reinterpret_cast<const float4*>(a.val);
  // lane state for its current node: quad range and the masks of its ends
  uint32_t x = lane, p = 0, qend = 0, y = 0, nq = 0, head = 0xfu, tail = 0xfu;
  uint64_t g = 0;  // buffer quad of position x
  for (uint32_t r0 = 0; r0 < total; r0 += 32 * kQuadRounds) {
    uint4 ix[kQuadRounds];
    float4 vx[kQuadRounds];
    uint32_t pn[kQuadRounds], mk[kQuadRounds];
#pragma unroll
    for (uint32_t u = 0; u < kQuadRounds; ++u) {
      pn[u] = kMiniMaxP;  // no entry
      mk[u] = 0;
      ix[u] = make_uint4(0, 0, 0, 0);
      vx[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (x < total) {
        if (x >= qend) {
          while (qpre[p + 1] <= x) ++p;
          qend = qpre[p + 1];
          const uint64_t e0 = (uint64_t)p * a.cap + lo[p], e1 = (uint64_t)p * a.cap + hi[p];
          nq = qend - qpre[p];
          y = x - qpre[p];
          g = (e0 >> 2) + y;
          head = (0xfu << (uint32_t)(e0 & 3)) & 0xfu;
          tail = (1u << (uint32_t)(((e1 - 1) & 3) + 1)) - 1u;
        }
        uint32_t mask = 0xfu;
        if (y == 0) mask &= head;
        if (y == nq - 1) mask &= tail;
        pn[u] = p;
        mk[u] = mask;
        if (4 * g + 4 <= buf_end) {
          ix[u] = ld_stream(idx4 + g);
          const uint4 vb = ld_stream(reinterpret_cast<const uint4*>(val4 + g));
          vx[u] = make_float4(__uint_as_float(vb.x), __uint_as_float(vb.y), __uint_as_float(vb.z),
                              __uint_as_float(vb.w));
        } else {  // the buffer's last, partial quad: its valid entries only
          const uint32_t* ie = a.idx + 4 * g;
          const float* ve = a.val + 4 * g;
          if (mask & 1u) { ix[u].x = ie[0]; vx[u].x = ve[0]; }
          if (mask & 2u) { ix[u].y = ie[1]; vx[u].y = ve[1]; }
          if (mask & 4u) { ix[u].z = ie[2]; vx[u].z = ve[2]; }
          if (mask & 8u) { ix[u].w = ie[3]; vx[u].w = ve[3]; }
        }
      }
      x += 32;
      y += 32;
      g += 32;
    }
    auto add = [&](uint32_t iv, float v) {
      const uint32_t off = iv - tile_lo;
      if (off < tile_n) {
        const uint32_t old = acc[off];
        acc[off] = __float_as_uint(op_fold(kop, old == kAbsent ? e : __uint_as_float(old), v));
      }
    };
    auto add_quad = [&](uint32_t u) {
      if (mk[u] & 1u) add(ix[u].x, vx[u].x);
      if (mk[u] & 2u) add(ix[u].y, vx[u].y);
      if (mk[u] & 4u) add(ix[u].z, vx[u].z);
      if (mk[u] & 8u) add(ix[u].w, vx[u].w);
    };
#pragma unroll
    for (uint32_t u = 0; u < kQuadRounds; ++u) {
      const uint32_t first = __shfl_sync(0xffffffffu, pn[u], 0);
      if (first == kMiniMaxP) break;  // warp-uniform: later rounds are empty too
      const bool live = pn[u] != kMiniMaxP;
      if (__all_sync(0xffffffffu, pn[u] == first || !live)) {  // one node: distinct indices
        if (live) add_quad(u);
      } else {
        const uint32_t last = __reduce_max_sync(0xffffffffu, live ? pn[u] : 0u);
        for (uint32_t q = first; q <= last; ++q) {  // one node at a time
          if (live && pn[u] == q) add_quad(u);
          __syncwarp();
        }
      }
      __syncwarp();
    }
  }
  if constexpr (LB) mini_epilogue_lookback(a, m, acc, active, sh, active ? presence_word(acc) : 0u);
  else mini_epilogue(a, m, acc, presence_word(acc));
}

// A hot tile (dense-first mode, more entries than hot_thr: a skewed,
// Zipf-like head): one CTA walks the nodes in ascending order. For node p the
// CTA takes the node's run of the tile, at most kMini entries with distinct
// indices, kMini / kHotThreads entries a thread, folds them into the shared
// accumulator, and a barrier orders node p before node p + 1, so every index
// is folded in node order. Loads run kHotAhead nodes ahead of the folds. Warp 0
// then writes the tile's dense slice, bitmap and union count like any warp
// tile. A CTA takes the hot tiles h, h + grid, ...
template <bool Q4, bool ANY>
__global__ void __launch_bounds__(kHotThreads)
reduce_hot_tile_kernel(ReduceArgs a) {
  griddep_wait();
  constexpr uint32_t R = kMini / kHotThreads;  // entries of a node's run per thread
  __shared__ __align__(16) uint32_t acc[kMini];
  __shared__ uint32_t run_lo[kMiniMaxP], run_n[kMiniMaxP];
  const uint32_t nhot = *a.hot_cnt;
  const int32_t kop = ANY ? a.op : kOpSum;
  const float e = op_neutral(kop);
  const uint32_t t = threadIdx.x;
  for (uint32_t h = blockIdx.x; h < nhot; h += gridDim.x) {  // CTA-uniform
    const uint32_t m = a.hot[h];
    const uint32_t tile_lo = m * kMini;
    const uint32_t tile_n = min(kMini, a.N - tile_lo);
    for (uint32_t i = t; i < kMini / 4; i += kHotThreads)
      reinterpret_cast<uint4*>(acc)[i] = make_uint4(kAbsent, kAbsent, kAbsent, kAbsent);
    if (t < (uint32_t)a.P) {
      const uint32_t n = (uint32_t)min((uint64_t)a.nnz[t], a.cap);
      const uint32_t l = min(a.split[(uint64_t)m * a.P + t], n);
      const uint32_t hi = min(a.split[(uint64_t)(m + 1) * a.P + t], n);
      run_lo[t] = l;
      run_n[t] = hi > l ? hi - l : 0u;  // beyond kMini only for an invalid stream (flagged)
    }
    __syncthreads();
    for (int32_t p0 = 0; p0 < a.P; p0 += kHotAhead) {
      uint32_t ix[kHotAhead][R];
      float vx[kHotAhead][R];
#pragma unroll
      for (uint32_t u = 0; u < kHotAhead; ++u) {
        const int32_t p = p0 + (int32_t)u;
#pragma unroll
        for (uint32_t r = 0; r < R; ++r) {
          ix[u][r] = ~0u;  // no entry: off is never below tile_n
          vx[u][r] = 0.0f;
          const uint32_t j = t + r * kHotThreads;
          if (p < a.P && j < run_n[p]) {
            const uint32_t jj = run_lo[p] + j;
            ix[u][r] = ld_stream(a.idx + (uint64_t)p * a.cap + jj);
            if constexpr (Q4) vx[u][r] = load_value<Q4>(a, (uint32_t)p, jj);
            else vx[u][r] = ld_stream(a.val + (uint64_t)p * a.cap + jj);
          }
        }
      }
#pragma unroll
      for (uint32_t u = 0; u < kHotAhead; ++u) {
#pragma unroll
        for (uint32_t r = 0; r < R; ++r) {
          const uint32_t off = ix[u][r] - tile_lo;
          if (ix[u][r] != ~0u && off < tile_n) {
            const uint32_t old = acc[off];
            acc[off] = __float_as_uint(op_fold(kop, old == kAbsent ? e : __uint_as_float(old), vx[u][r]));
          }
        }
        __syncthreads();  // node p0 + u is folded in before node p0 + u + 1
      }
    }
    if (t < 32) mini_epilogue(a, m, acc, presence_word(acc));
    __syncthreads();  // warp 0 has read acc and run_* before the next tile
  }
}

// Warp-tile mode, last pass: the union size U decides dense or sparse; a
// sparse result is compacted from the dense slices and bitmaps, groups of 8
// warp tiles per CTA taking their offsets by decoupled look-back.
__global__ void __launch_bounds__(kReduceThreads)
reduce_mini_compact_kernel(ReduceArgs a) {
  griddep_wait();
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t bc[3];
  const uint32_t U = *a.u_total;
  const bool dense = U > a.cap_sparse;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *a.out_nnz = U;
    *a.out_is_dense = dense ? 1 : 0;
  }
  if (dense) return;
  if (threadIdx.x == 0) bc[0] = atomicAdd(a.ticket, 1u);
  __syncthreads();
  const uint32_t g = bc[0];  // group of kReduceThreads bitmap words
  const uint64_t wi = (uint64_t)g * kReduceThreads + threadIdx.x;
  const uint64_t nwords = (uint64_t)a.ntiles * kMiniWords;
  const uint32_t word = wi < nwords ? a.tile_bm[wi] : 0u;
  uint32_t tot;
  const uint32_t ex = block_excl_scan(__popc(word), scratch, &tot);
  tile_lookback(a, g, tot, &bc[2]);
  __syncthreads();
  // Each warp writes its 32 words, lane b taking bit b of a word: the dense
  // slice is read in 128-byte rows and a word's entries go out side by side
  // (a full word, the Zipf head, costs one round). Eight words' values are
  // loaded before any of them is stored, so the loads overlap.
  const uint32_t lane = lane_id();
  const uint32_t pos0 = bc[2] + ex;
  const uint64_t wbase = (uint64_t)g * kReduceThreads + (threadIdx.x & ~31u);
  const uint32_t below = (1u << lane) - 1u;
  for (uint32_t k0 = 0; k0 < 32; k0 += 8) {
    uint32_t wk[8];
    float v[8];
#pragma unroll
    for (uint32_t u = 0; u < 8; ++u) {
      wk[u] = __shfl_sync(0xffffffffu, word, k0 + u);
      v[u] = (wk[u] >> lane) & 1u ? a.out_dense[(wbase + k0 + u) * 32 + lane] : 0.0f;
    }
#pragma unroll
    for (uint32_t u = 0; u < 8; ++u) {
      const uint32_t pk = __shfl_sync(0xffffffffu, pos0, k0 + u);
      if ((wk[u] >> lane) & 1u) {
        const uint32_t pos = pk + __popc(wk[u] & below);
        if (pos < a.cap_sparse) {
          a.out_idx[pos] = (uint32_t)((wbase + k0 + u) * 32 + lane);
          a.out_val[pos] = v[u];
        }
      }
    }
  }
}

// Dense-first mode: U = sum of the tiles' counts, the dense flag, and each
// tile's exclusive offset (one CTA).
__global__ void __launch_bounds__(1024)
reduce_finalize_kernel(uint2* __restrict__ tile_info, uint32_t ntiles, uint32_t cap_sparse,
                       uint32_t* __restrict__ out_nnz, int32_t* __restrict__ out_is_dense) {
  griddep_wait();
  __shared__ uint32_t scratch[34];
  uint32_t run = 0;
  for (uint32_t t0 = 0; t0 < ntiles; t0 += blockDim.x) {
    const uint32_t i = t0 + threadIdx.x;
    const uint32_t c = i < ntiles ? tile_info[i].y : 0u;
    uint32_t tot;
    const uint32_t ex = block_excl_scan(c, scratch, &tot);
    if (i < ntiles) tile_info[i].x = run + ex;
    run += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *out_nnz = run;
    *out_is_dense = run > cap_sparse ? 1 : 0;
  }
}

// Dense-first mode, sparse result after all: the tile's present entries,
// ascending, from its dense slice and saved bitmap (words_per_tile <= blockDim).
__global__ void __launch_bounds__(kReduceThreads)
reduce_compact_kernel(const int32_t* __restrict__ is_dense, const uint2* __restrict__ tile_info,
                      const uint32_t* __restrict__ tile_bm, const float* __restrict__ out_dense,
                      uint32_t* __restrict__ out_idx, float* __restrict__ out_val,
                      uint32_t words_per_tile) {
  griddep_wait();
  __shared__ uint32_t scratch[34];
  if (*is_dense) return;
  const uint32_t tile = blockIdx.x, tile_lo = tile * words_per_tile * 32;
  const uint32_t word = threadIdx.x < words_per_tile
                            ? tile_bm[(uint64_t)tile * words_per_tile + threadIdx.x] : 0u;
  uint32_t tot;
  uint32_t pos = tile_info[tile].x + block_excl_scan(__popc(word), scratch, &tot);
  uint32_t bits = word;
  while (bits) {
    const uint32_t b = __ffs(bits) - 1;
    bits &= bits - 1;
    const uint32_t i = tile_lo + threadIdx.x * 32 + b;
    out_idx[pos] = i;
    out_val[pos] = out_dense[i];
    ++pos;
  }
}

// Sparse regime: tiles of a.tile_w indices (up to kMaxTileW), chosen so a
// tile holds about two thousand entries. Shared memory scales with the
// tile's union, not its width: a presence bitmap is built first, its prefix
// popcounts give every present index a slot (its rank in the tile), and the
// sums go to a compact fp32 array of slots. Accumulation keeps ascending node
// order (barrier after each node with entries in a batch), so the bits equal
// the dense-accumulator kernel's. Tiles whose union exceeds kAccCap are
// accumulated in several slot windows.
constexpr uint32_t kMaxTileW = 1u << 17;
constexpr uint32_t kAccCap = 8192;
constexpr int32_t kMaxSparseP = 1024;

template <bool Q4, bool ANY>
__global__ void __launch_bounds__(kReduceThreads)
reduce_sparse_tile_kernel(ReduceArgs a) {
  griddep_wait();
  extern __shared__ __align__(16) uint32_t dyn[];
  const int32_t kop = ANY ? a.op : kOpSum;  // sum-only launches fold the branch away
  const uint32_t W = a.tile_w / 32;
  uint32_t* bm = dyn;                                    // [W] presence bits
  uint32_t* woff = bm + W;                               // [W] slots before each word
  float* acc = reinterpret_cast<float*>(woff + W);       // [kAccCap] compact sums
  uint32_t* lo = reinterpret_cast<uint32_t*>(acc + kAccCap);  // [P]
  uint32_t* pre = lo + a.P;                              // [P + 1]
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t bc[4];
  const uint32_t t = threadIdx.x, lane = lane_id();

  if (t == 0) {
    bc[0] = atomicAdd(a.ticket, 1u);
    bc[1] = 0;
  }
  for (uint32_t w = t; w < W; w += blockDim.x) bm[w] = 0;
  __syncthreads();
  const uint32_t tile = bc[0];
  const uint32_t tile_lo = tile * a.tile_w;
  const uint32_t tile_n = min(a.tile_w, a.N - tile_lo);
  const bool last = tile == a.ntiles - 1;
  for (int32_t p = t; p < a.P; p += blockDim.x) {
    uint32_t n = a.nnz[p];
    if (n > a.cap) {
      set_status(a.status, SPARCML_ERR_CAPACITY);
      n = (uint32_t)a.cap;
    }
    const uint32_t l = a.split[(uint64_t)tile * a.P + p];
    uint32_t h = a.split[(uint64_t)(tile + 1) * a.P + p];
    if (last && h < n) set_status(a.status, SPARCML_ERR_BAD_STREAM);  // idx >= N
    if (h < l) {
      set_status(a.status, SPARCML_ERR_BAD_STREAM);
      h = l;
    }
    lo[p] = l;
    pre[p] = h - l;
    atomicMax(&bc[1], n);
  }
  __syncthreads();
  uint32_t E = 0;
  for (int32_t base = 0; base < a.P; base += blockDim.x) {
    const int32_t p = base + (int32_t)t;
    const uint32_t c = p < a.P ? pre[p] : 0u;
    uint32_t tot;
    const uint32_t ex = block_excl_scan(c, scratch, &tot);
    if (p < a.P) pre[p] = E + ex;
    E += tot;
    __syncthreads();
  }
  if (t == 0) pre[a.P] = E;
  __syncthreads();
  const bool dense_certain = bc[1] > a.cap_sparse;
  auto node_of = [&](uint32_t v) {
    uint32_t l = 0, h = (uint32_t)a.P;
    while (h - l > 1) {
      const uint32_t m = (l + h) >> 1;
      if (pre[m] <= v) l = m; else h = m;
    }
    return l;
  };
  const uint32_t batch = blockDim.x * kUnroll;
  const bool resident = E <= batch;  // all entries stay in registers
  uint32_t iv[kUnroll], pv[kUnroll];
  float vv[kUnroll];
  // Load batch c0 into registers; entries that fail the stream checks get
  // pv = kNoNode and are skipped.
  constexpr uint32_t kNoNode = 0xffffffffu;
  auto load_batch = [&](uint32_t c0) {
#pragma unroll
    for (uint32_t u = 0; u < kUnroll; ++u) {
      const uint32_t v = c0 + u * blockDim.x + t;
      iv[u] = 0;
      vv[u] = 0.0f;
      pv[u] = kNoNode;
      if (v < E) {
        const uint32_t p = node_of(v);
        const uint32_t j = lo[p] + (v - pre[p]);
        iv[u] = a.idx[(uint64_t)p * a.cap + j];
        vv[u] = load_value<Q4>(a, p, j);
        pv[u] = p;
      }
    }
#pragma unroll
    for (uint32_t u = 0; u < kUnroll; ++u) {
      const uint32_t v = c0 + u * blockDim.x + t;
      uint32_t prev = __shfl_up_sync(0xffffffffu, iv[u], 1);
      if (v < E) {
        const uint32_t p = pv[u];
        const uint32_t j = lo[p] + (v - pre[p]);
        if ((lane == 0 || v == pre[p]) && j > 0) prev = a.idx[(uint64_t)p * a.cap + j - 1];
        if (!((j == 0 || prev < iv[u]) && iv[u] - tile_lo < tile_n)) {
          set_status(a.status, SPARCML_ERR_BAD_STREAM);
          pv[u] = kNoNode;
        }
      }
    }
  };
  // 1. presence bits
  for (uint32_t c0 = 0; c0 < E; c0 += batch) {
    load_batch(c0);
#pragma unroll
    for (uint32_t u = 0; u < kUnroll; ++u)
      if (pv[u] != kNoNode) {
        const uint32_t off = iv[u] - tile_lo;
        atomicOr(&bm[off >> 5], 1u << (off & 31));
      }
  }
  __syncthreads();
  // 2. slots: exclusive prefix of the words' popcounts (consecutive words per thread)
  const uint32_t wpt = (W + blockDim.x - 1) / blockDim.x;
  uint32_t cnt = 0;
  for (uint32_t i = 0; i < wpt; ++i) {
    const uint32_t w = t * wpt + i;
    cnt += w < W ? __popc(bm[w]) : 0u;
  }
  uint32_t U;
  uint32_t run = block_excl_scan(cnt, scratch, &U);
  for (uint32_t i = 0; i < wpt; ++i) {
    const uint32_t w = t * wpt + i;
    if (w < W) {
      woff[w] = run;
      run += __popc(bm[w]);
    }
  }
  // 3. the tile's output offset
  tile_lookback(a, tile, U, &bc[2]);
  __syncthreads();
  const uint32_t excl = bc[2];
  const uint32_t incl = excl + U;
  const bool dense = dense_certain || incl > a.cap_sparse;
  // 4. accumulate and emit, slot window by slot window
  for (uint32_t s0 = 0; s0 < U || (s0 == 0 && dense); s0 += kAccCap) {
    const uint32_t win = min(kAccCap, U - min(U, s0));
    for (uint32_t i = t; i < win; i += blockDim.x) acc[i] = op_neutral(kop);
    __syncthreads();
    for (uint32_t c0 = 0; c0 < E; c0 += batch) {
      if (!resident) load_batch(c0);
      const uint32_t c1 = min(c0 + batch, E);
      const uint32_t p_first = node_of(c0), p_last = node_of(c1 - 1);
      for (uint32_t p = p_first; p <= p_last; ++p) {
        if (pre[p + 1] == pre[p]) continue;  // no entries: no barrier needed
#pragma unroll
        for (uint32_t u = 0; u < kUnroll; ++u) {
          if (pv[u] == p) {
            const uint32_t off = iv[u] - tile_lo, w = off >> 5;
            const uint32_t slot = woff[w] + __popc(bm[w] & ((1u << (off & 31)) - 1u));
            if (slot - s0 < win) acc[slot - s0] = op_fold(kop, acc[slot - s0], vv[u]);
          }
        }
        __syncthreads();
      }
    }
    if (dense) {
      // every index of the tile once: present ones in the window of their slot,
      // absent ones (+0.0f) in the first window
      float* od = a.out_dense + tile_lo;
      for (uint32_t x = t; x < tile_n; x += blockDim.x) {
        const uint32_t w = x >> 5, bit = 1u << (x & 31);
        if (bm[w] & bit) {
          const uint32_t slot = woff[w] + __popc(bm[w] & (bit - 1u));
          if (slot - s0 < win) od[x] = acc[slot - s0];
        } else if (s0 == 0) {
          od[x] = op_neutral(kop);
        }
      }
    } else {
      for (uint32_t w = t; w < W; w += blockDim.x) {
        uint32_t bits = bm[w];
        uint32_t slot = woff[w];
        while (bits) {
          const uint32_t b = __ffs(bits) - 1;
          bits &= bits - 1;
          if (slot - s0 < win) {
            a.out_idx[excl + slot] = tile_lo + w * 32 + b;
            a.out_val[excl + slot] = acc[slot - s0];
          }
          ++slot;
        }
      }
    }
    __syncthreads();
  }
  if (t == 0) {
    a.tile_info[tile] = make_uint2(excl, U | (dense ? 0x80000000u : 0u));
    if (last) {
      *a.out_nnz = incl;
      *a.out_is_dense = dense ? 1 : 0;
    }
  }
}

// Dense result: rewrite the leading tiles that were emitted sparse.
__global__ void __launch_bounds__(256)
reduce_fixup_kernel(const int32_t* __restrict__ is_dense, const uint2* __restrict__ tile_info,
                    const uint32_t* __restrict__ out_idx, const float* __restrict__ out_val,
                    float* __restrict__ out_dense, uint32_t N, uint32_t tile_w, uint32_t ntiles,
                    float neutral) {
  griddep_wait();
  if (*is_dense == 0) return;
  for (uint32_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {  // block-uniform
    const uint2 info = tile_info[tile];
    if (info.y & 0x80000000u) continue;
    const uint32_t tile_lo = tile * tile_w;
    const uint32_t tile_n = min(tile_w, N - tile_lo);
    for (uint32_t x = threadIdx.x; x < tile_n; x += blockDim.x) out_dense[tile_lo + x] = neutral;
    __syncthreads();
    for (uint32_t e = threadIdx.x; e < info.y; e += blockDim.x) {
      const uint32_t i = out_idx[info.x + e];
      if (i - tile_lo < tile_n) out_dense[i] = out_val[info.x + e];
    }
    __syncthreads();
  }
}

// Blocks of the fix-up pass: each walks tiles; a sparse result exits at once.
inline unsigned fixup_grid(uint32_t ntiles) { return std::min<uint32_t>(ntiles, 1216u); }

struct ReduceLayout {
  size_t ticket, state, info, split, bm, hot, total;
};

ReduceLayout reduce_layout(int32_t P, uint64_t N) {
  // sized for the finest tiling any regime uses (kMini-index tiles)
  const size_t ntiles = (N + kMini - 1) / kMini;
  ReduceLayout l;
  l.ticket = 64;
  l.state = 256;
  l.info = align_up(l.state + 8 * ntiles, 256);
  l.split = align_up(l.info + 8 * ntiles, 256);
  l.bm = align_up(l.split + 4 * (ntiles + 1) * (size_t)P, 256);
  const size_t bm_words = std::max((N + kTile - 1) / kTile * (size_t)kWords, ntiles * 32);
  l.hot = align_up(l.bm + 4 * bm_words, 256);
  l.total = align_up(l.hot + 4 * ntiles, 256);
  return l;
}

template <bool Q4>
int launch_reduce(ReduceArgs a, void* ws, size_t ws_bytes, cudaStream_t s,
                  void* const* events) {
  auto mark = [&](int i) {
    if (events && events[i]) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
  };
  const ReduceLayout l = reduce_layout(a.P, a.N);
  if (ws_bytes < l.total) return SPARCML_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  a.status = reinterpret_cast<int32_t*>(w);
  a.ticket = reinterpret_cast<uint32_t*>(w + l.ticket);
  a.tile_state = reinterpret_cast<unsigned long long*>(w + l.state);
  a.tile_info = reinterpret_cast<uint2*>(w + l.info);
  uint32_t* split = reinterpret_cast<uint32_t*>(w + l.split);
  a.split = split;
  a.tile_bm = reinterpret_cast<uint32_t*>(w + l.bm);
  a.u_total = reinterpret_cast<uint32_t*>(w + 128);  // cleared with the ticket below
  a.hot_cnt = reinterpret_cast<uint32_t*>(w + 192);  // likewise
  a.hot = reinterpret_cast<uint32_t*>(w + l.hot);
  a.inject = reinterpret_cast<const uint32_t*>(w + kInjectOffset);
  // Clear the ticket and the look-back states (the status word is kept).
  if (cudaMemsetAsync(w + l.ticket, 0, l.info - l.ticket, s) != cudaSuccess)
    return SPARCML_ERR_CUDA;
  // Regime: the entries of an 8,192-index tile are at most P * cap * 8192 / N.
  // Sparse inputs take wide tiles (about 2,048 entries each) with a compact
  // accumulator; denser ones the dense-accumulator tile of kTile indices.
  const double est = (double)a.P * (double)a.cap * kTile / (double)a.N;
  uint32_t tile_w = kTile;
  // Few nodes covering at least N/16 indices: one warp per kMini-index tile.
  const bool mini = a.P <= kMiniMaxP && 16.0 * (double)a.P * (double)a.cap >= (double)a.N &&
                    a.op != kOpOr;  // warp tiles mark absent indices with a NaN pattern
  const bool sparse = !mini && a.P <= kMaxSparseP && est <= 2048.0;
  if (sparse) {
    while (tile_w < kMaxTileW && est * (2.0 * tile_w / kTile) <= 1024.0 && tile_w < a.N)
      tile_w *= 2;
  }
  if (mini) tile_w = kMini;
  a.tile_w = tile_w;
  a.hot_thr = (uint32_t)std::min<double>(
      std::max<double>(kHot, kHotRatio * (double)a.P * (double)a.cap * kMini / (double)a.N),
      (double)kMini * kMiniMaxP);
  a.ntiles = (uint32_t)((a.N + tile_w - 1) / tile_w);
  mark(0);
  if (mini) {
    // split table by one streaming pass (also validates the streams)
    const bool quads = (reinterpret_cast<uintptr_t>(a.idx) & 15) == 0 &&
                       ((uint64_t)a.P * a.cap) % 4 == 0 && a.cap <= (1ull << 31);
    const uint64_t per_block = quads ? 256 * 4 * kSplitQuads : 256 * kSplitBatch;
    const uint32_t gx = (uint32_t)std::max<uint64_t>(
        1, std::min<uint64_t>((a.cap + per_block - 1) / per_block, 2432 / (uint64_t)a.P));
    if (quads)
      launch_pdl(reduce_split_quad_kernel, dim3(gx, (unsigned)a.P), 256, 0, s,
          a.idx, a.nnz, a.P, a.cap, a.N, a.ntiles, split, a.status);
    else
      launch_pdl(reduce_split_stream_kernel, dim3(gx, (unsigned)a.P), 256, 0, s,
          a.idx, a.nnz, a.P, a.cap, a.N, a.ntiles, split, a.status);
    if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
    const unsigned grid = (a.ntiles + kMiniWarps - 1) / kMiniWarps;
    const bool vec = !Q4 && (reinterpret_cast<uintptr_t>(a.idx) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.val) & 15) == 0;
    const size_t smem =
        (size_t)kMiniWarps * (vec ? kMiniWarpWords : mini_warp_words(a.P)) * sizeof(uint32_t);
    // A possibly dense result (P * cap >= N / 4) is written dense-first; else
    // sparse-first with look-back and a fix-up if the union crosses after all.
    const bool lb = 4.0 * (double)a.P * (double)a.cap < (double)a.N;
    const bool any = a.op != kOpSum;
    auto go = [&](auto kernel) {
      if (!ensure_smem(reinterpret_cast<const void*>(kernel), smem)) return false;
      launch_pdl(kernel, grid, kMiniWarps * 32, smem, s, a);
      return true;
    };
    bool ok;
    if (vec)
      ok = lb ? (any ? go(reduce_mini_quad_kernel<true, true>) : go(reduce_mini_quad_kernel<true, false>))
              : (any ? go(reduce_mini_quad_kernel<false, true>) : go(reduce_mini_quad_kernel<false, false>));
    else
      ok = lb ? (any ? go(reduce_mini_kernel<Q4, true, true>) : go(reduce_mini_kernel<Q4, true, false>))
              : (any ? go(reduce_mini_kernel<Q4, false, true>) : go(reduce_mini_kernel<Q4, false, false>));
    if (!ok) return SPARCML_ERR_CUDA;
    if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
    mark(1);
    if (lb) {
      launch_pdl(reduce_fixup_kernel, fixup_grid(a.ntiles), 256, 0, s, a.out_is_dense, a.tile_info, a.out_idx,
                                                   a.out_val, a.out_dense, a.N, a.tile_w, a.ntiles,
        a.op == kOpMax ? -INFINITY : a.op == kOpMin ? INFINITY : 0.0f);
      if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
      mark(2);
      note_launches(3);
      return SPARCML_OK;
    }
    {  // the tiles too hot for one warp, a CTA each. A deferred tile holds more
       // than hot_thr - 8 P entries (quads cut at the runs' ends): hot_max bounds
       // how many there can be.
      const uint64_t least = std::max<uint64_t>(a.hot_thr / 2, 1);
      const uint64_t hot_max = std::min<uint64_t>(a.ntiles, (uint64_t)a.P * a.cap / least + 1);
      const unsigned hot_grid = (unsigned)std::min<uint64_t>(hot_max, kHotGrid);
      if (a.op != kOpSum)
        launch_pdl(reduce_hot_tile_kernel<Q4, true>, hot_grid, kHotThreads, 0, s, a);
      else
        launch_pdl(reduce_hot_tile_kernel<Q4, false>, hot_grid, kHotThreads, 0, s, a);
      if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
    }
    const uint64_t groups = ((uint64_t)a.ntiles * kMiniWords + kReduceThreads - 1) / kReduceThreads;
    launch_pdl(reduce_mini_compact_kernel, (unsigned)groups, kReduceThreads, 0, s, a);
    if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
    mark(2);
    note_launches(4);
    return SPARCML_OK;
  }
  const uint64_t nsplit = (uint64_t)(a.ntiles + 1) * a.P;  // one warp each
  launch_pdl(reduce_split_kernel, (unsigned)((nsplit * 32 + 255) / 256), 256, 0, s,
      a.idx, a.nnz, a.P, a.cap, a.N, a.ntiles, a.tile_w, split);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  if (sparse) {
    const size_t smem =
        (2 * (size_t)(tile_w / 32) + kAccCap + 2 * (size_t)a.P + 1) * sizeof(uint32_t);
    auto go = [&](auto kernel) {
      if (!ensure_smem(reinterpret_cast<const void*>(kernel), smem)) return false;
      launch_pdl(kernel, a.ntiles, kReduceThreads, smem, s, a);
      return true;
    };
    if (!(a.op != kOpSum ? go(reduce_sparse_tile_kernel<Q4, true>)
                         : go(reduce_sparse_tile_kernel<Q4, false>)))
      return SPARCML_ERR_CUDA;
  } else {
    const size_t smem = (kTile + kWords + 2 * kStages * kStageEntries + 3 * (size_t)a.P + 1) *
                        sizeof(uint32_t);
    auto go_dense = [&](auto kernel) {
      if (!ensure_smem(reinterpret_cast<const void*>(kernel), smem)) return false;
      launch_pdl(kernel, a.ntiles, kReduceThreads, smem, s, a);
      return true;
    };
    if ((double)a.P * (double)a.cap >= (double)a.N) {
      // dense-first: no look-back; U and the flag come from the finalize pass
      if (!(a.op != kOpSum ? go_dense(reduce_dense_tile_kernel<Q4, true, true>)
                           : go_dense(reduce_dense_tile_kernel<Q4, true, false>)))
        return SPARCML_ERR_CUDA;
      if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
      mark(1);
      launch_pdl(reduce_finalize_kernel, 1, 1024, 0, s, a.tile_info, a.ntiles, a.cap_sparse, a.out_nnz,
                                               a.out_is_dense);
      launch_pdl(reduce_compact_kernel, a.ntiles, kReduceThreads, 0, s,
          a.out_is_dense, a.tile_info, a.tile_bm, a.out_dense, a.out_idx, a.out_val, kWords);
      if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
      mark(2);
      note_launches(4);
      return SPARCML_OK;
    }
    if (!(a.op != kOpSum ? go_dense(reduce_dense_tile_kernel<Q4, false, true>)
                         : go_dense(reduce_dense_tile_kernel<Q4, false, false>)))
      return SPARCML_ERR_CUDA;
  }
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  mark(1);
  launch_pdl(reduce_fixup_kernel, fixup_grid(a.ntiles), 256, 0, s, a.out_is_dense, a.tile_info, a.out_idx,
                                               a.out_val, a.out_dense, a.N, a.tile_w, a.ntiles,
        a.op == kOpMax ? -INFINITY : a.op == kOpMin ? INFINITY : 0.0f);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  mark(2);
  note_launches(3);
  return SPARCML_OK;
}

int check_reduce_args(const uint32_t* idx, const uint32_t* nnz, int32_t P, uint64_t cap,
                      uint64_t N, uint32_t dens_num, uint32_t dens_den, uint32_t* out_idx,
                      float* out_val, uint64_t out_cap, float* out_dense, uint32_t* out_nnz,
                      int32_t* out_is_dense, void* ws) {
  if (!idx || !nnz || !out_idx || !out_val || !out_dense || !out_nnz || !out_is_dense || !ws)
    return SPARCML_ERR_INVALID_ARG;
  if (P < 1 || P > kMaxReduceP || N < 1 || N > 0xffffffffull || cap > 0xffffffffull ||
      dens_den < 1 || dens_num > dens_den)
    return SPARCML_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return SPARCML_ERR_INVALID_ARG;
  if (out_cap < N * dens_num / dens_den) return SPARCML_ERR_CAPACITY;
  return SPARCML_OK;
}

}  // namespace
}  // namespace sparcml

using namespace sparcml;

extern "C" size_t sparcml_sparse_reduce_workspace_size(int32_t P, uint64_t N) {
  if (P < 1 || P > kMaxReduceP || N < 1 || N > 0xffffffffull) return 0;
  return reduce_layout(P, N).total;
}

namespace sparcml {
namespace {
int reduce_fp32(const uint32_t* idx, const float* val, const uint32_t* nnz, int32_t P,
                uint64_t cap, uint64_t N, int32_t op, uint32_t dens_num, uint32_t dens_den,
                uint32_t* out_idx, float* out_val, uint64_t out_cap, float* out_dense,
                uint32_t* out_nnz, int32_t* out_is_dense, void* ws, size_t ws_bytes,
                void* stream, void* const* events) {
  const int st = check_reduce_args(idx, nnz, P, cap, N, dens_num, dens_den, out_idx, out_val,
                                   out_cap, out_dense, out_nnz, out_is_dense, ws);
  if (st != SPARCML_OK) return st;
  if (!val || op < kOpSum || op > kOpOr) return SPARCML_ERR_INVALID_ARG;
  ReduceArgs a = {};
  a.op = op;
  a.idx = idx;
  a.val = val;
  a.nnz = nnz;
  a.cap = cap;
  a.P = P;
  a.N = (uint32_t)N;
  a.ntiles = (uint32_t)((N + kTile - 1) / kTile);
  a.cap_sparse = (uint32_t)(N * dens_num / dens_den);
  a.out_idx = out_idx;
  a.out_val = out_val;
  a.out_dense = out_dense;
  a.out_nnz = out_nnz;
  a.out_is_dense = out_is_dense;
  return launch_reduce<false>(a, ws, ws_bytes, static_cast<cudaStream_t>(stream), events);
}
}  // namespace
}  // namespace sparcml

extern "C" int sparcml_sparse_reduce_traced(const uint32_t* idx, const float* val,
                                            const uint32_t* nnz, int32_t P, uint64_t cap,
                                            uint64_t N, uint32_t dens_num, uint32_t dens_den,
                                            uint32_t* out_idx, float* out_val, uint64_t out_cap,
                                            float* out_dense, uint32_t* out_nnz,
                                            int32_t* out_is_dense, void* ws, size_t ws_bytes,
                                            void* stream, void* const* events) {
  const ApiRange nvtx_range(__func__);
  return reduce_fp32(idx, val, nnz, P, cap, N, kOpSum, dens_num, dens_den, out_idx, out_val,
                     out_cap, out_dense, out_nnz, out_is_dense, ws, ws_bytes, stream, events);
}

extern "C" int sparcml_sparse_reduce_op(const uint32_t* idx, const float* val,
                                        const uint32_t* nnz, int32_t P, uint64_t cap, uint64_t N,
                                        int32_t op, uint32_t dens_num, uint32_t dens_den,
                                        uint32_t* out_idx, float* out_val, uint64_t out_cap,
                                        float* out_dense, uint32_t* out_nnz,
                                        int32_t* out_is_dense, void* ws, size_t ws_bytes,
                                        void* stream) {
  const ApiRange nvtx_range(__func__);
  return reduce_fp32(idx, val, nnz, P, cap, N, op, dens_num, dens_den, out_idx, out_val,
                     out_cap, out_dense, out_nnz, out_is_dense, ws, ws_bytes, stream, nullptr);
}

extern "C" int sparcml_sparse_reduce(const uint32_t* idx, const float* val, const uint32_t* nnz,
                                     int32_t P, uint64_t cap, uint64_t N, uint32_t dens_num,
                                     uint32_t dens_den, uint32_t* out_idx, float* out_val,
                                     uint64_t out_cap, float* out_dense, uint32_t* out_nnz,
                                     int32_t* out_is_dense, void* ws, size_t ws_bytes,
                                     void* stream) {
  return sparcml_sparse_reduce_traced(idx, val, nnz, P, cap, N, dens_num, dens_den, out_idx,
                                      out_val, out_cap, out_dense, out_nnz, out_is_dense, ws,
                                      ws_bytes, stream, nullptr);
}

namespace sparcml {
namespace {
int reduce_quantised(const uint32_t* idx, const uint8_t* codes, const float* scales,
                     const uint32_t* nnz, int32_t P, uint64_t cap, uint32_t bucket, uint32_t bits,
                     uint64_t N, uint32_t dens_num, uint32_t dens_den, uint32_t* out_idx,
                     float* out_val, uint64_t out_cap, float* out_dense, uint32_t* out_nnz,
                     int32_t* out_is_dense, void* ws, size_t ws_bytes, void* stream) {
  const int st = check_reduce_args(idx, nnz, P, cap, N, dens_num, dens_den, out_idx, out_val,
                                   out_cap, out_dense, out_nnz, out_is_dense, ws);
  if (st != SPARCML_OK) return st;
  if (bits != 2 && bits != 4 && bits != 8) return SPARCML_ERR_INVALID_ARG;
  const uint32_t per = 8 / bits;
  if (!codes || !scales || bucket < 1 || bucket % per != 0 || cap < 1)
    return SPARCML_ERR_INVALID_ARG;
  ReduceArgs a = {};
  a.idx = idx;
  a.codes = codes;
  a.scales = scales;
  a.nnz = nnz;
  a.cap = cap;
  a.code_stride = (cap + per - 1) / per;
  a.scale_stride = (cap + bucket - 1) / bucket;
  a.bucket = bucket;
  a.bucket_shift = (bucket & (bucket - 1)) == 0 ? (uint32_t)__builtin_ctz(bucket) : 32u;
  a.bits = bits;
  a.P = P;
  a.N = (uint32_t)N;
  a.ntiles = (uint32_t)((N + kTile - 1) / kTile);
  a.cap_sparse = (uint32_t)(N * dens_num / dens_den);
  a.out_idx = out_idx;
  a.out_val = out_val;
  a.out_dense = out_dense;
  a.out_nnz = out_nnz;
  a.out_is_dense = out_is_dense;
  return launch_reduce<true>(a, ws, ws_bytes, static_cast<cudaStream_t>(stream), nullptr);
}
}  // namespace
}  // namespace sparcml

extern "C" int sparcml_sparse_reduce_q4(const uint32_t* idx, const uint8_t* codes,
                                        const float* scales, const uint32_t* nnz, int32_t P,
                                        uint64_t cap, uint32_t bucket, uint64_t N,
                                        uint32_t dens_num, uint32_t dens_den, uint32_t* out_idx,
                                        float* out_val, uint64_t out_cap, float* out_dense,
                                        uint32_t* out_nnz, int32_t* out_is_dense, void* ws,
                                        size_t ws_bytes, void* stream) {
  const ApiRange nvtx_range(__func__);
  if (bucket < 2 || (bucket & 1)) return SPARCML_ERR_INVALID_ARG;
  return reduce_quantised(idx, codes, scales, nnz, P, cap, bucket, 4, N, dens_num, dens_den,
                          out_idx, out_val, out_cap, out_dense, out_nnz, out_is_dense, ws,
                          ws_bytes, stream);
}

extern "C" int sparcml_sparse_reduce_qb(const uint32_t* idx, const uint8_t* codes,
                                        const float* scales, const uint32_t* nnz, int32_t P,
                                        uint64_t cap, uint32_t bucket, uint32_t bits, uint64_t N,
                                        uint32_t dens_num, uint32_t dens_den, uint32_t* out_idx,
                                        float* out_val, uint64_t out_cap, float* out_dense,
                                        uint32_t* out_nnz, int32_t* out_is_dense, void* ws,
                                        size_t ws_bytes, void* stream) {
  const ApiRange nvtx_range(__func__);
  return reduce_quantised(idx, codes, scales, nnz, P, cap, bucket, bits, N, dens_num, dens_den,
                          out_idx, out_val, out_cap, out_dense, out_nnz, out_is_dense, ws,
                          ws_bytes, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free sparse reduce (the paper has no counterpart).
//
// For callers that cannot allocate device memory where they reduce: a plug-in
// inside a host framework that owns all device memory through its own pool,
// or a latency-critical path where cudaMalloc would synchronise the device.
// The reduce's scratch (ticket, look-back words, per-tile records) then comes
// from one fixed array compiled into this file. Every GPU that loads the
// library holds that array until the process exits. All calls share it, so
// calls whose work overlaps on the GPU race; the array keeps the last call's
// contents and each call clears the words that must start at zero.
// ---------------------------------------------------------------------------
#include <cuda.h>

#include <mutex>

namespace sparcml {
namespace {
constexpr uint64_t kNoAllocMaxN = SPARCML_NOALLOC_MAX_N;
constexpr size_t kNoAllocTiles = (kNoAllocMaxN + kTile - 1) / kTile;  // 16,384
constexpr size_t kNoAllocStateOff = 256;
constexpr size_t kNoAllocInfoOff = kNoAllocStateOff + 8 * kNoAllocTiles;
constexpr size_t kNoAllocBytes = kNoAllocInfoOff + 8 * kNoAllocTiles;  // 262,400 B
constexpr int kNoAllocMaxDevices = 64;
}  // namespace
}  // namespace sparcml

static __device__ __align__(256) unsigned char g_noalloc_scratch[sparcml::kNoAllocBytes];

namespace sparcml {
namespace {
std::mutex g_noalloc_mu;
struct NoAllocSlot {
  unsigned long long ctx_id;  // context the address belongs to (0: none yet)
  void* ptr;
};
NoAllocSlot g_noalloc[kNoAllocMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 if none or unknown).
// The driver functions come through the runtime's entry-point query, so the
// library does not link the driver library itself.
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current device's context. The
// first call on a device looks it up (cudaGetSymbolAddress: no allocation)
// and keeps it with the id of the context it belongs to; a later call in
// another context (after cudaDeviceReset, say) looks it up again. If the
// context id cannot be read, the address is looked up on every call.
int noalloc_scratch(char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
    return SPARCML_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocSlot& slot = g_noalloc[dev];
  unsigned long long id = current_ctx_id();
  if (id == 0 || slot.ctx_id != id || slot.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return SPARCML_ERR_CUDA;
    slot.ptr = p;
    slot.ctx_id = current_ctx_id();  // the lookup made the context current if it was not
  }
  *out = static_cast<char*>(slot.ptr);
  return SPARCML_OK;
}
}  // namespace
}  // namespace sparcml

extern "C" int sparcml_sparse_reduce_noalloc(const uint32_t* idx, const float* val,
                                             const uint32_t* nnz, int32_t P, uint64_t cap,
                                             uint64_t N, uint32_t dens_num, uint32_t dens_den,
                                             uint32_t* out_idx, float* out_val, uint64_t out_cap,
                                             float* out_dense, uint32_t* out_nnz,
                                             int32_t* out_is_dense, int32_t* status,
                                             void* stream) {
  const ApiRange nvtx_range(__func__);
  if (!idx || !val || !nnz || !out_idx || !out_val || !out_dense || !out_nnz || !out_is_dense)
    return SPARCML_ERR_INVALID_ARG;
  if (P < 1 || P > kMaxReduceP || N < 1 || N > 0xffffffffull || cap > 0xffffffffull ||
      dens_den < 1 || dens_num > dens_den)
    return SPARCML_ERR_INVALID_ARG;
  if (N > kNoAllocMaxN) return SPARCML_ERR_WORKSPACE;  // beyond the fixed scratch
  if (out_cap < N * dens_num / dens_den) return SPARCML_ERR_CAPACITY;
  char* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != SPARCML_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ReduceArgs a = {};
  a.idx = idx;
  a.val = val;
  a.nnz = nnz;
  a.cap = cap;
  a.P = P;
  a.N = (uint32_t)N;
  a.ntiles = (uint32_t)((N + kTile - 1) / kTile);
  a.tile_w = kTile;
  a.cap_sparse = (uint32_t)(N * dens_num / dens_den);
  a.out_idx = out_idx;
  a.out_val = out_val;
  a.out_dense = out_dense;
  a.out_nnz = out_nnz;
  a.out_is_dense = out_is_dense;
  a.status = status;
  a.ticket = reinterpret_cast<uint32_t*>(scratch + 64);
  a.tile_state = reinterpret_cast<unsigned long long*>(scratch + kNoAllocStateOff);
  a.tile_info = reinterpret_cast<uint2*>(scratch + kNoAllocInfoOff);
  // The ticket and this call's look-back words must start at zero.
  if (cudaMemsetAsync(scratch + 64, 0, kNoAllocStateOff - 64 + 8 * (size_t)a.ntiles, s) !=
      cudaSuccess)
    return SPARCML_ERR_CUDA;
  const size_t smem = (kTile + kWords + 2 * (size_t)a.P + 1) * sizeof(uint32_t);
  if (!ensure_smem(reinterpret_cast<const void*>(reduce_tile_kernel<false>), smem))
    return SPARCML_ERR_CUDA;
  launch_pdl(reduce_tile_kernel<false>, a.ntiles, kReduceThreads, smem, s, a);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  launch_pdl(reduce_fixup_kernel, fixup_grid(a.ntiles), 256, 0, s, a.out_is_dense, a.tile_info, a.out_idx,
                                               a.out_val, a.out_dense, a.N, a.tile_w, a.ntiles,
        a.op == kOpMax ? -INFINITY : a.op == kOpMin ? INFINITY : 0.0f);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  note_launches(2);
  return SPARCML_OK;
}
