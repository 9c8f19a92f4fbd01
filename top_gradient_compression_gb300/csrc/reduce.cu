// Sparse sum-reduction of P streams with the adaptive dense switch, sm_103a.
//
// "SparCML: High-Performance Sparse Communication for Machine Learning",
// §5.2 (allreduce of sparse vectors with a coordinate-wise associative op
// that has a neutral element: here fp32 sum, neutral +0.0), §5.3.2 (the
// split phase routes index ranges to owners: here each CTA owns a tile of
// the index space), §5.1 / §5.3.3 (switch to a dense representation once
// fill-in passes the threshold delta), App. B (the result size is the size
// of the union of the contributed index sets).
//
// One pass over the input, no sort, no floating-point atomics:
//
//  tile kernel   (one CTA per tile of kTile consecutive indices, tiles taken
//                in index order through a ticket). The CTA binary-searches
//                each node's sub-range for its tile, then adds the nodes'
//                entries into a shared-memory fp32 accumulator node by node
//                in ascending node order (indices are unique within a node,
//                so no two threads of one node touch the same word) and sets
//                a presence bitmap. Its union count is chained to the
//                previous tiles with a decoupled look-back (Merrill and
//                Garland, 2016) to get the tile's output offset. A tile whose
//                inclusive count still fits the sparse capacity writes its
//                entries ascending (bitmap + prefix popcount); once the
//                running count passes floor(N * num / den) the result is
//                certainly dense and the tile writes its dense slice.
//  fix-up kernel (one CTA per tile) runs only if the final result is dense:
//                the leading tiles that were written sparse are turned into
//                their dense slices (zeros, then a scatter of their entries).
//
// Every wait on a predecessor is bounded; on expiry the kernel records
// SPARCML_ERR_TIMEOUT and carries on, so a bad input can never hang the GPU.

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
constexpr uint32_t kSpinLimit = 1u << 21;

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
  int32_t* status;
};

__device__ __forceinline__ uint32_t lower_bound_u32(const uint32_t* a, uint32_t n, uint32_t x) {
  uint32_t lo = 0, hi = n;
  while (lo < hi) {
    const uint32_t mid = lo + ((hi - lo) >> 1);
    if (a[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Value of entry j of node p: fp32 as stored, or decoded from 4 bits.
template <bool Q4>
__device__ __forceinline__ float load_value(const ReduceArgs& a, uint32_t p, uint32_t j) {
  if constexpr (!Q4) {
    return a.val[(uint64_t)p * a.cap + j];
  } else {
    const uint8_t byte = a.codes[(uint64_t)p * a.code_stride + (j >> 1)];
    const uint32_t code = (j & 1) ? (byte >> 4) : (byte & 15u);
    const uint32_t level = code & 7u;
    if (level == 0) return 0.0f;
    const float scale = a.scales[(uint64_t)p * a.scale_stride + j / a.bucket];
    const float v = __fmul_rn(__fdiv_rn((float)level, 7.0f), scale);
    return (code & 8u) ? -v : v;
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
  if (tile == 0) {
    if (t == 0) atomicExch(&st[0], kFlagInc | count);
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
        if (++spins > kSpinLimit) {
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
  for (uint32_t w = t; w < kTile / 4; w += blockDim.x)
    reinterpret_cast<float4*>(acc)[w] = make_float4(0.f, 0.f, 0.f, 0.f);
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

// Sparse regime: tiles of a.tile_w indices (up to kMaxTileW), chosen so a
// tile holds about two thousand entries. Shared memory scales with the
// tile's union, not its width: a presence bitmap is built first, its prefix
// popcounts give every present index a slot (its rank in the tile), and the
// sums go to a compact fp32 array of slots. Accumulation keeps ascending node
// order (barrier after each node with entries in a batch), so the bits equal
// the dense-accumulator kernel's. Tiles whose union exceeds kAccCap are
// accumulated in several slot windows.
constexpr uint32_t kMaxTileW = 1u << 17;
constexpr uint32_t kMaxWords = kMaxTileW / 32;
constexpr uint32_t kAccCap = 8192;
constexpr int32_t kMaxSparseP = 1024;

template <bool Q4>
__global__ void __launch_bounds__(kReduceThreads)
reduce_sparse_tile_kernel(ReduceArgs a) {
  extern __shared__ __align__(16) uint32_t dyn[];
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
    for (uint32_t i = t; i < win; i += blockDim.x) acc[i] = 0.0f;
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
            if (slot - s0 < win) acc[slot - s0] = __fadd_rn(acc[slot - s0], vv[u]);
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
          od[x] = 0.0f;
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
                    float* __restrict__ out_dense, uint32_t N, uint32_t tile_w) {
  if (*is_dense == 0) return;
  const uint2 info = tile_info[blockIdx.x];
  if (info.y & 0x80000000u) return;
  const uint32_t tile_lo = blockIdx.x * tile_w;
  const uint32_t tile_n = min(tile_w, N - tile_lo);
  for (uint32_t x = threadIdx.x; x < tile_n; x += blockDim.x) out_dense[tile_lo + x] = 0.0f;
  __syncthreads();
  for (uint32_t e = threadIdx.x; e < info.y; e += blockDim.x) {
    const uint32_t i = out_idx[info.x + e];
    if (i - tile_lo < tile_n) out_dense[i] = out_val[info.x + e];
  }
}

struct ReduceLayout {
  size_t ticket, state, info, split, total;
};

ReduceLayout reduce_layout(int32_t P, uint64_t N) {
  const size_t ntiles = (N + kTile - 1) / kTile;
  ReduceLayout l;
  l.ticket = 64;
  l.state = 256;
  l.info = align_up(l.state + 8 * ntiles, 256);
  l.split = align_up(l.info + 8 * ntiles, 256);
  l.total = align_up(l.split + 4 * (ntiles + 1) * (size_t)P, 256);
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
  // Clear the ticket and the look-back states (the status word is kept).
  if (cudaMemsetAsync(w + l.ticket, 0, l.info - l.ticket, s) != cudaSuccess)
    return SPARCML_ERR_CUDA;
  // Regime: the entries of an 8,192-index tile are at most P * cap * 8192 / N.
  // Sparse inputs take wide tiles (about 2,048 entries each) with a compact
  // accumulator; denser ones the dense-accumulator tile of kTile indices.
  const double est = (double)a.P * (double)a.cap * kTile / (double)a.N;
  uint32_t tile_w = kTile;
  if (a.P <= kMaxSparseP && est <= 512.0) {
    while (tile_w < kMaxTileW && est * (2.0 * tile_w / kTile) <= 2048.0 && tile_w < a.N)
      tile_w *= 2;
  }
  a.tile_w = tile_w;
  a.ntiles = (uint32_t)((a.N + tile_w - 1) / tile_w);
  mark(0);
  const uint64_t nsplit = (uint64_t)(a.ntiles + 1) * a.P;  // one warp each
  reduce_split_kernel<<<(unsigned)((nsplit * 32 + 255) / 256), 256, 0, s>>>(
      a.idx, a.nnz, a.P, a.cap, a.N, a.ntiles, a.tile_w, split);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  if (tile_w > kTile) {
    const size_t smem =
        (2 * (size_t)(tile_w / 32) + kAccCap + 2 * (size_t)a.P + 1) * sizeof(uint32_t);
    if (!ensure_smem(reinterpret_cast<const void*>(reduce_sparse_tile_kernel<Q4>), smem))
      return SPARCML_ERR_CUDA;
    reduce_sparse_tile_kernel<Q4><<<a.ntiles, kReduceThreads, smem, s>>>(a);
  } else {
    const size_t smem = (kTile + kWords + 2 * (size_t)a.P + 1) * sizeof(uint32_t);
    if (!ensure_smem(reinterpret_cast<const void*>(reduce_tile_kernel<Q4, true>), smem))
      return SPARCML_ERR_CUDA;
    reduce_tile_kernel<Q4, true><<<a.ntiles, kReduceThreads, smem, s>>>(a);
  }
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  mark(1);
  reduce_fixup_kernel<<<a.ntiles, 256, 0, s>>>(a.out_is_dense, a.tile_info, a.out_idx,
                                               a.out_val, a.out_dense, a.N, a.tile_w);
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

extern "C" int sparcml_sparse_reduce_traced(const uint32_t* idx, const float* val,
                                            const uint32_t* nnz, int32_t P, uint64_t cap,
                                            uint64_t N, uint32_t dens_num, uint32_t dens_den,
                                            uint32_t* out_idx, float* out_val, uint64_t out_cap,
                                            float* out_dense, uint32_t* out_nnz,
                                            int32_t* out_is_dense, void* ws, size_t ws_bytes,
                                            void* stream, void* const* events) {
  const int st = check_reduce_args(idx, nnz, P, cap, N, dens_num, dens_den, out_idx, out_val,
                                   out_cap, out_dense, out_nnz, out_is_dense, ws);
  if (st != SPARCML_OK) return st;
  if (!val) return SPARCML_ERR_INVALID_ARG;
  ReduceArgs a = {};
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

extern "C" int sparcml_sparse_reduce_q4(const uint32_t* idx, const uint8_t* codes,
                                        const float* scales, const uint32_t* nnz, int32_t P,
                                        uint64_t cap, uint32_t bucket, uint64_t N,
                                        uint32_t dens_num, uint32_t dens_den, uint32_t* out_idx,
                                        float* out_val, uint64_t out_cap, float* out_dense,
                                        uint32_t* out_nnz, int32_t* out_is_dense, void* ws,
                                        size_t ws_bytes, void* stream) {
  const int st = check_reduce_args(idx, nnz, P, cap, N, dens_num, dens_den, out_idx, out_val,
                                   out_cap, out_dense, out_nnz, out_is_dense, ws);
  if (st != SPARCML_OK) return st;
  if (!codes || !scales || bucket < 2 || (bucket & 1) || cap < 1) return SPARCML_ERR_INVALID_ARG;
  ReduceArgs a = {};
  a.idx = idx;
  a.codes = codes;
  a.scales = scales;
  a.nnz = nnz;
  a.cap = cap;
  a.code_stride = (cap + 1) / 2;
  a.scale_stride = (cap + bucket - 1) / bucket;
  a.bucket = bucket;
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
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device. The first call
// on a device looks it up (cudaGetSymbolAddress, no allocation) and keeps it.
int noalloc_scratch(char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
    return SPARCML_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return SPARCML_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = static_cast<char*>(g_noalloc_ptr[dev]);
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
  reduce_tile_kernel<false><<<a.ntiles, kReduceThreads, smem, s>>>(a);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  reduce_fixup_kernel<<<a.ntiles, 256, 0, s>>>(a.out_is_dense, a.tile_info, a.out_idx,
                                               a.out_val, a.out_dense, a.N, a.tile_w);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  note_launches(2);
  return SPARCML_OK;
}
