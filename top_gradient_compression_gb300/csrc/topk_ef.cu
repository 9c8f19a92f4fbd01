// Top-k selection with error feedback, fused with packing, for sm_103a.
//
// "SparCML: High-Performance Sparse Communication for Machine Learning",
// §2.2 (Top-k SGD: each node sends its k largest-magnitude components and
// accumulates the rest for the next iteration), §4 (residual error), §5.1
// (sparse streams of index-value pairs), §8.4 (layer-wise sparsification:
// every segment of the caller's layer table keeps its own k_s).
//
// The host turns the caller's segment table into per-segment records and
// hands them to the GPU as the parameters of a small upload kernel (kernel
// parameters are copied at launch, so this needs no host-side staging, no
// allocation and no synchronisation). Then, stream-ordered:
//
//  1. init     chunk descriptors and the per-(node, segment) state.
//  2. guess    per (node, segment): acc = residual + grad on a sample (all of
//              a segment of up to 8,192 entries), and G = the r-th largest
//              sample key with its low 15 bits cleared, r chosen so that, with
//              overwhelming probability, at least k_s keys of the whole
//              segment are >= G (certainly so for a fully sampled segment).
//              Long segments also get a histogram scale from a second, higher
//              sample quantile, and a mid guess Gm of the k-th key itself:
//              the segment's k-th key in the last call made with the same
//              workspace, else the sample's estimate.
//  3. stream   the HBM-bound pass (one CTA per 8,192-entry chunk of a
//              segment): reads grad and residual once with 128-bit loads
//              aligned on the element grid, writes acc back into residual,
//              and compacts the candidates (key >= G) in index order into the
//              warp's own sub-slot. A segment that keeps everything (k = n) is
//              written straight to the stream here; one that keeps nothing
//              never has candidates. In long segments a stored candidate at or
//              above Gm gets +0.0f in the residual at once.
//  4. select   layer-sized segments: one CTA per segment selects among its
//              candidates in shared memory (four 8-bit radix digits) and
//              writes the kept entries in index order. Long segments, in
//              passes over ranges of sub-slots: a 2,048-bin histogram of
//              (key - G) >> shift; its boundary bin; the candidates in that
//              bin collected; the exact k-th key T and the index cut I_T
//              among keys equal to T (lowest indices first) from a select in
//              shared memory; an ordered write of every candidate with key >
//              T, or key == T and index <= I_T, which also zeroes the kept
//              candidates below Gm and restores acc at the stored ones at or
//              above Gm that are not kept. Whatever the candidates cannot decide (the guess
//              covered fewer than k_s entries, a sub-slot or the boundary
//              buffer overflowed) is decided again from the segment's acc
//              (now in residual) by a raw select: the answer is the same.
//
// The kept entries go to the node's stream in ascending index order, at the
// segment's offset (the sum of the k of the segments before it); the residual
// becomes +0.0f at every kept entry.

#include <cooperative_groups.h>

#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace sparcml {
namespace {

constexpr uint32_t kChunk = 8192;         // entries per stream-pass CTA
constexpr uint32_t kStreamThreads = 256;  // 8 warps x 1024 entries
constexpr uint32_t kWarpsPerChunk = kStreamThreads / 32;
constexpr uint32_t kSub = kChunk / kWarpsPerChunk;  // entries per warp sub-chunk: 1,024
constexpr uint32_t kRounds = kSub / (32 * 4);       // float4 rounds per warp
constexpr uint32_t kExactMax = 8192;      // segments sampled whole
constexpr uint32_t kLayerMax = 1u << 18;  // layer-sized: warp guess, one-CTA select
constexpr uint32_t kSampleLong = 8192;    // sample of one guess CTA
constexpr uint32_t kGuessCluster = 8;     // guess CTAs of a long segment (a cluster)
constexpr uint32_t kLongSample = kSampleLong * kGuessCluster;  // sample of a long segment
constexpr uint32_t kWarpSample = 2048;    // sample of a layer-sized segment
constexpr uint32_t kRun = 256;            // consecutive entries per sample run
constexpr uint32_t kGuessThreads = 256;
constexpr uint32_t kNone = 0xffffffffu;
constexpr uint32_t kBins = 2048;          // histogram of a long segment's candidates
constexpr uint32_t kRangeSubs = 256;      // sub-chunks per long-select range
constexpr uint32_t kBoundCap = 16384;     // boundary-bin entries per (node, long segment)
constexpr uint32_t kMaxRanges = 16384;    // ranges of one long segment (n < 2^32)
constexpr uint32_t kUploadWords = 7680;   // 30 KB of kernel parameters per upload launch
constexpr size_t kFallbackOffset = 68;     // workspace header: raw-select count of the last call

// Segment kinds (what the guess and select passes do with a segment).
enum : uint32_t { kKeepNone = 0, kKeepAll = 1, kExact = 2, kLayer = 3, kLong = 4 };

// One segment of the caller's table, identical for every node (12 words).
struct SegRec {
  uint32_t begin;   // node-local first entry
  uint32_t n;       // entries
  uint32_t k;       // entries kept
  uint32_t out0;    // offset of the segment's kept entries in a node's stream
  uint32_t chunk0;  // first node-local chunk
  uint32_t nchunk;  // chunks: ceil((n + 3) / kChunk) (quads aligned on the element grid)
  uint32_t slot;    // candidate entries per warp sub-slot, a multiple of 32
  uint32_t slot32;  // node-local base of the segment's sub-slots, in units of 32 entries
  uint32_t rank;    // guess rank r (low 16 bits) and histogram anchor rank (high 16 bits)
  uint32_t kind;
  uint32_t lidx;    // position among the long segments (kLong), else kNone
  uint32_t range0;  // first long-select range of the segment (kLong)
};
static_assert(sizeof(SegRec) == 48, "segment record layout");

// One chunk of a segment (two 16-byte words, loaded together).
struct ChunkDesc {
  uint32_t begin, end, seg, j;    // the segment's node-local range, its id, the chunk's place
  uint32_t slot, slot32, kind, aux;  // sub-slot size and base/32; kind; out0 (kKeepAll) or lidx
};
static_assert(sizeof(ChunkDesc) == 32, "chunk descriptor layout");

// Per (node, long segment): the select's state.
enum : uint32_t { kModeNormal = 0, kModeFallback = 1 };
struct LongSel {
  uint32_t mode, bin, rank, T, cut, overflow;
  uint32_t mid;  // the stream pass zeroes stored candidates at or above it
  uint32_t sig;  // signature of the segment whose T this record holds (kept across calls)
};

struct UploadBatch {
  uint32_t words[kUploadWords];
  uint32_t* dst;
  uint32_t count;
};

__global__ void __launch_bounds__(256) topk_upload_kernel(const __grid_constant__ UploadBatch b) {
  griddep_wait();
  for (uint32_t i = threadIdx.x; i < b.count; i += blockDim.x) b.dst[i] = b.words[i];
}

struct Args {
  const float* grad;
  float* residual;
  uint32_t* out_idx;
  float* out_val;
  uint32_t* out_nnz;
  int32_t* status;
  uint64_t N;
  uint64_t cap;
  uint64_t node_slots;  // candidate sub-slot entries per node
  int32_t P;
  uint32_t nseg, nchunk, nlong, nranges;
  uint32_t total_k;
  uint32_t vec;         // grad and residual 16-byte aligned: 128-bit loads on the element grid
  uint32_t u_L, u_m;    // equal segments of u_L entries and u_m chunks each (0: another table)
  const SegRec* recs;
  ChunkDesc* desc;
  const uint32_t* cta_list;   // segments guessed by one CTA (exact and long kinds)
  const uint32_t* warp_list;  // segments guessed by one warp (layer kind)
  const uint32_t* short_list; // segments selected by one CTA (exact and layer kinds)
  const uint32_t* long_list;  // long segments, by lidx
  const uint32_t* range_map;  // long-select range -> lidx << 16 | range within the segment
  uint2* guess;               // [P][nseg] (G, histogram shift)
  uint32_t* seg_cnt;          // [P][nseg] candidates
  uint32_t* seg_flag;         // [P][nseg] a sub-slot overflowed
  uint32_t* sub_cnt;          // [P][nchunk][8] candidates per warp sub-chunk
  uint32_t* cand_idx;         // [P][node_slots]
  float* cand_val;
  uint32_t* todo;             // layer-sized segments left to the raw select: p * nseg + s
  uint32_t* todo_cnt;
  uint32_t* fallbacks;        // (node, segment) pairs the raw select decided in this call
  uint32_t* hist;             // [P][nlong][kBins]
  LongSel* lsel;              // [P][nlong]
  uint32_t* bnd_cnt;          // [P][nlong]
  uint2* bnd;                 // [P][nlong][kBoundCap] (key, index)
  uint32_t* range_gt;         // [P][nranges]: candidates above the boundary bin
  uint32_t* range_off;        // [P][nranges]: output offset of the range in its segment
};

// Among bins ordered from high to low, find b with
//   above(b) = sum_{b' > b} h[b'] < r <= above(b) + h[b],   r >= 1.
// Block-wide (nbins % blockDim.x == 0); result in out[0] (kNone if the
// histogram holds fewer than r entries) and out[1] = above(b).
__device__ void find_from_top(const uint32_t* h, uint32_t nbins, uint32_t r, uint32_t* scratch,
                              uint32_t* out) {
  const uint32_t per = nbins / blockDim.x;
  const uint32_t t = threadIdx.x;
  uint32_t sum = 0;
  for (uint32_t i = 0; i < per; ++i) sum += h[nbins - 1 - (t * per + i)];
  if (t == 0) out[0] = kNone;
  uint32_t total;
  const uint32_t excl = block_excl_scan(sum, scratch, &total);
  if (excl < r && r <= excl + sum) {
    uint32_t acc = excl;
    for (uint32_t i = 0; i < per; ++i) {
      const uint32_t b = nbins - 1 - (t * per + i);
      if (acc + h[b] >= r) {
        out[0] = b;
        out[1] = acc;
        break;
      }
      acc += h[b];
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// 1. init: one grid-stride pass over every item of per-call state: the chunk
// descriptors (chunk -> segment by a binary search over the records), the
// per-(node, segment) counters and guesses of the trivial kinds, the
// long-select state and histograms, and the nodes' stream sizes.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) topk_init_kernel(Args a) {
  griddep_wait();
  const uint64_t n_desc = a.nchunk, n_seg = (uint64_t)a.P * a.nseg;
  const uint64_t n_long = (uint64_t)a.P * a.nlong, n_hist = n_long * kBins;
  const uint64_t total = n_desc + n_seg + n_long + n_hist + (uint64_t)a.P;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (uint64_t)gridDim.x * blockDim.x) {
    if (i < n_desc) {
      const uint32_t c = (uint32_t)i;
      uint32_t lo = 0, hi = a.nseg;  // the segment s with chunk0[s] <= c < chunk0[s + 1]
      while (hi - lo > 1) {
        const uint32_t m = (lo + hi) >> 1;
        if (a.recs[m].chunk0 <= c) lo = m; else hi = m;
      }
      const SegRec r = a.recs[lo];
      const uint32_t j = c - r.chunk0;
      ChunkDesc d;
      d.begin = r.begin;
      d.end = r.begin + r.n;
      d.seg = lo;
      d.j = j;
      d.slot = r.slot;
      d.slot32 = r.slot32 + j * kWarpsPerChunk * (r.slot / 32);
      d.kind = r.kind;
      d.aux = r.kind == kLong ? r.lidx : r.out0;
      a.desc[c] = d;
      continue;
    }
    uint64_t x = i - n_desc;
    if (x < n_seg) {
      const uint32_t s = (uint32_t)(x % a.nseg);
      const uint32_t kind = a.recs[s].kind;
      a.seg_cnt[x] = 0;
      a.seg_flag[x] = 0;
      if (kind == kKeepNone) a.guess[x] = make_uint2(kNone, 0);
      if (kind == kKeepAll) a.guess[x] = make_uint2(0, 0);
      continue;
    }
    x -= n_seg;
    if (x < n_long) {
      a.bnd_cnt[x] = 0;
      a.lsel[x].overflow = 0;
      a.lsel[x].mid = 0;  // zero everything stored until the long guess sets it
      continue;
    }
    x -= n_long;
    if (x < n_hist) {
      a.hist[x] = 0;
      continue;
    }
    x -= n_hist;
    a.out_nnz[x] = a.total_k;
    if (x == 0) {
      *a.todo_cnt = 0;
      *a.fallbacks = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// 2. guess.
// ---------------------------------------------------------------------------
// Largest G on the 2^15 grid with at least r of the block's keys >= G (the
// r-th largest key with its low 15 bits cleared), keys held KPT per thread.
// Over a cluster of CS CTAs (CS = 1: the block alone), the counts of each
// step summed through distributed shared memory.
template <uint32_t KPT>
__device__ uint32_t block_rank_key(const uint32_t (&key)[KPT], uint32_t r, uint32_t (*wsum)[8],
                                   cg::cluster_group& cluster, uint32_t CS) {
  constexpr uint32_t kWarps = kGuessThreads / 32;
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  uint32_t G = 0;
#pragma unroll 1
  for (int bit = 30; bit >= 15; --bit) {
    const uint32_t trial = G | (1u << bit);
    uint32_t c = 0;
#pragma unroll
    for (uint32_t q = 0; q < KPT; ++q) c += (key[q] != kNone && key[q] >= trial) ? 1u : 0u;
    c = warp_sum(c);
    uint32_t* ws = wsum[bit & 1];  // double-buffered: one barrier per bit
    if (lane == 0) ws[warp] = c;
    uint32_t tot = 0;
    if (CS == 1) {
      __syncthreads();
#pragma unroll
      for (uint32_t w = 0; w < kWarps; ++w) tot += ws[w];
    } else {
      cluster.sync();  // every CTA's counts of this bit are in
      for (uint32_t q = 0; q < CS; ++q) {
        const uint32_t* rw = cluster.map_shared_rank(ws, q);
#pragma unroll
        for (uint32_t w = 0; w < kWarps; ++w) tot += rw[w];
      }
    }
    if (tot >= r) G = trial;
  }
  if (CS > 1) cluster.sync();  // no CTA leaves while its counts may still be read
  return G;
}

// Histogram scale of a long segment: the smallest shift with
// (anchor - G) >> shift < kBins.
__device__ __forceinline__ uint32_t hist_shift(uint32_t G, uint32_t anchor) {
  if (anchor <= G) return 0;
  const uint32_t span = anchor - G;
  const uint32_t bits = 32 - __clz(span);
  return bits > 11 ? bits - 11 : 0;
}

// One CTA per (node, segment) of the exact and long kinds. Exact: the whole
// segment, r = k. Long: 32 runs of kRun consecutive entries spread evenly.
constexpr uint32_t kGuessKPT = kSampleLong / kGuessThreads;  // 32

// Segments sampled whole (the exact kind): one CTA per (node, segment).
__global__ void __launch_bounds__(kGuessThreads) topk_guess_cta_kernel(Args a, uint32_t nlist) {
  griddep_wait();
  __shared__ uint32_t wsum[2][8];
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t CS = 1, rank = 0;
  const uint32_t p = blockIdx.x / nlist, s = a.cta_list[blockIdx.x % nlist];
  const SegRec r = a.recs[s];
  const uint32_t t = threadIdx.x, lane = lane_id(), warp = t >> 5;
  const uint64_t base = (uint64_t)p * a.N + r.begin;
  const float* gp = a.grad + base;
  const float* rp = a.residual + base;
  const bool exact = r.kind == kExact;
  uint32_t pos[kGuessKPT];
  bool ok[kGuessKPT];
  if (exact) {
#pragma unroll
    for (uint32_t q = 0; q < kGuessKPT; ++q) {
      pos[q] = t + q * kGuessThreads;
      ok[q] = pos[q] < r.n;
    }
  } else {
    constexpr uint32_t kLinesPerRun = kRun / 32;
    const uint32_t nruns = (kSampleLong / kRun) * CS;
#pragma unroll
    for (uint32_t q = 0; q < kGuessKPT; q += kLinesPerRun) {
      const uint32_t run =
          rank * (kSampleLong / kRun) + warp * (kGuessKPT / kLinesPerRun) + q / kLinesPerRun;
      const uint32_t st =
          (uint32_t)(((uint64_t)run * (r.n - kRun) / (nruns - 1)) & ~(uint64_t)(kRun - 1));
#pragma unroll
      for (uint32_t l = 0; l < kLinesPerRun; ++l) {
        pos[q + l] = st + l * 32 + lane;
        ok[q + l] = true;
      }
    }
  }
  float ra[kGuessKPT], ga[kGuessKPT];
#pragma unroll
  for (uint32_t q = 0; q < kGuessKPT; ++q) {
    ra[q] = ok[q] ? rp[pos[q]] : 0.0f;
    ga[q] = ok[q] ? gp[pos[q]] : 0.0f;
  }
  uint32_t key[kGuessKPT];
#pragma unroll
  for (uint32_t q = 0; q < kGuessKPT; ++q) key[q] = ok[q] ? mag_key(__fadd_rn(ra[q], ga[q])) : kNone;
  const uint32_t G =
      block_rank_key<kGuessKPT>(key, exact ? r.k : (r.rank & 0xffffu), wsum, cluster, CS);
  uint32_t shift = 0;
  if (!exact) shift = hist_shift(G, block_rank_key<kGuessKPT>(key, r.rank >> 16, wsum, cluster, CS));
  if (t == 0 && rank == 0) a.guess[(uint64_t)p * a.nseg + s] = make_uint2(G, shift);
}

// Long segments: a cluster of CS CTAs per (node, segment), each sampling its
// own 32 runs of kRun entries (CS * 8,192 sample keys in all). G is the r-th
// largest sample key with its low 15 bits cleared, found as two radix digits
// (bits 30..20, then 19..15) from histograms summed over the cluster through
// distributed shared memory; the histogram anchor likewise with its rank.
// A long segment's signature (its begin, length and k), kept beside its T so
// that a later call with the same workspace and segment can start from it.
__device__ __forceinline__ uint32_t seg_signature(const SegRec& r) {
  return ((r.begin * 0x85ebca6bu) ^ (r.n * 0xc2b2ae35u) ^ (r.k * 0x27d4eb2fu)) | 1u;
}

__device__ __forceinline__ void warp_find_from_top32(const uint32_t* tot, uint32_t r,
                                                     uint32_t* bin) {
  // lanes hold bins 31 - lane (high to low); the bin where the count from the top reaches r
  const uint32_t lane = lane_id();
  const uint32_t v = tot[31 - lane];
  const uint32_t incl = warp_incl_sum(v);
  const uint32_t hit = __ballot_sync(0xffffffffu, incl >= r && incl - v < r);
  if (lane == 0) *bin = hit ? 31 - (__ffs(hit) - 1) : 0;
}

__global__ void __launch_bounds__(kGuessThreads) topk_guess_long_kernel(Args a) {
  griddep_wait();
  __shared__ uint32_t h1[2048];
  __shared__ uint32_t tot[2048];
  __shared__ uint32_t h2[3][32];
  __shared__ uint32_t t2[3][32];
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t res[2];
  __shared__ uint32_t pick[6];  // digit-1 bins of G, the anchor and the mid guess, ranks left
  __shared__ uint32_t pick2[3];
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t CS = cluster.num_blocks(), rank = cluster.block_rank();
  const uint32_t item = blockIdx.x / CS;
  const uint32_t p = item / a.nlong, s = a.long_list[item % a.nlong];
  const SegRec r = a.recs[s];
  const uint32_t t = threadIdx.x, lane = lane_id(), warp = t >> 5;
  for (uint32_t b = t; b < 2048; b += blockDim.x) h1[b] = 0;
  if (t < 96) (&h2[0][0])[t] = 0;
  const uint64_t base = (uint64_t)p * a.N + r.begin;
  const float* gp = a.grad + base;
  const float* rp = a.residual + base;
  constexpr uint32_t kLinesPerRun = kRun / 32;
  const uint32_t nruns = (kSampleLong / kRun) * CS;
  uint32_t key[kGuessKPT];
  {
    float ra[kGuessKPT], ga[kGuessKPT];
#pragma unroll
    for (uint32_t q = 0; q < kGuessKPT; q += kLinesPerRun) {
      const uint32_t run =
          rank * (kSampleLong / kRun) + warp * (kGuessKPT / kLinesPerRun) + q / kLinesPerRun;
      const uint32_t st =
          (uint32_t)(((uint64_t)run * (r.n - kRun) / (nruns - 1)) & ~(uint64_t)(kRun - 1));
#pragma unroll
      for (uint32_t l = 0; l < kLinesPerRun; ++l) {
        ra[q + l] = rp[st + l * 32 + lane];
        ga[q + l] = gp[st + l * 32 + lane];
      }
    }
#pragma unroll
    for (uint32_t q = 0; q < kGuessKPT; ++q) key[q] = mag_key(__fadd_rn(ra[q], ga[q]));
  }
  __syncthreads();
#pragma unroll
  for (uint32_t q = 0; q < kGuessKPT; ++q) atomicAdd(&h1[key[q] >> 20], 1u);
  __syncthreads();
  cluster.sync();  // every CTA's digit-1 histogram is in
  for (uint32_t b = t; b < 2048; b += blockDim.x) {
    uint32_t sum = 0;
    for (uint32_t q = 0; q < CS; ++q) sum += cluster.map_shared_rank(h1, q)[b];
    tot[b] = sum;
  }
  __syncthreads();
  const uint32_t rG = r.rank & 0xffffu, rA = r.rank >> 16;
  find_from_top(tot, 2048, rG, scratch, res);
  if (t == 0) {
    pick[0] = res[0] == kNone ? 0u : res[0];
    pick[1] = res[0] == kNone ? 1u : rG - res[1];
  }
  __syncthreads();
  find_from_top(tot, 2048, rA, scratch, res);
  if (t == 0) {
    pick[2] = res[0] == kNone ? 0u : res[0];
    pick[3] = res[0] == kNone ? 1u : rA - res[1];
  }
  __syncthreads();
  // the mid guess: rank k * S / n of the S sample keys, the sample's estimate of T
  const uint32_t S = nruns * kRun;
  const uint64_t rM64 = ((uint64_t)r.k * S + r.n / 2) / r.n;
  const uint32_t rM = rM64 < 1 ? 1u : (uint32_t)rM64;
  find_from_top(tot, 2048, rM, scratch, res);
  if (t == 0) {
    pick[4] = res[0] == kNone ? 0u : res[0];
    pick[5] = res[0] == kNone ? 1u : rM - res[1];
  }
  __syncthreads();
#pragma unroll
  for (uint32_t q = 0; q < kGuessKPT; ++q) {
    if ((key[q] >> 20) == pick[0]) atomicAdd(&h2[0][(key[q] >> 15) & 31u], 1u);
    if ((key[q] >> 20) == pick[2]) atomicAdd(&h2[1][(key[q] >> 15) & 31u], 1u);
    if ((key[q] >> 20) == pick[4]) atomicAdd(&h2[2][(key[q] >> 15) & 31u], 1u);
  }
  __syncthreads();
  cluster.sync();  // every CTA's digit-2 histograms are in
  if (t < 96) {
    uint32_t sum = 0;
    for (uint32_t q = 0; q < CS; ++q) sum += cluster.map_shared_rank(&h2[0][0], q)[t];
    (&t2[0][0])[t] = sum;
  }
  __syncthreads();
  if (warp == 0) warp_find_from_top32(t2[0], pick[1], &pick2[0]);
  if (warp == 1) warp_find_from_top32(t2[1], pick[3], &pick2[1]);
  if (warp == 2) warp_find_from_top32(t2[2], pick[5], &pick2[2]);
  __syncthreads();
  cluster.sync();  // no CTA leaves while its histograms may still be read
  if (t == 0 && rank == 0) {
    const uint32_t G = (pick[0] << 20) | (pick2[0] << 15);
    const uint32_t anchor = (pick[2] << 20) | (pick2[1] << 15);
    a.guess[(uint64_t)p * a.nseg + s] = make_uint2(G, hist_shift(G, anchor));
    // The zeroing threshold: the k-th key T of this segment in the last call
    // made with this workspace, if the record holds one (in error-feedback
    // training T moves little from step to step), else the sample's estimate.
    // It only decides which candidates the stream pass zeroes early.
    LongSel& L = a.lsel[(uint64_t)p * a.nlong + item % a.nlong];
    L.mid = L.sig == seg_signature(r) ? L.T : (pick[4] << 20) | (pick2[2] << 15);
  }
}

// Layer-sized segments: one warp per (node, segment), no block barrier. The
// 2,048-entry sample (8 runs of kRun) sits in registers, 64 keys per lane.
constexpr uint32_t kWarpKeys = kWarpSample / 32;

__global__ void __launch_bounds__(kGuessThreads) topk_guess_warp_kernel(Args a, uint32_t nlist) {
  griddep_wait();
  const uint32_t lane = lane_id();
  const uint64_t gw = (uint64_t)blockIdx.x * (kGuessThreads / 32) + (threadIdx.x >> 5);
  if (gw >= (uint64_t)a.P * nlist) return;  // warp-uniform
  const uint32_t p = (uint32_t)(gw / nlist), s = a.warp_list[gw % nlist];
  const SegRec r = a.recs[s];
  const uint64_t seg0 = (uint64_t)p * a.N + r.begin;
  // runs start on the element grid's 4-aligned positions inside the segment
  const uint32_t sh = (uint32_t)((4 - (seg0 & 3)) & 3);
  const float* gp = a.grad + seg0 + sh;
  const float* rp = a.residual + seg0 + sh;
  constexpr uint32_t nruns = kWarpSample / kRun;
  const uint32_t span = r.n - sh - kRun;  // n > kExactMax: positive
  auto run_at = [&](uint32_t run) { return (run * span / (nruns - 1)) & ~(kRun - 1); };
  uint32_t key[kWarpKeys];
  if (a.vec) {
    // a run is 64 float4, two per lane; four runs' loads in flight at once
    constexpr uint32_t kVecRuns = 4, kVecPer = kRun / 128;
#pragma unroll
    for (uint32_t r0 = 0; r0 < nruns; r0 += kVecRuns) {
      float4 x[kVecRuns * kVecPer], y[kVecRuns * kVecPer];
#pragma unroll
      for (uint32_t q = 0; q < kVecRuns * kVecPer; ++q) {
        const uint32_t i = run_at(r0 + q / kVecPer) + ((q % kVecPer) * 32 + lane) * 4;
        x[q] = *reinterpret_cast<const float4*>(rp + i);
        y[q] = *reinterpret_cast<const float4*>(gp + i);
      }
#pragma unroll
      for (uint32_t q = 0; q < kVecRuns * kVecPer; ++q) {
        uint32_t* kq = key + (r0 * kVecPer + q) * 4;
        kq[0] = mag_key(__fadd_rn(x[q].x, y[q].x));
        kq[1] = mag_key(__fadd_rn(x[q].y, y[q].y));
        kq[2] = mag_key(__fadd_rn(x[q].z, y[q].z));
        kq[3] = mag_key(__fadd_rn(x[q].w, y[q].w));
      }
    }
  } else {
    constexpr uint32_t kLines = kRun / 32, kBatchRuns = 2;
#pragma unroll
    for (uint32_t r0 = 0; r0 < nruns; r0 += kBatchRuns) {
      float x[kBatchRuns * kLines], y[kBatchRuns * kLines];
#pragma unroll
      for (uint32_t q = 0; q < kBatchRuns * kLines; ++q) {
        const uint32_t i = run_at(r0 + q / kLines) + (q % kLines) * 32 + lane;
        x[q] = rp[i];
        y[q] = gp[i];
      }
#pragma unroll
      for (uint32_t q = 0; q < kBatchRuns * kLines; ++q)
        key[r0 * kLines + q] = mag_key(__fadd_rn(x[q], y[q]));
    }
  }
  const uint32_t rr = r.rank & 0xffffu;
  uint32_t G = 0;
#pragma unroll 1
  for (int bit = 30; bit >= 15; --bit) {
    const uint32_t trial = G | (1u << bit);
    uint32_t c = 0;
#pragma unroll
    for (uint32_t q = 0; q < kWarpKeys; ++q) c += key[q] >= trial ? 1u : 0u;
    if (warp_sum(c) >= rr) G = trial;
  }
  if (lane == 0) a.guess[(uint64_t)p * a.nseg + s] = make_uint2(G, 0);
}

// ---------------------------------------------------------------------------
// 3. stream: one CTA per (node, chunk). Warp w owns the 1,024 grid positions
// [q0, q0 + 1024) with q0 = floor4(segment start) + j * kChunk + w * kSub,
// restricted to the segment: 8 rounds of one float4 per lane, in two
// batches of four whose 8 loads are in flight before the first is used. Quads wholly inside the segment use
// 128-bit accesses; the segment's ends go entry by entry. UNIFORM (a table of
// equal segments, the last one possibly shorter): the chunk's segment and
// place are arithmetic, so the data loads leave at once; otherwise they wait
// for the chunk's descriptor. The rest of the chunk's description is loaded
// after the data loads are in flight.
// ---------------------------------------------------------------------------
// A lane's candidates of one quad (bit q of `bits`: entry q of acc) into
// the warp's sub-slot at positions pos, pos + 1, ... in index order; those
// past the sub-slot's end are dropped (the segment then falls back to the raw
// select). Only the set bits are visited, and the value is picked by selects
// so acc stays in registers. Returns the bits of the entries stored.
__device__ __forceinline__ uint32_t store_candidates(uint32_t bits, uint32_t pos, uint32_t slot,
                                                     uint32_t* cidx, float* cval, uint32_t idx0,
                                                     const float4& acc, uint64_t keep) {
  uint32_t stored = bits;
  if (pos + __popc(bits) > slot) {  // the sub-slot fills up inside this quad (rare)
    stored = 0;
    uint32_t q_pos = pos;
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q)
      if (bits & (1u << q)) {
        if (q_pos < slot) stored |= 1u << q;
        ++q_pos;
      }
  }
  uint32_t m = stored;
  while (m) {
    const uint32_t q = __ffs(m) - 1;
    m &= m - 1;
    const float v = q == 0 ? acc.x : q == 1 ? acc.y : q == 2 ? acc.z : acc.w;
    st_keep(cidx + pos, idx0 + q, keep);
    st_keep(cval + pos, v, keep);
    ++pos;
  }
  return stored;
}

// Loads NB rounds, t0 .. t0 + NB - 1, of a warp's 1,024 entries: grad and
// residual as 128-bit loads inside the segment, entry by entry at its ends
// (zeros outside). All NB loads are issued before any is used.
template <uint32_t NB>
__device__ __forceinline__ void load_rounds(float4 (&gv)[NB], float4 (&rv)[NB], uint32_t t0,
                                            const float* gp, const float* rp, int32_t lo_r,
                                            int32_t hi_r, bool vec, uint32_t lane) {
#pragma unroll
  for (uint32_t u = 0; u < NB; ++u) {
    const int32_t e0 = (int32_t)(4 * ((t0 + u) * 32 + lane));
    if (vec && e0 >= lo_r && e0 + 4 <= hi_r) {
      gv[u] = __ldcs(reinterpret_cast<const float4*>(gp + e0));
      rv[u] = *reinterpret_cast<const float4*>(rp + e0);
    } else {
      float x[4] = {0.f, 0.f, 0.f, 0.f}, y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int32_t q = 0; q < 4; ++q)
        if (e0 + q >= lo_r && e0 + q < hi_r) {
          x[q] = gp[e0 + q];
          y[q] = rp[e0 + q];
        }
      gv[u] = make_float4(x[0], x[1], x[2], x[3]);
      rv[u] = make_float4(y[0], y[1], y[2], y[3]);
    }
  }
}

template <bool UNIFORM, bool ANY_LONG>
__global__ void __launch_bounds__(kStreamThreads, 4) topk_stream_kernel(Args a) {
  griddep_wait();
  const uint32_t gc = blockIdx.x;
  const uint32_t p = gc / a.nchunk, c = gc - p * a.nchunk;
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  uint32_t begin, end, seg, j;
  uint4 d1 = make_uint4(0, 0, 0, 0);
  if (UNIFORM) {
    seg = min(c / a.u_m, a.nseg - 1);
    j = c - seg * a.u_m;
    begin = seg * a.u_L;
    end = (uint32_t)min((uint64_t)begin + a.u_L, a.N);
  } else {
    const uint4 d0 = reinterpret_cast<const uint4*>(a.desc + c)[0];
    begin = d0.x;
    end = d0.y;
    seg = d0.z;
    j = d0.w;
  }
  const uint64_t row = (uint64_t)p * a.N;
  const uint64_t lo = row + begin, hi = row + end;
  const uint64_t q0 = ((lo & ~(uint64_t)3)) + (uint64_t)j * kChunk + (uint64_t)warp * kSub;
  // (only whether a position is below lo matters: lo_r is clamped to -1)
  const int32_t lo_r = (int32_t)max((int64_t)lo - (int64_t)q0, (int64_t)-1);
  const int32_t hi_r = (int32_t)max(min((int64_t)hi - (int64_t)q0, (int64_t)kSub + 4), (int64_t)-1);
  const float* gp = a.grad + q0;
  float* rp = a.residual + q0;
  // The warp's rounds in two batches of four whose 128-bit loads are all
  // issued before any of their entries is used, at four CTAs per SM (64
  // registers; five would spill).
  constexpr uint32_t kBatch = kRounds / 2;
  float4 gv[kBatch], rv[kBatch];
  load_rounds<kBatch>(gv, rv, 0, gp, rp, lo_r, hi_r, a.vec, lane);
  // the rest of the description, while the data loads are in flight
  uint32_t slot, slot32, kind, aux;
  if (UNIFORM) {
    const SegRec& r = a.recs[seg];
    slot = r.slot;
    kind = r.kind;
    aux = r.kind == kLong ? r.lidx : r.out0;
    slot32 = r.slot32 + j * kWarpsPerChunk * (slot / 32);
  } else {
    d1 = reinterpret_cast<const uint4*>(a.desc + c)[1];
    slot = d1.x;
    slot32 = d1.y;
    kind = d1.z;
    aux = d1.w;
  }
  const uint64_t gs = (uint64_t)p * a.nseg + seg;
  const uint32_t G = a.guess[gs].x;
  const uint32_t base_u = (uint32_t)(q0 - row);  // node-local index of q0, modulo 2^32
  if (kind == kKeepAll) {  // CTA-uniform. k = n: every entry goes to the stream, residual 0
    const uint64_t o = (uint64_t)p * a.cap + aux - begin;  // + node-local index
#pragma unroll
    for (uint32_t t = 0; t < kRounds; ++t) {
      const uint32_t u = t % kBatch;
      if (t > 0 && u == 0) load_rounds<kBatch>(gv, rv, t, gp, rp, lo_r, hi_r, a.vec, lane);
      const int32_t e0 = (int32_t)(4 * (t * 32 + lane));
      const float av[4] = {__fadd_rn(rv[u].x, gv[u].x), __fadd_rn(rv[u].y, gv[u].y),
                           __fadd_rn(rv[u].z, gv[u].z), __fadd_rn(rv[u].w, gv[u].w)};
#pragma unroll
      for (int32_t q = 0; q < 4; ++q)
        if (e0 + q >= lo_r && e0 + q < hi_r) {
          const uint32_t idx = base_u + (uint32_t)(e0 + q);
          a.out_idx[o + idx] = idx;
          a.out_val[o + idx] = av[q];
          rp[e0 + q] = 0.0f;
        }
    }
    return;
  }
  const uint64_t sub = (uint64_t)gc * kWarpsPerChunk + warp;
  const uint64_t slot0 = (uint64_t)p * a.node_slots + (uint64_t)slot32 * 32 + (uint64_t)warp * slot;
  // Long segments: the stream pass writes +0.0f (over the acc just stored)
  // for every candidate it stores at or above the mid guess Gm (an estimate
  // of T), and the select then zeroes the kept candidates below Gm and
  // restores acc at the stored ones at or above it that are not kept: few
  // scattered writes, where zeroing every kept candidate afterwards would
  // scatter k of them.
  const bool long_seg = ANY_LONG && kind == kLong;
  const uint32_t Gm = long_seg ? a.lsel[(uint64_t)p * a.nlong + aux].mid : 0u;
  uint32_t* const cidx = a.cand_idx + slot0;  // the warp's sub-slot
  float* const cval = a.cand_val + slot0;
  const uint64_t keep = l2_policy_evict_last();
  uint32_t run = 0;  // candidates so far in this sub-chunk (warp-uniform)
#pragma unroll
  for (uint32_t t = 0; t < kRounds; ++t) {
    const uint32_t u = t % kBatch;
    if (t > 0 && u == 0) load_rounds<kBatch>(gv, rv, t, gp, rp, lo_r, hi_r, a.vec, lane);
    const int32_t e0 = (int32_t)(4 * (t * 32 + lane));
    float4 acc;
    acc.x = __fadd_rn(rv[u].x, gv[u].x);
    acc.y = __fadd_rn(rv[u].y, gv[u].y);
    acc.z = __fadd_rn(rv[u].z, gv[u].z);
    acc.w = __fadd_rn(rv[u].w, gv[u].w);
    const float av[4] = {acc.x, acc.y, acc.z, acc.w};
    const bool full = a.vec && e0 >= lo_r && e0 + 4 <= hi_r;
    // the residual gets acc: stored first, then the candidates
    uint32_t bits = 0;
    if (full) {
      *reinterpret_cast<float4*>(rp + e0) = acc;
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) bits |= (mag_key(av[q]) >= G ? 1u : 0u) << q;
    } else {
#pragma unroll
      for (int32_t q = 0; q < 4; ++q)
        if (e0 + q >= lo_r && e0 + q < hi_r) {
          rp[e0 + q] = av[q];
          bits |= (mag_key(av[q]) >= G ? 1u : 0u) << q;
        }
    }
    if (__ballot_sync(0xffffffffu, bits) == 0) continue;  // warp-uniform
    uint32_t tot;
    const uint32_t pos = run + warp_excl_small(__popc(bits), &tot);
    run += tot;
    const uint32_t stored =
        store_candidates(bits, pos, slot, cidx, cval, base_u + (uint32_t)e0, acc, keep);
    if constexpr (ANY_LONG) {
      if (long_seg) {
#pragma unroll
        for (uint32_t q = 0; q < 4; ++q)
          if (((stored >> q) & 1u) && mag_key(av[q]) >= Gm) rp[e0 + q] = 0.0f;
      }
    }
  }
  // Pad the sub-slot's last 32-byte sector: every sector of candidates is
  // written whole, so no later eviction from L2 leaves a half-written sector.
  const uint32_t pad_end = min((run + 7u) & ~7u, slot);
  if (run + lane < pad_end) {
    st_keep(cidx + run + lane, kNone, keep);
    st_keep(cval + run + lane, 0.0f, keep);
  }
  if (lane == 0) {
    a.sub_cnt[sub] = run;
    if (run > slot) atomicOr(&a.seg_flag[gs], 1u);
  }
  if constexpr (ANY_LONG) {
    // A long segment's chunks all add to one counter: one add per CTA (the
    // chunk's warps summed in shared memory), not per warp, keeps that L2
    // sector from serialising the launch.
    __shared__ uint32_t cta_run[kWarpsPerChunk];
    if (lane == 0) cta_run[warp] = run;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t sum = 0;
#pragma unroll
      for (uint32_t w = 0; w < kWarpsPerChunk; ++w) sum += cta_run[w];
      if (sum) atomicAdd(&a.seg_cnt[gs], sum);
    }
  } else {
    if (lane == 0 && run) atomicAdd(&a.seg_cnt[gs], run);
  }
}

// ---------------------------------------------------------------------------
// 4a. select of a layer-sized segment whose candidates were all kept in
// their sub-slots (at most kShortCands over at most kShortSubs sub-chunks):
// one CTA of kSegThreads per (node, segment):
//  1. each thread copies its sub-chunks' candidates into shared memory with
//     cp.async (every copy in flight at once), at the sub-chunks' offsets;
//  2. four radix digits (8, 8, 8, 7 bits) of the k-th key T, each from one
//     256-bin histogram over the shared copy (warp-aggregated adds), its
//     bins scanned from the top by warp 0;
//  3. thread t writes the kept entries of its contiguous candidate range in
//     index order at the offset given by a block scan of its counts (keys
//     > T, and keys == T up to tie_take, lowest indices first); then the
//     offsets are resolved to indices and the residual is zeroed there.
// Segments that do not qualify go to the to-do list of the raw select.
// ---------------------------------------------------------------------------
constexpr uint32_t kSegThreads = 128;
constexpr uint32_t kShortSubs = 3 * kSegThreads;  // 33 chunks of a layer-sized segment fit
constexpr uint32_t kShortCands = 8192;
// Layer-sized segments expected to leave more candidates than this go to the
// range-parallel long select instead (their guess then samples 8,192 entries).
constexpr uint32_t kShortExpect = 6144;

__device__ __forceinline__ uint32_t warp_excl_sum(uint32_t v, uint32_t* total) {
  const uint32_t incl = warp_incl_sum(v);
  *total = __shfl_sync(0xffffffffu, incl, 31);
  return incl - v;
}

__global__ void __launch_bounds__(kSegThreads) topk_select_short_kernel(Args a, uint32_t nlist) {
  griddep_wait();
  __shared__ uint32_t wpre[kShortSubs + 1];
  __shared__ float vals[kShortCands];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t dig[2];
  const uint32_t t = threadIdx.x, lane = lane_id(), warp = t >> 5;
  const uint32_t p = blockIdx.x / nlist, s = a.short_list[blockIdx.x % nlist];
  const SegRec r = a.recs[s];
  const uint64_t gs = (uint64_t)p * a.nseg + s;
  const uint32_t k = r.k, nsub = r.nchunk * kWarpsPerChunk;
  const uint32_t cnt = a.seg_cnt[gs];
  if (a.seg_flag[gs] != 0 || cnt < k || cnt > kShortCands || nsub > kShortSubs) {
    if (t == 0) a.todo[atomicAdd(a.todo_cnt, 1u)] = (uint32_t)gs;  // CTA-uniform
    return;
  }
  const uint64_t sub0 = ((uint64_t)p * a.nchunk + r.chunk0) * kWarpsPerChunk;
  const uint64_t slot_base = (uint64_t)p * a.node_slots + (uint64_t)r.slot32 * 32;
  const uint32_t* cidx = a.cand_idx + slot_base;
  const float* cval = a.cand_val + slot_base;
  // 1. offsets of the sub-chunks' candidates (thread t: sub-chunks 3t .. 3t + 2)
  uint32_t c3[3], csum = 0;
#pragma unroll
  for (uint32_t i = 0; i < 3; ++i) {
    const uint32_t w = 3 * t + i;
    c3[i] = w < nsub ? a.sub_cnt[sub0 + w] : 0u;
    csum += c3[i];
  }
  uint32_t M;
  uint32_t off = block_excl_scan(csum, scratch, &M);
#pragma unroll
  for (uint32_t i = 0; i < 3; ++i) {
    const uint32_t w = 3 * t + i;
    if (w < nsub) wpre[w] = off;
    for (uint32_t e = 0; e < c3[i]; ++e) cp_async4(vals + off + e, cval + (uint64_t)w * r.slot + e);
    off += c3[i];
  }
  if (t == 0) wpre[nsub] = M;
  cp_async_wait_all();
  __syncthreads();
  // 2. radix digits of T (bits 30..23, 22..15, 14..7, 6..0)
  uint32_t prefix = 0, rem = k;
  for (int d = 0; d < 4; ++d) {
    const uint32_t shift = d == 3 ? 0 : 23 - 8 * d;
    const uint32_t wbits = d == 3 ? 7 : 8, hi_shift = shift + wbits;
    for (uint32_t i = t; i < 256; i += kSegThreads) hist[i] = 0;
    __syncthreads();
    for (uint32_t v0 = 0; v0 < M; v0 += kSegThreads) {
      const uint32_t v = v0 + t;
      const uint32_t key = v < M ? mag_key(vals[v]) : 0u;
      const bool match = v < M && (d == 0 || (key >> hi_shift) == prefix);
      hist_add(hist, (key >> shift) & ((1u << wbits) - 1u), match);
    }
    __syncthreads();
    if (warp == 0) {  // bins from high to low: lane covers 8 of them
      uint32_t hb[8], sum = 0;
#pragma unroll
      for (uint32_t i = 0; i < 8; ++i) {
        hb[i] = hist[255 - (8 * lane + i)];
        sum += hb[i];
      }
      uint32_t tot;
      const uint32_t excl = warp_excl_sum(sum, &tot);
      uint32_t b = 0xffffffffu, ab = 0;
      if (excl < rem && rem <= excl + sum) {
        uint32_t acc = excl;
#pragma unroll
        for (uint32_t i = 0; i < 8; ++i) {
          if (b == 0xffffffffu && acc + hb[i] >= rem) {
            b = 255 - (8 * lane + i);
            ab = acc;
          }
          acc += hb[i];
        }
      }
      const uint32_t found = __ballot_sync(0xffffffffu, b != 0xffffffffu);
      if (lane == 0 && !found) {  // cannot happen for consistent counts
        set_status(a.status, SPARCML_ERR_BAD_STREAM);
        dig[0] = 0;
        dig[1] = rem;
      }
      if (found && lane == __ffs(found) - 1) {
        dig[0] = b;
        dig[1] = rem - ab;
      }
    }
    __syncthreads();
    prefix = (prefix << wbits) | dig[0];
    rem = dig[1];
  }
  const uint32_t T = prefix, tie_take = rem;  // keys == T to keep, lowest indices first
  // 3. ordered write of this thread's contiguous range
  const uint32_t per = (M + kSegThreads - 1) / kSegThreads;
  const uint32_t v_lo = min(t * per, M), v_hi = min(v_lo + per, M);
  uint32_t n_gt = 0, n_eq = 0;
  for (uint32_t v = v_lo; v < v_hi; ++v) {
    const uint32_t key = mag_key(vals[v]);
    n_gt += key > T ? 1u : 0u;
    n_eq += key == T ? 1u : 0u;
  }
  uint32_t tot;  // both counts in one scan: M <= kShortCands < 2^16
  const uint32_t ex = block_excl_scan((n_gt << 16) | n_eq, scratch, &tot);
  uint32_t e_gt = ex >> 16, e_eq = ex & 0xffffu;
  float* rp = a.residual + (uint64_t)p * a.N;
  const uint64_t out0 = (uint64_t)p * a.cap + r.out0;
  uint32_t* oi = a.out_idx + out0;
  const uint64_t keep = l2_policy_evict_last();
  uint32_t w = 0;  // sub-chunk of v_lo: the largest w with wpre[w] <= v_lo
  for (uint32_t step = 256; step > 0; step >>= 1)
    if (w + step <= nsub && wpre[w + step] <= v_lo) w += step;
  for (uint32_t v = v_lo; v < v_hi; ++v) {
    const float x = vals[v];
    const uint32_t key = mag_key(x);
    const bool gt = key > T, eq = key == T;
    if (gt || (eq && e_eq < tie_take)) {
      const uint32_t pos = e_gt + min(e_eq, tie_take);
      while (wpre[w + 1] <= v) ++w;
      if (pos < k) {
        oi[pos] = w * r.slot + (v - wpre[w]);  // slot offset for now
        st_keep(a.out_val + out0 + pos, x, keep);
      } else {
        set_status(a.status, SPARCML_ERR_BAD_STREAM);
      }
    }
    e_gt += gt ? 1u : 0u;
    e_eq += eq ? 1u : 0u;
  }
  __syncthreads();  // the offsets written above are visible to the whole CTA
  // offsets -> indices; the residual is zeroed at each kept index. (Every
  // position below k was written above when the counts are consistent; an
  // offset out of the segment's sub-slots is skipped, not followed.)
  const uint32_t span = nsub * r.slot;
  for (uint32_t i = t; i < k; i += kSegThreads) {
    const uint32_t o = oi[i];
    if (o >= span) {
      set_status(a.status, SPARCML_ERR_BAD_STREAM);
      continue;
    }
    const uint32_t idx = cidx[o];
    st_keep(oi + i, idx, keep);
    if (idx - r.begin < r.n) rp[idx] = 0.0f;
  }
}

// ---------------------------------------------------------------------------
// 4b. select of a long segment from its candidates.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bin_of(uint32_t key, uint32_t G, uint32_t shift) {
  return min((key - G) >> shift, kBins - 1);
}

// The boundary bin from the histogram the stream pass built; a segment whose
// candidates cannot decide its select is handed to the raw select.
__global__ void __launch_bounds__(256) long_find_kernel(Args a) {
  griddep_wait();
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t res[2];
  const uint32_t p = blockIdx.x / a.nlong, ls = blockIdx.x % a.nlong;
  const uint32_t s = a.long_list[ls];
  const SegRec r = a.recs[s];
  const uint64_t gs = (uint64_t)p * a.nseg + s, pl = (uint64_t)p * a.nlong + ls;
  LongSel& L = a.lsel[pl];
  if (a.seg_flag[gs] != 0 || a.seg_cnt[gs] < r.k) {  // CTA-uniform
    if (threadIdx.x == 0) L.mode = kModeFallback;
    return;
  }
  find_from_top(a.hist + pl * kBins, kBins, r.k, scratch, res);
  if (threadIdx.x == 0) {
    if (res[0] == kNone) {  // counts disagree with the candidates: decide it again raw
      L.mode = kModeFallback;
    } else {
      L.mode = kModeNormal;
      L.bin = res[0];
      L.rank = r.k - res[1];
    }
  }
}

// The candidates of one range (kRangeSubs sub-chunks) of a long segment,
// warp w taking its 32 sub-chunks' candidates as one sequence: f(v, idx_ptr,
// val_ptr) for v = 0 .. its count, in index order, 32 lanes at a time.
struct RangeView {
  uint32_t p, ls, s, rr;  // node, long segment, segment id, range within the segment
  SegRec rec;
  uint64_t gs, pl;
  uint32_t excl;          // candidates of this lane's sub-chunk before it in the warp
  uint32_t own;           // candidates of this lane's sub-chunk
  uint32_t count;         // this warp's candidates
  uint64_t slot_base;     // this warp's first sub-slot
};

// Range gr = p * nranges + rid, seen by warp `warp` (0..7) of its 8 warps.
__device__ __forceinline__ bool range_view_at(const Args& a, RangeView* v, uint32_t gr,
                                              uint32_t warp) {
  const uint32_t rid = gr % a.nranges;
  v->p = gr / a.nranges;
  const uint32_t m = a.range_map[rid];
  v->ls = m >> 16;
  v->rr = m & 0xffffu;
  v->s = a.long_list[v->ls];
  v->rec = a.recs[v->s];
  v->gs = (uint64_t)v->p * a.nseg + v->s;
  v->pl = (uint64_t)v->p * a.nlong + v->ls;
  const uint32_t lane = lane_id();
  const uint32_t nsub = v->rec.nchunk * kWarpsPerChunk;
  const uint32_t w0 = v->rr * kRangeSubs + warp * 32;  // the warp's first sub-chunk
  const uint32_t w = w0 + lane;
  const uint64_t sub0 = ((uint64_t)v->p * a.nchunk + v->rec.chunk0) * kWarpsPerChunk;
  const uint32_t c = w < nsub ? min(a.sub_cnt[sub0 + w], v->rec.slot) : 0u;
  const uint32_t incl = warp_incl_sum(c);
  v->excl = incl - c;
  v->own = c;
  v->count = __shfl_sync(0xffffffffu, incl, 31);
  v->slot_base = (uint64_t)v->p * a.node_slots + (uint64_t)v->rec.slot32 * 32 +
                 (uint64_t)w0 * v->rec.slot;
  return true;
}

// The range of a CTA of 256 threads: blockIdx.x.
__device__ __forceinline__ bool range_view(const Args& a, RangeView* v) {
  return range_view_at(a, v, blockIdx.x, threadIdx.x >> 5);
}

// Offset (from the warp's first sub-slot) of the warp's candidate number x:
// sub-chunk i = the last lane whose exclusive count is <= x (five shuffles),
// then x - excl_i into it. Below 32 * 1,024: 32 bits.
__device__ __forceinline__ uint32_t range_off(const RangeView& v, uint32_t x) {
  uint32_t i = 0;
#pragma unroll
  for (uint32_t step = 16; step > 0; step >>= 1) {
    const uint32_t cand = i + step;
    const uint32_t e = __shfl_sync(0xffffffffu, v.excl, cand & 31u);
    if (cand < 32 && e <= x) i = cand;
  }
  const uint32_t e = __shfl_sync(0xffffffffu, v.excl, i);
  return i * v.rec.slot + (x - e);
}

// The same offsets for the warp's first kTab candidates, as a table in
// shared memory that each lane fills for its own sub-chunk: a candidate
// x < kTab then takes one shared load instead of the search above.
constexpr uint32_t kTab = 512;
__device__ __forceinline__ void range_table(const RangeView& v, uint32_t* tab /* [kTab] */) {
  const uint32_t lane = lane_id();
  const uint32_t end = min(v.excl + v.own, kTab);
  const uint32_t base = lane * v.rec.slot - v.excl;  // offset of x is base + x (mod 2^32)
  for (uint32_t x = v.excl; x < end; ++x) tab[x] = base + x;
  __syncwarp();
}

// Candidates a lane holds in registers at once: a warp's first 512 are all
// loaded before any is used (a warp of 32 sub-chunks holds about 500 at 1.5 %
// density); any beyond are taken in further batches.
constexpr uint32_t kHold = 16;
static_assert(kTab == 32 * kHold, "the held candidates are the tabled ones");

// Per range: the candidates' bins, (key - G) >> shift (the top bin takes
// everything above), counted in shared memory and added to the (node,
// segment) histogram. A segment whose sub-slots overflowed is skipped: its
// select falls back to the raw select.
__global__ void __launch_bounds__(256) long_hist_kernel(Args a) {
  griddep_wait();
  __shared__ uint32_t h[kBins];
  for (uint32_t b = threadIdx.x; b < kBins; b += blockDim.x) h[b] = 0;
  __syncthreads();
  RangeView v;
  range_view(a, &v);
  if (a.seg_flag[v.gs] != 0) return;  // CTA-uniform
  const uint32_t lane = lane_id();
  const uint2 gsh = a.guess[v.gs];
  const float* cv = a.cand_val + v.slot_base;
  __shared__ uint32_t tabs[kStreamThreads / 32][kTab];
  uint32_t* tab = tabs[threadIdx.x >> 5];
  range_table(v, tab);
  for (uint32_t x0 = 0; x0 < v.count; x0 += 32 * kHold) {
    float xv[kHold];
#pragma unroll
    for (uint32_t u = 0; u < kHold; ++u) {
      const uint32_t x = x0 + u * 32 + lane;
      const uint32_t xm = min(x, v.count - 1);
      const uint32_t o = x0 == 0 ? tab[xm] : range_off(v, xm);  // x0: warp-uniform
      xv[u] = x < v.count ? cv[o] : 0.0f;
    }
#pragma unroll
    for (uint32_t u = 0; u < kHold; ++u)
      if (x0 + u * 32 + lane < v.count) atomicAdd(&h[bin_of(mag_key(xv[u]), gsh.x, gsh.y)], 1u);
  }
  __syncthreads();
  uint32_t* gh = a.hist + v.pl * kBins;
  for (uint32_t b = threadIdx.x; b < kBins; b += blockDim.x)
    if (h[b]) atomicAdd(gh + b, h[b]);  // result unused: a reduction in L2
}

// Per range: candidates above the boundary bin are counted; those in it are
// appended (key, index) to the segment's boundary buffer.
__global__ void __launch_bounds__(256, 4) long_collect_kernel(Args a) {
  griddep_wait();
  __shared__ uint32_t wgt[8];
  RangeView v;
  range_view(a, &v);
  if (a.lsel[v.pl].mode != kModeNormal) return;  // CTA-uniform
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint2 gsh = a.guess[v.gs];
  const uint32_t bstar = a.lsel[v.pl].bin;
  uint2* bnd = a.bnd + v.pl * kBoundCap;
  const float* cv = a.cand_val + v.slot_base;
  const uint32_t* ci = a.cand_idx + v.slot_base;
  __shared__ uint32_t tabs[kStreamThreads / 32][kTab];
  uint32_t* tab = tabs[warp];
  range_table(v, tab);
  uint32_t gt = 0;
  for (uint32_t x0 = 0; x0 < v.count; x0 += 32 * kHold) {
    float xv[kHold];
#pragma unroll
    for (uint32_t u = 0; u < kHold; ++u) {
      const uint32_t x = x0 + u * 32 + lane;
      const uint32_t xm = min(x, v.count - 1);
      const uint32_t o = x0 == 0 ? tab[xm] : range_off(v, xm);  // x0: warp-uniform
      xv[u] = x < v.count ? cv[o] : 0.0f;
    }
#pragma unroll
    for (uint32_t u = 0; u < kHold; ++u) {
      const uint32_t x = x0 + u * 32 + lane;
      if (x0 + u * 32 >= v.count) break;  // warp-uniform
      const uint32_t key = mag_key(xv[u]);
      const uint32_t b = bin_of(key, gsh.x, gsh.y);
      gt += (x < v.count && b > bstar) ? 1u : 0u;
      const bool inb = x < v.count && b == bstar;
      const uint32_t m = __ballot_sync(0xffffffffu, inb);
      if (m) {
        const uint32_t xm = min(x, v.count - 1);
        const uint32_t o = x0 == 0 ? tab[xm] : range_off(v, xm);  // the whole warp
        uint32_t base = 0;
        if (lane == 0) base = atomicAdd(&a.bnd_cnt[v.pl], (uint32_t)__popc(m));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (inb) {
          const uint32_t pos = base + __popc(m & lanemask_lt());
          if (pos < kBoundCap) bnd[pos] = make_uint2(key, ci[o]);
          else atomicOr(&a.lsel[v.pl].overflow, 1u);
        }
      }
    }
  }
  gt = warp_sum(gt);
  if (lane == 0) wgt[warp] = gt;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t sum = 0;
    for (uint32_t w = 0; w < 8; ++w) sum += wgt[w];
    a.range_gt[(uint64_t)v.p * a.nranges + blockIdx.x % a.nranges] = sum;
  }
}

// Per (node, long segment), one CTA of 1,024 threads: the exact k-th key T
// among the boundary bin's candidates (three radix digits in shared memory),
// the index cut I_T (keys equal to T are kept up to the tie_take-th lowest
// index: four 8-bit digits of the index), the kept boundary entries counted
// per range, and the output offset of every range (a scan over the ranges).
constexpr uint32_t kExactThreads = 1024;

__global__ void __launch_bounds__(kExactThreads) long_exact_kernel(Args a) {
  griddep_wait();
  extern __shared__ __align__(16) uint32_t dyn[];
  uint32_t* skey = dyn;                     // [kBoundCap]
  uint32_t* sidx = skey + kBoundCap;        // [kBoundCap]
  uint32_t* rkeep = sidx + kBoundCap;       // [kMaxRanges] kept boundary entries per range
  uint32_t* hist = rkeep + kMaxRanges;      // [2048]
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t res[2];
  const uint32_t t = threadIdx.x;
  const uint32_t p = blockIdx.x / a.nlong, ls = blockIdx.x % a.nlong;
  const uint32_t s = a.long_list[ls];
  const SegRec r = a.recs[s];
  const uint64_t pl = (uint64_t)p * a.nlong + ls;
  LongSel& L = a.lsel[pl];
  if (L.mode != kModeNormal) return;  // CTA-uniform
  const uint32_t M = a.bnd_cnt[pl];
  if (L.overflow || M > kBoundCap || M < L.rank) {
    __syncthreads();
    if (t == 0) L.mode = kModeFallback;
    return;
  }
  const uint2* bnd = a.bnd + pl * kBoundCap;
  for (uint32_t i = t; i < M; i += kExactThreads) {
    const uint2 e = bnd[i];
    skey[i] = e.x;
    sidx[i] = e.y;
  }
  const uint32_t nr = (r.nchunk * kWarpsPerChunk + kRangeSubs - 1) / kRangeSubs;
  for (uint32_t i = t; i < nr; i += kExactThreads) rkeep[i] = 0;
  __syncthreads();
  // the rank-th largest key: digits of 11, 11 and 9 bits
  uint32_t prefix = 0, rem = L.rank;
  for (int d = 0; d < 3; ++d) {
    const uint32_t width = d < 2 ? 11 : 9, shift = d == 0 ? 20 : (d == 1 ? 9 : 0);
    const uint32_t nb = 1u << width, hi_shift = shift + width;
    for (uint32_t b = t; b < 2048; b += kExactThreads) hist[b] = 0;
    __syncthreads();
    for (uint32_t i = t; i < M; i += kExactThreads) {
      const uint32_t key = skey[i];
      if (d == 0 || (key >> hi_shift) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    find_from_top(hist, 2048, rem, scratch, res);  // bins past nb stay zero
    uint32_t b = res[0];
    if (b == kNone) {  // cannot happen for consistent counts
      set_status(a.status, SPARCML_ERR_BAD_STREAM);
      b = 0;
    } else {
      rem -= res[1];
    }
    prefix = (prefix << width) | b;
    __syncthreads();
  }
  const uint32_t T = prefix, tie_take = rem;  // keys == T to keep, lowest indices first
  // index cut among keys == T: the tie_take-th smallest index (4 digits of 8 bits)
  uint32_t n_eq = 0;
  for (uint32_t i = t; i < M; i += kExactThreads) n_eq += skey[i] == T ? 1u : 0u;
  uint32_t eq_total;
  block_excl_scan(n_eq, scratch, &eq_total);
  uint32_t cut = 0xffffffffu;
  if (tie_take < eq_total) {
    uint32_t ip = 0, irem = tie_take;  // smallest first: count from the bottom
    for (int d = 0; d < 4; ++d) {
      const uint32_t shift = 24 - 8 * d;
      for (uint32_t b = t; b < 2048; b += kExactThreads) hist[b] = 0;
      __syncthreads();
      for (uint32_t i = t; i < M; i += kExactThreads) {
        const uint32_t x = sidx[i];
        if (skey[i] == T && (d == 0 || (x >> (shift + 8)) == ip))
          atomicAdd(&hist[2047 - ((x >> shift) & 255u)], 1u);  // reversed: smallest on top
      }
      __syncthreads();
      find_from_top(hist, 2048, irem, scratch, res);
      uint32_t b = res[0];
      if (b == kNone) {
        set_status(a.status, SPARCML_ERR_BAD_STREAM);
        b = 2047;
      } else {
        irem -= res[1];
      }
      ip = (ip << 8) | (2047 - b);
      __syncthreads();
    }
    cut = ip;
  }
  // kept boundary entries per range
  const uint64_t row = (uint64_t)p * a.N;
  const uint64_t A = (row + r.begin) & ~3ull;
  for (uint32_t i = t; i < M; i += kExactThreads) {
    const uint32_t key = skey[i], x = sidx[i];
    if (key > T || (key == T && x <= cut)) {
      const uint32_t sub = (uint32_t)((row + x - A) / kSub);
      atomicAdd(&rkeep[sub / kRangeSubs], 1u);
    }
  }
  __syncthreads();
  // output offsets of the ranges: above-bin counts plus kept boundary entries
  const uint64_t rg0 = (uint64_t)p * a.nranges + r.range0;
  uint32_t run = 0;
  for (uint32_t i0 = 0; i0 < nr; i0 += kExactThreads) {
    const uint32_t i = i0 + t;
    const uint32_t c = i < nr ? a.range_gt[rg0 + i] + rkeep[i] : 0u;
    uint32_t tot;
    const uint32_t ex = block_excl_scan(c, scratch, &tot);
    if (i < nr) a.range_off[rg0 + i] = run + ex;
    run += tot;
    __syncthreads();
  }
  if (t == 0) {
    if (run != r.k) {  // the counts do not add up: decide the segment again raw
      L.mode = kModeFallback;
    } else {
      L.T = T;
      L.cut = cut;
      L.sig = seg_signature(r);
    }
  }
}

// Per range: every candidate with key > T, or key == T and index <= I_T, in
// index order at the range's offset. The residual: the stream pass zeroed the
// candidates with key >= Gm (the mid guess); a kept one below Gm is zeroed
// here and a stored one at or above Gm that is not kept gets its acc back. Each warp loads its
// first 512 candidates' values and indices together (both are needed:
// the index is the output or the restore address) and holds them between
// the count and the write; any beyond are read again.
__global__ void __launch_bounds__(256) long_write_kernel(Args a) {
  griddep_wait();
  __shared__ uint32_t wcnt[8];
  __shared__ uint32_t wbase[8];
  __shared__ uint32_t roff;
  RangeView v;
  range_view(a, &v);
  if (a.lsel[v.pl].mode != kModeNormal) return;  // CTA-uniform
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) roff = a.range_off[(uint64_t)v.p * a.nranges + blockIdx.x % a.nranges];
  const LongSel L = a.lsel[v.pl];
  const uint32_t T = L.T, cut = L.cut, Gm = L.mid;
  const float* cv = a.cand_val + v.slot_base;
  const uint32_t* ci = a.cand_idx + v.slot_base;
  auto kept = [&](float x, uint32_t idx, bool valid) {
    const uint32_t key = mag_key(x);
    return valid && (key > T || (key == T && idx <= cut));
  };
  __shared__ uint32_t tabs[kStreamThreads / 32][kTab];
  range_table(v, tabs[warp]);
  float xv[kHold];
  uint32_t iv[kHold];
#pragma unroll
  for (uint32_t u = 0; u < kHold; ++u) {
    const uint32_t x = u * 32 + lane;
    const uint32_t o = tabs[warp][min(x, v.count - 1)];
    xv[u] = x < v.count ? cv[o] : 0.0f;
    iv[u] = x < v.count ? ci[o] : 0u;
  }
  uint32_t kb = 0, n = 0;
#pragma unroll
  for (uint32_t u = 0; u < kHold; ++u) {
    const bool k_ = kept(xv[u], iv[u], u * 32 + lane < v.count);
    kb |= (k_ ? 1u : 0u) << u;
    n += k_ ? 1u : 0u;
  }
  for (uint32_t x0 = 32 * kHold; x0 < v.count; x0 += 32) {
    const uint32_t x = x0 + lane;
    const uint32_t o = range_off(v, min(x, v.count - 1));
    n += kept(x < v.count ? cv[o] : 0.0f, x < v.count ? ci[o] : 0u, x < v.count) ? 1u : 0u;
  }
  n = warp_sum(n);
  if (lane == 0) wcnt[warp] = n;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t run = roff;
    for (uint32_t w = 0; w < 8; ++w) {
      wbase[w] = run;
      run += wcnt[w];
    }
  }
  __syncthreads();
  uint32_t pos = wbase[warp];
  const uint64_t out0 = (uint64_t)v.p * a.cap + v.rec.out0;
  float* rp = a.residual + (uint64_t)v.p * a.N;
  const uint64_t keep = l2_policy_evict_last();
  auto emit = [&](bool valid, bool k_, uint32_t idx, float val) {
    const uint32_t m = __ballot_sync(0xffffffffu, k_);
    const bool zeroed = mag_key(val) >= Gm;
    if (k_) {
      const uint32_t o = pos + __popc(m & lanemask_lt());
      if (o < v.rec.k) {
        st_keep(a.out_idx + out0 + o, idx, keep);
        st_keep(a.out_val + out0 + o, val, keep);
      } else {
        set_status(a.status, SPARCML_ERR_BAD_STREAM);
      }
      if (!zeroed) rp[idx] = 0.0f;
    } else if (valid && zeroed) {
      rp[idx] = val;
    }
    pos += __popc(m);
  };
#pragma unroll
  for (uint32_t u = 0; u < kHold; ++u) emit(u * 32 + lane < v.count, (kb >> u) & 1u, iv[u], xv[u]);
  for (uint32_t x0 = 32 * kHold; x0 < v.count; x0 += 32) {
    const uint32_t x = x0 + lane;
    const uint32_t o = range_off(v, min(x, v.count - 1));
    const float val = x < v.count ? cv[o] : 0.0f;
    const uint32_t idx = x < v.count ? ci[o] : 0u;
    emit(x < v.count, kept(val, idx, x < v.count), idx, val);
  }
}

// Before the raw select re-reads a long segment that fell back: every
// candidate the stream pass stored (and zeroed in the residual) gets its acc
// back, so the residual holds acc over the whole segment again.
__global__ void __launch_bounds__(256) long_restore_kernel(Args a) {
  griddep_wait();
  {  // most segments did not fall back: look at the mode before the range's records
    const uint32_t ls = a.range_map[blockIdx.x % a.nranges] >> 16;
    if (a.lsel[(uint64_t)(blockIdx.x / a.nranges) * a.nlong + ls].mode != kModeFallback) return;
  }
  RangeView v;
  range_view(a, &v);
  const uint32_t lane = lane_id();
  const float* cv = a.cand_val + v.slot_base;
  const uint32_t* ci = a.cand_idx + v.slot_base;
  float* rp = a.residual + (uint64_t)v.p * a.N;
  for (uint32_t x0 = 0; x0 < v.count; x0 += 32) {
    const uint32_t x = x0 + lane;
    const uint32_t o = range_off(v, min(x, v.count - 1));
    if (x < v.count) rp[ci[o]] = cv[o];
  }
}

// ---------------------------------------------------------------------------
// 4c. raw select: the segment decided from its acc (already in residual), by
// a cluster of CS CTAs (CTA q owns the q-th of CS equal parts). Three radix
// digits (11, 11, 9 bits) of the exact k-th key T, the histograms summed
// through distributed shared memory; then each CTA's counts of keys > T and
// == T, their prefix over the cluster, and an ordered compaction.
// ---------------------------------------------------------------------------
constexpr uint32_t kRawThreads = 256;
constexpr uint32_t kRawCluster = 8;

struct RawShared {
  uint32_t hist[2048];
  uint32_t tot[2048];
  uint32_t scratch[34];
  uint32_t res[2];
  uint32_t cnt[2];  // this CTA's (> T, == T) counts, read by higher ranks
};

__device__ void select_raw(const Args& a, RawShared& sh, cg::cluster_group& cluster, uint32_t p,
                           uint32_t s, uint32_t rank, uint32_t CS) {
  const SegRec r = a.recs[s];
  const uint32_t t = threadIdx.x, k = r.k;
  if (t == 0 && rank == 0) atomicAdd(a.fallbacks, 1u);
  const uint32_t lo = r.begin + (uint32_t)((uint64_t)r.n * rank / CS);
  const uint32_t hi = r.begin + (uint32_t)((uint64_t)r.n * (rank + 1) / CS);
  const float* rp0 = a.residual + (uint64_t)p * a.N;
  float* rp = a.residual + (uint64_t)p * a.N;
  auto for_each = [&](auto&& body) {
    for (uint32_t v0 = lo; v0 < hi; v0 += blockDim.x) {
      const uint32_t i = v0 + t;
      const bool valid = i < hi;
      body(valid, i, valid ? rp0[i] : 0.0f);
    }
  };
  uint32_t prefix = 0, rem = k;
  for (int d = 0; d < 3; ++d) {
    const uint32_t width = d < 2 ? 11 : 9, shift = d == 0 ? 20 : (d == 1 ? 9 : 0);
    const uint32_t nb = 1u << width, hi_shift = shift + width;
    for (uint32_t b = t; b < 2048; b += blockDim.x) sh.hist[b] = 0;
    __syncthreads();
    for_each([&](bool valid, uint32_t, float x) {
      const uint32_t key = mag_key(x);
      hist_add(sh.hist, (key >> shift) & (nb - 1), valid && (d == 0 || (key >> hi_shift) == prefix));
    });
    __syncthreads();
    if (CS > 1) cluster.sync();
    for (uint32_t b = t; b < 2048; b += blockDim.x) {
      uint32_t sum = 0;
      if (b < nb) {
        if (CS > 1) {
          for (uint32_t q = 0; q < CS; ++q) sum += cluster.map_shared_rank(sh.hist, q)[b];
        } else {
          sum = sh.hist[b];
        }
      }
      sh.tot[b] = sum;
    }
    __syncthreads();
    find_from_top(sh.tot, 2048, rem, sh.scratch, sh.res);
    uint32_t b = sh.res[0];
    if (b == kNone) {  // cannot happen for consistent counts; keep going safely
      set_status(a.status, SPARCML_ERR_BAD_STREAM);
      b = 0;
    } else {
      rem -= sh.res[1];
    }
    prefix = (prefix << width) | b;
    if (CS > 1) cluster.sync();  // every CTA is done reading this CTA's histogram
  }
  const uint32_t T = prefix, tie_take = rem;
  uint32_t n_gt = 0, n_eq = 0;
  for_each([&](bool valid, uint32_t, float x) {
    const uint32_t key = mag_key(x);
    n_gt += (valid && key > T) ? 1u : 0u;
    n_eq += (valid && key == T) ? 1u : 0u;
  });
  {
    uint32_t tot;
    block_excl_scan(n_gt, sh.scratch, &tot);
    __syncthreads();
    if (t == 0) sh.cnt[0] = tot;
    block_excl_scan(n_eq, sh.scratch, &tot);
    if (t == 0) sh.cnt[1] = tot;
    __syncthreads();
  }
  uint32_t gt_pre = 0, eq_pre = 0;
  if (CS > 1) {
    cluster.sync();
    for (uint32_t q = 0; q < rank; ++q) {
      const uint32_t* rc = cluster.map_shared_rank(sh.cnt, q);
      gt_pre += rc[0];
      eq_pre += rc[1];
    }
    cluster.sync();  // peers may exit or reuse their shared memory after this
  }
  const uint64_t out0 = (uint64_t)p * a.cap + r.out0;
  uint32_t run_gt = gt_pre, run_eq = eq_pre;
  for_each([&](bool valid, uint32_t i, float x) {
    const uint32_t key = mag_key(x);
    const bool gt = valid && key > T;
    const bool eq = valid && key == T;
    uint32_t tot;
    const uint32_t ex = block_excl_scan((gt ? 1u : 0u) | (eq ? 0x10000u : 0u), sh.scratch, &tot);
    const uint32_t e_gt = run_gt + (ex & 0xffffu), e_eq = run_eq + (ex >> 16);
    if (gt || (eq && e_eq < tie_take)) {
      const uint32_t pos = e_gt + min(e_eq, tie_take);
      if (pos < k) {
        a.out_idx[out0 + pos] = i;
        a.out_val[out0 + pos] = x;
        rp[i] = 0.0f;
      } else {
        set_status(a.status, SPARCML_ERR_BAD_STREAM);
      }
    }
    run_gt += tot & 0xffffu;
    run_eq += tot >> 16;
    __syncthreads();
  });
}

// mode 0: the layer-sized segments on the to-do list, one CTA each (grid-
// stride); mode 1: the long segments in fallback mode, one cluster each.
__global__ void __launch_bounds__(kRawThreads) topk_select_raw_kernel(Args a, int mode) {
  griddep_wait();
  __shared__ RawShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  if (mode == 0) {
    const uint32_t n_todo = *a.todo_cnt;
    for (uint32_t i = blockIdx.x; i < n_todo; i += gridDim.x) {
      const uint32_t gs = a.todo[i];
      select_raw(a, sh, cluster, gs / a.nseg, gs % a.nseg, 0, 1);
      __syncthreads();
    }
    return;
  }
  const uint32_t CS = cluster.num_blocks();
  const uint32_t pl = blockIdx.x / CS;
  const uint32_t p = pl / a.nlong, ls = pl % a.nlong;
  if (a.lsel[pl].mode != kModeFallback) return;  // uniform over the cluster
  select_raw(a, sh, cluster, p, a.long_list[ls], cluster.block_rank(), CS);
}

// ---------------------------------------------------------------------------
// Host side: the plan of one call.
// ---------------------------------------------------------------------------
// Rank of the guess in a sample of S of a segment's n entries with k kept:
// r = ceil(lambda + 4 sqrt(lambda) + 8) with lambda = k S / n, the expected
// number of sampled keys among the top k plus four standard deviations and a
// margin, so the r-th largest sample key is very likely at or below the k-th
// key of the segment.
uint32_t sample_rank(uint32_t k, uint32_t n, uint32_t S) {
  if (n == 0) return 0;
  const double lam = (double)k * (double)S / (double)n;
  const double rr = std::ceil(lam + 4.0 * std::sqrt(lam) + 8.0);
  return rr >= (double)S ? S : (uint32_t)rr;
}

// Rank of the histogram's upper anchor: half of the sample count that is
// very likely still above the k-th key, at least 1.
uint32_t anchor_rank(uint32_t k, uint32_t n, uint32_t S) {
  const double lam = (double)k * (double)S / (double)n;
  const double lo = lam - 4.0 * std::sqrt(lam) - 8.0;
  return lo >= 2.0 ? (uint32_t)(lo / 2.0) : 1u;
}

struct Plan {
  int32_t P;
  uint64_t N;
  uint32_t nseg, nchunk, nlong, nranges;
  uint64_t total_k, node_slots;
  std::vector<uint32_t> blob;  // records, then the lists
  size_t w_recs, w_cta, w_warp, w_short, w_long, w_rmap;  // word offsets in the blob
  uint32_t n_cta, n_warp, n_short;
  uint32_t u_L, u_m;  // equal segments (the last one possibly shorter), else 0
  // workspace byte offsets
  size_t o_blob, o_desc, o_guess, o_cnt, o_flag, o_todo, o_sub, o_cidx, o_cval, o_hist, o_lsel,
      o_bcnt, o_bnd, o_rgt, o_roff, total;
};

// Builds the plan; returns SPARCML_OK or the error of the arguments.
int make_plan(int32_t P, uint64_t N, const uint64_t* seg_begin, const uint32_t* seg_k,
              uint32_t nseg, Plan* pl) {
  if (P < 1 || P > 65535 || N < 1 || N > 0xffffffffull || !seg_begin || !seg_k || nseg < 1 ||
      seg_begin[0] != 0 || seg_begin[nseg] != N)
    return SPARCML_ERR_INVALID_ARG;
  Plan& q = *pl;
  q.P = P;
  q.N = N;
  q.nseg = nseg;
  std::vector<SegRec> recs(nseg);
  std::vector<uint32_t> cta, warp, shrt, lng, rmap;
  uint64_t chunks = 0, slots = 0, out = 0;
  for (uint32_t s = 0; s < nseg; ++s) {
    if (seg_begin[s + 1] <= seg_begin[s]) return SPARCML_ERR_INVALID_ARG;
    const uint64_t n = seg_begin[s + 1] - seg_begin[s];
    if (seg_k[s] > n) return SPARCML_ERR_INVALID_ARG;
    SegRec& r = recs[s];
    r.begin = (uint32_t)seg_begin[s];
    r.n = (uint32_t)n;
    r.k = seg_k[s];
    r.out0 = (uint32_t)out;
    out += r.k;
    if (out > 0xffffffffull) return SPARCML_ERR_CAPACITY;
    r.chunk0 = (uint32_t)chunks;
    r.nchunk = (uint32_t)((n + 3 + kChunk - 1) / kChunk);
    chunks += r.nchunk;
    r.kind = r.k == 0 ? kKeepNone : r.k == n ? kKeepAll
             : n <= kExactMax ? kExact : n <= kLayerMax ? kLayer : kLong;
    if (r.kind == kLayer &&
        (double)sample_rank(r.k, r.n, kWarpSample) * (double)n / kWarpSample > kShortExpect)
      r.kind = kLong;
    // sub-slot: about twice the density plus an eighth of a sub-chunk, at most
    // what a sub-chunk of the segment can hold; none for the trivial kinds
    uint32_t slot = 0;
    if (r.kind != kKeepNone && r.kind != kKeepAll) {
      const double want = (double)kSub * (2.0 * r.k / (double)n) + kSub / 8.0;
      const double most = (double)std::min<uint64_t>(kSub, n + 3);
      slot = (uint32_t)(std::ceil(std::min(want, most) / 32.0) * 32.0);
      slot = std::max<uint32_t>(slot, 32);
    }
    r.slot = slot;
    r.slot32 = (uint32_t)(slots / 32);
    slots += (uint64_t)r.nchunk * kWarpsPerChunk * slot;
    r.lidx = kNone;
    r.range0 = 0;
    r.rank = 0;
    if (r.kind == kExact) {
      r.rank = r.k;
      cta.push_back(s);
      shrt.push_back(s);
    } else if (r.kind == kLayer) {
      r.rank = sample_rank(r.k, r.n, kWarpSample);
      warp.push_back(s);
      shrt.push_back(s);
    } else if (r.kind == kLong) {
      // both ranks in 16 bits: a rank of the whole sample becomes the one below
      // it (a guess slightly higher; too few candidates send the segment to the
      // raw select)
      r.rank = std::min<uint32_t>(sample_rank(r.k, r.n, kLongSample), 0xffffu) |
               (std::min<uint32_t>(anchor_rank(r.k, r.n, kLongSample), 0xffffu) << 16);
      r.lidx = (uint32_t)lng.size();
      r.range0 = (uint32_t)rmap.size();
      const uint32_t nr = (r.nchunk * kWarpsPerChunk + kRangeSubs - 1) / kRangeSubs;
      if (nr > kMaxRanges || r.lidx > 0xffffu) return SPARCML_ERR_INVALID_ARG;
      for (uint32_t i = 0; i < nr; ++i) rmap.push_back((r.lidx << 16) | i);
      lng.push_back(s);
    }
  }
  if (chunks > 0xffffffffull || (uint64_t)P * chunks > 0x7fffffffull ||
      (uint64_t)P * nseg > 0x7fffffffull || slots / 32 > 0xffffffffull ||
      (uint64_t)P * rmap.size() > 0x7fffffffull)
    return SPARCML_ERR_INVALID_ARG;
  q.nchunk = (uint32_t)chunks;
  q.node_slots = slots;
  q.u_L = q.u_m = 0;
  {
    bool eq = true;
    for (uint32_t s = 1; s + 1 < nseg && eq; ++s) eq = recs[s].n == recs[0].n;
    if (eq && recs[nseg - 1].n <= recs[0].n) {
      q.u_L = recs[0].n;
      q.u_m = recs[0].nchunk;
    }
  }
  q.total_k = out;
  q.nlong = (uint32_t)lng.size();
  q.nranges = (uint32_t)rmap.size();
  q.n_cta = (uint32_t)cta.size();
  q.n_warp = (uint32_t)warp.size();
  q.n_short = (uint32_t)shrt.size();
  // the blob: records then lists, each list 4-word aligned
  auto pad4 = [](size_t w) { return (w + 3) / 4 * 4; };
  q.w_recs = 0;
  q.w_cta = pad4(q.w_recs + (size_t)nseg * 12);
  q.w_warp = pad4(q.w_cta + cta.size());
  q.w_short = pad4(q.w_warp + warp.size());
  q.w_long = pad4(q.w_short + shrt.size());
  q.w_rmap = pad4(q.w_long + lng.size());
  q.blob.assign(pad4(q.w_rmap + rmap.size()), 0u);
  std::copy(reinterpret_cast<const uint32_t*>(recs.data()),
            reinterpret_cast<const uint32_t*>(recs.data()) + (size_t)nseg * 12, q.blob.begin());
  std::copy(cta.begin(), cta.end(), q.blob.begin() + q.w_cta);
  std::copy(warp.begin(), warp.end(), q.blob.begin() + q.w_warp);
  std::copy(shrt.begin(), shrt.end(), q.blob.begin() + q.w_short);
  std::copy(lng.begin(), lng.end(), q.blob.begin() + q.w_long);
  std::copy(rmap.begin(), rmap.end(), q.blob.begin() + q.w_rmap);
  // workspace layout
  const uint64_t pseg = (uint64_t)P * nseg, psub = (uint64_t)P * chunks * kWarpsPerChunk;
  const uint64_t plong = (uint64_t)P * q.nlong, prng = (uint64_t)P * q.nranges;
  size_t o = 256;  // status word, fault-injection word, to-do counter
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  q.o_blob = take(4 * q.blob.size());
  q.o_desc = take(sizeof(ChunkDesc) * (size_t)chunks);
  q.o_guess = take(8 * pseg);
  q.o_cnt = take(4 * pseg);
  q.o_flag = take(4 * pseg);
  q.o_todo = take(4 * pseg);
  q.o_sub = take(4 * psub);
  q.o_cidx = take(4 * (uint64_t)P * slots);
  q.o_cval = take(4 * (uint64_t)P * slots);
  q.o_hist = take(4 * plong * kBins);
  q.o_lsel = take(sizeof(LongSel) * plong);
  q.o_bcnt = take(4 * plong);
  q.o_bnd = take(8 * plong * kBoundCap);
  q.o_rgt = take(4 * prng);
  q.o_roff = take(4 * prng);
  q.total = o;
  return SPARCML_OK;
}

int launch_topk(const Plan& q, const float* grad, float* residual, uint32_t* out_idx,
                float* out_val, uint32_t* out_nnz, uint64_t cap, void* ws, size_t ws_bytes,
                cudaStream_t s, void* const* events) {
  char* w = static_cast<char*>(ws);
  auto mark = [&](int i) {
    if (events && events[i]) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
  };
  Args a = {};
  a.grad = grad;
  a.residual = residual;
  a.out_idx = out_idx;
  a.out_val = out_val;
  a.out_nnz = out_nnz;
  a.status = reinterpret_cast<int32_t*>(w);
  a.N = q.N;
  a.cap = cap;
  a.node_slots = q.node_slots;
  a.P = q.P;
  a.nseg = q.nseg;
  a.nchunk = q.nchunk;
  a.nlong = q.nlong;
  a.nranges = q.nranges;
  a.total_k = (uint32_t)q.total_k;
  a.vec = ((reinterpret_cast<uintptr_t>(grad) | reinterpret_cast<uintptr_t>(residual)) & 15) == 0;
  a.u_L = q.u_L;
  a.u_m = q.u_m;
  uint32_t* blob = reinterpret_cast<uint32_t*>(w + q.o_blob);
  a.recs = reinterpret_cast<const SegRec*>(blob + q.w_recs);
  a.cta_list = blob + q.w_cta;
  a.warp_list = blob + q.w_warp;
  a.short_list = blob + q.w_short;
  a.long_list = blob + q.w_long;
  a.range_map = blob + q.w_rmap;
  a.desc = reinterpret_cast<ChunkDesc*>(w + q.o_desc);
  a.guess = reinterpret_cast<uint2*>(w + q.o_guess);
  a.seg_cnt = reinterpret_cast<uint32_t*>(w + q.o_cnt);
  a.seg_flag = reinterpret_cast<uint32_t*>(w + q.o_flag);
  a.todo = reinterpret_cast<uint32_t*>(w + q.o_todo);
  a.todo_cnt = reinterpret_cast<uint32_t*>(w + 64);
  a.fallbacks = reinterpret_cast<uint32_t*>(w + kFallbackOffset);
  a.sub_cnt = reinterpret_cast<uint32_t*>(w + q.o_sub);
  a.cand_idx = reinterpret_cast<uint32_t*>(w + q.o_cidx);
  a.cand_val = reinterpret_cast<float*>(w + q.o_cval);
  a.hist = reinterpret_cast<uint32_t*>(w + q.o_hist);
  a.lsel = reinterpret_cast<LongSel*>(w + q.o_lsel);
  a.bnd_cnt = reinterpret_cast<uint32_t*>(w + q.o_bcnt);
  a.bnd = reinterpret_cast<uint2*>(w + q.o_bnd);
  a.range_gt = reinterpret_cast<uint32_t*>(w + q.o_rgt);
  a.range_off = reinterpret_cast<uint32_t*>(w + q.o_roff);
  uint64_t launches = 0;

  mark(0);
  // the plan's records and lists travel as kernel parameters
  for (size_t i = 0; i < q.blob.size(); i += kUploadWords) {
    UploadBatch b;
    b.count = (uint32_t)std::min<size_t>(kUploadWords, q.blob.size() - i);
    b.dst = blob + i;
    std::copy(q.blob.begin() + i, q.blob.begin() + i + b.count, b.words);
    topk_upload_kernel<<<1, 256, 0, s>>>(b);
    ++launches;
  }
  {
    const uint64_t items = q.nchunk + (uint64_t)q.P * q.nseg + (uint64_t)q.P * q.nlong * (kBins + 1) +
                           (uint64_t)q.P;
    launch_pdl(topk_init_kernel, (unsigned)std::min<uint64_t>((items + 255) / 256, 4 * 152), 256, 0, s, a);
    ++launches;
  }
  if (q.n_cta) {
    launch_pdl(topk_guess_cta_kernel, (unsigned)((uint64_t)q.P * q.n_cta), kGuessThreads, 0, s,
        a, q.n_cta);
    ++launches;
  }
  if (q.nlong) {  // a cluster of kGuessCluster CTAs per (node, long segment)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((uint64_t)q.P * q.nlong * kGuessCluster), 1, 1);
    cfg.blockDim = dim3(kGuessThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kGuessCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, topk_guess_long_kernel, a) != cudaSuccess)
      return SPARCML_ERR_CUDA;
    ++launches;
  }
  if (q.n_warp) {
    const uint64_t warps = (uint64_t)q.P * q.n_warp, wpc = kGuessThreads / 32;
    launch_pdl(topk_guess_warp_kernel, (unsigned)((warps + wpc - 1) / wpc), kGuessThreads, 0, s, a, q.n_warp);
    ++launches;
  }
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  mark(1);
  {
    const unsigned grid = (unsigned)((uint64_t)q.P * q.nchunk);
    // (the compiler drops the long-segment path from tables without one)
    if (q.u_L && q.nlong)
      launch_pdl(topk_stream_kernel<true, true>, grid, kStreamThreads, 0, s, a);
    else if (q.u_L)
      launch_pdl(topk_stream_kernel<true, false>, grid, kStreamThreads, 0, s, a);
    else if (q.nlong)
      launch_pdl(topk_stream_kernel<false, true>, grid, kStreamThreads, 0, s, a);
    else
      launch_pdl(topk_stream_kernel<false, false>, grid, kStreamThreads, 0, s, a);
    ++launches;
  }
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  mark(2);
  if (q.n_short) {
    launch_pdl(topk_select_short_kernel, (unsigned)((uint64_t)q.P * q.n_short), kSegThreads, 0, s,
        a, q.n_short);
    launch_pdl(topk_select_raw_kernel, (unsigned)std::min<uint64_t>((uint64_t)q.P * q.n_short, 2 * 152),
                             kRawThreads, 0, s, a, 0);
    launches += 2;
    if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  }
  if (q.nlong) {
    const unsigned pl = (unsigned)((uint64_t)q.P * q.nlong);
    const unsigned pr = (unsigned)((uint64_t)q.P * q.nranges);
    launch_pdl(long_hist_kernel, pr, 256, 0, s, a);
    launch_pdl(long_find_kernel, pl, 256, 0, s, a);
    launch_pdl(long_collect_kernel, pr, 256, 0, s, a);
    const size_t smem = (2 * (size_t)kBoundCap + kMaxRanges + 2048) * sizeof(uint32_t);
    if (!ensure_smem(reinterpret_cast<const void*>(long_exact_kernel), smem))
      return SPARCML_ERR_CUDA;
    launch_pdl(long_exact_kernel, pl, kExactThreads, smem, s, a);
    launch_pdl(long_write_kernel, pr, 256, 0, s, a);
    launch_pdl(long_restore_kernel, pr, 256, 0, s, a);
    launches += 6;
    if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl * kRawCluster, 1, 1);
    cfg.blockDim = dim3(kRawThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kRawCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, topk_select_raw_kernel, a, 1) != cudaSuccess)
      return SPARCML_ERR_CUDA;
    ++launches;
  }
  mark(3);
  note_launches(launches);
  return SPARCML_OK;
}

int topk_call(const float* grad, float* residual, int32_t P, uint64_t N, const uint64_t* seg_begin,
              const uint32_t* seg_k, uint32_t nseg, uint32_t* out_idx, float* out_val,
              uint32_t* out_nnz, uint64_t cap, void* ws, size_t ws_bytes, void* stream,
              void* const* events) {
  if (!grad || !residual || !out_idx || !out_val || !out_nnz || !ws) return SPARCML_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return SPARCML_ERR_INVALID_ARG;
  Plan q;
  const int st = make_plan(P, N, seg_begin, seg_k, nseg, &q);
  if (st != SPARCML_OK) return st;
  if (ws_bytes < q.total) return SPARCML_ERR_WORKSPACE;
  if (q.total_k > cap) return SPARCML_ERR_CAPACITY;
  return launch_topk(q, grad, residual, out_idx, out_val, out_nnz, cap, ws, ws_bytes,
                     static_cast<cudaStream_t>(stream), events);
}

// The equal-segment table: segment s = [s L, min((s + 1) L, N)), k_s =
// floor(n_s k_num / k_den) (the last segment takes the remainder).
bool uniform_table(uint64_t N, uint64_t seg_len, uint32_t k_num, uint32_t k_den,
                   std::vector<uint64_t>* begin, std::vector<uint32_t>* ks) {
  if (N < 1 || N > 0xffffffffull || seg_len < 1 || k_den < 1 || k_num > k_den) return false;
  const uint64_t L = std::min<uint64_t>(seg_len, N);
  begin->clear();
  ks->clear();
  for (uint64_t b = 0; b < N; b += L) {
    begin->push_back(b);
    ks->push_back((uint32_t)(std::min<uint64_t>(L, N - b) * k_num / k_den));
  }
  begin->push_back(N);
  return true;
}

}  // namespace
}  // namespace sparcml

using namespace sparcml;

extern "C" uint32_t sparcml_topk_uniform_segments(uint64_t N, uint64_t seg_len, uint32_t k_num,
                                                  uint32_t k_den, uint64_t* seg_begin,
                                                  uint32_t* seg_k) {
  std::vector<uint64_t> b;
  std::vector<uint32_t> k;
  if (!uniform_table(N, seg_len, k_num, k_den, &b, &k) || k.size() > 0xffffffffull) return 0;
  if (seg_begin) std::copy(b.begin(), b.end(), seg_begin);
  if (seg_k) std::copy(k.begin(), k.end(), seg_k);
  return (uint32_t)k.size();
}

extern "C" uint64_t sparcml_topk_total_k(const uint32_t* seg_k, uint32_t nseg) {
  uint64_t t = 0;
  if (seg_k)
    for (uint32_t s = 0; s < nseg; ++s) t += seg_k[s];
  return t;
}

extern "C" size_t sparcml_topk_ef_workspace_size(int32_t P, uint64_t N, const uint64_t* seg_begin,
                                                 const uint32_t* seg_k, uint32_t nseg) {
  Plan q;
  if (make_plan(P, N, seg_begin, seg_k, nseg, &q) != SPARCML_OK) return 0;
  return q.total;
}

extern "C" int sparcml_topk_ef_traced(const float* grad, float* residual, int32_t P, uint64_t N,
                                      const uint64_t* seg_begin, const uint32_t* seg_k,
                                      uint32_t nseg, uint32_t* out_idx, float* out_val,
                                      uint32_t* out_nnz, uint64_t cap, void* ws, size_t ws_bytes,
                                      void* stream, void* const* events) {
  const ApiRange nvtx_range(__func__);
  return topk_call(grad, residual, P, N, seg_begin, seg_k, nseg, out_idx, out_val, out_nnz, cap,
                   ws, ws_bytes, stream, events);
}

extern "C" int sparcml_topk_ef(const float* grad, float* residual, int32_t P, uint64_t N,
                               const uint64_t* seg_begin, const uint32_t* seg_k, uint32_t nseg,
                               uint32_t* out_idx, float* out_val, uint32_t* out_nnz, uint64_t cap,
                               void* ws, size_t ws_bytes, void* stream) {
  return topk_call(grad, residual, P, N, seg_begin, seg_k, nseg, out_idx, out_val, out_nnz, cap,
                   ws, ws_bytes, stream, nullptr);
}

extern "C" size_t sparcml_topk_ef_uniform_workspace_size(int32_t P, uint64_t N, uint64_t seg_len,
                                                         uint32_t k_num, uint32_t k_den) {
  std::vector<uint64_t> b;
  std::vector<uint32_t> k;
  if (!uniform_table(N, seg_len, k_num, k_den, &b, &k) || k.size() > 0xffffffffull) return 0;
  return sparcml_topk_ef_workspace_size(P, N, b.data(), k.data(), (uint32_t)k.size());
}

extern "C" int sparcml_topk_ef_uniform_traced(const float* grad, float* residual, int32_t P,
                                              uint64_t N, uint64_t seg_len, uint32_t k_num,
                                              uint32_t k_den, uint32_t* out_idx, float* out_val,
                                              uint32_t* out_nnz, uint64_t cap, void* ws,
                                              size_t ws_bytes, void* stream,
                                              void* const* events) {
  const ApiRange nvtx_range(__func__);
  std::vector<uint64_t> b;
  std::vector<uint32_t> k;
  if (!uniform_table(N, seg_len, k_num, k_den, &b, &k) || k.size() > 0xffffffffull)
    return SPARCML_ERR_INVALID_ARG;
  return topk_call(grad, residual, P, N, b.data(), k.data(), (uint32_t)k.size(), out_idx,
                   out_val, out_nnz, cap, ws, ws_bytes, stream, events);
}

extern "C" int sparcml_topk_ef_uniform(const float* grad, float* residual, int32_t P, uint64_t N,
                                       uint64_t seg_len, uint32_t k_num, uint32_t k_den,
                                       uint32_t* out_idx, float* out_val, uint32_t* out_nnz,
                                       uint64_t cap, void* ws, size_t ws_bytes, void* stream) {
  return sparcml_topk_ef_uniform_traced(grad, residual, P, N, seg_len, k_num, k_den, out_idx,
                                        out_val, out_nnz, cap, ws, ws_bytes, stream, nullptr);
}

extern "C" int64_t sparcml_topk_ef_fallbacks(const void* ws, void* stream) {
  if (!ws) return -1;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return -1;
  uint32_t h = 0;
  if (cudaMemcpy(&h, static_cast<const char*>(ws) + kFallbackOffset, sizeof h,
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return -1;
  return h;
}
