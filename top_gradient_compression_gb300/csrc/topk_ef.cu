// Top-k selection with error feedback, fused with packing, for sm_103a.
//
// "SparCML: High-Performance Sparse Communication for Machine Learning",
// §2.2 (Top-k SGD: each node sends its k largest-magnitude components and
// accumulates the rest for the next iteration), §4 (residual error), §5.1
// (sparse streams of index-value pairs), §8.4 (layer-wise sparsification,
// here: segments), App. A (the last part takes the remainder).
//
// Exact selection in three launches, all stream-ordered:
//
//  1. guess  (one CTA per segment). Computes acc = residual + grad on a
//     sample of the segment (all of it when it is short, else 256 runs of
//     32 consecutive entries) and picks a key G low enough that, with
//     overwhelming probability, at least k_s entries of the whole segment
//     have |acc| key >= G. For a fully sampled segment G <= the exact k-th
//     key, so coverage is certain.
//
//  2. stream (one CTA per 8192-entry chunk, the HBM-bound pass). Reads grad
//     and residual once with 128-bit loads, writes acc back into residual
//     with 128-bit stores, and compacts the chunk's candidates (key >= G)
//     into a per-chunk slot in index order (warp ballots). Counts go to the
//     chunk and to its segment.
//
//  3. select (one thread-block cluster per segment). If the candidates do
//     not cover k_s (or a chunk slot overflowed) the cluster falls back to
//     reading the segment's acc directly; the answer is the same either
//     way. A three-digit radix select over the candidates, with the
//     histograms summed through distributed shared memory, gives the exact
//     k-th key T and how many entries equal to T to keep (lowest indices
//     first). An ordered compaction then writes the kept entries ascending
//     and sets residual = +0.0f at each of them.
//
// Only the stream pass touches all of grad and residual: 12 bytes per
// entry plus a few percent for candidates.

#include <cooperative_groups.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace sparcml {
namespace {

constexpr uint32_t kChunk = 8192;         // entries per stream-pass CTA
constexpr uint32_t kStreamThreads = 256;  // 8 warps x 1024 entries
constexpr uint32_t kWarpsPerChunk = kStreamThreads / 32;
constexpr uint32_t kSub = kChunk / kWarpsPerChunk;            // entries per warp: 1,024
constexpr uint32_t kRounds = kSub / (32 * 4);                  // float4 rounds per warp
constexpr uint32_t kSampleMax = 8192;     // sample of a long segment
constexpr uint32_t kSampleShort = 4096;   // sample of a layer-sized segment
constexpr uint32_t kShortSegment = 1u << 18;
constexpr uint32_t kRun = 256;  // consecutive entries per sample run (1 KB per array)
constexpr uint32_t kGuessThreads = 256;
constexpr uint32_t kSelectThreads = 256;
constexpr uint32_t kSmallCands = 4096;  // candidates a select CTA keeps in shared memory
constexpr uint32_t kWin = 1024;  // chunks per window in the select pass
constexpr uint32_t kNone = 0xffffffffu;

struct Geo {
  uint64_t N;        // entries per node
  uint64_t cap;      // stream capacity per node
  uint32_t L;        // segment length (last segment may be shorter)
  uint32_t L_last;
  uint32_t nseg;     // segments per node
  uint32_t m;        // chunks per full segment
  uint32_t m_last;   // chunks in the last segment
  uint32_t nchunk;   // chunks per node
  uint32_t k_full;   // k of a full segment
  uint32_t k_last;   // k of the last segment
  uint32_t slot;     // candidate slot capacity per warp sub-chunk
  int32_t P;
  // rank r of the guess in a sample (see sample_rank), per segment kind:
  // the warp guess's sample and the CTA guess's sample
  uint32_t r_warp_full, r_warp_last, r_cta_full, r_cta_last;
};

__device__ __forceinline__ uint32_t seg_n(const Geo& g, uint32_t s) {
  return s == g.nseg - 1 ? g.L_last : g.L;
}
__device__ __forceinline__ uint32_t seg_k(const Geo& g, uint32_t s) {
  return s == g.nseg - 1 ? g.k_last : g.k_full;
}
__device__ __forceinline__ uint32_t seg_chunks(const Geo& g, uint32_t s) {
  return s == g.nseg - 1 ? g.m_last : g.m;
}
// Node-local chunk c -> segment s, chunk j inside it.
__device__ __forceinline__ void chunk_pos(const Geo& g, uint32_t c, uint32_t* s, uint32_t* j) {
  const uint32_t full = (g.nseg - 1) * g.m;
  if (c >= full) {
    *s = g.nseg - 1;
    *j = c - full;
  } else {
    *s = c / g.m;
    *j = c % g.m;
  }
}

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
// 1. guess: one CTA per (node, segment). The sample keys stay in registers
// (KPT per thread); G = the r-th largest sample key with its low 15 bits
// cleared, found bit by bit (16 block-wide counts, no histogram).
// ---------------------------------------------------------------------------
template <uint32_t KPT>
__global__ void __launch_bounds__(kGuessThreads)
topk_guess_kernel(const float* __restrict__ grad, const float* __restrict__ residual, Geo g,
                  uint32_t* __restrict__ guess, uint32_t* __restrict__ seg_cnt,
                  uint32_t* __restrict__ seg_flag, uint32_t* __restrict__ out_nnz,
                  uint32_t total_k, uint32_t* __restrict__ todo_cnt) {
  constexpr uint32_t kWarps = kGuessThreads / 32;
  __shared__ uint32_t wsum[2][kWarps];

  const uint32_t gs = blockIdx.x;
  const uint32_t p = gs / g.nseg, s = gs % g.nseg;
  const uint32_t n = seg_n(g, s), k = seg_k(g, s);
  const uint32_t t = threadIdx.x, lane = lane_id(), warp = t >> 5;
  if (t == 0) {
    if (gs == 0) *todo_cnt = 0;
    seg_cnt[gs] = 0;
    seg_flag[gs] = 0;
    if (s == 0) out_nnz[p] = total_k;
  }
  if (k == 0) {
    if (t == 0) guess[gs] = kNone;  // no key reaches it: no candidates
    return;
  }
  if (k >= n) {
    if (t == 0) guess[gs] = 0;  // everything is kept
    return;
  }
  const uint64_t base = (uint64_t)p * g.N + (uint64_t)s * g.L;
  const float* gp = grad + base;
  const float* rp = residual + base;

  // Sample: all of a segment of at most kSampleMax entries; else runs of kRun
  // consecutive entries (1 KB per array: whole DRAM bursts), fewer for
  // layer-sized segments whose candidate sets are small anyway.
  const bool exact = n <= kSampleMax;
  const uint32_t S = exact ? n : (n <= kShortSegment ? kSampleShort : kSampleMax);
  const uint32_t r = exact ? k : (s == g.nseg - 1 ? g.r_cta_last : g.r_cta_full);
  // All sample loads are issued before any is used.
  uint32_t pos[KPT];
  bool ok[KPT];
  if (exact) {
#pragma unroll
    for (uint32_t q = 0; q < KPT; ++q) {
      pos[q] = t + q * kGuessThreads;
      ok[q] = pos[q] < S;
    }
  } else {
    // Runs of kRun consecutive entries spread evenly over the segment; warp w
    // reads runs w * (KPT / kLinesPerRun) + ..., each as kRun / 32 coalesced
    // 128-byte lines per array.
    const uint32_t nruns = S / kRun;
    constexpr uint32_t kLinesPerRun = kRun / 32;
#pragma unroll
    for (uint32_t q = 0; q < KPT; q += kLinesPerRun) {
      const uint32_t run = warp * (KPT / kLinesPerRun) + q / kLinesPerRun;
      const uint32_t st =
          run < nruns
              ? (uint32_t)(((uint64_t)run * (n - kRun) / (nruns - 1)) & ~(uint64_t)(kRun - 1))
              : 0u;
#pragma unroll
      for (uint32_t l = 0; l < kLinesPerRun; ++l) {
        pos[q + l] = st + l * 32 + lane;
        ok[q + l] = run < nruns;
      }
    }
  }
  float ra[KPT], ga[KPT];
#pragma unroll
  for (uint32_t q = 0; q < KPT; ++q) {
    ra[q] = ok[q] ? rp[pos[q]] : 0.0f;
    ga[q] = ok[q] ? gp[pos[q]] : 0.0f;
  }
  uint32_t key[KPT];
#pragma unroll
  for (uint32_t q = 0; q < KPT; ++q) key[q] = ok[q] ? mag_key(__fadd_rn(ra[q], ga[q])) : kNone;
  // Bitwise radix select on the 2^15 grid: the largest G with at least r
  // sample keys >= G, i.e. the r-th largest key with its low 15 bits cleared.
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
    __syncthreads();
    uint32_t tot = 0;
#pragma unroll
    for (uint32_t w = 0; w < kWarps; ++w) tot += ws[w];
    if (tot >= r) G = trial;
  }
  const uint32_t prefix = G >> 15;
  if (t == 0) guess[gs] = prefix << 15;
}

// Layer-sized segments (kSampleMax < n <= kShortSegment): one warp per
// segment, no block barrier. The 2,048-entry sample (8 runs of kRun) sits in
// registers, 64 keys per lane; G is the same function of the sample as in
// topk_guess_kernel (the r-th largest key with its low 15 bits cleared).
constexpr uint32_t kWarpSample = 2048;
constexpr uint32_t kWarpKeys = kWarpSample / 32;

__global__ void __launch_bounds__(kGuessThreads)
topk_guess_warp_kernel(const float* __restrict__ grad, const float* __restrict__ residual, Geo g,
                       uint32_t* __restrict__ guess, uint32_t* __restrict__ seg_cnt,
                       uint32_t* __restrict__ seg_flag, uint32_t* __restrict__ out_nnz,
                       uint32_t total_k, uint32_t* __restrict__ todo_cnt) {
  const uint32_t lane = lane_id();
  const uint32_t gs = blockIdx.x * (kGuessThreads / 32) + (threadIdx.x >> 5);
  if (gs >= (uint32_t)g.P * g.nseg) return;  // warp-uniform
  const uint32_t p = gs / g.nseg, s = gs % g.nseg;
  const uint32_t n = seg_n(g, s), k = seg_k(g, s);
  if (lane == 0) {
    if (gs == 0) *todo_cnt = 0;
    seg_cnt[gs] = 0;
    seg_flag[gs] = 0;
    if (s == 0) out_nnz[p] = total_k;
  }
  if (k == 0 || k >= n) {
    if (lane == 0) guess[gs] = k == 0 ? kNone : 0u;
    return;
  }
  const uint64_t base = (uint64_t)p * g.N + (uint64_t)s * g.L;
  const float* gp = grad + base;
  const float* rp = residual + base;
  constexpr uint32_t nruns = kWarpSample / kRun, kLines = kRun / 32, kBatchRuns = 2;
  const uint32_t r = s == g.nseg - 1 ? g.r_warp_last : g.r_warp_full;
  uint32_t key[kWarpKeys];
  // run start (n <= kShortSegment, so run * (n - kRun) fits in 32 bits)
  auto run_at = [&](uint32_t run) { return (run * (n - kRun) / (nruns - 1)) & ~(kRun - 1); };
  if (((reinterpret_cast<uintptr_t>(gp) | reinterpret_cast<uintptr_t>(rp)) & 15) == 0) {
    // 16-byte aligned segment: a run is 64 float4, two per lane; four runs'
    // loads (16 of them) in flight at once
    constexpr uint32_t kVecRuns = 4, kVecPer = kRun / 128;  // float4 per lane per run
#pragma unroll
    for (uint32_t r0 = 0; r0 < nruns; r0 += kVecRuns) {
      float4 a[kVecRuns * kVecPer], b[kVecRuns * kVecPer];
#pragma unroll
      for (uint32_t q = 0; q < kVecRuns * kVecPer; ++q) {
        const uint32_t i = run_at(r0 + q / kVecPer) + ((q % kVecPer) * 32 + lane) * 4;
        a[q] = *reinterpret_cast<const float4*>(rp + i);
        b[q] = *reinterpret_cast<const float4*>(gp + i);
      }
#pragma unroll
      for (uint32_t q = 0; q < kVecRuns * kVecPer; ++q) {
        uint32_t* kq = key + (r0 * kVecPer + q) * 4;
        kq[0] = mag_key(__fadd_rn(a[q].x, b[q].x));
        kq[1] = mag_key(__fadd_rn(a[q].y, b[q].y));
        kq[2] = mag_key(__fadd_rn(a[q].z, b[q].z));
        kq[3] = mag_key(__fadd_rn(a[q].w, b[q].w));
      }
    }
  } else {
#pragma unroll
    for (uint32_t r0 = 0; r0 < nruns; r0 += kBatchRuns) {
      float a[kBatchRuns * kLines], b[kBatchRuns * kLines];
#pragma unroll
      for (uint32_t q = 0; q < kBatchRuns * kLines; ++q) {
        const uint32_t i = run_at(r0 + q / kLines) + (q % kLines) * 32 + lane;
        a[q] = rp[i];
        b[q] = gp[i];
      }
#pragma unroll
      for (uint32_t q = 0; q < kBatchRuns * kLines; ++q)
        key[r0 * kLines + q] = mag_key(__fadd_rn(a[q], b[q]));
    }
  }
  uint32_t G = 0;
#pragma unroll 1
  for (int bit = 30; bit >= 15; --bit) {
    const uint32_t trial = G | (1u << bit);
    uint32_t c = 0;
#pragma unroll
    for (uint32_t q = 0; q < kWarpKeys; ++q) c += key[q] >= trial ? 1u : 0u;
    if (warp_sum(c) >= r) G = trial;
  }
  if (lane == 0) guess[gs] = G;
}

// ---------------------------------------------------------------------------
// 2. stream: one CTA per chunk of kChunk entries (a chunk never crosses a
// segment boundary). Warp w owns the contiguous sub-chunk of kSub entries
// [start + kSub w, start + kSub (w + 1)), read as kRounds rounds of 32 float4,
// and compacts its candidates in index order straight from registers into its
// own sub-slot: no barrier, no second read.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kStreamThreads)
topk_stream_kernel(const float* __restrict__ grad, float* __restrict__ residual, Geo g,
                   const uint32_t* __restrict__ guess, uint32_t* __restrict__ seg_cnt,
                   uint32_t* __restrict__ seg_flag, uint32_t* __restrict__ sub_cnt,
                   uint32_t* __restrict__ cand_idx, float* __restrict__ cand_val) {
  const uint32_t gc = blockIdx.x;
  const uint32_t p = gc / g.nchunk, c = gc % g.nchunk;
  uint32_t s, j;
  chunk_pos(g, c, &s, &j);
  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  const uint32_t seg_start = s * g.L;
  const uint64_t start64 = (uint64_t)seg_start + (uint64_t)j * kChunk + warp * kSub;
  const uint64_t seg_end = (uint64_t)seg_start + seg_n(g, s);
  const uint32_t nn = start64 < seg_end ? (uint32_t)min((uint64_t)kSub, seg_end - start64) : 0u;
  const uint32_t start = nn ? (uint32_t)start64 : 0u;  // this warp's first entry
  const uint32_t G = guess[p * g.nseg + s];
  const float* gp = grad + (uint64_t)p * g.N + start;
  float* rp = residual + (uint64_t)p * g.N + start;
  const bool aligned =
      ((reinterpret_cast<uintptr_t>(gp) | reinterpret_cast<uintptr_t>(rp)) & 15) == 0;

  float4 gv[kRounds], rv[kRounds];
#pragma unroll
  for (uint32_t t = 0; t < kRounds; ++t) {
    const uint32_t e0 = 4 * (t * 32 + lane);  // sub-chunk local
    if (aligned && e0 + 4 <= nn) {
      gv[t] = __ldcs(reinterpret_cast<const float4*>(gp + e0));
      rv[t] = *reinterpret_cast<const float4*>(rp + e0);
    } else {
      float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q)
        if (e0 + q < nn) {
          a[q] = gp[e0 + q];
          b[q] = rp[e0 + q];
        }
      gv[t] = make_float4(a[0], a[1], a[2], a[3]);
      rv[t] = make_float4(b[0], b[1], b[2], b[3]);
    }
  }
  const uint64_t sub = (uint64_t)gc * kWarpsPerChunk + warp;
  const uint64_t slot0 = sub * g.slot;
  uint32_t run = 0;  // candidates so far in this sub-chunk (warp-uniform)
#pragma unroll
  for (uint32_t t = 0; t < kRounds; ++t) {
    const uint32_t e0 = 4 * (t * 32 + lane);
    float4 a;
    a.x = __fadd_rn(rv[t].x, gv[t].x);
    a.y = __fadd_rn(rv[t].y, gv[t].y);
    a.z = __fadd_rn(rv[t].z, gv[t].z);
    a.w = __fadd_rn(rv[t].w, gv[t].w);
    const float av[4] = {a.x, a.y, a.z, a.w};
    uint32_t bits = 0;
    if (aligned && e0 + 4 <= nn) {
      *reinterpret_cast<float4*>(rp + e0) = a;
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) bits |= (mag_key(av[q]) >= G ? 1u : 0u) << q;
    } else {
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q)
        if (e0 + q < nn) {
          rp[e0 + q] = av[q];
          bits |= (mag_key(av[q]) >= G ? 1u : 0u) << q;
        }
    }
    if (__ballot_sync(0xffffffffu, bits) == 0) continue;  // warp-uniform
    uint32_t tot;
    uint32_t pos = run + warp_excl_small(__popc(bits), &tot);
    run += tot;
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q)
      if (bits & (1u << q)) {
        if (pos < g.slot) {
          const uint64_t keep = l2_policy_evict_last();
          st_keep(cand_idx + slot0 + pos, start + e0 + q, keep);
          st_keep(cand_val + slot0 + pos, av[q], keep);
        }
        ++pos;
      }
  }
  if (lane == 0) {
    sub_cnt[sub] = run;
    if (run) atomicAdd(&seg_cnt[p * g.nseg + s], run);
    if (run > g.slot) atomicOr(&seg_flag[p * g.nseg + s], 1u);
  }
}

// ---------------------------------------------------------------------------
// 3. select: one cluster of CS CTAs per (node, segment). CTA r of the
// cluster owns chunks [ms*r/CS, ms*(r+1)/CS) of the segment.
// ---------------------------------------------------------------------------
struct SelectArgs {
  uint32_t CS;         // CTAs per segment (a thread-block cluster when > 1)
  uint32_t warp_done;  // topk_select_short_kernel ran: only the segments in `todo` remain
  uint32_t raw_only;   // the long-segment passes ran: only fallback segments remain
  uint32_t* todo;      // segments the short kernel left to topk_select_kernel
  uint32_t* todo_cnt;
  float* residual;
  const uint32_t* seg_cnt;
  const uint32_t* seg_flag;
  const uint32_t* sub_cnt;  // candidates per warp sub-chunk
  const uint32_t* guess;    // per-segment lower bound G of the k-th key
  const uint32_t* cand_idx;
  const float* cand_val;
  uint32_t* out_idx;
  float* out_val;
  int32_t* status;
  Geo g;
};

struct SelectShared {
  uint32_t hist[2048];
  uint32_t tot[2048];
  uint32_t wpre[kWin + 1];  // prefix of sub-chunk counts of a window
  uint32_t scratch[34];
  uint32_t res[2];
  uint32_t cnt[2];  // this CTA's (> T, == T) counts, read by higher ranks
};

// Exclusive prefix of the candidate counts of nw consecutive sub-chunks into
// sh.wpre[0..nw]; returns the window total.
__device__ uint32_t load_window(SelectShared& sh, const uint32_t* cc, uint32_t nw) {
  const uint32_t per = (kWin + kSelectThreads - 1) / kSelectThreads;
  const uint32_t t = threadIdx.x;
  uint32_t v[per], sum = 0;
#pragma unroll
  for (uint32_t i = 0; i < per; ++i) {
    const uint32_t w = t * per + i;
    v[i] = w < nw ? cc[w] : 0u;
    sum += v[i];
  }
  uint32_t total;
  uint32_t ex = block_excl_scan(sum, sh.scratch, &total);
#pragma unroll
  for (uint32_t i = 0; i < per; ++i) {
    const uint32_t w = t * per + i;
    if (w < nw) sh.wpre[w] = ex;
    ex += v[i];
  }
  if (t == 0) sh.wpre[nw] = total;
  __syncthreads();
  return total;
}

// Position v of a window -> its sub-chunk (largest w with wpre[w] <= v).
__device__ __forceinline__ uint32_t window_chunk(const SelectShared& sh, uint32_t nw, uint32_t v) {
  uint32_t lo = 0, hi = nw;  // invariant: wpre[lo] <= v < wpre[hi]
  while (hi - lo > 1) {
    const uint32_t mid = (lo + hi) >> 1;
    if (sh.wpre[mid] <= v) lo = mid; else hi = mid;
  }
  return lo;
}

// Select for a layer-sized segment whose candidates were all kept in their
// sub-slots (at most kShortCands of them, over at most kShortSubs
// sub-chunks): one CTA of kSegThreads per segment (4 warps share the work of
// each phase, so a segment's chain of phases is short):
//  1. thread t copies sub-chunk t's candidates into shared memory with
//     cp.async (every copy in flight at once), at the sub-chunk's offset;
//  2. four radix digits (8, 8, 8, 7 bits) of the k-th key T, each from one
//     256-bin histogram over the shared copy (warp-aggregated adds), its
//     bins scanned from the top by warp 0;
//  3. thread t writes the kept entries of its contiguous candidate range in
//     index order at the offset given by a block scan of its counts (keys
//     > T, and keys == T up to tie_take, lowest indices first); then the
//     offsets are resolved to indices and the residual is zeroed there.
// Segments that do not qualify go to the to-do list of topk_select_kernel.
constexpr uint32_t kShortSubs = 128;
constexpr uint32_t kShortCands = 2048;
constexpr uint32_t kSegThreads = 128;  // = kShortSubs: one sub-chunk per thread in phase 1

__device__ __forceinline__ bool short_select_eligible(const SelectArgs& a, uint32_t gs, uint32_t k,
                                                      uint32_t ms) {
  return a.CS == 1 && a.seg_flag[gs] == 0 && a.seg_cnt[gs] >= k &&
         ms * kWarpsPerChunk <= kShortSubs && a.seg_cnt[gs] <= kShortCands;
}

__device__ __forceinline__ uint32_t warp_excl_sum(uint32_t v, uint32_t* total) {
  const uint32_t incl = warp_incl_sum(v);
  *total = __shfl_sync(0xffffffffu, incl, 31);
  return incl - v;
}

__global__ void __launch_bounds__(kSegThreads)
topk_select_short_kernel(SelectArgs a) {
  __shared__ uint32_t wpre[kShortSubs + 1];
  __shared__ float vals[kShortCands];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t dig[2];
  const Geo& g = a.g;
  const uint32_t t = threadIdx.x, lane = lane_id(), warp = t >> 5;
  const uint32_t gs = blockIdx.x;
  const uint32_t p = gs / g.nseg, s = gs % g.nseg;
  const uint32_t k = seg_k(g, s), ms = seg_chunks(g, s);
  if (k == 0) return;                                // CTA-uniform
  if (!short_select_eligible(a, gs, k, ms)) {        // CTA-uniform: to topk_select_kernel
    if (t == 0) a.todo[atomicAdd(a.todo_cnt, 1u)] = gs;
    return;
  }
  const uint32_t nsub = ms * kWarpsPerChunk;
  const uint64_t sub0 = ((uint64_t)p * g.nchunk + (uint64_t)s * g.m) * kWarpsPerChunk;
  const uint32_t* cidx = a.cand_idx + sub0 * g.slot;
  const float* cval = a.cand_val + sub0 * g.slot;
  // 1. offsets of the sub-chunks' candidates, then the copies
  const uint32_t c = t < nsub ? a.sub_cnt[sub0 + t] : 0u;
  uint32_t M;
  const uint32_t off = block_excl_scan(c, scratch, &M);
  if (t < nsub) wpre[t] = off;
  if (t == 0) wpre[nsub] = M;
  for (uint32_t i = 0; i < c; ++i) cp_async4(vals + off + i, cval + (uint64_t)t * g.slot + i);
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
      if (lane == 0) {
        if (!found) {
          set_status(a.status, SPARCML_ERR_BAD_STREAM);
          dig[0] = 0;
          dig[1] = rem;
        }
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
  float* rp = a.residual + (uint64_t)p * g.N;
  const uint64_t out0 = (uint64_t)p * g.cap + (uint64_t)s * g.k_full;
  uint32_t* oi = a.out_idx + out0;
  const uint64_t keep = l2_policy_evict_last();
  uint32_t w = 0;  // sub-chunk of v_lo: the largest w with wpre[w] <= v_lo
  for (uint32_t step = kShortSubs / 2; step > 0; step >>= 1)
    if (w + step <= nsub && wpre[w + step] <= v_lo) w += step;
  for (uint32_t v = v_lo; v < v_hi; ++v) {
    const float x = vals[v];
    const uint32_t key = mag_key(x);
    const bool gt = key > T, eq = key == T;
    if (gt || (eq && e_eq < tie_take)) {
      const uint32_t pos = e_gt + min(e_eq, tie_take);
      while (wpre[w + 1] <= v) ++w;
      if (pos < k) {
        oi[pos] = w * g.slot + (v - wpre[w]);  // slot offset for now
        st_keep(a.out_val + out0 + pos, x, keep);
      } else {
        set_status(a.status, SPARCML_ERR_BAD_STREAM);
      }
    }
    e_gt += gt ? 1u : 0u;
    e_eq += eq ? 1u : 0u;
  }
  __syncthreads();  // the offsets written above are visible to the whole CTA
  // offsets -> indices; the residual is zeroed at each kept index.
  for (uint32_t j = t; j < k; j += kSegThreads) {
    const uint32_t idx = cidx[oi[j]];
    st_keep(oi + j, idx, keep);
    rp[idx] = 0.0f;
  }
}

// Select for segment gs by CTA `rank` of the CS CTAs (a cluster when CS > 1)
// that share it. Every CTA of a cluster calls this for the same segment.
__device__ __forceinline__ void select_segment(const SelectArgs& a, SelectShared& sh,
                                               cg::cluster_group& cluster, uint32_t gs,
                                               uint32_t rank) {
  const uint32_t CS = a.CS;
  const Geo& g = a.g;
  const uint32_t p = gs / g.nseg, s = gs % g.nseg;
  const uint32_t n = seg_n(g, s), k = seg_k(g, s);
  if (k == 0) return;  // uniform over the cluster
  const uint32_t t = threadIdx.x;
  const bool raw = a.seg_flag[gs] != 0 || a.seg_cnt[gs] < k;
  if (a.raw_only && !raw) return;  // done by the long-segment passes
  const uint32_t ms = seg_chunks(g, s);
  const uint32_t c_first = s * g.m;  // node-local id of the segment's first chunk
  const uint32_t ca = c_first + (uint32_t)((uint64_t)ms * rank / CS);
  const uint32_t cb = c_first + (uint32_t)((uint64_t)ms * (rank + 1) / CS);
  const uint32_t seg_start = s * g.L;
  const uint64_t seg_end = (uint64_t)seg_start + n;
  const uint32_t raw_lo =
      (uint32_t)min((uint64_t)seg_start + (uint64_t)(ca - c_first) * kChunk, seg_end);
  const uint32_t raw_hi =
      (uint32_t)min((uint64_t)seg_start + (uint64_t)(cb - c_first) * kChunk, seg_end);
  float* rp = a.residual + (uint64_t)p * g.N;
  const uint64_t node_sub0 = (uint64_t)p * g.nchunk * kWarpsPerChunk;
  const uint32_t sa = ca * kWarpsPerChunk, sb = cb * kWarpsPerChunk;  // this CTA's sub-chunks

  // Fast path: one CTA owns the segment and all its candidates fit in shared
  // memory. They are read from global memory once, in index order; the
  // radix select and the ordered compaction then run on the shared copy.
  if (CS == 1 && !raw && ms * kWarpsPerChunk <= kWin && a.seg_cnt[gs] <= kSmallCands) {
    extern __shared__ uint32_t dsm[];
    uint32_t* s_idx = dsm;
    float* s_val = reinterpret_cast<float*>(dsm + kSmallCands);
    const uint32_t nsub = ms * kWarpsPerChunk;
    const uint32_t M = load_window(sh, a.sub_cnt + node_sub0 + sa, nsub);
    constexpr uint32_t kLoadBatch = 4;  // candidate loads in flight per thread
    for (uint32_t v0 = 0; v0 < M; v0 += blockDim.x * kLoadBatch) {
      uint32_t li[kLoadBatch];
      float lv[kLoadBatch];
#pragma unroll
      for (uint32_t u = 0; u < kLoadBatch; ++u) {
        const uint32_t v = v0 + u * blockDim.x + t;
        li[u] = 0;
        lv[u] = 0.0f;
        if (v < M) {
          const uint32_t w = window_chunk(sh, nsub, v);
          const uint64_t slot = (node_sub0 + sa + w) * g.slot + (v - sh.wpre[w]);
          li[u] = a.cand_idx[slot];
          lv[u] = a.cand_val[slot];
        }
      }
#pragma unroll
      for (uint32_t u = 0; u < kLoadBatch; ++u) {
        const uint32_t v = v0 + u * blockDim.x + t;
        if (v < M) {
          s_idx[v] = li[u];
          s_val[v] = lv[u];
        }
      }
    }
    __syncthreads();
    // Four 8-bit digits (bits 30..23, 22..15, 14..7, 6..0): 256 bins, one
    // per thread, so zeroing and scanning a histogram costs one step.
    uint32_t prefix = 0, rem = k;
    for (int d = 0; d < 4; ++d) {
      const uint32_t shift = d == 3 ? 0 : 23 - 8 * d;
      const uint32_t nb = d == 3 ? 128 : 256, hi_shift = d == 0 ? 31 : shift + (d == 3 ? 7 : 8);
      for (uint32_t b = t; b < 256; b += blockDim.x) sh.hist[b] = 0;
      __syncthreads();
      for (uint32_t v0 = 0; v0 < M; v0 += blockDim.x) {
        const uint32_t v = v0 + t;
        const uint32_t key = v < M ? mag_key(s_val[v]) : 0u;
        const bool match = v < M && (d == 0 || (key >> hi_shift) == prefix);
        hist_add(sh.hist, (key >> shift) & (nb - 1), match);
      }
      __syncthreads();
      find_from_top(sh.hist, 256, rem, sh.scratch, sh.res);
      uint32_t b = sh.res[0];
      if (b == kNone) {
        set_status(a.status, SPARCML_ERR_BAD_STREAM);
        b = 0;
      } else {
        rem -= sh.res[1];
      }
      prefix = (prefix << (d == 3 ? 7 : 8)) | b;
    }
    const uint32_t T = prefix, tie_take = rem;
    const uint64_t out0 = (uint64_t)p * g.cap + (uint64_t)s * g.k_full;
    uint32_t run_gt = 0, run_eq = 0;
    for (uint32_t v0 = 0; v0 < M; v0 += blockDim.x) {
      const uint32_t v = v0 + t;
      const float x = v < M ? s_val[v] : 0.0f;
      const uint32_t key = mag_key(x);
      const bool gt = v < M && key > T;
      const bool eq = v < M && key == T;
      uint32_t tot;
      const uint32_t ex =
          block_excl_scan((gt ? 1u : 0u) | (eq ? 0x10000u : 0u), sh.scratch, &tot);
      const uint32_t e_gt = run_gt + (ex & 0xffffu), e_eq = run_eq + (ex >> 16);
      if (gt || (eq && e_eq < tie_take)) {
        const uint32_t pos = e_gt + min(e_eq, tie_take);
        if (pos < k) {
          const uint32_t i = s_idx[v];
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
    }
    return;
  }

  // Visit every candidate of this CTA as (index, value), window by window.
  // `ordered` passes see them in ascending index order, blockDim at a time.
  auto for_each = [&](auto&& body) {
    if (raw) {
      const uint32_t total = raw_hi > raw_lo ? raw_hi - raw_lo : 0;
      for (uint32_t v0 = 0; v0 < total; v0 += blockDim.x) {
        const uint32_t v = v0 + t;
        const bool valid = v < total;
        const uint32_t i = raw_lo + v;
        body(valid, i, valid ? rp[i] : 0.0f);
      }
    } else {
      for (uint32_t w0 = sa; w0 < sb; w0 += kWin) {
        const uint32_t nw = min(kWin, sb - w0);
        const uint32_t total = load_window(sh, a.sub_cnt + node_sub0 + w0, nw);
        for (uint32_t v0 = 0; v0 < total; v0 += blockDim.x) {
          const uint32_t v = v0 + t;
          const bool valid = v < total;
          uint32_t i = 0;
          float x = 0.0f;
          if (valid) {
            const uint32_t w = window_chunk(sh, nw, v);
            const uint64_t slot = (node_sub0 + w0 + w) * g.slot + (v - sh.wpre[w]);
            i = a.cand_idx[slot];
            x = a.cand_val[slot];
          }
          body(valid, i, x);
        }
        __syncthreads();  // wpre is rewritten by the next window
      }
    }
  };

  // Radix select of the k-th largest key: digits of 11, 11 and 9 bits.
  uint32_t prefix = 0, rem = k;
  for (int d = 0; d < 3; ++d) {
    const uint32_t width = d < 2 ? 11 : 9, shift = d == 0 ? 20 : (d == 1 ? 9 : 0);
    const uint32_t nb = 1u << width, hi_shift = shift + width;
    for (uint32_t b = t; b < 2048; b += blockDim.x) sh.hist[b] = 0;
    __syncthreads();
    for_each([&](bool valid, uint32_t, float x) {
      const uint32_t key = mag_key(x);
      const bool match = valid && (d == 0 || (key >> hi_shift) == prefix);
      hist_add(sh.hist, (key >> shift) & (nb - 1), match);
    });
    __syncthreads();
    if (CS > 1) cluster.sync();
    for (uint32_t b = t; b < nb; b += blockDim.x) {
      uint32_t sum = 0;
      if (CS > 1) {
        for (uint32_t q = 0; q < CS; ++q) sum += cluster.map_shared_rank(sh.hist, q)[b];
      } else {
        sum = sh.hist[b];
      }
      sh.tot[b] = sum;
    }
    __syncthreads();
    find_from_top(sh.tot, nb, rem, sh.scratch, sh.res);
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
  const uint32_t T = prefix;     // exact k-th largest key
  const uint32_t tie_take = rem;  // keys == T to keep, lowest indices first

  // Counts of this CTA: keys > T and keys == T.
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

  // Ordered compaction of the kept entries.
  const uint64_t out0 = (uint64_t)p * g.cap + (uint64_t)s * g.k_full;
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

// ---------------------------------------------------------------------------
// Long segments (thousands of chunks): the exact select as a sequence of
// grid-wide passes, each CTA owning a range of kRangeSubs warp sub-chunks of
// one segment (a few hundred candidates), so the whole GPU works on every
// pass:
//   long_hist  x3  histogram of one radix digit (11, 11, 9 bits) of the keys
//                  that match the prefix so far, per CTA in shared memory,
//                  flushed into the segment's global histogram;
//   long_find  x3  one CTA per segment: the boundary bin -> prefix, rank left;
//   long_count     per range: keys > T and keys == T;
//   long_scan      one CTA per segment: exclusive prefix over its ranges;
//   long_write     per range: the kept entries in index order, residual = 0.
// Segments whose candidates do not cover k (or overflowed a slot) are left to
// topk_select_kernel, which reads their acc directly.
// ---------------------------------------------------------------------------
constexpr uint32_t kRangeSubs = 256;
constexpr uint32_t kHistWords = 2048 + 2048 + 512;  // per segment: the three digits

struct LongArgs {
  Geo g;
  const uint32_t* seg_cnt;
  const uint32_t* seg_flag;
  const uint32_t* sub_cnt;
  const uint32_t* cand_idx;
  const float* cand_val;
  float* residual;
  uint32_t* out_idx;
  float* out_val;
  int32_t* status;
  uint32_t* hist;       // [P * nseg][kHistWords]
  uint32_t* sel;        // [P * nseg][2]: prefix so far, rank left (then T, tie_take)
  uint32_t* range_cnt;  // [P * nseg][nr][2]: keys > T, keys == T (then their prefixes)
  uint32_t nr;          // ranges of a full segment
};

__device__ __forceinline__ bool long_eligible(const LongArgs& a, uint32_t gs, uint32_t k) {
  return k > 0 && a.seg_flag[gs] == 0 && a.seg_cnt[gs] >= k;
}

// The candidates of range r of segment gs: per-sub-chunk prefix in spre,
// returns their count (0 if the range is empty or the segment is not handled).
__device__ uint32_t long_range_setup(const LongArgs& a, uint32_t gs, uint32_t r, uint32_t* spre,
                                     uint32_t* scratch, uint64_t* sub_base) {
  const Geo& g = a.g;
  const uint32_t s = gs % g.nseg, p = gs / g.nseg;
  const uint32_t nsub = seg_chunks(g, s) * kWarpsPerChunk;
  const uint32_t sa = r * kRangeSubs;
  if (sa >= nsub || !long_eligible(a, gs, seg_k(g, s))) return 0;  // CTA-uniform
  const uint32_t nr = min(kRangeSubs, nsub - sa);
  *sub_base = ((uint64_t)p * g.nchunk + (uint64_t)s * g.m) * kWarpsPerChunk + sa;
  const uint32_t c = threadIdx.x < nr ? a.sub_cnt[*sub_base + threadIdx.x] : 0u;
  uint32_t tot;
  const uint32_t ex = block_excl_scan(c, scratch, &tot);
  if (threadIdx.x < nr) spre[threadIdx.x] = ex;
  if (threadIdx.x == 0) spre[nr] = tot;
  for (uint32_t i = nr + 1 + threadIdx.x; i <= kRangeSubs; i += blockDim.x) spre[i] = tot;
  __syncthreads();
  return tot;
}

__device__ __forceinline__ uint64_t long_slot(const LongArgs& a, const uint32_t* spre,
                                              uint64_t sub_base, uint32_t v) {
  uint32_t w = 0;
#pragma unroll
  for (uint32_t step = kRangeSubs / 2; step > 0; step >>= 1)
    if (spre[w + step] <= v) w += step;
  return (sub_base + w) * a.g.slot + (v - spre[w]);
}

__global__ void __launch_bounds__(kSelectThreads)
long_hist_kernel(LongArgs a, int d) {
  __shared__ uint32_t spre[kRangeSubs + 1];
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t hist[2048];
  const uint32_t gs = blockIdx.x / a.nr, r = blockIdx.x % a.nr;
  uint64_t sub_base = 0;
  const uint32_t M = long_range_setup(a, gs, r, spre, scratch, &sub_base);
  if (M == 0) return;
  const uint32_t width = d < 2 ? 11 : 9, shift = d == 0 ? 20 : (d == 1 ? 9 : 0);
  const uint32_t nb = 1u << width, hi_shift = shift + width;
  const uint32_t prefix = d == 0 ? 0u : a.sel[2 * gs];
  for (uint32_t b = threadIdx.x; b < nb; b += blockDim.x) hist[b] = 0;
  __syncthreads();
  constexpr uint32_t kB = 4;
  for (uint32_t v0 = 0; v0 < M; v0 += blockDim.x * kB) {
    float x[kB];
#pragma unroll
    for (uint32_t q = 0; q < kB; ++q) {
      const uint32_t v = v0 + q * blockDim.x + threadIdx.x;
      x[q] = v < M ? a.cand_val[long_slot(a, spre, sub_base, v)] : 0.0f;
    }
#pragma unroll
    for (uint32_t q = 0; q < kB; ++q) {
      const uint32_t v = v0 + q * blockDim.x + threadIdx.x;
      const uint32_t key = mag_key(x[q]);
      hist_add(hist, (key >> shift) & (nb - 1),
               v < M && (d == 0 || (key >> hi_shift) == prefix));
    }
  }
  __syncthreads();
  uint32_t* gh = a.hist + (uint64_t)gs * kHistWords + (d == 0 ? 0 : (d == 1 ? 2048 : 4096));
  for (uint32_t b = threadIdx.x; b < nb; b += blockDim.x)
    if (hist[b]) atomicAdd(&gh[b], hist[b]);
}

__global__ void __launch_bounds__(kSelectThreads)
long_find_kernel(LongArgs a, int d) {
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t res[2];
  const uint32_t gs = blockIdx.x;
  const Geo& g = a.g;
  const uint32_t k = seg_k(g, gs % g.nseg);
  if (!long_eligible(a, gs, k)) return;
  const uint32_t width = d < 2 ? 11 : 9, nb = 1u << width;
  const uint32_t* gh = a.hist + (uint64_t)gs * kHistWords + (d == 0 ? 0 : (d == 1 ? 2048 : 4096));
  const uint32_t prefix = d == 0 ? 0u : a.sel[2 * gs];
  const uint32_t rem = d == 0 ? k : a.sel[2 * gs + 1];
  find_from_top(gh, nb, rem, scratch, res);
  if (threadIdx.x == 0) {
    uint32_t b = res[0], above = res[1];
    if (b == kNone) {  // cannot happen for consistent counts
      set_status(a.status, SPARCML_ERR_BAD_STREAM);
      b = 0;
      above = 0;
    }
    a.sel[2 * gs] = (prefix << width) | b;
    a.sel[2 * gs + 1] = rem - above;
  }
}

__global__ void __launch_bounds__(kSelectThreads)
long_count_kernel(LongArgs a) {
  __shared__ uint32_t spre[kRangeSubs + 1];
  __shared__ uint32_t scratch[34];
  const uint32_t gs = blockIdx.x / a.nr, r = blockIdx.x % a.nr;
  uint64_t sub_base = 0;
  const uint32_t M = long_range_setup(a, gs, r, spre, scratch, &sub_base);
  if (M == 0) {
    if (threadIdx.x == 0) {
      a.range_cnt[2 * ((uint64_t)gs * a.nr + r)] = 0;
      a.range_cnt[2 * ((uint64_t)gs * a.nr + r) + 1] = 0;
    }
    return;
  }
  const uint32_t T = a.sel[2 * gs];
  uint32_t n_gt = 0, n_eq = 0;
  constexpr uint32_t kB = 4;
  for (uint32_t v0 = 0; v0 < M; v0 += blockDim.x * kB) {
    float x[kB];
#pragma unroll
    for (uint32_t q = 0; q < kB; ++q) {
      const uint32_t v = v0 + q * blockDim.x + threadIdx.x;
      x[q] = v < M ? a.cand_val[long_slot(a, spre, sub_base, v)] : 0.0f;
    }
#pragma unroll
    for (uint32_t q = 0; q < kB; ++q) {
      const uint32_t v = v0 + q * blockDim.x + threadIdx.x;
      const uint32_t key = mag_key(x[q]);
      n_gt += (v < M && key > T) ? 1u : 0u;
      n_eq += (v < M && key == T) ? 1u : 0u;
    }
  }
  uint32_t tg, te;
  block_excl_scan(n_gt, scratch, &tg);
  __syncthreads();
  block_excl_scan(n_eq, scratch, &te);
  if (threadIdx.x == 0) {
    a.range_cnt[2 * ((uint64_t)gs * a.nr + r)] = tg;
    a.range_cnt[2 * ((uint64_t)gs * a.nr + r) + 1] = te;
  }
}

__global__ void __launch_bounds__(1024)
long_scan_kernel(LongArgs a) {
  __shared__ uint32_t scratch[34];
  const uint32_t gs = blockIdx.x;
  const Geo& g = a.g;
  if (!long_eligible(a, gs, seg_k(g, gs % g.nseg))) return;
  uint32_t* rc = a.range_cnt + 2 * (uint64_t)gs * a.nr;
  uint32_t run_gt = 0, run_eq = 0;
  for (uint32_t r0 = 0; r0 < a.nr; r0 += blockDim.x) {
    const uint32_t r = r0 + threadIdx.x;
    const uint32_t cg_ = r < a.nr ? rc[2 * r] : 0u, ce = r < a.nr ? rc[2 * r + 1] : 0u;
    uint32_t tg, te;
    const uint32_t eg = block_excl_scan(cg_, scratch, &tg);
    __syncthreads();
    const uint32_t ee = block_excl_scan(ce, scratch, &te);
    if (r < a.nr) {
      rc[2 * r] = run_gt + eg;
      rc[2 * r + 1] = run_eq + ee;
    }
    run_gt += tg;
    run_eq += te;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kSelectThreads)
long_write_kernel(LongArgs a) {
  __shared__ uint32_t spre[kRangeSubs + 1];
  __shared__ uint32_t scratch[34];
  const uint32_t gs = blockIdx.x / a.nr, r = blockIdx.x % a.nr;
  uint64_t sub_base = 0;
  const uint32_t M = long_range_setup(a, gs, r, spre, scratch, &sub_base);
  if (M == 0) return;
  const Geo& g = a.g;
  const uint32_t p = gs / g.nseg, s = gs % g.nseg, k = seg_k(g, s);
  const uint32_t T = a.sel[2 * gs], tie_take = a.sel[2 * gs + 1];
  uint32_t run_gt = a.range_cnt[2 * ((uint64_t)gs * a.nr + r)];
  uint32_t run_eq = a.range_cnt[2 * ((uint64_t)gs * a.nr + r) + 1];
  float* rp = a.residual + (uint64_t)p * g.N;
  const uint64_t out0 = (uint64_t)p * g.cap + (uint64_t)s * g.k_full;
  const uint64_t keep = l2_policy_evict_last();
  for (uint32_t v0 = 0; v0 < M; v0 += blockDim.x) {
    const uint32_t v = v0 + threadIdx.x;
    uint64_t slot = 0;
    float x = 0.0f;
    if (v < M) {
      slot = long_slot(a, spre, sub_base, v);
      x = a.cand_val[slot];
    }
    const uint32_t key = mag_key(x);
    const bool gt = v < M && key > T, eq = v < M && key == T;
    uint32_t tot;
    const uint32_t ex = block_excl_scan((gt ? 1u : 0u) | (eq ? 0x10000u : 0u), scratch, &tot);
    const uint32_t e_gt = run_gt + (ex & 0xffffu), e_eq = run_eq + (ex >> 16);
    if (gt || (eq && e_eq < tie_take)) {
      const uint32_t pos = e_gt + min(e_eq, tie_take);
      if (pos < k) {
        const uint32_t i = a.cand_idx[slot];
        st_keep(a.out_idx + out0 + pos, i, keep);
        st_keep(a.out_val + out0 + pos, x, keep);
        rp[i] = 0.0f;
      } else {
        set_status(a.status, SPARCML_ERR_BAD_STREAM);
      }
    }
    run_gt += tot & 0xffffu;
    run_eq += tot >> 16;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kSelectThreads)
topk_select_kernel(SelectArgs a) {
  __shared__ SelectShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  if (a.warp_done) {  // only the segments the short kernel handed over
    const uint32_t n_todo = *a.todo_cnt;
    for (uint32_t i = blockIdx.x; i < n_todo; i += gridDim.x) {
      select_segment(a, sh, cluster, a.todo[i], 0);
      __syncthreads();
    }
  } else {
    select_segment(a, sh, cluster, blockIdx.x / a.CS, a.CS > 1 ? cluster.block_rank() : 0u);
  }
}

struct Layout {
  size_t todo_cnt, guess, seg_cnt, seg_flag, todo, chunk_cnt, cand_idx, cand_val;
  size_t lhist, lsel, lrange, total;
  uint32_t nr;  // long-segment ranges of a full segment
};

// Rank of the guess in a sample of S of a segment's n entries with k kept:
// r = ceil(lambda + 4 sqrt(lambda) + 8) with lambda = k S / n, the expected
// number of sampled keys among the top k plus four standard deviations and a
// margin, so the r-th largest sample key is very likely at or below the k-th
// key of the segment. Computed once on the host (double precision is slow on
// this GPU's cores).
uint32_t sample_rank(uint32_t k, uint32_t n, uint32_t S) {
  if (n == 0) return 0;
  const double lam = (double)k * (double)S / (double)n;
  const double rr = std::ceil(lam + 4.0 * std::sqrt(lam) + 8.0);
  return rr >= (double)S ? S : (uint32_t)rr;
}

bool make_geo(int32_t P, uint64_t N, uint64_t seg_len, uint32_t k_num, uint32_t k_den, Geo* g) {
  if (P < 1 || P > 65535 || N < 1 || N > 0xffffffffull || seg_len < 1 || k_den < 1 ||
      k_num > k_den)
    return false;
  const uint64_t L = std::min<uint64_t>(seg_len, N);
  g->N = N;
  g->L = (uint32_t)L;
  g->nseg = (uint32_t)((N + L - 1) / L);
  g->L_last = (uint32_t)(N - (uint64_t)(g->nseg - 1) * L);
  g->m = (uint32_t)((L + kChunk - 1) / kChunk);
  g->m_last = (g->L_last + kChunk - 1) / kChunk;
  const uint64_t nchunk = (uint64_t)(g->nseg - 1) * g->m + g->m_last;
  if (nchunk > 0xffffffffull || (uint64_t)P * g->nseg > 0x7fffffffull ||
      (uint64_t)P * nchunk > 0x7fffffffull)
    return false;
  g->nchunk = (uint32_t)nchunk;
  g->k_full = (uint32_t)(L * k_num / k_den);
  g->k_last = (uint32_t)((uint64_t)g->L_last * k_num / k_den);
  // Expected candidates are about d + a few per cent of a chunk; the slot
  // holds 2d + 1/8 of it (or all of it), and overflow falls back safely.
  const double want = (double)kSub * (2.0 * k_num / k_den) + kSub / 8.0;
  uint32_t slot = (uint32_t)std::min<double>(kSub, std::ceil(want / 32.0) * 32.0);
  g->slot = std::max<uint32_t>(slot, 32);
  g->P = P;
  auto cta_sample = [](uint32_t n) { return n <= kShortSegment ? kSampleShort : kSampleMax; };
  g->r_warp_full = sample_rank(g->k_full, g->L, kWarpSample);
  g->r_warp_last = sample_rank(g->k_last, g->L_last, kWarpSample);
  g->r_cta_full = sample_rank(g->k_full, g->L, cta_sample(g->L));
  g->r_cta_last = sample_rank(g->k_last, g->L_last, cta_sample(g->L_last));
  return true;
}

Layout make_layout(const Geo& g) {
  Layout l;
  size_t o = 256;  // status word and padding
  const size_t nsegs = (size_t)g.P * g.nseg, nch = (size_t)g.P * g.nchunk * kWarpsPerChunk;
  l.todo_cnt = 64;
  l.guess = o; o = align_up(o + 4 * nsegs, 256);
  l.todo = o; o = align_up(o + 4 * nsegs, 256);
  l.seg_cnt = o; o = align_up(o + 4 * nsegs, 256);
  l.seg_flag = o; o = align_up(o + 4 * nsegs, 256);
  l.chunk_cnt = o; o = align_up(o + 4 * nch, 256);
  l.cand_idx = o; o = align_up(o + 4 * nch * g.slot, 256);
  l.cand_val = o; o = align_up(o + 4 * nch * g.slot, 256);
  l.nr = (uint32_t)(((uint64_t)g.m * kWarpsPerChunk + kRangeSubs - 1) / kRangeSubs);
  l.lhist = o; o = align_up(o + 4 * nsegs * kHistWords, 256);
  l.lsel = o; o = align_up(o + 8 * nsegs, 256);
  l.lrange = o; o = align_up(o + 8 * nsegs * l.nr, 256);
  l.total = o;
  return l;
}

}  // namespace
}  // namespace sparcml

using namespace sparcml;

extern "C" size_t sparcml_topk_ef_workspace_size(int32_t P, uint64_t N, uint64_t seg_len,
                                                 uint32_t k_num, uint32_t k_den) {
  Geo g;
  if (!make_geo(P, N, seg_len, k_num, k_den, &g)) return 0;
  return make_layout(g).total;
}

extern "C" int sparcml_topk_ef_traced(const float* grad, float* residual, int32_t P,
                                      uint64_t N, uint64_t seg_len, uint32_t k_num,
                                      uint32_t k_den, uint32_t* out_idx, float* out_val,
                                      uint32_t* out_nnz, uint64_t cap, void* ws, size_t ws_bytes,
                                      void* stream, void* const* events) {
  Geo g;
  if (!grad || !residual || !out_idx || !out_val || !out_nnz || !ws ||
      !make_geo(P, N, seg_len, k_num, k_den, &g))
    return SPARCML_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return SPARCML_ERR_INVALID_ARG;
  const Layout l = make_layout(g);
  if (ws_bytes < l.total) return SPARCML_ERR_WORKSPACE;
  const uint64_t total_k = (uint64_t)(g.nseg - 1) * g.k_full + g.k_last;
  if (total_k > cap || total_k > 0xffffffffull) return SPARCML_ERR_CAPACITY;
  g.cap = cap;
  char* w = static_cast<char*>(ws);
  uint32_t* guess = reinterpret_cast<uint32_t*>(w + l.guess);
  uint32_t* seg_cnt = reinterpret_cast<uint32_t*>(w + l.seg_cnt);
  uint32_t* seg_flag = reinterpret_cast<uint32_t*>(w + l.seg_flag);
  uint32_t* chunk_cnt = reinterpret_cast<uint32_t*>(w + l.chunk_cnt);
  uint32_t* cand_idx = reinterpret_cast<uint32_t*>(w + l.cand_idx);
  float* cand_val = reinterpret_cast<float*>(w + l.cand_val);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  uint32_t* todo = reinterpret_cast<uint32_t*>(w + l.todo);
  uint32_t* todo_cnt = reinterpret_cast<uint32_t*>(w + l.todo_cnt);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto mark = [&](int i) {
    if (events && events[i]) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
  };

  mark(0);
  const uint32_t nsegs = (uint32_t)P * g.nseg;
  if (g.L > kSampleMax && g.L <= kShortSegment && g.L_last > kSampleMax) {
    // layer-sized segments: one warp each
    const uint32_t wpc = kGuessThreads / 32;
    topk_guess_warp_kernel<<<(nsegs + wpc - 1) / wpc, kGuessThreads, 0, s>>>(
        grad, residual, g, guess, seg_cnt, seg_flag, out_nnz, (uint32_t)total_k, todo_cnt);
  } else {
    // Keys per guess thread: the largest sample of any segment / kGuessThreads.
    auto sample_size = [](uint32_t n) {
      return n <= kSampleMax ? n : (n <= kShortSegment ? kSampleShort : kSampleMax);
    };
    const uint32_t smax = std::max(sample_size(g.L), sample_size(g.L_last));
    if (smax <= 16 * kGuessThreads)
      topk_guess_kernel<16><<<nsegs, kGuessThreads, 0, s>>>(
          grad, residual, g, guess, seg_cnt, seg_flag, out_nnz, (uint32_t)total_k, todo_cnt);
    else
      topk_guess_kernel<kSampleMax / kGuessThreads><<<nsegs, kGuessThreads, 0, s>>>(
          grad, residual, g, guess, seg_cnt, seg_flag, out_nnz, (uint32_t)total_k, todo_cnt);
  }
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  mark(1);
  topk_stream_kernel<<<(unsigned)((uint64_t)P * g.nchunk), kStreamThreads, 0, s>>>(
      grad, residual, g, guess, seg_cnt, seg_flag, chunk_cnt, cand_idx, cand_val);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  mark(2);

  // Cluster size: enough CTAs per segment to spread its chunks (<= 8).
  uint32_t CS = 1;
  while (CS < 8 && (uint64_t)g.m / (CS * 2) >= 64) CS *= 2;
  SelectArgs a{CS, CS == 1 ? 1u : 0u, CS > 1 ? 1u : 0u, todo, todo_cnt, residual, seg_cnt,
               seg_flag, chunk_cnt, guess, cand_idx, cand_val, out_idx, out_val, status, g};
  if (CS == 1) {  // layer-sized segments: one CTA each
    topk_select_short_kernel<<<nsegs, kSegThreads, 0, s>>>(a);
    if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  } else {  // long segments: grid-wide passes
    LongArgs la{g, seg_cnt, seg_flag, chunk_cnt, cand_idx, cand_val, residual, out_idx, out_val,
                status, reinterpret_cast<uint32_t*>(w + l.lhist),
                reinterpret_cast<uint32_t*>(w + l.lsel),
                reinterpret_cast<uint32_t*>(w + l.lrange), l.nr};
    if (cudaMemsetAsync(la.hist, 0, 4 * (size_t)nsegs * kHistWords, s) != cudaSuccess)
      return SPARCML_ERR_CUDA;
    const unsigned ranges = nsegs * l.nr;
    for (int d = 0; d < 3; ++d) {
      long_hist_kernel<<<ranges, kSelectThreads, 0, s>>>(la, d);
      long_find_kernel<<<nsegs, kSelectThreads, 0, s>>>(la, d);
    }
    long_count_kernel<<<ranges, kSelectThreads, 0, s>>>(la);
    long_scan_kernel<<<nsegs, 1024, 0, s>>>(la);
    long_write_kernel<<<ranges, kSelectThreads, 0, s>>>(la);
    if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  }
  // CS == 1: a small grid walks the segments the short kernel handed over.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS == 1 ? std::min<unsigned>(nsegs, 2 * 152)
                             : (unsigned)((uint64_t)P * g.nseg * CS), 1, 1);
  cfg.blockDim = dim3(kSelectThreads, 1, 1);
  cfg.dynamicSmemBytes = 2 * kSmallCands * sizeof(uint32_t);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!ensure_smem(reinterpret_cast<const void*>(topk_select_kernel), cfg.dynamicSmemBytes))
    return SPARCML_ERR_CUDA;
  if (CS == 1) {
    topk_select_kernel<<<cfg.gridDim, cfg.blockDim, cfg.dynamicSmemBytes, s>>>(a);
    if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  } else if (cudaLaunchKernelEx(&cfg, topk_select_kernel, a) != cudaSuccess) {
    return SPARCML_ERR_CUDA;
  }
  mark(3);
  note_launches(CS == 1 ? 4 : 3 + 9);
  return SPARCML_OK;
}

extern "C" int sparcml_topk_ef(const float* grad, float* residual, int32_t P, uint64_t N,
                               uint64_t seg_len, uint32_t k_num, uint32_t k_den,
                               uint32_t* out_idx, float* out_val, uint32_t* out_nnz,
                               uint64_t cap, void* ws, size_t ws_bytes, void* stream) {
  return sparcml_topk_ef_traced(grad, residual, P, N, seg_len, k_num, k_den, out_idx, out_val,
                                out_nnz, cap, ws, ws_bytes, stream, nullptr);
}
