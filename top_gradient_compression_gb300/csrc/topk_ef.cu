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
constexpr uint32_t kRounds = kChunk / (kStreamThreads * 4);  // float4 rounds per warp
constexpr uint32_t kSampleMax = 8192;     // sample of a long segment
constexpr uint32_t kSampleShort = 2048;   // sample of a layer-sized segment
constexpr uint32_t kShortSegment = 1u << 18;
constexpr uint32_t kRun = 32;
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
  uint32_t slot;     // candidate slot capacity per chunk
  int32_t P;
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
// 1. guess: one CTA per (node, segment).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kGuessThreads)
topk_guess_kernel(const float* __restrict__ grad, const float* __restrict__ residual, Geo g,
                  uint32_t* __restrict__ guess, uint32_t* __restrict__ seg_cnt,
                  uint32_t* __restrict__ seg_flag, uint32_t* __restrict__ out_nnz,
                  uint32_t total_k) {
  __shared__ uint32_t keys[kSampleMax];
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t scratch[34];
  __shared__ uint32_t res[2];

  const uint32_t gs = blockIdx.x;
  const uint32_t p = gs / g.nseg, s = gs % g.nseg;
  const uint32_t n = seg_n(g, s), k = seg_k(g, s);
  const uint32_t t = threadIdx.x;
  if (t == 0) {
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

  // Sample size: all of a short segment; else runs of 32 consecutive entries
  // (one 128-byte line per array per run), fewer for layer-sized segments
  // whose candidate sets are small anyway.
  const bool exact = n <= kSampleMax;
  const uint32_t S = exact ? n : (n <= kShortSegment ? kSampleShort : kSampleMax);
  uint32_t r;
  if (exact) {
    r = k;
  } else {
    const double lam = (double)k * (double)S / (double)n;
    const double rr = ceil(lam + 4.0 * sqrt(lam) + 8.0);
    r = rr >= (double)S ? S : (uint32_t)rr;
  }
  if (exact) {
#pragma unroll 4
    for (uint32_t i = t; i < S; i += blockDim.x) keys[i] = mag_key(__fadd_rn(rp[i], gp[i]));
  } else {
    // Warp w loads runs w, w + 8, ...: 4 runs (8 coalesced lines) in flight per lane.
    const uint32_t nruns = S / kRun, lane = lane_id(), warp = t >> 5, nw = blockDim.x >> 5;
    for (uint32_t r0 = warp; r0 < nruns; r0 += 4 * nw) {
      float a[4], b[4];
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) {
        const uint32_t run = r0 + q * nw;
        a[q] = b[q] = 0.0f;
        if (run < nruns) {
          const uint32_t st =
              (uint32_t)(((uint64_t)run * (n - kRun) / (nruns - 1)) & ~(uint64_t)(kRun - 1));
          a[q] = rp[st + lane];
          b[q] = gp[st + lane];
        }
      }
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) {
        const uint32_t run = r0 + q * nw;
        if (run < nruns) keys[run * kRun + lane] = mag_key(__fadd_rn(a[q], b[q]));
      }
    }
  }
  __syncthreads();
  // Two radix digits (bits 30..20, then 19..9) of the r-th largest key.
  uint32_t prefix = 0, rem = r;
  for (int d = 0; d < 2; ++d) {
    const uint32_t shift = d == 0 ? 20 : 9;
    for (uint32_t b = t; b < 2048; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    const uint32_t iters = (S + blockDim.x - 1) / blockDim.x;
    for (uint32_t it = 0; it < iters; ++it) {
      const uint32_t i = it * blockDim.x + t;
      const bool valid = i < S;
      const uint32_t key = valid ? keys[i] : 0;
      const bool match = valid && (d == 0 || (key >> 20) == prefix);
      hist_add(hist, (key >> shift) & 2047u, match);
    }
    __syncthreads();
    find_from_top(hist, 2048, rem, scratch, res);
    const uint32_t b = res[0] == kNone ? 0 : res[0];
    rem -= res[0] == kNone ? 0 : res[1];
    prefix = d == 0 ? b : ((prefix << 11) | b);
    __syncthreads();
  }
  if (t == 0) guess[gs] = prefix << 9;
}

// ---------------------------------------------------------------------------
// 2. stream: one CTA per chunk of kChunk entries (a chunk never crosses a
// segment boundary). Warp w owns the contiguous entries
// [start + 1024 w, start + 1024 (w + 1)), read as kRounds rounds of 32 float4.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kStreamThreads)
topk_stream_kernel(const float* __restrict__ grad, float* __restrict__ residual, Geo g,
                   const uint32_t* __restrict__ guess, uint32_t* __restrict__ seg_cnt,
                   uint32_t* __restrict__ seg_flag, uint32_t* __restrict__ chunk_cnt,
                   uint32_t* __restrict__ cand_idx, float* __restrict__ cand_val) {
  __shared__ uint32_t warp_tot[kStreamThreads / 32];
  const uint32_t gc = blockIdx.x;
  const uint32_t p = gc / g.nchunk, c = gc % g.nchunk;
  uint32_t s, j;
  chunk_pos(g, c, &s, &j);
  const uint32_t seg_start = s * g.L;
  const uint32_t start = seg_start + j * kChunk;
  const uint32_t nn = min(kChunk, seg_start + seg_n(g, s) - start);  // entries in this chunk
  const uint32_t G = guess[p * g.nseg + s];
  const float* gp = grad + (uint64_t)p * g.N + start;
  float* rp = residual + (uint64_t)p * g.N + start;
  const bool aligned =
      ((reinterpret_cast<uintptr_t>(gp) | reinterpret_cast<uintptr_t>(rp)) & 15) == 0;

  const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
  uint32_t mask = 0;  // bit 4t+q: entry q of round t is a candidate

  // Phase A: load, accumulate, write back, flag candidates.
  float4 gv[kRounds], rv[kRounds];
#pragma unroll
  for (uint32_t t = 0; t < kRounds; ++t) {
    const uint32_t e0 = 4 * (warp * (kRounds * 32) + t * 32 + lane);  // chunk-local
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
#pragma unroll
  for (uint32_t t = 0; t < kRounds; ++t) {
    const uint32_t e0 = 4 * (warp * (kRounds * 32) + t * 32 + lane);
    float4 a;
    a.x = __fadd_rn(rv[t].x, gv[t].x);
    a.y = __fadd_rn(rv[t].y, gv[t].y);
    a.z = __fadd_rn(rv[t].z, gv[t].z);
    a.w = __fadd_rn(rv[t].w, gv[t].w);
    const float av[4] = {a.x, a.y, a.z, a.w};
    if (aligned && e0 + 4 <= nn) {
      *reinterpret_cast<float4*>(rp + e0) = a;
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) mask |= (mag_key(av[q]) >= G ? 1u : 0u) << (4 * t + q);
    } else {
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q)
        if (e0 + q < nn) {
          rp[e0 + q] = av[q];
          mask |= (mag_key(av[q]) >= G ? 1u : 0u) << (4 * t + q);
        }
    }
  }
  const uint32_t my = __popc(mask);
  const uint32_t wsum = warp_sum(my);
  if (lane == 0) warp_tot[warp] = wsum;
  __syncthreads();
  uint32_t base = 0, total = 0;
#pragma unroll
  for (uint32_t w = 0; w < kStreamThreads / 32; ++w) {
    base += w < warp ? warp_tot[w] : 0u;
    total += warp_tot[w];
  }
  if (threadIdx.x == 0) {
    chunk_cnt[gc] = total;
    if (total) atomicAdd(&seg_cnt[p * g.nseg + s], total);
    if (total > g.slot) atomicOr(&seg_flag[p * g.nseg + s], 1u);
  }

  // Phase B: ordered compaction of the warp's candidates into the slot.
  if (wsum == 0) return;
  const uint64_t slot0 = (uint64_t)gc * g.slot;
  uint32_t run = base;
#pragma unroll
  for (uint32_t t = 0; t < kRounds; ++t) {
    const uint32_t bits = (mask >> (4 * t)) & 15u;
    uint32_t tot;
    uint32_t pos = run + warp_excl_small(__popc(bits), &tot);
    run += tot;
    if (bits) {
      const uint32_t e0 = 4 * (warp * (kRounds * 32) + t * 32 + lane);
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q)
        if (bits & (1u << q)) {
          if (pos < g.slot) {
            cand_idx[slot0 + pos] = start + e0 + q;
            cand_val[slot0 + pos] = rp[e0 + q];
          }
          ++pos;
        }
    }
  }
}

// ---------------------------------------------------------------------------
// 3. select: one cluster of CS CTAs per (node, segment). CTA r of the
// cluster owns chunks [ms*r/CS, ms*(r+1)/CS) of the segment.
// ---------------------------------------------------------------------------
struct SelectArgs {
  float* residual;
  const uint32_t* seg_cnt;
  const uint32_t* seg_flag;
  const uint32_t* chunk_cnt;
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
  uint32_t wpre[kWin + 1];
  uint32_t scratch[34];
  uint32_t res[2];
  uint32_t cnt[2];  // this CTA's (> T, == T) counts, read by higher ranks
};

// Exclusive prefix of the candidate counts of chunks [c0, c0 + nw) into
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

// Position v of a window -> its chunk (largest w with wpre[w] <= v).
__device__ __forceinline__ uint32_t window_chunk(const SelectShared& sh, uint32_t nw, uint32_t v) {
  uint32_t lo = 0, hi = nw;  // invariant: wpre[lo] <= v < wpre[hi]
  while (hi - lo > 1) {
    const uint32_t mid = (lo + hi) >> 1;
    if (sh.wpre[mid] <= v) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kSelectThreads)
topk_select_kernel(SelectArgs a) {
  __shared__ SelectShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t CS = cluster.num_blocks();
  const uint32_t rank = cluster.block_rank();
  const Geo& g = a.g;
  const uint32_t gs = blockIdx.x / CS;
  const uint32_t p = gs / g.nseg, s = gs % g.nseg;
  const uint32_t n = seg_n(g, s), k = seg_k(g, s);
  if (k == 0) return;  // uniform over the cluster
  const uint32_t t = threadIdx.x;
  const bool raw = a.seg_flag[gs] != 0 || a.seg_cnt[gs] < k;
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
  const uint64_t node_chunk0 = (uint64_t)p * g.nchunk;

  // Fast path: one CTA owns the segment and all its candidates fit in shared
  // memory. They are read from global memory once, in index order; the
  // radix select and the ordered compaction then run on the shared copy.
  if (CS == 1 && !raw && ms <= kWin && a.seg_cnt[gs] <= kSmallCands) {
    extern __shared__ uint32_t dsm[];
    uint32_t* s_idx = dsm;
    float* s_val = reinterpret_cast<float*>(dsm + kSmallCands);
    const uint32_t M = load_window(sh, a.chunk_cnt + node_chunk0 + c_first, ms);
    for (uint32_t v = t; v < M; v += blockDim.x) {
      const uint32_t w = window_chunk(sh, ms, v);
      const uint64_t slot = (node_chunk0 + c_first + w) * g.slot + (v - sh.wpre[w]);
      s_idx[v] = a.cand_idx[slot];
      s_val[v] = a.cand_val[slot];
    }
    __syncthreads();
    const uint32_t shifts[3] = {20, 9, 0};
    const uint32_t widths[3] = {11, 11, 9};
    uint32_t prefix = 0, rem = k;
    for (int d = 0; d < 3; ++d) {
      const uint32_t shift = shifts[d], nb = 1u << widths[d], hi_shift = shift + widths[d];
      for (uint32_t b = t; b < nb; b += blockDim.x) sh.hist[b] = 0;
      __syncthreads();
      for (uint32_t v0 = 0; v0 < M; v0 += blockDim.x) {
        const uint32_t v = v0 + t;
        const uint32_t key = v < M ? mag_key(s_val[v]) : 0u;
        const bool match = v < M && (d == 0 || (key >> hi_shift) == prefix);
        hist_add(sh.hist, (key >> shift) & (nb - 1), match);
      }
      __syncthreads();
      find_from_top(sh.hist, nb, rem, sh.scratch, sh.res);
      uint32_t b = sh.res[0];
      if (b == kNone) {
        set_status(a.status, SPARCML_ERR_BAD_STREAM);
        b = 0;
      } else {
        rem -= sh.res[1];
      }
      prefix = (prefix << widths[d]) | b;
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
      for (uint32_t w0 = ca; w0 < cb; w0 += kWin) {
        const uint32_t nw = min(kWin, cb - w0);
        const uint32_t total = load_window(sh, a.chunk_cnt + node_chunk0 + w0, nw);
        for (uint32_t v0 = 0; v0 < total; v0 += blockDim.x) {
          const uint32_t v = v0 + t;
          const bool valid = v < total;
          uint32_t i = 0;
          float x = 0.0f;
          if (valid) {
            const uint32_t w = window_chunk(sh, nw, v);
            const uint64_t slot = (node_chunk0 + w0 + w) * g.slot + (v - sh.wpre[w]);
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
  const uint32_t shifts[3] = {20, 9, 0};
  const uint32_t widths[3] = {11, 11, 9};
  uint32_t prefix = 0, rem = k;
  for (int d = 0; d < 3; ++d) {
    const uint32_t shift = shifts[d], nb = 1u << widths[d], hi_shift = shift + widths[d];
    for (uint32_t b = t; b < 2048; b += blockDim.x) sh.hist[b] = 0;
    __syncthreads();
    for_each([&](bool valid, uint32_t, float x) {
      const uint32_t key = mag_key(x);
      const bool match = valid && (d == 0 || (key >> hi_shift) == prefix);
      hist_add(sh.hist, (key >> shift) & (nb - 1), match);
    });
    __syncthreads();
    cluster.sync();
    for (uint32_t b = t; b < nb; b += blockDim.x) {
      uint32_t sum = 0;
      for (uint32_t q = 0; q < CS; ++q) sum += cluster.map_shared_rank(sh.hist, q)[b];
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
    prefix = (prefix << widths[d]) | b;
    cluster.sync();  // every CTA is done reading this CTA's histogram
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
  cluster.sync();
  uint32_t gt_pre = 0, eq_pre = 0;
  for (uint32_t q = 0; q < rank; ++q) {
    const uint32_t* rc = cluster.map_shared_rank(sh.cnt, q);
    gt_pre += rc[0];
    eq_pre += rc[1];
  }
  cluster.sync();  // peers may exit or reuse their shared memory after this

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

struct Layout {
  size_t guess, seg_cnt, seg_flag, chunk_cnt, cand_idx, cand_val, total;
};

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
  const double want = (double)kChunk * (2.0 * k_num / k_den) + kChunk / 8.0;
  uint32_t slot = (uint32_t)std::min<double>(kChunk, std::ceil(want / 32.0) * 32.0);
  g->slot = std::max<uint32_t>(slot, 32);
  g->P = P;
  return true;
}

Layout make_layout(const Geo& g) {
  Layout l;
  size_t o = 256;  // status word and padding
  const size_t nsegs = (size_t)g.P * g.nseg, nch = (size_t)g.P * g.nchunk;
  l.guess = o; o = align_up(o + 4 * nsegs, 256);
  l.seg_cnt = o; o = align_up(o + 4 * nsegs, 256);
  l.seg_flag = o; o = align_up(o + 4 * nsegs, 256);
  l.chunk_cnt = o; o = align_up(o + 4 * nch, 256);
  l.cand_idx = o; o = align_up(o + 4 * nch * g.slot, 256);
  l.cand_val = o; o = align_up(o + 4 * nch * g.slot, 256);
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
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto mark = [&](int i) {
    if (events && events[i]) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
  };

  mark(0);
  topk_guess_kernel<<<(unsigned)(P * g.nseg), kGuessThreads, 0, s>>>(
      grad, residual, g, guess, seg_cnt, seg_flag, out_nnz, (uint32_t)total_k);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  mark(1);
  topk_stream_kernel<<<(unsigned)((uint64_t)P * g.nchunk), kStreamThreads, 0, s>>>(
      grad, residual, g, guess, seg_cnt, seg_flag, chunk_cnt, cand_idx, cand_val);
  if (launch_status() != SPARCML_OK) return SPARCML_ERR_CUDA;
  mark(2);

  // Cluster size: enough CTAs per segment to spread its chunks (<= 8).
  uint32_t CS = 1;
  while (CS < 8 && (uint64_t)g.m / (CS * 2) >= 64) CS *= 2;
  SelectArgs a{residual, seg_cnt, seg_flag, chunk_cnt, cand_idx, cand_val,
               out_idx, out_val, status, g};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((uint64_t)P * g.nseg * CS), 1, 1);
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
  if (cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)cfg.dynamicSmemBytes) != cudaSuccess)
    return SPARCML_ERR_CUDA;
  if (cudaLaunchKernelEx(&cfg, topk_select_kernel, a) != cudaSuccess) return SPARCML_ERR_CUDA;
  mark(3);
  note_launches(3);
  return SPARCML_OK;
}

extern "C" int sparcml_topk_ef(const float* grad, float* residual, int32_t P, uint64_t N,
                               uint64_t seg_len, uint32_t k_num, uint32_t k_den,
                               uint32_t* out_idx, float* out_val, uint32_t* out_nnz,
                               uint64_t cap, void* ws, size_t ws_bytes, void* stream) {
  return sparcml_topk_ef_traced(grad, residual, P, N, seg_len, k_num, k_den, out_idx, out_val,
                                out_nnz, cap, ws, ws_bytes, stream, nullptr);
}
