// CPU oracle for the SparCML sparse-reduction hot path.
//
// TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
// statement of what the hot path computes. Only the test-suite, the smoke
// check and the benchmark's CPU-baseline leg may load it. It shares no code,
// header, table or constant generator with the CUDA library.
//
// Source: "SparCML: High-Performance Sparse Communication for Machine
// Learning" (Renggli, Ashkboos, Aghagolzadeh, Alistarh, Hoefler), as
// summarised section by section on its abstract page:
//   §2.2   Top-k SGD keeps the k largest-magnitude components per node and
//          carries the rest forward (error feedback); quantisation Q is an
//          element-wise stochastic operator with zero-mean noise.
//   §4     each node carries its unapplied components as a residual.
//   §5.1   sparse streams of index-value pairs, dense once fill-in passes a
//          threshold delta.
//   §5.2   reduction with any coordinate-wise associative op that has a
//          neutral element (here: fp32 sum, neutral element +0.0).
//   §6     stochastic QSGD quantisation in buckets with one full-precision
//          scale per bucket.
//   App. A floor(N/P)-style partitions with the remainder in the last part.
//
// Readings where the summary is silent (each one is also listed in the
// design notes): ties at the Top-k boundary go to the lowest index; exactly
// k_s = floor(n_s * k_num / k_den) entries are kept per segment even if some
// are zero; streams are strictly ascending; the sum runs over nodes in
// ascending order starting from +0.0f; the result is dense iff
// U * dens_den > N * dens_num; the 4-bit code is sign<<3 | level with 7
// levels of the bucket's max |v|; the rounding draw is SplitMix64 keyed by
// (seed, node, index).
//
// Status codes returned (0 = OK): 1 invalid argument, 3 capacity exceeded,
// 4 bad stream (index out of range or not strictly ascending).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <atomic>
#include <map>
#include <thread>
#include <utility>
#include <vector>

namespace {

enum { OK = 0, INVALID = 1, CAPACITY = 3, BAD_STREAM = 4 };

// Magnitude ordering key: the IEEE-754 bit pattern of |x|. For non-negative
// floats the unsigned bit pattern orders like the value.
uint32_t magnitude_key(float x) {
  uint32_t u;
  std::memcpy(&u, &x, sizeof u);
  return u & 0x7fffffffu;
}

// SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014; the 64-bit finaliser from Vigna's splitmix64):
// advance the state by the golden-ratio increment, then mix it.
uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9e3779b97f4a7c15ULL;
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

uint64_t segment_k(uint64_t n_s, uint64_t k_num, uint64_t k_den) {
  return n_s * k_num / k_den;  // floor(d * n_s) with d = k_num / k_den
}

// One fp32 addition, round to nearest even. IEEE 754 leaves the payload of a
// NaN result open; the reading used throughout is that every NaN produced by
// an addition is the quiet NaN with all payload bits set (0x7fffffff), so
// that the bits of a result do not depend on which input NaN a machine
// propagates.
float add_f32(float a, float b) {
  float r = a + b;
  if (r != r) {
    const uint32_t canonical = 0x7fffffffu;
    std::memcpy(&r, &canonical, sizeof r);
  }
  return r;
}

}  // namespace

extern "C" {

uint64_t oracle_splitmix64(uint64_t x) { return splitmix64(x); }

// Top-k with error feedback (§2.2, §4) of one segment [b, e) of one node,
// keeping k_s entries: acc = residual + grad over the segment; the k_s
// entries with the largest magnitude key (ties: lower index first) go to
// out_idx/out_val in ascending index order; the residual becomes acc with
// the kept positions set to +0.0f.
static void topk_segment(const float* g, float* r, uint64_t b, uint64_t e, uint64_t k_s,
                         uint32_t* out_idx, float* out_val) {
  const uint64_t n_s = e - b;
  std::vector<float> acc(n_s);
  // Error feedback: the accumulated gradient is residual + new gradient.
  for (uint64_t i = 0; i < n_s; ++i) acc[i] = add_f32(r[b + i], g[b + i]);
  std::vector<std::pair<uint32_t, uint32_t>> keyed;  // (key, index)
  keyed.reserve(n_s);
  for (uint64_t i = 0; i < n_s; ++i)
    keyed.emplace_back(magnitude_key(acc[i]), (uint32_t)(b + i));
  // Largest magnitude first; among equal magnitudes the lower index first.
  std::sort(keyed.begin(), keyed.end(),
            [](const std::pair<uint32_t, uint32_t>& x, const std::pair<uint32_t, uint32_t>& y) {
              if (x.first != y.first) return x.first > y.first;
              return x.second < y.second;
            });
  std::vector<uint32_t> chosen;
  for (uint64_t j = 0; j < k_s; ++j) chosen.push_back(keyed[j].second);
  std::sort(chosen.begin(), chosen.end());
  for (uint64_t j = 0; j < chosen.size(); ++j) {
    out_idx[j] = chosen[j];
    out_val[j] = acc[chosen[j] - b];
  }
  // Transmitted components leave the residual; the rest stay in it.
  for (uint32_t i : chosen) acc[i - b] = 0.0f;
  for (uint64_t i = 0; i < n_s; ++i) r[b + i] = acc[i];
}

// Checks a segment table: seg_begin[0] = 0 < seg_begin[1] < ... <
// seg_begin[nseg] = N and seg_k[s] <= n_s; returns the sum of the k_s in
// *total_k.
static int check_segments(uint64_t N, const uint64_t* seg_begin, const uint64_t* seg_k,
                          uint64_t nseg, uint64_t* total_k) {
  if (nseg == 0 || seg_begin[0] != 0 || seg_begin[nseg] != N) return INVALID;
  uint64_t t = 0;
  for (uint64_t s = 0; s < nseg; ++s) {
    if (seg_begin[s + 1] <= seg_begin[s]) return INVALID;
    if (seg_k[s] > seg_begin[s + 1] - seg_begin[s]) return INVALID;
    t += seg_k[s];
  }
  *total_k = t;
  return OK;
}

// Per-node Top-k with error feedback over an arbitrary segment table, the
// layer-wise sparsification of §8.4: segment s of every node is
// [seg_begin[s], seg_begin[s + 1]) and keeps seg_k[s] entries.
//   grad, residual: [P][N] fp32 row-major; residual is updated in place.
//   out_idx/out_val: [P][cap]; node p's stream holds the segments' kept
//   entries one segment after the other (so ascending), starting at p*cap;
//   out_nnz[p] = sum of seg_k.
int oracle_topk_ef_segments(const float* grad, float* residual, int32_t P, uint64_t N,
                            const uint64_t* seg_begin, const uint64_t* seg_k, uint64_t nseg,
                            uint32_t* out_idx, float* out_val, uint32_t* out_nnz,
                            uint64_t cap) {
  if (P <= 0 || N == 0 || N > 0xffffffffULL) return INVALID;
  uint64_t total_k = 0;
  const int st = check_segments(N, seg_begin, seg_k, nseg, &total_k);
  if (st != OK) return st;
  if (total_k > cap) return CAPACITY;
  for (int32_t p = 0; p < P; ++p) {
    uint64_t written = 0;
    for (uint64_t s = 0; s < nseg; ++s) {
      topk_segment(grad + (uint64_t)p * N, residual + (uint64_t)p * N, seg_begin[s],
                   seg_begin[s + 1], seg_k[s], out_idx + (uint64_t)p * cap + written,
                   out_val + (uint64_t)p * cap + written);
      written += seg_k[s];
    }
    out_nnz[p] = (uint32_t)written;
  }
  return OK;
}

// Per-node Top-k with error feedback (§2.2, §4) over equal segments: segment
// s is [s*seg_len, min((s+1)*seg_len, N)) (the last one takes the remainder,
// App. A) and keeps k_s = floor(n_s * k_num / k_den) entries.
int oracle_topk_ef(const float* grad, float* residual, int32_t P, uint64_t N,
                   uint64_t seg_len, uint64_t k_num, uint64_t k_den,
                   uint32_t* out_idx, float* out_val, uint32_t* out_nnz,
                   uint64_t cap) {
  if (P <= 0 || N == 0 || N > 0xffffffffULL || seg_len == 0 || k_den == 0 ||
      k_num > k_den || k_den > 0xffffffffULL)
    return INVALID;
  std::vector<uint64_t> begin, ks;
  for (uint64_t b = 0; b < N; b += seg_len) {
    begin.push_back(b);
    ks.push_back(segment_k(std::min(seg_len, N - b), k_num, k_den));
  }
  begin.push_back(N);
  return oracle_topk_ef_segments(grad, residual, P, N, begin.data(), ks.data(), ks.size(),
                                 out_idx, out_val, out_nnz, cap);
}

// Select entries with |x| > thr (thr = 0 keeps the nonzeros), ascending.
// If a node has more than cap such entries, the first cap are kept and
// CAPACITY is returned; out_nnz[p] = min(count, cap).
int oracle_pack(const float* x, int32_t P, uint64_t N, float thr, uint32_t* out_idx,
                float* out_val, uint32_t* out_nnz, uint64_t cap) {
  if (P <= 0 || N > 0xffffffffULL || !(thr >= 0.0f)) return INVALID;
  int status = OK;
  for (int32_t p = 0; p < P; ++p) {
    uint64_t n = 0;
    for (uint64_t i = 0; i < N; ++i) {
      const float v = x[(uint64_t)p * N + i];
      if (std::fabs(v) > thr) {
        if (n < cap) {
          out_idx[(uint64_t)p * cap + n] = (uint32_t)i;
          out_val[(uint64_t)p * cap + n] = v;
        }
        ++n;
      }
    }
    if (n > cap) status = CAPACITY;
    out_nnz[p] = (uint32_t)std::min<uint64_t>(n, cap);
  }
  return status;
}

// 4-bit stochastic quantisation of each node's stream values (§2.2, §6).
// Buckets are runs of `bucket` consecutive stream entries (the last one may
// be short). scale = max |v| over the bucket. With r = (|v| / scale) * 7 in
// fp32, the level is floor(r) rounded up with probability frac(r), the draw
// being u = (h >> 40) * 2^-24 for h = sm(sm(sm(seed) ^ node) ^ index).
// Code = (v < 0 ? 8 : 0) | level; two codes per byte, even entry in the low
// nibble. codes: [P][ceil(cap/2)], scales: [P][ceil(cap/bucket)].
int oracle_quantize4(const uint32_t* idx, const float* val, const uint32_t* nnz,
                     int32_t P, uint64_t cap, uint32_t bucket, uint64_t seed,
                     uint8_t* codes, float* scales) {
  if (P <= 0 || bucket == 0 || cap == 0) return INVALID;
  const uint64_t code_stride = (cap + 1) / 2;
  const uint64_t scale_stride = (cap + bucket - 1) / bucket;
  const uint64_t seed_mix = splitmix64(seed);
  for (int32_t p = 0; p < P; ++p) {
    if (nnz[p] > cap) return INVALID;
    const uint64_t node_mix = splitmix64(seed_mix ^ (uint64_t)(uint32_t)p);
    const uint32_t* ip = idx + (uint64_t)p * cap;
    const float* vp = val + (uint64_t)p * cap;
    uint8_t* cp = codes + (uint64_t)p * code_stride;
    for (uint64_t b0 = 0; b0 < nnz[p]; b0 += bucket) {
      const uint64_t b1 = std::min<uint64_t>(b0 + bucket, nnz[p]);
      float scale = 0.0f;
      for (uint64_t j = b0; j < b1; ++j) scale = std::max(scale, std::fabs(vp[j]));
      scales[(uint64_t)p * scale_stride + b0 / bucket] = scale;
      for (uint64_t j = b0; j < b1; ++j) {
        const float v = vp[j];
        uint32_t level = 0;
        if (scale > 0.0f) {
          const float r = (std::fabs(v) / scale) * 7.0f;
          const float f = std::floor(r);
          const float frac = r - f;
          const uint64_t h = splitmix64(node_mix ^ (uint64_t)ip[j]);
          const float u = (float)(h >> 40) * (1.0f / 16777216.0f);
          level = (uint32_t)f + (u < frac ? 1u : 0u);
          if (level > 7) level = 7;
        }
        const uint8_t code = (uint8_t)((v < 0.0f ? 8u : 0u) | level);
        uint8_t& byte = cp[j / 2];
        if ((j & 1) == 0)
          byte = (uint8_t)((byte & 0xf0) | code);
        else
          byte = (uint8_t)((byte & 0x0f) | (code << 4));
      }
    }
  }
  return OK;
}

// Inverse of the 4-bit code: v = +-(level / 7) * scale, level 0 -> +0.0f.
int oracle_dequantize4(const uint8_t* codes, const float* scales, const uint32_t* nnz,
                       int32_t P, uint64_t cap, uint32_t bucket, float* val_out) {
  if (P <= 0 || bucket == 0 || cap == 0) return INVALID;
  const uint64_t code_stride = (cap + 1) / 2;
  const uint64_t scale_stride = (cap + bucket - 1) / bucket;
  float level_value[8];
  for (int l = 0; l < 8; ++l) level_value[l] = (float)l / 7.0f;
  for (int32_t p = 0; p < P; ++p) {
    if (nnz[p] > cap) return INVALID;
    for (uint64_t j = 0; j < nnz[p]; ++j) {
      const uint8_t byte = codes[(uint64_t)p * code_stride + j / 2];
      const uint32_t code = (j & 1) ? (byte >> 4) : (byte & 0x0f);
      const uint32_t level = code & 7u;
      const float scale = scales[(uint64_t)p * scale_stride + j / bucket];
      float v = 0.0f;
      if (level != 0) {
        v = level_value[level] * scale;
        if (code & 8u) v = -v;
      }
      val_out[(uint64_t)p * cap + j] = v;
    }
  }
  return OK;
}

// b-bit stochastic quantisation (§6: QSGD-style buckets with one fp32 scale,
// 2-, 4- and 8-bit outputs), of stream values or of dense rows. With
// s = 2^(b-1) - 1 levels: scale = max |v| over the bucket, r = (|v| / scale)
// * s in fp32, level = floor(r) rounded up with probability frac(r) (the
// same SplitMix64 draw as the 4-bit form, keyed by (seed, node, index)), code
// = (v < 0) << (b-1) | level. 8/b codes per byte, the earliest entry in the
// lowest bits. Dense rows (idx == nullptr) use the position j as the index;
// nnz == nullptr means every row holds cap entries. If err_out is given it
// receives v - dequantised(v) per entry (quantisation-error feedback).
// codes: [P][ceil(cap / (8/b))], scales: [P][ceil(cap / bucket)].
int oracle_quantize(const uint32_t* idx, const float* val, const uint32_t* nnz, int32_t P,
                    uint64_t cap, uint32_t bucket, uint32_t bits, uint64_t seed,
                    uint8_t* codes, float* scales, float* err_out) {
  if (P <= 0 || cap == 0 || (bits != 2 && bits != 4 && bits != 8)) return INVALID;
  const uint32_t per_byte = 8 / bits;
  if (bucket == 0 || bucket % per_byte != 0) return INVALID;
  const uint32_t s = (1u << (bits - 1)) - 1;
  const uint64_t code_stride = (cap + per_byte - 1) / per_byte;
  const uint64_t scale_stride = (cap + bucket - 1) / bucket;
  const uint64_t seed_mix = splitmix64(seed);
  for (int32_t p = 0; p < P; ++p) {
    const uint64_t n = nnz ? nnz[p] : cap;
    if (n > cap) return INVALID;
    const uint64_t node_mix = splitmix64(seed_mix ^ (uint64_t)(uint32_t)p);
    const float* vp = val + (uint64_t)p * cap;
    uint8_t* cp = codes + (uint64_t)p * code_stride;
    for (uint64_t b0 = 0; b0 < n; b0 += bucket) {
      const uint64_t b1 = std::min<uint64_t>(b0 + bucket, n);
      float scale = 0.0f;
      for (uint64_t j = b0; j < b1; ++j) scale = std::max(scale, std::fabs(vp[j]));
      scales[(uint64_t)p * scale_stride + b0 / bucket] = scale;
      for (uint64_t j = b0; j < b1; ++j) {
        const float v = vp[j];
        const uint64_t index = idx ? idx[(uint64_t)p * cap + j] : j;
        uint32_t level = 0;
        if (scale > 0.0f) {
          const float r = (std::fabs(v) / scale) * (float)s;
          const float f = std::floor(r);
          const float frac = r - f;
          const uint64_t h = splitmix64(node_mix ^ index);
          const float u = (float)(h >> 40) * (1.0f / 16777216.0f);
          level = (uint32_t)f + (u < frac ? 1u : 0u);
          if (level > s) level = s;
        }
        const uint32_t sign = v < 0.0f ? 1u : 0u;
        const uint32_t code = (sign << (bits - 1)) | level;
        const uint32_t shift = (uint32_t)(j % per_byte) * bits;
        uint8_t& byte = cp[j / per_byte];
        const uint32_t mask = ((1u << bits) - 1u) << shift;
        byte = (uint8_t)((byte & ~mask) | (code << shift));
        if (err_out) {
          float q = 0.0f;
          if (level != 0) {
            q = ((float)level / (float)s) * scale;
            if (sign) q = -q;
          }
          err_out[(uint64_t)p * cap + j] = v - q;
        }
      }
    }
  }
  return OK;
}

// Inverse of the b-bit code: v = +-(level / s) * scale, level 0 -> +0.0f.
int oracle_dequantize(const uint8_t* codes, const float* scales, const uint32_t* nnz,
                      int32_t P, uint64_t cap, uint32_t bucket, uint32_t bits, float* val_out) {
  if (P <= 0 || cap == 0 || (bits != 2 && bits != 4 && bits != 8)) return INVALID;
  const uint32_t per_byte = 8 / bits;
  if (bucket == 0 || bucket % per_byte != 0) return INVALID;
  const uint32_t s = (1u << (bits - 1)) - 1;
  const uint64_t code_stride = (cap + per_byte - 1) / per_byte;
  const uint64_t scale_stride = (cap + bucket - 1) / bucket;
  for (int32_t p = 0; p < P; ++p) {
    const uint64_t n = nnz ? nnz[p] : cap;
    if (n > cap) return INVALID;
    for (uint64_t j = 0; j < n; ++j) {
      const uint8_t byte = codes[(uint64_t)p * code_stride + j / per_byte];
      const uint32_t code = (byte >> ((j % per_byte) * bits)) & ((1u << bits) - 1u);
      const uint32_t level = code & s;
      const float scale = scales[(uint64_t)p * scale_stride + j / bucket];
      float v = 0.0f;
      if (level != 0) {
        v = ((float)level / (float)s) * scale;
        if (code >> (bits - 1)) v = -v;
      }
      val_out[(uint64_t)p * cap + j] = v;
    }
  }
  return OK;
}

// Sum-reduction of P sparse streams (§5.2) with the dense switch (§5.1,
// §5.3.3). The sum for an index runs over the nodes that hold it, in
// ascending node order, starting from +0.0f. U = size of the index union.
// Dense iff U * dens_den > N * dens_num; then out_dense[N] holds the sums
// and +0.0f elsewhere. Otherwise out_idx/out_val hold the U sums ascending
// (out_cap must be >= U). out_nnz = U in both cases.
int oracle_sparse_reduce(const uint32_t* idx, const float* val, const uint32_t* nnz,
                         int32_t P, uint64_t cap, uint64_t N, uint32_t dens_num,
                         uint32_t dens_den, uint32_t* out_idx, float* out_val,
                         uint64_t out_cap, float* out_dense, uint64_t* out_nnz,
                         int32_t* out_is_dense) {
  if (P <= 0 || N == 0 || N > 0xffffffffULL || dens_den == 0) return INVALID;
  std::map<uint32_t, float> sum;
  for (int32_t p = 0; p < P; ++p) {
    if (nnz[p] > cap) return INVALID;
    for (uint64_t j = 0; j < nnz[p]; ++j) {
      const uint32_t i = idx[(uint64_t)p * cap + j];
      if (i >= N) return BAD_STREAM;
      if (j > 0 && i <= idx[(uint64_t)p * cap + j - 1]) return BAD_STREAM;
      const float v = val[(uint64_t)p * cap + j];
      auto it = sum.find(i);
      if (it == sum.end())
        sum.emplace(i, add_f32(0.0f, v));
      else
        it->second = add_f32(it->second, v);
    }
  }
  const uint64_t U = sum.size();
  const bool dense = U * (uint64_t)dens_den > N * (uint64_t)dens_num;
  *out_nnz = U;
  *out_is_dense = dense ? 1 : 0;
  if (dense) {
    for (uint64_t i = 0; i < N; ++i) out_dense[i] = 0.0f;
    for (const auto& kv : sum) out_dense[kv.first] = kv.second;
  } else {
    if (U > out_cap) return CAPACITY;
    uint64_t j = 0;
    for (const auto& kv : sum) {
      out_idx[j] = kv.first;
      out_val[j] = kv.second;
      ++j;
    }
  }
  return OK;
}

// Reduction of P sparse streams with another coordinate-wise associative
// operation that has a neutral element (§5.2): a stream stands for the
// vector whose unlisted coordinates hold the neutral element, and
//   op 0 sum: a + b,                          neutral +0.0f
//   op 1 max: b if b > a else a (fp32 order),  neutral -inf
//   op 2 min: b if b < a else a,               neutral +inf
//   op 3 or:  bitwise or of the fp32 bit patterns, neutral +0.0f (all bits 0)
// applied over the nodes that hold an index in ascending node order,
// starting from the neutral element. Union size, dense switch and output
// layout as in oracle_sparse_reduce; a dense result holds the neutral element
// where no node has the index. op 0 is oracle_sparse_reduce.
static float fold(int32_t op, float a, float b) {
  switch (op) {
    case 0: return add_f32(a, b);
    case 1: return b > a ? b : a;
    case 2: return b < a ? b : a;
    default: {
      uint32_t x, y;
      std::memcpy(&x, &a, 4);
      std::memcpy(&y, &b, 4);
      x |= y;
      float r;
      std::memcpy(&r, &x, 4);
      return r;
    }
  }
}

static float neutral(int32_t op) {
  if (op == 1) return -std::numeric_limits<float>::infinity();
  if (op == 2) return std::numeric_limits<float>::infinity();
  return 0.0f;
}

int oracle_sparse_reduce_op(const uint32_t* idx, const float* val, const uint32_t* nnz,
                            int32_t P, uint64_t cap, uint64_t N, int32_t op, uint32_t dens_num,
                            uint32_t dens_den, uint32_t* out_idx, float* out_val,
                            uint64_t out_cap, float* out_dense, uint64_t* out_nnz,
                            int32_t* out_is_dense) {
  if (P <= 0 || N == 0 || N > 0xffffffffULL || dens_den == 0 || op < 0 || op > 3)
    return INVALID;
  const float e = neutral(op);
  std::map<uint32_t, float> acc;
  for (int32_t p = 0; p < P; ++p) {
    if (nnz[p] > cap) return INVALID;
    for (uint64_t j = 0; j < nnz[p]; ++j) {
      const uint32_t i = idx[(uint64_t)p * cap + j];
      if (i >= N) return BAD_STREAM;
      if (j > 0 && i <= idx[(uint64_t)p * cap + j - 1]) return BAD_STREAM;
      const float v = val[(uint64_t)p * cap + j];
      auto it = acc.find(i);
      if (it == acc.end())
        acc.emplace(i, fold(op, e, v));
      else
        it->second = fold(op, it->second, v);
    }
  }
  const uint64_t U = acc.size();
  const bool dense = U * (uint64_t)dens_den > N * (uint64_t)dens_num;
  *out_nnz = U;
  *out_is_dense = dense ? 1 : 0;
  if (dense) {
    for (uint64_t i = 0; i < N; ++i) out_dense[i] = e;
    for (const auto& kv : acc) out_dense[kv.first] = kv.second;
  } else {
    if (U > out_cap) return CAPACITY;
    uint64_t j = 0;
    for (const auto& kv : acc) {
      out_idx[j] = kv.first;
      out_val[j] = kv.second;
      ++j;
    }
  }
  return OK;
}

// Static sparse allreduce by recursive doubling (SSAR, §5.3.1), emulated on
// one host: at stage s = 0 .. log2(P) - 1 every node i combines its current
// sparse partial result with the one of node i XOR 2^s; both obtain the same
// result, so a stage keeps one result per group of 2^(s+1) nodes. Combining
// two partial results A (lower group) and B is the two-stream sum reduce:
// for every index of A ∪ B, (+0.0f + a) + b, or +0.0f + the single value.
// The result never switches to dense (static sparse). out gets the final
// result (ascending, out_nnz entries); stage_nnz[s] the total number of
// entries held after stage s over the distinct partial results (fill-in).
// P must be a power of two >= 2.
int oracle_ssar(const uint32_t* idx, const float* val, const uint32_t* nnz, int32_t P,
                uint64_t cap, uint64_t N, uint32_t* out_idx, float* out_val, uint64_t out_cap,
                uint64_t* out_nnz, uint64_t* stage_nnz) {
  if (P < 2 || (P & (P - 1)) != 0 || N == 0 || N > 0xffffffffULL) return INVALID;
  std::vector<std::map<uint32_t, float>> part((size_t)P);
  for (int32_t p = 0; p < P; ++p) {
    if (nnz[p] > cap) return INVALID;
    for (uint64_t j = 0; j < nnz[p]; ++j) {
      const uint32_t i = idx[(uint64_t)p * cap + j];
      if (i >= N) return BAD_STREAM;
      if (j > 0 && i <= idx[(uint64_t)p * cap + j - 1]) return BAD_STREAM;
      part[(size_t)p].emplace(i, val[(uint64_t)p * cap + j]);
    }
  }
  // group g of a stage holds the partial result of nodes [g * 2^s, (g + 1) * 2^s)
  int stage = 0;
  while (part.size() > 1) {
    std::vector<std::map<uint32_t, float>> next(part.size() / 2);
    uint64_t fill = 0;
    for (size_t g = 0; g < next.size(); ++g) {
      const auto& A = part[2 * g];
      const auto& B = part[2 * g + 1];
      auto& C = next[g];
      for (const auto& kv : A) C.emplace(kv.first, add_f32(0.0f, kv.second));
      for (const auto& kv : B) {
        auto it = C.find(kv.first);
        if (it == C.end())
          C.emplace(kv.first, add_f32(0.0f, kv.second));
        else
          it->second = add_f32(it->second, kv.second);
      }
      fill += C.size();
    }
    stage_nnz[stage++] = fill;
    part.swap(next);
  }
  const auto& R = part[0];
  *out_nnz = R.size();
  if (R.size() > out_cap) return CAPACITY;
  uint64_t j = 0;
  for (const auto& kv : R) {
    out_idx[j] = kv.first;
    out_val[j] = kv.second;
    ++j;
  }
  return OK;
}

// Scatter each node's stream into a dense [P][N] vector, +0.0f elsewhere.
int oracle_densify(const uint32_t* idx, const float* val, const uint32_t* nnz, int32_t P,
                   uint64_t cap, uint64_t N, float* dense) {
  if (P <= 0 || N > 0xffffffffULL) return INVALID;
  for (int32_t p = 0; p < P; ++p) {
    if (nnz[p] > cap) return INVALID;
    float* d = dense + (uint64_t)p * N;
    for (uint64_t i = 0; i < N; ++i) d[i] = 0.0f;
    for (uint64_t j = 0; j < nnz[p]; ++j) {
      const uint32_t i = idx[(uint64_t)p * cap + j];
      if (i >= N) return BAD_STREAM;
      d[i] = val[(uint64_t)p * cap + j];
    }
  }
  return OK;
}

// ---------------------------------------------------------------------------
// Host-core timing drivers: the CPU baseline on every core. They split the
// work into pieces that do not interact and run each piece with the same
// code as the sequential functions above, so the results are identical.
// ---------------------------------------------------------------------------

// oracle_topk_ef_segments with the (node, segment) pairs spread over
// nthreads threads (each pair is independent: its own slice of residual,
// grad and output stream).
int oracle_topk_ef_segments_mt(const float* grad, float* residual, int32_t P, uint64_t N,
                               const uint64_t* seg_begin, const uint64_t* seg_k, uint64_t nseg,
                               uint32_t* out_idx, float* out_val, uint32_t* out_nnz,
                               uint64_t cap, int32_t nthreads) {
  if (P <= 0 || N == 0 || N > 0xffffffffULL || nthreads < 1) return INVALID;
  uint64_t total_k = 0;
  const int st = check_segments(N, seg_begin, seg_k, nseg, &total_k);
  if (st != OK) return st;
  if (total_k > cap) return CAPACITY;
  std::vector<uint64_t> out0(nseg + 1, 0);
  for (uint64_t s = 0; s < nseg; ++s) out0[s + 1] = out0[s] + seg_k[s];
  const uint64_t tasks = (uint64_t)P * nseg;
  std::atomic<uint64_t> next{0};
  auto work = [&]() {
    for (uint64_t t = next++; t < tasks; t = next++) {
      const uint64_t p = t / nseg, s = t % nseg;
      topk_segment(grad + p * N, residual + p * N, seg_begin[s], seg_begin[s + 1], seg_k[s],
                   out_idx + p * cap + out0[s], out_val + p * cap + out0[s]);
    }
  };
  std::vector<std::thread> pool;
  for (int32_t i = 1; i < nthreads; ++i) pool.emplace_back(work);
  work();
  for (auto& th : pool) th.join();
  for (int32_t p = 0; p < P; ++p) out_nnz[p] = (uint32_t)total_k;
  return OK;
}

// oracle_sparse_reduce with the index space cut into nthreads ranges: each
// thread owns [N t / T, N (t + 1) / T), walks every node's entries in that
// range in ascending node order into its own std::map, so every index gets
// the same sum in the same order as in the sequential function.
int oracle_sparse_reduce_mt(const uint32_t* idx, const float* val, const uint32_t* nnz,
                            int32_t P, uint64_t cap, uint64_t N, uint32_t dens_num,
                            uint32_t dens_den, uint32_t* out_idx, float* out_val,
                            uint64_t out_cap, float* out_dense, uint64_t* out_nnz,
                            int32_t* out_is_dense, int32_t nthreads) {
  if (P <= 0 || N == 0 || N > 0xffffffffULL || dens_den == 0 || nthreads < 1) return INVALID;
  for (int32_t p = 0; p < P; ++p)
    if (nnz[p] > cap) return INVALID;
  const int32_t T = nthreads;
  std::vector<int> bad(T, 0);
  std::vector<std::map<uint32_t, float>> part(T);
  auto work = [&](int32_t t) {
    // streams: strictly ascending and below N (each thread checks a slice)
    for (int32_t p = 0; p < P; ++p) {
      const uint32_t* row = idx + (uint64_t)p * cap;
      const uint64_t n = nnz[p], j0 = n * t / T, j1 = n * (t + 1) / T;
      for (uint64_t j = j0; j < j1; ++j)
        if (row[j] >= N || (j > 0 && row[j] <= row[j - 1])) bad[t] = 1;
    }
    const uint64_t r0 = N * t / T, r1 = N * (t + 1) / T;
    auto& sum = part[t];
    for (int32_t p = 0; p < P; ++p) {
      const uint32_t* row = idx + (uint64_t)p * cap;
      const uint32_t* lo = std::lower_bound(row, row + nnz[p], (uint32_t)r0);
      // the last range also takes any entry >= N (rejected above anyway)
      const uint32_t* hi =
          t == T - 1 ? row + nnz[p] : std::lower_bound(row, row + nnz[p], (uint32_t)r1);
      for (const uint32_t* q = lo; q < hi; ++q) {
        const float v = val[(uint64_t)p * cap + (uint64_t)(q - row)];
        auto it = sum.find(*q);
        if (it == sum.end())
          sum.emplace(*q, add_f32(0.0f, v));
        else
          it->second = add_f32(it->second, v);
      }
    }
  };
  std::vector<std::thread> pool;
  for (int32_t t = 1; t < T; ++t) pool.emplace_back(work, t);
  work(0);
  for (auto& th : pool) th.join();
  for (int32_t t = 0; t < T; ++t)
    if (bad[t]) return BAD_STREAM;
  uint64_t U = 0;
  for (int32_t t = 0; t < T; ++t) U += part[t].size();
  const bool dense = U * (uint64_t)dens_den > N * (uint64_t)dens_num;
  *out_nnz = U;
  *out_is_dense = dense ? 1 : 0;
  if (dense) {
    for (uint64_t i = 0; i < N; ++i) out_dense[i] = 0.0f;
    for (int32_t t = 0; t < T; ++t)
      for (const auto& kv : part[t]) out_dense[kv.first] = kv.second;
  } else {
    if (U > out_cap) return CAPACITY;
    uint64_t j = 0;
    for (int32_t t = 0; t < T; ++t)
      for (const auto& kv : part[t]) {
        out_idx[j] = kv.first;
        out_val[j] = kv.second;
        ++j;
      }
  }
  return OK;
}

}  // extern "C"
