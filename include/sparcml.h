/*
 * sparcml.h - C ABI of the GB300 (sm_103a) sparse-reduction hot path.
 *
 * The operations follow "SparCML: High-Performance Sparse Communication for
 * Machine Learning" (Renggli, Ashkboos, Aghagolzadeh, Alistarh, Hoefler):
 * P data-parallel nodes each hold a fp32 gradient of N entries. Each node
 * keeps its k largest-magnitude components and carries the rest forward as
 * a residual (Top-k with error feedback, §2.2 and §4), sends them as a
 * sparse stream of index-value pairs (§5.1), optionally quantised to 4 bits
 * with stochastic rounding (§2.2, §6), and the P streams are sum-reduced
 * (§5.2) into a sparse result that switches to a dense fp32 vector once its
 * fill-in passes a threshold (§5.1, §5.3.3). Here the P nodes are slices of
 * one GPU's memory and the "network" is the reduce kernel.
 *
 * Conventions shared by every entry point:
 *   - Layout. A node-major batch of P vectors of N fp32 values is one
 *     row-major [P][N] array: node p starts at element p*N. A batch of P
 *     sparse streams is idx uint32 [P][cap], val float [P][cap] and nnz
 *     uint32 [P]: node p's entries are idx[p*cap + j], val[p*cap + j] for
 *     j < nnz[p], with idx strictly ascending and < N (node-local indices).
 *   - Memory. Every array argument is DEVICE memory owned by the caller,
 *     except where a parameter says "host". The library never allocates,
 *     frees or keeps device memory between calls: scratch space comes from
 *     the caller as a workspace (`ws`, `ws_bytes`), sized by the matching
 *     *_workspace_size function. A workspace may be reused by later calls
 *     but not by two calls in flight at the same time.
 *   - Streams. `stream` is a cudaStream_t (NULL = legacy default stream).
 *     All work is enqueued on it and the call returns without waiting:
 *     the calls are non-blocking in the sense of §7 (MPI-3 style
 *     non-blocking collectives). Only sparcml_get_status synchronises.
 *   - Workspace header. The first 256 bytes of every workspace hold the
 *     device status word (bytes 0..3) and the fault-injection word (bytes
 *     32..35, see sparcml_set_fault_injection). Zero the first 64 bytes when
 *     a workspace is created; the library keeps them from then on.
 *   - Errors. A return value other than SPARCML_OK means nothing was
 *     enqueued (bad argument, workspace too small, capacity too small) or
 *     a CUDA launch failed (SPARCML_ERR_CUDA). Problems found on the device
 *     (an index out of range or out of order, a selection that does not
 *     fit, a wait that ran out) never trap: the first one is recorded in a
 *     device status word (the first 4 bytes of the workspace, or the
 *     explicit `status` pointer) and read back by sparcml_get_status.
 *   - Limits. 1 <= P <= 65535, 1 <= N <= 2^32 - 1 (indices are uint32),
 *     unless an entry point states its own bound on P.
 *
 * Results are deterministic: the same inputs give the same bits on every
 * run (fixed summation order, no floating-point atomics).
 */
#ifndef SPARCML_H
#define SPARCML_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum sparcml_status {
  SPARCML_OK = 0,
  SPARCML_ERR_INVALID_ARG = 1, /* bad pointer, size or parameter           */
  SPARCML_ERR_WORKSPACE = 2,   /* ws_bytes below the *_workspace_size     */
  SPARCML_ERR_CAPACITY = 3,    /* an output does not fit its capacity     */
  SPARCML_ERR_BAD_STREAM = 4,  /* index >= N, or not strictly ascending   */
  SPARCML_ERR_NONFINITE = 5,   /* a checked input holds a NaN or an inf   */
  SPARCML_ERR_TIMEOUT = 6,     /* a bounded device-side wait ran out      */
  SPARCML_ERR_CUDA = 7         /* a CUDA runtime call or launch failed    */
};

/* Human-readable name of a status code (static string, never NULL). */
const char* sparcml_status_string(int status);

/* Number of GPU kernels this library has launched in this process so far
 * (all devices, all threads). Lets a caller count the kernels inside a
 * timed region. */
uint64_t sparcml_launch_count(void);

/* Testing hook for the failure-detection path (the pages describe no fault
 * tolerance; this exercises the library's own bounded waits). Writes the
 * fault-injection word of a workspace (bytes 32..35) on `stream`:
 *   mode SPARCML_INJECT_WITHHOLD_FIRST: in later sparse-reduce and SSAR
 *     calls made with this workspace, the first tile (reduce) or each
 *     pair's first chunk (SSAR) of every decoupled look-back chain withholds
 *     its published prefix, and every bounded wait gives up after a few
 *     thousand polls (milliseconds) instead of about two million. The
 *     waiting tiles record SPARCML_ERR_TIMEOUT in the status word and carry
 *     on; the outputs of such a call are unspecified, but every memory
 *     access stays in bounds and the call always completes.
 *   mode 0: clears it (later calls are normal again).
 * The word stays as written across calls. A workspace whose first 64 bytes
 * were zeroed when it was created has no fault armed.
 * Returns SPARCML_ERR_INVALID_ARG for another mode or a workspace pointer
 * that is NULL or not 256-byte aligned. */
#define SPARCML_INJECT_WITHHOLD_FIRST 1
int sparcml_set_fault_injection(void* ws, int32_t mode, void* stream);

/* Synchronises `stream`, then returns the first device-detected error
 * recorded in the status word at `status_word` (a workspace pointer, or the
 * explicit status pointer given to densify/quantize/dequantize) and resets
 * it to SPARCML_OK. Returns SPARCML_ERR_CUDA if synchronisation fails. */
int sparcml_get_status(void* status_word, void* stream);

/* ------------------------------------------------------------------------
 * Top-k selection with error feedback, fused with packing (§2.2, §4, §5.1),
 * over a table of segments: the layer-wise sparsification of §8.4, where
 * every layer of the model keeps its own number of components.
 *
 * For every node p and every element i:
 *     acc = residual[p][i] + grad[p][i]            (one fp32 add, RN; a NaN
 *                                                   result is 0x7fffffff)
 * Segment s of every node is [seg_begin[s], seg_begin[s+1]) and keeps
 * exactly seg_k[s] entries: those with the largest |acc|, comparing the bit
 * patterns of |acc| as unsigned integers (so any NaN ranks above +-inf, which
 * rank above every finite value), ties going to the lowest index. Node p's
 * stream holds the kept entries of segment 0, then segment 1, ..., each in
 * ascending index order (so the stream is ascending), with val = acc;
 * out_nnz[p] = sum of seg_k. residual[p][i] becomes +0.0f at kept entries
 * and acc everywhere else.
 *
 *   grad      [P][N] fp32, read only.
 *   residual  [P][N] fp32, read and overwritten in place (the EF state).
 *   seg_begin HOST array of nseg + 1 entries: seg_begin[0] = 0 <
 *             seg_begin[1] < ... < seg_begin[nseg] = N (no empty segment).
 *   seg_k     HOST array of nseg entries, seg_k[s] <= seg_begin[s+1] -
 *             seg_begin[s] (0 keeps nothing, the length keeps everything).
 *             Both host arrays are read during the call only; the library
 *             copies what the GPU needs into the workspace on `stream`
 *             through kernel parameters (no host-side staging buffer, no
 *             synchronisation).
 *   out_idx, out_val  [P][cap]; out_nnz [P]. cap >= sparcml_topk_total_k,
 *             else SPARCML_ERR_CAPACITY.
 *   ws        >= sparcml_topk_ef_workspace_size(P, N, seg_begin, seg_k, nseg)
 *             bytes, 256-byte aligned; the same table must be passed to both.
 * A table that breaks the rules above returns SPARCML_ERR_INVALID_ARG.
 * 128-bit loads are used when grad and residual are 16-byte aligned
 * (whatever the segment offsets); other pointers take a slower scalar path.
 * ------------------------------------------------------------------------ */
size_t sparcml_topk_ef_workspace_size(int32_t P, uint64_t N, const uint64_t* seg_begin,
                                      const uint32_t* seg_k, uint32_t nseg);
int sparcml_topk_ef(const float* grad, float* residual, int32_t P, uint64_t N,
                    const uint64_t* seg_begin, const uint32_t* seg_k, uint32_t nseg,
                    uint32_t* out_idx, float* out_val, uint32_t* out_nnz, uint64_t cap,
                    void* ws, size_t ws_bytes, void* stream);

/* Same as sparcml_topk_ef, plus a profiling hook: `events` is a host array
 * of 4 cudaEvent_t (entries may be NULL; the array itself may be NULL),
 * recorded on `stream` before the table upload and guess kernels, before the
 * stream kernel, before the select kernels and after them, so a caller can
 * time each phase with CUDA events on the launching stream. */
int sparcml_topk_ef_traced(const float* grad, float* residual, int32_t P, uint64_t N,
                           const uint64_t* seg_begin, const uint32_t* seg_k, uint32_t nseg,
                           uint32_t* out_idx, float* out_val, uint32_t* out_nnz, uint64_t cap,
                           void* ws, size_t ws_bytes, void* stream, void* const* events);

/* Diagnostic: synchronises `stream`, then returns how many (node, segment)
 * pairs the last sparcml_topk_ef call made with workspace `ws` decided by
 * re-reading the segment (the raw select), because its sampled guess did not
 * leave enough candidates, a candidate sub-slot overflowed or the boundary
 * bin was too large; -1 on a CUDA error. The results are the same either
 * way; a count above zero on ordinary data means lost speed, not accuracy. */
int64_t sparcml_topk_ef_fallbacks(const void* ws, void* stream);

/* Capacity a stream needs for a table: the sum of seg_k (0 for NULL). */
uint64_t sparcml_topk_total_k(const uint32_t* seg_k, uint32_t nseg);

/* The equal-segment table (App. A: the last segment takes the remainder):
 * segment s = [s*L, min((s+1)*L, N)) with L = min(seg_len, N), keeping
 * k_s = floor(n_s * k_num / k_den) entries (density d = k_num / k_den).
 * Returns nseg (0 for N = 0, N >= 2^32, seg_len = 0, k_den = 0 or
 * k_num > k_den) and, where the host pointers are not NULL, writes
 * seg_begin[0 .. nseg] and seg_k[0 .. nseg - 1]. */
uint32_t sparcml_topk_uniform_segments(uint64_t N, uint64_t seg_len, uint32_t k_num,
                                       uint32_t k_den, uint64_t* seg_begin, uint32_t* seg_k);

/* Convenience forms over the equal-segment table above: identical to
 * sparcml_topk_ef(_traced) called with that table. */
size_t sparcml_topk_ef_uniform_workspace_size(int32_t P, uint64_t N, uint64_t seg_len,
                                              uint32_t k_num, uint32_t k_den);
int sparcml_topk_ef_uniform(const float* grad, float* residual, int32_t P, uint64_t N,
                            uint64_t seg_len, uint32_t k_num, uint32_t k_den,
                            uint32_t* out_idx, float* out_val, uint32_t* out_nnz, uint64_t cap,
                            void* ws, size_t ws_bytes, void* stream);
int sparcml_topk_ef_uniform_traced(const float* grad, float* residual, int32_t P, uint64_t N,
                                   uint64_t seg_len, uint32_t k_num, uint32_t k_den,
                                   uint32_t* out_idx, float* out_val, uint32_t* out_nnz,
                                   uint64_t cap, void* ws, size_t ws_bytes, void* stream,
                                   void* const* events);

/* ------------------------------------------------------------------------
 * Pack a naturally sparse dense batch into streams (§5.1): node p's stream
 * holds every i with |x[p][i]| > thr, ascending (thr = 0 keeps nonzeros;
 * -0.0 is not kept). thr must be >= 0 and not NaN.
 * If a node has more than cap such entries, its first cap (lowest indices)
 * are written, out_nnz[p] = cap and SPARCML_ERR_CAPACITY is recorded in the
 * workspace status word.
 *   x [P][N] fp32;  out_* as above;  ws >= sparcml_pack_workspace_size(P, N).
 * ------------------------------------------------------------------------ */
size_t sparcml_pack_workspace_size(int32_t P, uint64_t N);
int sparcml_pack(const float* x, int32_t P, uint64_t N, float thr, uint32_t* out_idx,
                 float* out_val, uint32_t* out_nnz, uint64_t cap, void* ws,
                 size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * 4-bit stochastic quantisation of stream values (QSGD-style, §2.2 and §6;
 * the pages give 2/4/8-bit outputs and buckets with one full-precision
 * scale each).
 *
 * Node p's entries are cut into buckets of `bucket` consecutive stream
 * entries (the last may be short). scale = max |val| over the bucket (fp32).
 * For each entry with value v and index i:
 *     r     = (|v| / scale) * 7            (fp32, RN, no contraction)
 *     level = floor(r) + (u < r - floor(r)),  clamped to 7;  level = 0 if
 *             scale == 0
 *     u     = (h >> 40) * 2^-24,  h = sm(sm(sm(seed) ^ p) ^ i)
 * where sm(x) is one SplitMix64 output for state x (x + 0x9e3779b97f4a7c15
 * through the SplitMix64 finaliser). code = (v < 0 ? 8 : 0) | level, two
 * codes per byte, the even entry in the low nibble.
 *   idx, val, nnz  input streams [P][cap], [P][cap], [P].
 *   bucket   entries per bucket, even, >= 2.
 *   codes    [P][ceil(cap/2)] bytes: bytes past ceil(nnz[p]/2) untouched.
 *   scales   [P][ceil(cap/bucket)] fp32: entries past the last bucket
 *            untouched.
 *   status   device int32 status word (may be NULL): records
 *            SPARCML_ERR_CAPACITY if some nnz[p] > cap (that node is
 *            treated as having cap entries).
 * ------------------------------------------------------------------------ */
int sparcml_quantize4(const uint32_t* idx, const float* val, const uint32_t* nnz,
                      int32_t P, uint64_t cap, uint32_t bucket, uint64_t seed,
                      uint8_t* codes, float* scales, int32_t* status, void* stream);

/* Inverse map: val_out[p][j] = (code & 8 ? -1 : 1) * (level / 7.0f) * scale,
 * with level / 7.0f rounded to fp32 first and level 0 giving +0.0f.
 * val_out [P][cap]; entries past nnz[p] untouched. */
int sparcml_dequantize4(const uint8_t* codes, const float* scales, const uint32_t* nnz,
                        int32_t P, uint64_t cap, uint32_t bucket, float* val_out,
                        int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * b-bit stochastic quantisation, b in {2, 4, 8} (§6: QSGD with 2-, 4- and
 * 8-bit outputs; §2.2 zero-mean noise), of stream values or of dense rows
 * (for example the dense reduced result, quantised before it is shared as
 * in the second half of DSAR, §6). The 4-bit form of sparcml_quantize4
 * with s = 2^(b-1) - 1 levels (1, 7, 127):
 *     r     = (|v| / scale) * s            (fp32, RN, no contraction)
 *     level = floor(r) + (u < r - floor(r)),  clamped to s;  0 if scale == 0
 *     code  = (v < 0) << (b-1) | level,  8/b codes per byte, the earliest
 *             entry of the byte in its lowest bits
 * with u and the SplitMix64 key as in sparcml_quantize4.
 *   idx      [P][cap] stream indices, or NULL for dense rows: the rounding
 *            key of entry j is then j itself.
 *   val      [P][cap] values.
 *   nnz      [P] entries per row, or NULL: every row holds cap entries.
 *   bucket   entries per bucket, >= 1, a multiple of 8/b.
 *   codes    [P][ceil(cap / (8/b))] bytes; scales [P][ceil(cap/bucket)].
 *   err_out  [P][cap] or NULL: receives v - dequantised(v) (one fp32 RN
 *            subtraction) per entry, for quantisation-error feedback.
 *   status   as for sparcml_quantize4.
 * SPARCML_ERR_INVALID_ARG for another b or a bucket that splits a byte.
 * ------------------------------------------------------------------------ */
int sparcml_quantize(const uint32_t* idx, const float* val, const uint32_t* nnz, int32_t P,
                     uint64_t cap, uint32_t bucket, uint32_t bits, uint64_t seed,
                     uint8_t* codes, float* scales, float* err_out, int32_t* status,
                     void* stream);

/* Inverse map of sparcml_quantize: val_out[p][j] = +-(level / s) * scale,
 * level / s rounded to fp32 first, level 0 giving +0.0f. nnz may be NULL
 * (full rows). Entries past nnz[p] untouched. */
int sparcml_dequantize(const uint8_t* codes, const float* scales, const uint32_t* nnz,
                       int32_t P, uint64_t cap, uint32_t bucket, uint32_t bits, float* val_out,
                       int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Sparse sum-reduction of P streams with the adaptive dense switch
 * (§5.2 sum with neutral element 0; §5.1 / §5.3.3 switch to dense; the
 * result size U is the size of the index union, App. B).
 *
 * For every index i in the union of the P streams:
 *     out[i] = ((+0.0f + v_p0) + v_p1) + ...   over the nodes p0 < p1 < ...
 *              that hold i, in ascending node order (fp32 RN adds).
 * U = number of distinct indices. The result is dense iff
 *     U * dens_den > N * dens_num          (dens_num/dens_den = 1/4: > 25%)
 * Sparse result: out_idx/out_val [0, U) ascending; out_dense holds
 * unspecified values (it may be used as scratch).
 * Dense result: out_dense [N] holds out[i], +0.0f where no node has i;
 * out_idx/out_val hold unspecified values.
 * *out_nnz = U and *out_is_dense = 0/1 in both cases (device scalars).
 *   P        1 .. 4,096 (above: SPARCML_ERR_INVALID_ARG, and the workspace
 *            size function returns 0); cap < 2^32.
 *   out_cap  capacity of out_idx/out_val, >= floor(N * dens_num / dens_den)
 *            (enough for any sparse result).
 *   ws       >= sparcml_sparse_reduce_workspace_size(P, N) bytes.
 * Streams must be strictly ascending with indices < N; otherwise
 * SPARCML_ERR_BAD_STREAM is recorded in the workspace and the outputs are
 * unspecified (all memory accesses stay in bounds).
 * ------------------------------------------------------------------------ */
size_t sparcml_sparse_reduce_workspace_size(int32_t P, uint64_t N);
int sparcml_sparse_reduce(const uint32_t* idx, const float* val, const uint32_t* nnz,
                          int32_t P, uint64_t cap, uint64_t N, uint32_t dens_num,
                          uint32_t dens_den, uint32_t* out_idx, float* out_val,
                          uint64_t out_cap, float* out_dense, uint32_t* out_nnz,
                          int32_t* out_is_dense, void* ws, size_t ws_bytes, void* stream);

/* Same as sparcml_sparse_reduce, plus a profiling hook: `events` is a host
 * array of 3 cudaEvent_t (entries may be NULL), recorded on `stream` before
 * the split and tile kernels, between them and the finishing kernel (dense
 * fix-up or compaction), and after it. */
int sparcml_sparse_reduce_traced(const uint32_t* idx, const float* val, const uint32_t* nnz,
                                 int32_t P, uint64_t cap, uint64_t N, uint32_t dens_num,
                                 uint32_t dens_den, uint32_t* out_idx, float* out_val,
                                 uint64_t out_cap, float* out_dense, uint32_t* out_nnz,
                                 int32_t* out_is_dense, void* ws, size_t ws_bytes, void* stream,
                                 void* const* events);

/* Same reduction with another coordinate-wise associative operation that
 * has a neutral element (§5.2). A stream stands for the vector holding the
 * neutral element at its unlisted indices; for every index in the union,
 *     out[i] = e op v_p0 op v_p1 op ...   (nodes p0 < p1 < ... holding i)
 * with
 *     SPARCML_OP_SUM 0  a + b (fp32 RN)                       e = +0.0f
 *     SPARCML_OP_MAX 1  b if b > a else a (ties keep a)       e = -inf
 *     SPARCML_OP_MIN 2  b if b < a else a (ties keep a)       e = +inf
 *     SPARCML_OP_OR  3  bitwise or of the fp32 bit patterns   e = +0.0f
 * U, the dense switch, layouts and error behaviour as in
 * sparcml_sparse_reduce; a dense result holds e where no node has the
 * index. op = SPARCML_OP_SUM is sparcml_sparse_reduce. Another op value:
 * SPARCML_ERR_INVALID_ARG. */
#define SPARCML_OP_SUM 0
#define SPARCML_OP_MAX 1
#define SPARCML_OP_MIN 2
#define SPARCML_OP_OR 3
int sparcml_sparse_reduce_op(const uint32_t* idx, const float* val, const uint32_t* nnz,
                             int32_t P, uint64_t cap, uint64_t N, int32_t op, uint32_t dens_num,
                             uint32_t dens_den, uint32_t* out_idx, float* out_val,
                             uint64_t out_cap, float* out_dense, uint32_t* out_nnz,
                             int32_t* out_is_dense, void* ws, size_t ws_bytes, void* stream);

/* Same reduction, with each stream's values given in the 4-bit form of
 * sparcml_quantize4 (codes, scales, bucket) and decoded on load exactly as
 * sparcml_dequantize4 does. Bit-identical to dequantize4 followed by
 * sparcml_sparse_reduce. */
int sparcml_sparse_reduce_q4(const uint32_t* idx, const uint8_t* codes, const float* scales,
                             const uint32_t* nnz, int32_t P, uint64_t cap, uint32_t bucket,
                             uint64_t N, uint32_t dens_num, uint32_t dens_den,
                             uint32_t* out_idx, float* out_val, uint64_t out_cap,
                             float* out_dense, uint32_t* out_nnz, int32_t* out_is_dense,
                             void* ws, size_t ws_bytes, void* stream);

/* Same reduction with values in the b-bit form of sparcml_quantize (b in
 * {2, 4, 8}; codes, scales, bucket as there), decoded on load exactly as
 * sparcml_dequantize does: bit-identical to sparcml_dequantize followed by
 * sparcml_sparse_reduce. bits = 4 is sparcml_sparse_reduce_q4. */
int sparcml_sparse_reduce_qb(const uint32_t* idx, const uint8_t* codes, const float* scales,
                             const uint32_t* nnz, int32_t P, uint64_t cap, uint32_t bucket,
                             uint32_t bits, uint64_t N, uint32_t dens_num, uint32_t dens_den,
                             uint32_t* out_idx, float* out_val, uint64_t out_cap,
                             float* out_dense, uint32_t* out_nnz, int32_t* out_is_dense,
                             void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Static sparse allreduce by recursive doubling (SSAR, §5.3.1), emulated on
 * one GPU. In stage s = 0 .. log2(P) - 1 each node combines its sparse
 * partial result with that of node i XOR 2^s; both get the same result, so
 * stage s keeps one partial result per group of 2^(s+1) nodes. Combining the
 * lower group's A with the upper group's B is the two-stream sum reduce:
 *     out[i] = (+0.0f + a) + b   if i is in both,   +0.0f + v otherwise.
 * The result stays sparse at every stage (no dense switch).
 *   idx, val, nnz  P input streams [P][cap] (strictly ascending, < N).
 *   P        a power of two, 2 .. 65,536; cap <= 2^31 - 1.
 *   out_idx/out_val  the final result, ascending; out_cap >=
 *            min(N, P * cap); *out_nnz = its size (device scalar).
 *   stage_nnz  device [log2 P] or NULL: entries held after each stage over
 *            its distinct partial results (the fill-in).
 *   ws       >= sparcml_ssar_workspace_size(P, cap, N) bytes, 256-aligned.
 * Device-side errors (bad stream, an expired bounded wait) go to the
 * workspace's status word (sparcml_get_status(ws, stream)).
 * ------------------------------------------------------------------------ */
size_t sparcml_ssar_workspace_size(int32_t P, uint64_t cap, uint64_t N);
int sparcml_ssar_allreduce(const uint32_t* idx, const float* val, const uint32_t* nnz, int32_t P,
                           uint64_t cap, uint64_t N, uint32_t* out_idx, float* out_val,
                           uint64_t out_cap, uint32_t* out_nnz, unsigned long long* stage_nnz,
                           void* ws, size_t ws_bytes, void* stream);

/* Same, plus a profiling hook: `events` is a host array of log2(P) + 1
 * cudaEvent_t (entries may be NULL), recorded on `stream` before each stage
 * and after the last. */
int sparcml_ssar_allreduce_traced(const uint32_t* idx, const float* val, const uint32_t* nnz,
                                  int32_t P, uint64_t cap, uint64_t N, uint32_t* out_idx,
                                  float* out_val, uint64_t out_cap, uint32_t* out_nnz,
                                  unsigned long long* stage_nnz, void* ws, size_t ws_bytes,
                                  void* stream, void* const* events);

/* ------------------------------------------------------------------------
 * Allocation-free sparse reduce. The paper has no counterpart: this entry
 * point exists for callers of this library that cannot allocate device
 * memory where they reduce (a plug-in inside a host framework that owns all
 * device memory through its own pool, or a latency-critical path where a
 * cudaMalloc would synchronise the device), so they cannot provide the
 * workspace that sparcml_sparse_reduce needs.
 *
 * Same arguments and results as sparcml_sparse_reduce, without ws/ws_bytes.
 * Its scratch is one fixed array compiled into the library (262,400 bytes,
 * enough for N <= SPARCML_NOALLOC_MAX_N); every GPU that loads the library
 * holds it until the process exits. The call allocates and frees nothing.
 *   - N > SPARCML_NOALLOC_MAX_N returns SPARCML_ERR_WORKSPACE and enqueues
 *     nothing.
 *   - Device-side errors go to *status (device int32, may be NULL).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture. The address is kept with the id of the
 *     context it belongs to: a call in a new context of that device (after
 *     cudaDeviceReset, say) looks it up again.
 *   - All calls share the array: calls whose work can overlap on the GPU
 *     (different streams, different host threads) race and must be
 *     serialised by the caller. Each call clears what must start at zero.
 * ------------------------------------------------------------------------ */
#define SPARCML_NOALLOC_MAX_N (1ull << 27)
int sparcml_sparse_reduce_noalloc(const uint32_t* idx, const float* val, const uint32_t* nnz,
                                  int32_t P, uint64_t cap, uint64_t N, uint32_t dens_num,
                                  uint32_t dens_den, uint32_t* out_idx, float* out_val,
                                  uint64_t out_cap, float* out_dense, uint32_t* out_nnz,
                                  int32_t* out_is_dense, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Densify (§5.1 representation switch): dense[p][i] = val of node p's
 * entry with index i, +0.0f where the stream has none. dense [P][N].
 * Entries with idx >= N are skipped and SPARCML_ERR_BAD_STREAM is recorded
 * in *status (may be NULL). Duplicate indices: one of them wins.
 * ------------------------------------------------------------------------ */
int sparcml_densify(const uint32_t* idx, const float* val, const uint32_t* nnz, int32_t P,
                    uint64_t cap, uint64_t N, float* dense, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Checked mode for inputs (the pages define no behaviour for non-finite
 * gradients or values: every operation above passes NaN and inf through by
 * its rules, e.g. a NaN key ranks above every finite one in Top-k). A caller
 * that wants such inputs flagged scans them first: SPARCML_ERR_NONFINITE is
 * recorded in *status if any of x[0 .. n) is a NaN or +-inf.
 *   x       device fp32 array, any 4-byte alignment (16-byte aligned arrays
 *           are read with 128-bit loads); n = 0 checks nothing.
 *   status  device int32 status word (e.g. a workspace head), required.
 * Stream-ordered and non-blocking like every other call; read the result
 * with sparcml_get_status.
 * ------------------------------------------------------------------------ */
int sparcml_check_finite(const float* x, uint64_t n, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARCML_H */
