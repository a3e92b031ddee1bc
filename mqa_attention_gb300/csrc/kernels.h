// Internal interface between the C-ABI host code (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

namespace gbattn {

// Launches `kernel` with programmatic stream serialisation: its grid may be scheduled
// while the kernel before it in the stream is still running. Every kernel launched
// this way calls gb::pdl_wait() before its first global-memory access, which blocks
// until that kernel has completed and its writes are visible.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kTile = 128;  // query / key tile rows of the main kernels

// ---------------------------------------------------------------- fp16 scaling
// The backward runs its tensor-core products in fp16 (2^-11 relative
// rounding of P and dS instead of bf16's 2^-9). Each fp16 operand tensor is
// multiplied by an exact power of two chosen from the tensor's largest
// magnitude, so that nothing overflows and the scaling adds no rounding:
//   q~, k~ : largest |value| below 2^14   (|R x| <= sqrt(2) max|x|)
//   v, dO  : largest |value| below 2^3, so |dP| <= 64 D and |dS| <= 128 D < 2^15.
// Index of each tensor's maximum in the 4-float array written by the
// abs-max pass.
enum { kMaxQ = 0, kMaxK = 1, kMaxV = 2, kMaxDO = 3 };
constexpr int kTargetQK = 14;
constexpr int kTargetVDO = 3;
constexpr int kMaxScaleExp = 40;

// Exponent e (|e| <= kMaxScaleExp) with m * 2^e < 2^target for a finite m >= 0.
__host__ __device__ inline int pow2_exponent(float m, int target) {
  uint32_t bits;
  memcpy(&bits, &m, 4);
  const int ex = static_cast<int>((bits >> 23) & 0xffu);
  int e;
  if (ex == 255) e = 0;                       // inf / nan: outputs are non-finite anyway
  else if (ex == 0) e = kMaxScaleExp;         // zero or subnormal maximum
  else e = target - (ex - 126);               // m < 2^(ex - 126)
  return e < -kMaxScaleExp ? -kMaxScaleExp : (e > kMaxScaleExp ? kMaxScaleExp : e);
}
// 2^e as a float, |e| <= 126.
__host__ __device__ inline float exp2i(int e) {
  const uint32_t bits = static_cast<uint32_t>(127 + e) << 23;
  float f;
  memcpy(&f, &bits, 4);
  return f;
}
struct BwdExponents {
  int q, k, v, dout;
};
__host__ __device__ inline BwdExponents bwd_exponents(const float* maxes) {
  BwdExponents x;
  x.q = pow2_exponent(maxes[kMaxQ] * 1.4142136f, kTargetQK);
  x.k = pow2_exponent(maxes[kMaxK] * 1.4142136f, kTargetQK);
  x.v = pow2_exponent(maxes[kMaxV], kTargetVDO);
  x.dout = pow2_exponent(maxes[kMaxDO], kTargetVDO);
  return x;
}

// Device address of the library's status word on the current device (a static device
// variable: looking it up allocates nothing). Returns an ATTN_* code.
int device_status_word(int** out);

// ---------------------------------------------------------------- row kernels
// RoPE table for positions 0..S-1: four fp32 arrays [S][D/2], n floats apart (n >=
// S*D/2): cos hi, sin hi, cos lo, sin lo, where hi + lo is the fp64 value to about
// 48 significant bits (hi alone: the fp64 value rounded to fp32).
cudaError_t launch_rope_table(float* tab, long long n, int S, int D, double theta,
                              cudaStream_t stream);

// Largest |value| of up to four bf16 tensors, atomically max-ed into maxes[i]
// (which the caller zeroes first).
struct AbsMaxParams {
  const void* x[4];
  long long n[4];  // element counts, multiples of 8
  float* maxes;
  int blk0[5];     // CTAs [blk0[t], blk0[t+1]) read tensor t (set by launch_absmax)
};
cudaError_t launch_absmax(const AbsMaxParams& p, cudaStream_t stream);
cudaError_t launch_zero_words(void* w, int n, cudaStream_t stream);  // n <= 32

// Row pre-pass over the query rows (segment 0) and key rows (segment 1) of one
// call, in one launch. Forward (bwd == 0): y = bf16(R x) for both segments.
// Backward (bwd == 1):
//   query rows: y = fp16(bf16(R q) 2^eq), y2 = fp16(dout 2^edo),
//               delta = (dout . out) 2^(edo+ev), lse2 = lse log2(e), dqacc row = 0
//   key rows:   y = fp16(bf16(R k) 2^ek),  y2 = fp16(v 2^ev)
struct RowSegment {
  const void* x;
  void* y;
  const void* x2;  // backward: dout (query rows) or v (key rows)
  void* y2;
  long long rows;  // output rows (Sp per head)
  int S;     // input rows per head; input row h*S + i sits at position pos0 + i
  int Sp;    // output rows per head (S, or S rounded up to whole tiles)
  int pos0;
};
struct RowPrepParams {
  int bwd;
  int rope_interleaved;  // 0: half-split pairs (i, i + D/2); 1: pairs (2i, 2i + 1)
  int exact;             // 1: rotated rows rounded as the exact rotation rounds (else fp32)
  RowSegment seg[2];
  int D;
  const float* cos_tab;  // table hi parts
  const float* sin_tab;
  const float* cos_lo;   // table lo parts
  const float* sin_lo;
  int tab_rows;          // positions the table holds
  const float* maxes;  // backward
  const void* out;     // backward, query rows (null: delta is written by the delta pass)
  float* delta;
  const float* lse;
  float* lse2;
  float* dqacc;
  float* dk_zero;  // backward, key rows: zeroed when the main kernel sums dK/dV partials
  float* dv_zero;
  int dk_zero_rows;  // with dk_zero: rows [0, dk_zero_rows) of each head are zeroed
  int* status;       // device status word (a wait that expired)
  int* zero_word;    // forward: set to 0 (the next forward launch's unit counter), or null
};
cudaError_t launch_row_prep(const RowPrepParams& p, cudaStream_t stream);

// dq = scale * 2^-(edo+ev+ek) * R_iᵀ dqacc (fp32 in; fp32 out, or bf16 rounded to
// nearest even when dq_bf16); row r sits at position pos0 + r % S.
cudaError_t launch_dq_finalize(const float* dqacc, void* dq, bool dq_bf16, long long rows, int S,
                               int Sp, int pos0, int D, float scale, const float* maxes, const float* cos_tab,
                               const float* sin_tab, int tab_rows, int rope_interleaved,
                               int* status, cudaStream_t stream);
// Merge of two partial attention results of the same rows (bf16 out, fp32 lse);
// o / l may be oa / la.
cudaError_t launch_merge(const void* oa, const float* la, const void* ob, const float* lb, void* o,
                         float* l, long long rows, int D, cudaStream_t stream);
// dst[h*S + i] = src[h*Sp + i] for rows of `words` 4-byte words (rows = heads * S);
// to_bf16: fp32 source rows written as bf16 rows.
cudaError_t launch_unpad_rows(const void* src, void* dst, long long rows, int S, int Sp, int words,
                              bool to_bf16, cudaStream_t stream);
// y = bf16(x) (nearest even), n a multiple of 8.
cudaError_t launch_f32_to_bf16(const float* x, void* y, long long n, cudaStream_t stream);

// ---------------------------------------------------------------- main kernels
struct FwdParams {
  CUtensorMap map_q;    // rotated q (bf16), box {64, 128}
  CUtensorMap map_k;    // rotated k (bf16), box {64, 128}
  CUtensorMap map_v;    // v (bf16), box {64, 128}
  CUtensorMap map_out;  // out (bf16), box {64, 128}
  void* out;            // the same rows, for query tiles that see no key
  float* lse;
  int* status;
  // Query block of Sq rows per head at positions 128*q_tile0 + i; K/V block of Skv
  // rows at 128*kv_tile0 + j (self-attention: Sq = Skv = S, both tiles 0).
  int B, Hq, Hkv, Sq, Skv, D;
  int q_tile0, kv_tile0;
  int kv_valid;      // keys per head that exist (< Skv when the block is padded)
  float scale_log2;  // scale * log2(e)
  int causal;
  int inject_timeout;
  // D = 64: query tiles handed out to the persistent CTAs beyond their first (zeroed by
  // the RoPE pre-pass before the launch); null: one CTA per query tile
  int* unit_counter;
};
cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream);

constexpr int kMaxBwdPlan = 64;  // key tiles a work-order table can hold
struct BwdParams {
  CUtensorMap map_q;   // scaled rotated q (fp16), box {64, BQ}
  CUtensorMap map_do;  // scaled dout (fp16), box {64, BQ}
  CUtensorMap map_k;   // scaled rotated k (fp16), box {64, 128}
  CUtensorMap map_v;   // scaled v (fp16), box {64, 128}
  CUtensorMap map_dk;  // dk (fp32) [B*Hkv*S, D], box {32, 128}
  CUtensorMap map_dv;  // dv (fp32) [B*Hkv*S, D], box {32, 128}
  CUtensorMap map_cos; // RoPE cos table (fp32) [positions, D/2], box {32, 128}
  CUtensorMap map_sin; // RoPE sin table, the same
  CUtensorMap map_dqacc;  // D = 64: the dQ accumulator (fp32) [B*Hq*S, D], box {32, 128}
  const float* lse2;   // lse * log2(e), [B*Hq*S]
  const float* delta;  // scaled delta, [B*Hq*S]
  const float* maxes;  // the abs-max pass's four maxima
  float* dqacc;        // [B*Hq*S][D] fp32, accumulated with atomics (scaled)
  float* dk;           // [B*Hkv*S][D] fp32
  float* dv;           // [B*Hkv*S][D] fp32
  const float* cos_tab;
  const float* sin_tab;
  int tab_rows;        // positions the cos / sin tables (and their maps) hold
  int* status;
  int B, Hq, Hkv, Sq, Skv, D;  // query and K/V blocks as in FwdParams
  int q_tile0, kv_tile0;
  float scale;
  float scale_log2;
  int causal;
  int inject_timeout;
  int hsplit;  // CTAs sharing one (KV head, key tile): 1, or 2 (dK/dV summed with reductions)
  int rope_interleaved;  // rotation pairs of the dk epilogue (see RowPrepParams)
  // Work order, heaviest unit first. nplan > 0: entry e is key tile plan_kt[e] with
  // plan_parts[e] CTAs per (batch, KV head) — 1, or 2 each taking half of the group's
  // query heads and adding its dK/dV partials — and hsplit is unused. nplan = 0: key
  // tile blockIdx / (B*Hkv*hsplit), hsplit CTAs each.
  int nplan;
  short plan_kt[kMaxBwdPlan];
  signed char plan_parts[kMaxBwdPlan];
};
// Exact delta pass: delta_i = sum_j P_ij dP_ij over the visible keys of each query row,
// from the backward pre-pass's fp16 operands (self-attention, S rows per head, a
// multiple of 128). Written scaled by 2^(edo+ev), as the main kernel reads delta.
struct DeltaParams {
  CUtensorMap map_q;   // scaled rotated q (fp16), box {64, 128}
  CUtensorMap map_do;  // scaled dout (fp16), box {64, 128}
  CUtensorMap map_k;   // scaled rotated k (fp16), box {64, 128}
  CUtensorMap map_v;   // scaled v (fp16), box {64, 128}
  const float* lse2;   // lse * log2(e), [B*Hq*S] (+inf on padding rows)
  const float* maxes;  // the abs-max pass's four maxima
  float* delta;        // [B*Hq*S], written
  int* status;
  int B, Hq, Hkv, S, D;
  float scale_log2;    // scale * log2(e)
  int causal;
  int inject_timeout;
};
cudaError_t launch_delta(const DeltaParams& p, cudaStream_t stream);

// Query-tile rows used by the backward main kernel for head dimension D.
inline int bwd_query_tile(int) { return 64; }
cudaError_t launch_bwd_main(const BwdParams& p, cudaStream_t stream);

// Decode-shape forward: Sq query rows per head at positions q_pos0 + i against a
// cache of Skv rotated keys / values; chunks of tiles_per_chunk key tiles per CTA.
struct DecParams {
  CUtensorMap map_q;  // q (bf16, rotated in the kernel) rows [B*Hq*Sq, D], box {64, 128}
  CUtensorMap map_k;  // rotated key cache (bf16) rows [B*Hkv*Skv, D], box {64, 128}
  CUtensorMap map_v;  // value cache (bf16), same rows
  float* part_out;    // [nchunks][rows][D] fp32: each chunk's out (divided by its row sum)
  float* part_lse;    // [nchunks][rows]: each chunk's lse (-inf: no key seen)
  void* out;          // [rows][D] bf16
  float* lse;         // [rows]
  const float* cos_tab;  // table hi parts
  const float* sin_tab;
  const float* cos_lo;   // table lo parts
  const float* sin_lo;
  int rope_interleaved;
  int exact;             // 1: the query rows rounded as the exact rotation rounds
  int tab_rows;          // positions the table holds
  int* status;
  int B, Hq, Hkv, Sq, Skv, D;
  int q_pos0;
  int tiles_per_chunk, nchunks;
  long long rows;     // B * Hq * Sq
  float scale_log2;
};
// The chunk kernel and the merge of the chunks into out / lse.
cudaError_t launch_decode(const DecParams& p, cudaStream_t stream);

}  // namespace gbattn
