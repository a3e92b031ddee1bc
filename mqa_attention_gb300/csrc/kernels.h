// Internal interface between the C-ABI host code (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gbattn {

constexpr int kTile = 128;  // query / key tile rows of the main kernels

// RoPE cos/sin table, [S][D/2] fp32 each, built in fp64.
cudaError_t launch_rope_table(float* cos_tab, float* sin_tab, int S, int D, double theta,
                              cudaStream_t stream);

// Rotates rows of x (bf16 [rows][D], position = row % S) into y (bf16).
// When `delta` is non-null it also writes delta[row] = sum_d a[row][d] * b[row][d]
// (bf16 a, b), lse2[row] = lse[row] * log2(e), and zeroes dqacc[row][:] (fp32).
struct RowPrepParams {
  const void* x;
  void* y;
  long long rows;
  int S, D;
  const float* cos_tab;
  const float* sin_tab;
  // optional backward extras (query rows only)
  const void* a;  // out
  const void* b;  // dout
  float* delta;
  const float* lse;
  float* lse2;
  float* dqacc;
};
cudaError_t launch_row_prep(const RowPrepParams& p, cudaStream_t stream);

// dq = scale * R_iᵀ dqacc (fp32 in, fp32 out).
cudaError_t launch_dq_finalize(const float* dqacc, float* dq, long long rows, int S, int D,
                               float scale, const float* cos_tab, const float* sin_tab,
                               cudaStream_t stream);

struct FwdParams {
  CUtensorMap map_q;    // rotated q, box {64, 128}
  CUtensorMap map_k;    // rotated k, box {64, 128}
  CUtensorMap map_v;    // v, box {64, 128}
  CUtensorMap map_out;  // out, box {64, 128}
  float* lse;
  int* status;
  int B, Hq, Hkv, S, D;
  float scale_log2;  // scale * log2(e)
  int causal;
  int inject_timeout;
};
cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream);

struct BwdParams {
  CUtensorMap map_q;   // rotated q, box {64, BQ}
  CUtensorMap map_do;  // dout, box {64, BQ}
  CUtensorMap map_k;   // rotated k, box {64, 128}
  CUtensorMap map_v;   // v, box {64, 128}
  const float* lse2;   // lse * log2(e), [B*Hq*S]
  const float* delta;  // [B*Hq*S]
  float* dqacc;        // [B*Hq*S][D] fp32, accumulated with atomics
  float* dk;           // [B*Hkv*S][D] fp32
  float* dv;           // [B*Hkv*S][D] fp32
  const float* cos_tab;
  const float* sin_tab;
  int* status;
  int B, Hq, Hkv, S, D;
  float scale;
  float scale_log2;
  int causal;
  int inject_timeout;
};
// Query-tile rows used by the backward main kernel for head dimension D.
inline int bwd_query_tile(int D) { return D == 128 ? 64 : 128; }
cudaError_t launch_bwd_main(const BwdParams& p, cudaStream_t stream);

}  // namespace gbattn
