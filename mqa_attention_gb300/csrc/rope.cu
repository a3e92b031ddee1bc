// HBM-bound row kernels around the attention main kernels:
//   * the RoPE cos/sin table (built once per (S, D, theta) in fp64, stored fp32),
//   * the abs-max pass that fixes the backward's power-of-two fp16 scales,
//   * the RoPE pre-pass that rotates q and k rows (bf16 for the forward; for the
//     backward bf16-rounded, scaled and stored fp16, fused with the fp16 copies of
//     dout and v, delta_i = dout_i . out_i, lse in base 2 and the zeroing of the
//     fp32 dq accumulator),
//   * the dq finalisation dq_i = scale * R_iᵀ dq~_i.
// RoPE is the half-split rotation x*cos + rotate_half(x)*sin with
// rotate_half(x) = cat(-x2, x1) and inverse frequencies theta^(-2i/D)
// ("Picotron模型实现解析Llama架构与Flash Attention集成", §1 嵌入层与位置编码;
//  "ColossalAI 中的 PaLM 教学实现…", §2.3 RotaryEmbedding), or, in the interleaved
// mode, the rotation of the complex pairs x_2i + j x_2i+1 by the same angles
// ("深度学习系统设计llama3-from-scratch：并行计算架构", §RoPE).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "rope_math.cuh"

namespace gbattn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSitePrep = 60;  // status-word site of the pre-pass's wait
// index checks of the debug build
constexpr int kChkPrepIn = 61, kChkPrepOut = 62, kChkPrepTab = 63, kChkFinal = 64;

// cos and sin of p * theta^(-2i/D), p < S, i < D/2, evaluated in fp64 and stored as
// fp32 pairs: hi = fp32(x), lo = fp32(x - hi), so that hi + lo carries about 48
// significant bits of the fp64 value. The four arrays [S][D/2] are cos hi, sin hi,
// cos lo, sin lo, n = S*D/2 floats apart.
__global__ void rope_table_kernel(float* __restrict__ tab, long long n, int S, int D,
                                  double theta) {
  gb::pdl_wait();  // the previous kernel in the stream has completed
  gb::pdl_launch_dependents();
  const int half = D / 2;
  const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (idx >= (long long)S * half) return;
  const int p = static_cast<int>(idx / half);
  const int i = static_cast<int>(idx % half);
  const double inv_freq = pow(theta, -2.0 * i / static_cast<double>(D));
  double sv, cv;
  sincos(static_cast<double>(p) * inv_freq, &sv, &cv);
  const float ch = static_cast<float>(cv), sh = static_cast<float>(sv);
  tab[idx] = ch;
  tab[n + idx] = sh;
  tab[2 * n + idx] = static_cast<float>(cv - static_cast<double>(ch));
  tab[3 * n + idx] = static_cast<float>(sv - static_cast<double>(sh));
}

struct alignas(16) Vec8x16 {
  uint32_t w[4];
};

__device__ __forceinline__ void load8(const float* p, float (&o)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void store8(float* p, const float (&o)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(o[0], o[1], o[2], o[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(o[4], o[5], o[6], o[7]);
}
__device__ __forceinline__ void load8_bf16(const void* p, float (&o)[8]) {
  const Vec8x16 x = *reinterpret_cast<const Vec8x16*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.w[i]));
    o[2 * i] = f.x;
    o[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void store8_bf16(void* p, const float (&o)[8]) {
  Vec8x16 x;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
    x.w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<Vec8x16*>(p) = x;
}
// Rounds to bf16 (nearest even), multiplies by the power of two s (exact) and
// stores as fp16 (exact while the result is a normal fp16 number).
__device__ __forceinline__ void store8_bf16_scaled_f16(void* p, const float (&o)[8], float s) {
  Vec8x16 x;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = __bfloat162float(__float2bfloat16_rn(o[2 * i])) * s;
    const float b = __bfloat162float(__float2bfloat16_rn(o[2 * i + 1])) * s;
    __half2 h = __floats2half2_rn(a, b);
    x.w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<Vec8x16*>(p) = x;
}

// Largest |x| of bf16 tensors. For a non-negative bf16 value the bit pattern
// orders like the value, so the maximum is taken on the 15-bit magnitudes of
// packed pairs (__vmaxu2) and converted back to float once per CTA. The CTAs are
// shared out among the tensors in proportion to their sizes; each reads one
// contiguous slab of its tensor, eight 16-byte loads in flight per thread.
constexpr int kAbsMaxThreads = 256;
constexpr int kAbsMaxUnroll = 8;

__global__ void __launch_bounds__(kAbsMaxThreads) absmax_kernel(const AbsMaxParams p) {
  gb::pdl_wait();  // the previous kernel in the stream has completed
  gb::pdl_launch_dependents();
  __shared__ uint32_t red[kAbsMaxThreads / 32];
  const int blk = static_cast<int>(blockIdx.x);
  // the CTA's tensor t (selected without indexing the parameter arrays at run time)
  const int t = blk >= p.blk0[3] ? 3 : blk >= p.blk0[2] ? 2 : blk >= p.blk0[1] ? 1 : 0;
  auto pick = [t](auto a0, auto a1, auto a2, auto a3) {
    return t == 0 ? a0 : t == 1 ? a1 : t == 2 ? a2 : a3;
  };
  const long long chunks = pick(p.n[0], p.n[1], p.n[2], p.n[3]) / 8;
  const int b0 = pick(p.blk0[0], p.blk0[1], p.blk0[2], p.blk0[3]);
  const int b1 = pick(p.blk0[1], p.blk0[2], p.blk0[3], p.blk0[4]);
  const long long per = (chunks + (b1 - b0) - 1) / (b1 - b0);
  const long long lo = (blk - b0) * per;
  const long long hi = lo + per < chunks ? lo + per : chunks;
  const uint4* src = static_cast<const uint4*>(pick(p.x[0], p.x[1], p.x[2], p.x[3]));
  uint32_t acc = 0u;
  for (long long c0 = lo + threadIdx.x; c0 < hi; c0 += kAbsMaxThreads * kAbsMaxUnroll) {
    uint4 v[kAbsMaxUnroll];
#pragma unroll
    for (int u = 0; u < kAbsMaxUnroll; ++u) {
      const long long c = c0 + u * kAbsMaxThreads;
      v[u] = c < hi ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kAbsMaxUnroll; ++u)
      acc = __vmaxu2(acc, __vmaxu2(__vmaxu2(v[u].x & 0x7fff7fffu, v[u].y & 0x7fff7fffu),
                                   __vmaxu2(v[u].z & 0x7fff7fffu, v[u].w & 0x7fff7fffu)));
  }
  uint32_t m = max(acc & 0xffffu, acc >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0u;
    for (int w = 0; w < kAbsMaxThreads / 32; ++w) b = max(b, red[w]);
    // bf16 magnitude bits -> float bits; non-negative floats order like their bits
    atomicMax(reinterpret_cast<unsigned int*>(p.maxes + t), b << 16);
  }
}

// Rotation pairs per thread of the row pre-pass (its table entries are loaded once).
constexpr int kRopePairs = 4;

template <int N>
struct alignas(4 * N) Bf16xN {  // N bf16 / fp16 values
  uint32_t w[N / 2];
};
template <int N>
__device__ __forceinline__ void storen_bf16(void* p, const float (&o)[N]) {
  Bf16xN<N> x;
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
    x.w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<Bf16xN<N>*>(p) = x;
}
// Rounds to bf16 (nearest even), multiplies by the power of two s (exact) and stores
// as fp16 (exact while the result is a normal fp16 number).
template <int N>
__device__ __forceinline__ void storen_bf16_scaled_f16(void* p, const float (&o)[N], float s) {
  Bf16xN<N> x;
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const float a = __bfloat162float(__float2bfloat16_rn(o[2 * i])) * s;
    const float b = __bfloat162float(__float2bfloat16_rn(o[2 * i + 1])) * s;
    __half2 h = __floats2half2_rn(a, b);
    x.w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<Bf16xN<N>*>(p) = x;
}
__device__ __forceinline__ void load4(const float* p, float (&o)[4]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
}
__device__ __forceinline__ void zero4(float* p) {
  *reinterpret_cast<float4*>(p) = make_float4(0.f, 0.f, 0.f, 0.f);
}

// The default row pre-pass: one thread per (output row, c) with c < D/16 and the two
// 8-element groups of rope_off_a / rope_off_b, the rotation in fp32 with the table's
// hi parts (rope_rotate16) and one rounding to bf16. Rows [0, seg[0].rows) are query
// rows, the next seg[1].rows are key rows; a segment's outputs hold Sp rows per head,
// of which the first S are its input rows (the rest, when the sequence is padded to
// whole tiles, are written as rows that contribute nothing, as above).
template <int D, bool kBwd, bool kPad>
__global__ void __launch_bounds__(256) row_prep_kernel(const RowPrepParams p) {
  gb::pdl_wait();  // the previous kernel in the stream has completed
  gb::pdl_launch_dependents();
  if (p.zero_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *p.zero_word = 0;
  constexpr int T = D / 16;  // threads per row
  constexpr int H = D / 2;
  const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long grow = t / T;
  const int c = static_cast<int>(t % T);
  const bool is_q = grow < p.seg[0].rows;
  const RowSegment& sg = is_q ? p.seg[0] : p.seg[1];
  const long long row0 = is_q ? grow : grow - p.seg[0].rows;
  // Threads past the last row read row 0 of the segment (a valid address), take
  // part in the shuffles below and write nothing.
  bool live = row0 < sg.rows;
  // output row, its head and row within the head (rows < 2^31: 32-bit division)
  const unsigned ro32 = live ? static_cast<unsigned>(row0) : 0u;
  const unsigned head = ro32 / static_cast<unsigned>(sg.Sp);
  const int i = static_cast<int>(ro32 - head * static_cast<unsigned>(sg.Sp));
  const long long ro = ro32;
  const bool real = !kPad || i < sg.S;  // kPad = false: every output row is an input row
  long long ri =  // input row
      !kPad ? ro : (real ? static_cast<long long>(head) * sg.S + i : 0);
  int pos = sg.pos0 + (real ? i : 0);
  {
    const long long in_rows = kPad ? (sg.rows / sg.Sp) * sg.S : sg.rows;
    // (threads past the last row read row 0 on purpose and write nothing)
    const bool ok = gb::bounds_ok(!live || ri < in_rows, p.status, kChkPrepIn) &&
                    gb::bounds_ok(!live || pos < p.tab_rows, p.status, kChkPrepTab);
    if (!ok) {  // read row 0 and position 0 instead, write nothing
      ri = 0;
      pos = 0;
      live = false;
    }
  }
  const bool inter = p.rope_interleaved != 0;
  const int oa = rope_off_a(c, inter), ob = rope_off_b(c, D, inter);
  const long long e1 = ri * D + oa, e2 = ri * D + ob;  // input elements
  const long long f1 = ro * D + oa, f2 = ro * D + ob;  // output elements
  const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float x1[8], x2[8], cs[8], sn[8], y1[8], y2[8];
  load8_bf16(static_cast<const __nv_bfloat16*>(sg.x) + e1, x1);
  load8_bf16(static_cast<const __nv_bfloat16*>(sg.x) + e2, x2);
  load8(p.cos_tab + (long long)pos * H + 8 * c, cs);
  load8(p.sin_tab + (long long)pos * H + 8 * c, sn);
  rope_rotate16(x1, x2, cs, sn, inter, 1.f, y1, y2);
  if (!real) {
#pragma unroll
    for (int k = 0; k < 8; ++k) y1[k] = y2[k] = 0.f;
  }
  if constexpr (!kBwd) {
    if (live) {
      store8_bf16(static_cast<__nv_bfloat16*>(sg.y) + f1, y1);
      store8_bf16(static_cast<__nv_bfloat16*>(sg.y) + f2, y2);
      if (sg.y2 != nullptr) {  // padded copy of v (key rows)
        float a1[8], a2[8];
        load8_bf16(static_cast<const __nv_bfloat16*>(sg.x2) + e1, a1);
        load8_bf16(static_cast<const __nv_bfloat16*>(sg.x2) + e2, a2);
        if (!real) {
#pragma unroll
          for (int k = 0; k < 8; ++k) a1[k] = a2[k] = 0.f;
        }
        store8_bf16(static_cast<__nv_bfloat16*>(sg.y2) + f1, a1);
        store8_bf16(static_cast<__nv_bfloat16*>(sg.y2) + f2, a2);
      }
    }
  } else {
    const BwdExponents ex = bwd_exponents(p.maxes);
    const float s_rot = exp2i(is_q ? ex.q : ex.k);
    const float s_x2 = exp2i(is_q ? ex.dout : ex.v);
    float a1[8], a2[8];
    load8_bf16(static_cast<const __nv_bfloat16*>(sg.x2) + e1, a1);
    load8_bf16(static_cast<const __nv_bfloat16*>(sg.x2) + e2, a2);
    if (!real) {
#pragma unroll
      for (int k = 0; k < 8; ++k) a1[k] = a2[k] = 0.f;
    }
    if (live) {
      store8_bf16_scaled_f16(static_cast<__half*>(sg.y) + f1, y1, s_rot);
      store8_bf16_scaled_f16(static_cast<__half*>(sg.y) + f2, y2, s_rot);
      // x2 is already bf16: scaling by a power of two and storing fp16 is exact
      store8_bf16_scaled_f16(static_cast<__half*>(sg.y2) + f1, a1, s_x2);
      store8_bf16_scaled_f16(static_cast<__half*>(sg.y2) + f2, a2, s_x2);
    }
    // delta for query rows, unless the exact delta pass writes it (out is then null:
    // the same for every thread). Every thread computes it and takes part in the
    // shuffle (a warp may straddle the query/key boundary); key rows read row 0 of
    // `out` and write nothing.
    float dot = 0.f;
    if (p.out != nullptr) {
      float o1[8], o2[8];
      const long long eo = is_q ? 0 : ri * D;
      load8_bf16(static_cast<const __nv_bfloat16*>(p.out) + (e1 - eo), o1);
      load8_bf16(static_cast<const __nv_bfloat16*>(p.out) + (e2 - eo), o2);
#pragma unroll
      for (int k = 0; k < 8; ++k) dot += a1[k] * o1[k] + a2[k] * o2[k];
#pragma unroll
      for (int o = T / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    }
    if (!is_q && live && p.dk_zero != nullptr && i < p.dk_zero_rows) {
      store8(p.dk_zero + f1, z);
      store8(p.dk_zero + f2, z);
      store8(p.dv_zero + f1, z);
      store8(p.dv_zero + f2, z);
    }
    if (is_q && live) {
      if (c == 0) {
        if (p.out != nullptr) p.delta[ro] = real ? dot * exp2i(ex.dout + ex.v) : 0.f;
        p.lse2[ro] = real ? p.lse[ri] * kLog2e : INFINITY;
      }
      store8(p.dqacc + f1, z);
      store8(p.dqacc + f2, z);
    }
  }
}

// The row pre-pass streams its rows through shared memory. One CTA per SM takes a
// contiguous range of items, an item being kBlockRows positions of kBlockHeads heads of
// one segment. A producer warp keeps the next items' rows in flight with bulk copies
// into a ring of stages (mbarriers with byte counts), so that the bytes in flight are
// held in shared memory, not registers, and the table rows of a position block are
// loaded once for every head group of those positions (two table slots). Sixteen compute
// warps rotate kRopePairs pairs of one row per thread at a time from shared memory and
// store the results with coalesced 8-byte stores.
constexpr int kBlockRows = 16;
constexpr int kBlockHeads = 4;
constexpr int kPrepCompute = 512;                 // compute threads (16 warps)
constexpr int kPrepThreads = kPrepCompute + 32;   // + the producer warp

template <int D, bool kBwd>
struct PrepCfg {
  static constexpr int H = D / 2;
  static constexpr int kTabFloats = kBlockRows * H;        // one table array's block
  static constexpr int kTabBytes = 4 * kTabFloats * 4;     // cos hi, sin hi, cos lo, sin lo
  static constexpr int kTensors = kBwd ? 3 : 2;            // row blocks an item holds at most
  static constexpr int kRowElems = kBlockRows * D;         // one head's rows of an item
  static constexpr int kLseOff = kTensors * kBlockHeads * kRowElems * 2;
  static constexpr int kStageBytes = kLseOff + (kBwd ? kBlockHeads * kBlockRows * 4 : 0);
  static constexpr int kStagesFit = (220 * 1024 - 2 * kTabBytes) / kStageBytes;
  static constexpr int kStages = kStagesFit > 6 ? 6 : kStagesFit;
  static constexpr int kSmemBytes = 2 * kTabBytes + kStages * kStageBytes + 128;
  static_assert(kStages >= 2, "row pre-pass ring");
};

struct PrepItem {
  int seg, p0, h0, nh, nrows, nreal;
};
template <bool kPad>
__device__ __forceinline__ PrepItem prep_item(const RowPrepParams& p, long long n, long long n0,
                                              int ng0, int ng1) {
  PrepItem it;
  it.seg = n < n0 ? 0 : 1;
  const RowSegment& sg = p.seg[it.seg];
  const long long m = it.seg ? n - n0 : n;
  const int ng = it.seg ? ng1 : ng0;
  it.p0 = static_cast<int>(m / ng) * kBlockRows;
  it.h0 = static_cast<int>(m % ng) * kBlockHeads;
  const int heads = static_cast<int>(sg.rows / sg.Sp);
  it.nh = min(kBlockHeads, heads - it.h0);
  it.nrows = min(kBlockRows, sg.Sp - it.p0);  // the last block of a head may be short
  // input rows that exist (the rest of a padded head is written as zeros)
  it.nreal = !kPad ? it.nrows : max(0, min(it.nrows, sg.S - it.p0));
  return it;
}

// The exact-rotation row pre-pass (RowPrepParams::exact): query rows (segment 0) and
// key rows (segment 1) of one call, each output row the rotated input row of its head
// and position, rounded to bf16 as the exact rotation rounds (rope_rotate_fast). A
// segment's outputs hold Sp rows per head, of which the first S are its input rows;
// when the sequence is padded to whole tiles the rest are written as rows that
// contribute nothing (zero operands, delta 0 and, in the backward, lse * log2 e = +inf
// so that their probabilities are 0).
template <int D, bool kBwd, bool kPad>
__global__ void __launch_bounds__(kPrepThreads, 1) row_prep_exact_kernel(const RowPrepParams p) {
  using C = PrepCfg<D, kBwd>;
  constexpr int NP = kRopePairs;
  constexpr int T = D / (2 * NP);  // threads per row
  constexpr int H = D / 2;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar_full[C::kStages], bar_empty[C::kStages];
  __shared__ __align__(8) uint64_t bar_tab_full[2], bar_tab_empty[2];
  __shared__ int abort_flag;
  float* tabs = reinterpret_cast<float*>(smem);                    // [2][4][R][H]
  uint8_t* stages = smem + 2 * C::kTabBytes;                       // [kStages][kStageBytes]
  volatile int* abort_ptr = &abort_flag;

  // items: segment 0 then 1, position blocks then head groups; this CTA's range
  const int ng0 = p.seg[0].rows ? static_cast<int>((p.seg[0].rows / p.seg[0].Sp + kBlockHeads - 1) / kBlockHeads) : 0;
  const int ng1 = p.seg[1].rows ? static_cast<int>((p.seg[1].rows / p.seg[1].Sp + kBlockHeads - 1) / kBlockHeads) : 0;
  const long long n0 = p.seg[0].rows ? static_cast<long long>((p.seg[0].Sp + kBlockRows - 1) / kBlockRows) * ng0 : 0;
  const long long n1 = p.seg[1].rows ? static_cast<long long>((p.seg[1].Sp + kBlockRows - 1) / kBlockRows) * ng1 : 0;
  const long long nall = n0 + n1;
  const long long first = nall * blockIdx.x / gridDim.x;
  const long long last = nall * (blockIdx.x + 1) / gridDim.x;
  const bool dot = kBwd && p.out != nullptr;  // delta from out (query rows)

  const int tid = threadIdx.x;
  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < C::kStages; ++i) {
      gb::mbar_init(gb::smem_u32(&bar_full[i]), 1);
      gb::mbar_init(gb::smem_u32(&bar_empty[i]), kPrepCompute);
    }
    for (int i = 0; i < 2; ++i) {
      gb::mbar_init(gb::smem_u32(&bar_tab_full[i]), 1);
      gb::mbar_init(gb::smem_u32(&bar_tab_empty[i]), kPrepCompute);
    }
    gb::fence_mbar_init();
  }
  __syncthreads();
  gb::pdl_wait();  // the previous kernel in the stream has completed
  gb::pdl_launch_dependents();
  if (p.zero_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *p.zero_word = 0;

  if (tid >= kPrepCompute) {
    // ================================================================ producer
    if (tid == kPrepCompute) {
      int tgen = -1, pseg = -1, pp0 = -1;
      long long issued = 0;
      for (long long n = first; n < last; ++n) {
        const PrepItem it = prep_item<kPad>(p, n, n0, ng0, ng1);
        const RowSegment& sg = p.seg[it.seg];
        if (it.seg != pseg || it.p0 != pp0) {  // a new position block: its table rows
          ++tgen;
          const int ts = tgen & 1;
          if (!gb::bounded_wait(gb::smem_u32(&bar_tab_empty[ts]), ((tgen >> 1) & 1) ^ 1, abort_ptr,
                                p.status, kSitePrep))
            break;
          const uint32_t tb = static_cast<uint32_t>(it.nrows) * H * 4;
          const uint32_t full = gb::smem_u32(&bar_tab_full[ts]);
          gb::mbar_arrive_expect_tx(full, 4 * tb);
          const long long te = static_cast<long long>(sg.pos0 + it.p0) * H;
          const float* src[4] = {p.cos_tab, p.sin_tab, p.cos_lo, p.sin_lo};
          if (gb::bounds_ok(sg.pos0 + it.p0 + it.nrows <= p.tab_rows, p.status, kChkPrepTab))
            for (int a = 0; a < 4; ++a)
              gb::bulk_load(gb::smem_u32(tabs + (ts * 4 + a) * C::kTabFloats), src[a] + te, tb, full);
          pseg = it.seg;
          pp0 = it.p0;
        }
        const int st = static_cast<int>(issued % C::kStages);
        if (!gb::bounded_wait(gb::smem_u32(&bar_empty[st]), ((issued / C::kStages) & 1) ^ 1,
                              abort_ptr, p.status, kSitePrep))
          break;
        const bool q = it.seg == 0;
        const bool x2_in = kBwd || sg.y2 != nullptr;
        const int ntens = 1 + (x2_in ? 1 : 0) + (dot && q ? 1 : 0);
        const bool lse_in = kBwd && q && !kPad;  // lse rows (padded: read in the loop)
        const uint32_t rb = static_cast<uint32_t>(it.nreal) * D * 2;
        const uint32_t lb = lse_in ? static_cast<uint32_t>(it.nreal) * 4 : 0u;
        const uint32_t full = gb::smem_u32(&bar_full[st]);
        gb::mbar_arrive_expect_tx(full, static_cast<uint32_t>(it.nh) * (ntens * rb + lb));
        uint8_t* stg = stages + st * C::kStageBytes;
        const void* src[3] = {sg.x, x2_in ? sg.x2 : p.out, p.out};
        const long long in_rows = (sg.rows / sg.Sp) * (kPad ? sg.S : sg.Sp);
        if (rb > 0) {
          for (int k = 0; k < it.nh; ++k) {
            const long long r = static_cast<long long>(it.h0 + k) * (kPad ? sg.S : sg.Sp) + it.p0;
            if (!gb::bounds_ok(r + it.nreal <= in_rows, p.status, kChkPrepIn)) continue;
            for (int m = 0; m < ntens; ++m)
              gb::bulk_load(gb::smem_u32(stg + ((m * kBlockHeads + k) * C::kRowElems) * 2),
                            static_cast<const __nv_bfloat16*>(src[m]) + r * D, rb, full);
            if (lb > 0)
              gb::bulk_load(gb::smem_u32(stg + C::kLseOff + k * kBlockRows * 4), p.lse + r, lb,
                            full);
          }
        }
        ++issued;
      }
      // copies already issued land before the CTA releases its shared memory
      for (long long i = issued - C::kStages > 0 ? issued - C::kStages : 0; i < issued; ++i) {
        const uint64_t t0 = gb::globaltimer_ns();
        while (!gb::mbar_try_wait(gb::smem_u32(&bar_full[i % C::kStages]), (i / C::kStages) & 1) &&
               gb::globaltimer_ns() - t0 < gb::kWaitLimitNs / 4) {
        }
      }
    }
    return;
  }

  // ================================================================ compute warps
  BwdExponents ex{0, 0, 0, 0};
  if constexpr (kBwd) ex = bwd_exponents(p.maxes);
  const bool inter = p.rope_interleaved != 0;
  const int c = tid % T;
  const int oa = rope_off_a_n<NP>(c, inter), ob = rope_off_b_n<NP>(c, D, inter);
  const unsigned lane = tid & 31u;
  const unsigned row_mask = ((1u << T) - 1u) << (lane & ~static_cast<unsigned>(T - 1));
  auto lds = [](const __nv_bfloat16* q, float (&o)[NP]) {  // NP bf16 values from shared memory
    const Bf16xN<NP> v = *reinterpret_cast<const Bf16xN<NP>*>(q);
#pragma unroll
    for (int e = 0; e < NP / 2; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.w[e]));
      o[2 * e] = f.x;
      o[2 * e + 1] = f.y;
    }
  };
  int tgen = -1, pseg = -1, pp0 = -1;
  long long used = 0;
  for (long long n = first; n < last; ++n) {
    const PrepItem it = prep_item<kPad>(p, n, n0, ng0, ng1);
    const RowSegment& sg = p.seg[it.seg];
    const bool q = it.seg == 0;
    if (it.seg != pseg || it.p0 != pp0) {
      if (tgen >= 0) gb::mbar_arrive(gb::smem_u32(&bar_tab_empty[tgen & 1]));
      ++tgen;
      if (!gb::bounded_wait(gb::smem_u32(&bar_tab_full[tgen & 1]), (tgen >> 1) & 1, abort_ptr,
                            p.status, kSitePrep))
        break;
      pseg = it.seg;
      pp0 = it.p0;
    }
    const int st = static_cast<int>(used % C::kStages);
    if (!gb::bounded_wait(gb::smem_u32(&bar_full[st]), (used / C::kStages) & 1, abort_ptr, p.status,
                          kSitePrep))
      break;
    const float* tab = tabs + (tgen & 1) * 4 * C::kTabFloats;
    const uint8_t* stg = stages + st * C::kStageBytes;
    const __nv_bfloat16* xs = reinterpret_cast<const __nv_bfloat16*>(stg);
    const bool x2_in = kBwd || sg.y2 != nullptr;
    const float s_rot = exp2i(q ? ex.q : ex.k);
    const float s_x2 = exp2i(q ? ex.dout : ex.v);
#pragma unroll 1
    for (int row = tid / T; row < it.nh * kBlockRows; row += kPrepCompute / T) {
      const int k = row / kBlockRows, il = row % kBlockRows;
      if (il >= it.nrows) continue;
      const int i = it.p0 + il;  // row within the head
      const bool real = il < it.nreal;
      const long long ro = static_cast<long long>(it.h0 + k) * sg.Sp + i;  // output row
      if (!gb::bounds_ok(ro < sg.rows, p.status, kChkPrepOut)) continue;
      const long long f1 = ro * D + oa, f2 = ro * D + ob;
      float chi[NP], clo[NP], shi[NP], slo[NP];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float4 v = *reinterpret_cast<const float4*>(tab + a * C::kTabFloats + il * H + NP * c);
        float* dst = a == 0 ? chi : a == 1 ? shi : a == 2 ? clo : slo;
        dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
      }
      const __nv_bfloat16* xr = xs + k * C::kRowElems + il * D;
      float x1[NP], x2[NP], y1[NP], y2[NP], a1[NP], a2[NP];
      if (real) {
        lds(xr + oa, x1);
        lds(xr + ob, x2);
        if (x2_in) {
          lds(xr + kBlockHeads * C::kRowElems + oa, a1);
          lds(xr + kBlockHeads * C::kRowElems + ob, a2);
        }
      } else {
#pragma unroll
        for (int e = 0; e < NP; ++e) x1[e] = x2[e] = a1[e] = a2[e] = 0.f;
      }
      rope_rotate_fast<NP>(x1, x2, chi, clo, shi, slo, inter, y1, y2);
      if constexpr (!kBwd) {
        storen_bf16<NP>(static_cast<__nv_bfloat16*>(sg.y) + f1, y1);
        storen_bf16<NP>(static_cast<__nv_bfloat16*>(sg.y) + f2, y2);
        if (sg.y2 != nullptr) {  // padded copy of v (key rows)
          storen_bf16<NP>(static_cast<__nv_bfloat16*>(sg.y2) + f1, a1);
          storen_bf16<NP>(static_cast<__nv_bfloat16*>(sg.y2) + f2, a2);
        }
      } else {
        storen_bf16_scaled_f16<NP>(static_cast<__half*>(sg.y) + f1, y1, s_rot);
        storen_bf16_scaled_f16<NP>(static_cast<__half*>(sg.y) + f2, y2, s_rot);
        // x2 is already bf16: scaling by a power of two and storing fp16 is exact
        storen_bf16_scaled_f16<NP>(static_cast<__half*>(sg.y2) + f1, a1, s_x2);
        storen_bf16_scaled_f16<NP>(static_cast<__half*>(sg.y2) + f2, a2, s_x2);
        if (q) {
          // delta_i = dout_i . out_i (unless the exact delta pass writes it instead)
          if (dot) {
            float o1[NP], o2[NP];
            if (real) {
              lds(xr + 2 * kBlockHeads * C::kRowElems + oa, o1);
              lds(xr + 2 * kBlockHeads * C::kRowElems + ob, o2);
            } else {
#pragma unroll
              for (int e = 0; e < NP; ++e) o1[e] = o2[e] = 0.f;
            }
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < NP; ++e) d += a1[e] * o1[e] + a2[e] * o2[e];
#pragma unroll
            for (int o = T / 2; o > 0; o >>= 1) d += __shfl_xor_sync(row_mask, d, o);
            if (c == 0) p.delta[ro] = d * exp2i(ex.dout + ex.v);
          }
          if (c == 0) {
            float l = INFINITY;
            if (real) {
              if constexpr (kPad)
                l = p.lse[static_cast<long long>(it.h0 + k) * sg.S + i];
              else
                l = reinterpret_cast<const float*>(stg + C::kLseOff)[k * kBlockRows + il];
              l *= kLog2e;
            }
            p.lse2[ro] = l;
          }
          zero4(p.dqacc + f1);
          zero4(p.dqacc + f2);
        } else if (p.dk_zero != nullptr && i < p.dk_zero_rows) {
          zero4(p.dk_zero + f1);
          zero4(p.dk_zero + f2);
          zero4(p.dv_zero + f1);
          zero4(p.dv_zero + f2);
        }
      }
    }
    gb::mbar_arrive(gb::smem_u32(&bar_empty[st]));
    ++used;
  }
  if (tgen >= 0) gb::mbar_arrive(gb::smem_u32(&bar_tab_empty[tgen & 1]));
}

// dq in fp32, or rounded to bf16 (nearest even) when kBf16.
template <int D, bool kBf16>
__global__ void __launch_bounds__(256)
    dq_finalize_kernel(const float* __restrict__ dqacc, void* __restrict__ dq, long long rows,
                       int S, int Sp, int pos0, float scale, const float* __restrict__ maxes,
                       const float* __restrict__ cos_tab, const float* __restrict__ sin_tab,
                       int tab_rows, int rope_interleaved, int* status) {
  gb::pdl_wait();  // the previous kernel in the stream has completed
  gb::pdl_launch_dependents();
  constexpr int T = D / 16;
  constexpr int H = D / 2;
  const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long row = t / T;
  if (row >= rows) return;
  const int c = static_cast<int>(t % T);
  // dq row `row` (S rows per head); its accumulator row has Sp rows per head
  // (rows < 2^31: 32-bit division)
  const unsigned head = static_cast<unsigned>(row) / static_cast<unsigned>(S);
  const int i = static_cast<int>(static_cast<unsigned>(row) - head * static_cast<unsigned>(S));
  const int pos = pos0 + i;
  if (!gb::bounds_ok(pos < tab_rows, status, kChkFinal)) return;
  const bool inter = rope_interleaved != 0;
  const long long racc = static_cast<long long>(head) * Sp + i;
  const long long e1 = row * D + rope_off_a(c, inter);
  const long long e2 = row * D + rope_off_b(c, D, inter);
  const long long a1 = racc * D + rope_off_a(c, inter);
  const long long a2 = racc * D + rope_off_b(c, D, inter);
  const BwdExponents ex = bwd_exponents(maxes);
  const float f = scale * exp2i(-(ex.dout + ex.v + ex.k));
  float x1[8], x2[8], cs[8], sn[8], y1[8], y2[8];
  load8(dqacc + a1, x1);
  load8(dqacc + a2, x2);
  load8(cos_tab + (long long)pos * H + 8 * c, cs);
  load8(sin_tab + (long long)pos * H + 8 * c, sn);
  rope_rotate16(x1, x2, cs, sn, inter, -1.f, y1, y2);  // transpose: rotation by -angle
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    y1[i] *= f;
    y2[i] *= f;
  }
  if constexpr (kBf16) {
    store8_bf16(static_cast<__nv_bfloat16*>(dq) + e1, y1);
    store8_bf16(static_cast<__nv_bfloat16*>(dq) + e2, y2);
  } else {
    store8(static_cast<float*>(dq) + e1, y1);
    store8(static_cast<float*>(dq) + e2, y2);
  }
}

// Merge of two partial attention results over disjoint key sets of the same
// query rows: lse = ln(e^lse_a + e^lse_b), out = e^(lse_a - lse) out_a +
// e^(lse_b - lse) out_b (a row with lse_a = lse_b = -inf gets out = 0, lse = -inf).
// One thread per 8 elements of a row; the D/8 threads of a row share a warp and
// read everything before any of them writes, so out / lse may be out_a / lse_a.
template <int D>
__global__ void __launch_bounds__(256)
    merge_kernel(const void* oa, const float* la, const void* ob, const float* lb, void* o,
                 float* l, long long rows) {
  gb::pdl_wait();  // the previous kernel in the stream has completed
  gb::pdl_launch_dependents();
  constexpr int T = D / 8;
  const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long row = t / T;
  const int c = static_cast<int>(t % T);
  const bool live = row < rows;
  const long long rr = live ? row : 0;
  const float a = la[rr], b = lb[rr];
  float xa[8], xb[8];
  load8_bf16(static_cast<const __nv_bfloat16*>(oa) + rr * D + 8 * c, xa);
  load8_bf16(static_cast<const __nv_bfloat16*>(ob) + rr * D + 8 * c, xb);
  __syncwarp();
  if (!live) return;
  const float m = fmaxf(a, b);
  float wa = 0.f, wb = 0.f, lse = -INFINITY;
  if (m != -INFINITY) {
    wa = expf(a - m);
    wb = expf(b - m);
    const float sum = wa + wb;
    lse = m + logf(sum);
    wa /= sum;
    wb /= sum;
  }
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = wa * xa[i] + wb * xb[i];
  store8_bf16(static_cast<__nv_bfloat16*>(o) + row * D + 8 * c, y);
  if (c == 0) l[row] = lse;
}

// Rows of a padded layout (Sp rows per head) to the unpadded one (S rows per
// head): dst[h*S + i] = src[h*Sp + i], i < S, rows of `words` 4-byte words; with
// to_bf16, fp32 rows become bf16 rows (nearest even) of words/2 words.
__global__ void __launch_bounds__(256)
    unpad_rows_kernel(const uint32_t* __restrict__ src, uint32_t* __restrict__ dst, long long rows,
                      int S, int Sp, int words, int to_bf16) {
  gb::pdl_wait();  // the previous kernel in the stream has completed
  gb::pdl_launch_dependents();
  const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const int per_row = to_bf16 ? words / 2 : words;
  const long long row = t / per_row;
  if (row >= rows) return;
  const int w = static_cast<int>(t % per_row);
  const long long srow = (row / S) * Sp + row % S;
  if (to_bf16) {
    const float a = __uint_as_float(src[srow * words + 2 * w]);
    const float b = __uint_as_float(src[srow * words + 2 * w + 1]);
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    dst[row * per_row + w] = *reinterpret_cast<uint32_t*>(&h);
  } else {
    dst[row * per_row + w] = src[srow * words + w];
  }
}

// y = bf16(x), nearest even; n a multiple of 8.
__global__ void __launch_bounds__(256)
    f32_to_bf16_kernel(const float* __restrict__ x, void* __restrict__ y, long long n8) {
  gb::pdl_wait();  // the previous kernel in the stream has completed
  gb::pdl_launch_dependents();
  const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (t >= n8) return;
  float v[8];
  load8(x + 8 * t, v);
  store8_bf16(static_cast<__nv_bfloat16*>(y) + 8 * t, v);
}

long long blocks_for(long long threads) { return (threads + 255) / 256; }

}  // namespace

cudaError_t launch_rope_table(float* tab, long long n, int S, int D, double theta,
                              cudaStream_t stream) {
  const long long cnt = (long long)S * (D / 2);
  return launch_pdl(rope_table_kernel, dim3((unsigned)blocks_for(cnt)), dim3(256), 0, stream, tab,
                    n, S, D, theta);
}

cudaError_t launch_absmax(const AbsMaxParams& p_in, cudaStream_t stream) {
  // About 8 CTAs per SM over all tensors, at least one per present tensor and
  // none for an absent one (its slab is empty).
  AbsMaxParams p = p_in;
  long long total = 0;
  for (int t = 0; t < 4; ++t) total += p.x[t] ? p.n[t] : 0;
  const long long want = 152 * 8;
  p.blk0[0] = 0;
  for (int t = 0; t < 4; ++t) {
    long long nb = 0;
    if (p.x[t] && p.n[t] > 0) {
      nb = total > 0 ? (want * p.n[t] + total - 1) / total : 1;
      nb = nb < 1 ? 1 : nb;
    }
    p.blk0[t + 1] = p.blk0[t] + static_cast<int>(nb);
  }
  if (p.blk0[4] == 0) return cudaSuccess;
  return launch_pdl(absmax_kernel, dim3(static_cast<unsigned>(p.blk0[4])), dim3(kAbsMaxThreads),
                    0, stream, p);
}

// Zeroes n <= 32 words (the abs-max pass's maxima) as a launch of its own: a memset
// node between two kernels would hold back the abs-max pass's programmatic early start.
__global__ void zero_words_kernel(uint32_t* __restrict__ w, int n) {
  gb::pdl_wait();  // the previous kernel in the stream has completed
  gb::pdl_launch_dependents();
  if (static_cast<int>(threadIdx.x) < n) w[threadIdx.x] = 0u;
}

cudaError_t launch_zero_words(void* w, int n, cudaStream_t stream) {
  if (n <= 0 || n > 32) return cudaErrorInvalidValue;
  return launch_pdl(zero_words_kernel, dim3(1), dim3(32), 0, stream, static_cast<uint32_t*>(w), n);
}

cudaError_t launch_row_prep(const RowPrepParams& p, cudaStream_t stream) {
  const bool pad = p.seg[0].S != p.seg[0].Sp || p.seg[1].S != p.seg[1].Sp;
  if (!p.exact) {
    const long long threads = (p.seg[0].rows + p.seg[1].rows) * (p.D / 16);
    if (threads == 0) return cudaSuccess;
    const unsigned grid = (unsigned)blocks_for(threads);
#define GB_PREP(DD, BW, PD) \
  return launch_pdl(row_prep_kernel<DD, BW, PD>, dim3(grid), dim3(256), 0, stream, p)
    if (p.D == 128) {
      if (p.bwd) { if (pad) GB_PREP(128, true, true); else GB_PREP(128, true, false); }
      else { if (pad) GB_PREP(128, false, true); else GB_PREP(128, false, false); }
    } else {
      if (p.bwd) { if (pad) GB_PREP(64, true, true); else GB_PREP(64, true, false); }
      else { if (pad) GB_PREP(64, false, true); else GB_PREP(64, false, false); }
    }
#undef GB_PREP
  }
  auto items = [](const RowSegment& sg) {
    if (sg.rows == 0) return 0LL;
    const long long heads = sg.rows / sg.Sp;
    return static_cast<long long>((sg.Sp + kBlockRows - 1) / kBlockRows) *
           ((heads + kBlockHeads - 1) / kBlockHeads);
  };
  const long long n = items(p.seg[0]) + items(p.seg[1]);
  if (n == 0) return cudaSuccess;
  int dev = 0, nsm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(n < nsm ? n : nsm);  // one CTA per SM
#define GB_PREP(DD, BW, PD)                                                                     \
  do {                                                                                          \
    constexpr int smem = PrepCfg<DD, BW>::kSmemBytes;                                           \
    e = cudaFuncSetAttribute(row_prep_exact_kernel<DD, BW, PD>,                                 \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);                \
    if (e != cudaSuccess) return e;                                                             \
    return launch_pdl(row_prep_exact_kernel<DD, BW, PD>, dim3(grid), dim3(kPrepThreads), smem,  \
                      stream, p);                                                               \
  } while (0)
  if (p.D == 128) {
    if (p.bwd) { if (pad) GB_PREP(128, true, true); else GB_PREP(128, true, false); }
    else { if (pad) GB_PREP(128, false, true); else GB_PREP(128, false, false); }
  } else {
    if (p.bwd) { if (pad) GB_PREP(64, true, true); else GB_PREP(64, true, false); }
    else { if (pad) GB_PREP(64, false, true); else GB_PREP(64, false, false); }
  }
#undef GB_PREP
}

cudaError_t launch_dq_finalize(const float* dqacc, void* dq, bool dq_bf16, long long rows, int S,
                               int Sp, int pos0, int D, float scale, const float* maxes, const float* cos_tab,
                               const float* sin_tab, int tab_rows, int rope_interleaved,
                               int* status, cudaStream_t stream) {
  const long long threads = rows * (D / 16);
  const unsigned grid = (unsigned)blocks_for(threads);
#define GB_FIN(DD, BF)                                                                       \
  return launch_pdl(dq_finalize_kernel<DD, BF>, dim3(grid), dim3(256), 0, stream, dqacc, dq, rows, \
                    S, Sp, pos0, scale, maxes, cos_tab, sin_tab, tab_rows, rope_interleaved, status)
  if (D == 128) {
    if (dq_bf16) GB_FIN(128, true);
    else GB_FIN(128, false);
  } else {
    if (dq_bf16) GB_FIN(64, true);
    else GB_FIN(64, false);
  }
#undef GB_FIN
}

cudaError_t launch_merge(const void* oa, const float* la, const void* ob, const float* lb, void* o,
                         float* l, long long rows, int D, cudaStream_t stream) {
  const unsigned grid = (unsigned)blocks_for(rows * (D / 8));
  if (D == 128) return launch_pdl(merge_kernel<128>, dim3(grid), dim3(256), 0, stream, oa, la, ob, lb, o, l, rows);
  return launch_pdl(merge_kernel<64>, dim3(grid), dim3(256), 0, stream, oa, la, ob, lb, o, l, rows);
}

cudaError_t launch_unpad_rows(const void* src, void* dst, long long rows, int S, int Sp, int words,
                              bool to_bf16, cudaStream_t stream) {
  const long long n = rows * (to_bf16 ? words / 2 : words);
  if (n == 0) return cudaSuccess;
  return launch_pdl(unpad_rows_kernel, dim3((unsigned)blocks_for(n)), dim3(256), 0, stream,
                    static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst), rows, S, Sp,
                    words, to_bf16 ? 1 : 0);
}

cudaError_t launch_f32_to_bf16(const float* x, void* y, long long n, cudaStream_t stream) {
  const long long n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  return launch_pdl(f32_to_bf16_kernel, dim3((unsigned)blocks_for(n8)), dim3(256), 0, stream, x, y,
                    n8);
}

}  // namespace gbattn
