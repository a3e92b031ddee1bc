// The RoPE rotation of 8 (value, partner) pairs, shared by every kernel that
// rotates rows (the pre-passes, decode, the dq finalisation, the dk epilogue), so
// that a row rotated in two places rounds identically. The products and the fused
// adds are spelled out: a contraction chosen differently by the compiler in two
// kernels would change the last bit.
//
// Half-split ("Picotron模型实现解析Llama架构与Flash Attention集成", §1 嵌入层与位置编码;
// "ColossalAI 中的 PaLM 教学实现…", §2.3 RotaryEmbedding): pair i is (a_i, b_i) at
// frequency i, x*cos + rotate_half(x)*sin. Interleaved ("深度学习系统设计llama3-from-
// scratch：并行计算架构", §RoPE): pairs (a_2j, a_2j+1) at frequency j and
// (b_2j, b_2j+1) at 4 + j, the complex product by e^(i angle). cs / sn hold the 8
// table entries of the frequencies; sgn = 1 rotates by +angle, -1 by -angle.
//
// Rotated operands that are rounded to bf16 (q~, k~) go through the exact form
// below: the table holds each cosine and sine as an fp32 pair hi + lo (about 48
// significant bits of the fp64 value), the rotation is evaluated with error-free
// products and sums, and the result is nudged off a bf16 rounding midpoint when
// the exact value lies beside it. The bf16 value is then the one the exact
// rotation rounds to (to within about 2^-47 of a midpoint), whichever kernel
// computes it and in whatever order, and equal to rounding the fp64 rotation.
// Gradients (fp32 outputs) take the plain fp32 form with the hi parts.
#pragma once

#include <cstdint>

// One pair (a, b) rotated by the angle with cosine c and sine s (fp32).
__device__ __forceinline__ void rope_rotate_pair(float a, float b, float c, float s, float sgn,
                                                 float& ya, float& yb) {
  ya = __fmaf_rn(a, c, -sgn * __fmul_rn(b, s));
  yb = __fmaf_rn(b, c, sgn * __fmul_rn(a, s));
}

__device__ __forceinline__ void rope_rotate16(const float (&a)[8], const float (&b)[8],
                                              const float (&cs)[8], const float (&sn)[8],
                                              bool inter, float sgn, float (&ya)[8],
                                              float (&yb)[8]) {
  if (!inter) {
#pragma unroll
    for (int i = 0; i < 8; ++i) rope_rotate_pair(a[i], b[i], cs[i], sn[i], sgn, ya[i], yb[i]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      rope_rotate_pair(a[2 * j], a[2 * j + 1], cs[j], sn[j], sgn, ya[2 * j], ya[2 * j + 1]);
      rope_rotate_pair(b[2 * j], b[2 * j + 1], cs[4 + j], sn[4 + j], sgn, yb[2 * j],
                       yb[2 * j + 1]);
    }
  }
}

// x*(ch+cl) + y*(sh+sl) for bf16-valued x, y (so every product below is formed
// from exact operands), returned as an fp32 value that rounds to bf16 like the
// exact value does.
//   p1 + e1 = x*ch, p2 + e2 = y*sh exactly (products with their rounding errors);
//   s + t = p1 + p2 exactly (two-sum); tail = t + e1 + e2 + x*cl + y*sl.
// r = fl(s + tail) is within one fp32 ulp of the exact value, so a bf16 rounding
// of r can only differ from that of the exact value when r sits exactly on a bf16
// midpoint (low 16 bits 0x8000); then the residual (s - r) + tail (s - r is exact)
// says on which side the exact value lies, and r moves one fp32 ulp that way.
__device__ __forceinline__ float rope_dot2_exact(float x, float ch, float cl, float y, float sh,
                                                 float sl) {
  const float p1 = __fmul_rn(x, ch);
  const float e1 = __fmaf_rn(x, ch, -p1);
  const float p2 = __fmul_rn(y, sh);
  const float e2 = __fmaf_rn(y, sh, -p2);
  const float s = __fadd_rn(p1, p2);
  const float bb = __fsub_rn(s, p1);
  const float t = __fadd_rn(__fsub_rn(p1, __fsub_rn(s, bb)), __fsub_rn(p2, bb));
  const float tail = __fmaf_rn(x, cl, __fmaf_rn(y, sl, __fadd_rn(__fadd_rn(t, e1), e2)));
  float r = __fadd_rn(s, tail);
  const uint32_t u = __float_as_uint(r);
  if ((u & 0xffffu) == 0x8000u) {
    const float res = __fadd_rn(__fsub_rn(s, r), tail);
    if (res != 0.f) {
      // away from zero when the exact value is further from zero than r
      const bool away = (res > 0.f) == (r > 0.f);
      r = __uint_as_float(away ? u + 1u : u - 1u);
    }
  }
  return r;
}

// Packed fp32 pairs: one instruction for two lanes' worth of the same operation,
// each lane rounded as the scalar form.
__device__ __forceinline__ unsigned long long rope_pk(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void rope_upk(unsigned long long r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ unsigned long long rope_mul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long rope_fma2(unsigned long long a, unsigned long long b,
                                                      unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long rope_add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long rope_sub2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// One pair (x, y) rotated by +angle for a bf16 result, both outputs at once (lane 0:
// x cos - y sin, lane 1: y cos + x sin): the steps of rope_dot2_exact on packed lanes,
// (x, y) * (ch, ch) + (-y, x) * (sh, sh) with the lo parts in the tail, then the
// midpoint check per output.
__device__ __forceinline__ void rope_pair_exact(float x, float y, float ch, float cl, float sh,
                                                float sl, float& rx, float& ry) {
  const unsigned long long X = rope_pk(x, y);
  const unsigned long long Y = rope_pk(-y, x);
  const unsigned long long C = rope_pk(ch, ch), CL = rope_pk(cl, cl);
  const unsigned long long SN = rope_pk(sh, sh), SL = rope_pk(sl, sl);
  const unsigned long long p1 = rope_mul2(X, C);
  const unsigned long long e1 = rope_fma2(X, C, p1 ^ 0x8000000080000000ull);   // X*C - p1
  const unsigned long long p2 = rope_mul2(Y, SN);
  const unsigned long long e2 = rope_fma2(Y, SN, p2 ^ 0x8000000080000000ull);  // Y*S - p2
  const unsigned long long s = rope_add2(p1, p2);
  const unsigned long long bb = rope_sub2(s, p1);
  const unsigned long long t = rope_add2(rope_sub2(p1, rope_sub2(s, bb)), rope_sub2(p2, bb));
  const unsigned long long tail =
      rope_fma2(X, CL, rope_fma2(Y, SL, rope_add2(rope_add2(t, e1), e2)));
  const unsigned long long r = rope_add2(s, tail);
  float r0, r1;
  rope_upk(r, r0, r1);
  const uint32_t u0 = __float_as_uint(r0), u1 = __float_as_uint(r1);
  if (((u0 & 0xffffu) == 0x8000u) | ((u1 & 0xffffu) == 0x8000u)) {
    // an output on a bf16 midpoint: the residual (s - r) + tail says on which side
    // of it the exact value lies (rare: about 2^-16 of the outputs)
    float s0, s1, t0, t1;
    rope_upk(s, s0, s1);
    rope_upk(tail, t0, t1);
    auto nudge = [](float rr, float ss, float tt) {
      const uint32_t u = __float_as_uint(rr);
      if ((u & 0xffffu) != 0x8000u) return rr;
      const float res = __fadd_rn(__fsub_rn(ss, rr), tt);
      if (res == 0.f) return rr;
      const bool away = (res > 0.f) == (rr > 0.f);
      return __uint_as_float(away ? u + 1u : u - 1u);
    };
    r0 = nudge(r0, s0, t0);
    r1 = nudge(r1, s1, t1);
  }
  rx = r0;
  ry = r1;
}

// NP pairs rotated by +angle for a bf16 result: ya = a cos - b sin, yb = b cos + a sin,
// each exact up to the final rounding (see rope_dot2_exact); the caller rounds to bf16
// (nearest even). c_hi/c_lo, s_hi/s_lo: the NP table entries as hi + lo pairs.
// Half-split: pair i is (a_i, b_i) at frequency i; interleaved: (a_2j, a_2j+1) at j and
// (b_2j, b_2j+1) at NP/2 + j.
template <int NP>
__device__ __forceinline__ void rope_rotate_exact(const float (&a)[NP], const float (&b)[NP],
                                                  const float (&c_hi)[NP], const float (&c_lo)[NP],
                                                  const float (&s_hi)[NP], const float (&s_lo)[NP],
                                                  bool inter, float (&ya)[NP], float (&yb)[NP]) {
  if (!inter) {
#pragma unroll
    for (int i = 0; i < NP; ++i)
      rope_pair_exact(a[i], b[i], c_hi[i], c_lo[i], s_hi[i], s_lo[i], ya[i], yb[i]);
  } else {
    constexpr int H = NP / 2;
#pragma unroll
    for (int j = 0; j < H; ++j) {
      rope_pair_exact(a[2 * j], a[2 * j + 1], c_hi[j], c_lo[j], s_hi[j], s_lo[j], ya[2 * j],
                      ya[2 * j + 1]);
      rope_pair_exact(b[2 * j], b[2 * j + 1], c_hi[H + j], c_lo[H + j], s_hi[H + j], s_lo[H + j],
                      yb[2 * j], yb[2 * j + 1]);
    }
  }
}

__device__ __forceinline__ void rope_rotate16_exact(const float (&a)[8], const float (&b)[8],
                                                    const float (&c_hi)[8], const float (&c_lo)[8],
                                                    const float (&s_hi)[8], const float (&s_lo)[8],
                                                    bool inter, float (&ya)[8], float (&yb)[8]) {
  rope_rotate_exact<8>(a, b, c_hi, c_lo, s_hi, s_lo, inter, ya, yb);
}

// The same result at the cost of the plain fp32 rotation for almost every pair: y =
// fl(x c_hi - fl(y s_hi)) differs from the exact value by less than 2^-22 (|x| + |y|)
// (two roundings of at most 2^-24 of a magnitude below |x| + |y|, and the hi parts'
// own error, 2^-24 of a value below 1, times |x| and |y|). When neither output of the
// pair lies within 2^-21 (|x| + |y|) of a bf16 rounding midpoint (low 16 bits 0x8000),
// the exact value rounds to bf16 like the plain one; otherwise (about 1 pair in 10^4)
// the pair is recomputed exactly (rope_pair_exact).
__device__ __forceinline__ bool rope_far_from_midpoint(float r, float t) {
  const float mid = __uint_as_float((__float_as_uint(r) & 0xffff0000u) | 0x8000u);
  return fabsf(__fsub_rn(r, mid)) > t;
}
__device__ __forceinline__ void rope_pair_fast(float x, float y, float ch, float cl, float sh,
                                               float sl, float& rx, float& ry) {
  const float px = __fmaf_rn(x, ch, -__fmul_rn(y, sh));
  const float py = __fmaf_rn(y, ch, __fmul_rn(x, sh));
  const float t = __fmul_rn(__fadd_rn(fabsf(x), fabsf(y)), 4.76837158203125e-7f);  // 2^-21
  if (rope_far_from_midpoint(px, t) & rope_far_from_midpoint(py, t)) {
    rx = px;
    ry = py;
  } else {
    rope_pair_exact(x, y, ch, cl, sh, sl, rx, ry);
  }
}

// rope_rotate_exact's result through rope_pair_fast.
template <int NP>
__device__ __forceinline__ void rope_rotate_fast(const float (&a)[NP], const float (&b)[NP],
                                                 const float (&c_hi)[NP], const float (&c_lo)[NP],
                                                 const float (&s_hi)[NP], const float (&s_lo)[NP],
                                                 bool inter, float (&ya)[NP], float (&yb)[NP]) {
  if (!inter) {
#pragma unroll
    for (int i = 0; i < NP; ++i)
      rope_pair_fast(a[i], b[i], c_hi[i], c_lo[i], s_hi[i], s_lo[i], ya[i], yb[i]);
  } else {
    constexpr int H = NP / 2;
#pragma unroll
    for (int j = 0; j < H; ++j) {
      rope_pair_fast(a[2 * j], a[2 * j + 1], c_hi[j], c_lo[j], s_hi[j], s_lo[j], ya[2 * j],
                     ya[2 * j + 1]);
      rope_pair_fast(b[2 * j], b[2 * j + 1], c_hi[H + j], c_lo[H + j], s_hi[H + j], s_lo[H + j],
                     yb[2 * j], yb[2 * j + 1]);
    }
  }
}

// Element offsets (within a row) of the two NP-element groups of chunk c < D/(2 NP):
// half-split [NP c, NP c + NP) and [D/2 + NP c, +NP); interleaved [2 NP c, +NP) and
// [2 NP c + NP, +NP). Both use the table entries [NP c, NP c + NP) of the row's position.
template <int NP>
__device__ __forceinline__ int rope_off_a_n(int c, bool inter) { return inter ? 2 * NP * c : NP * c; }
template <int NP>
__device__ __forceinline__ int rope_off_b_n(int c, int D, bool inter) {
  return inter ? 2 * NP * c + NP : D / 2 + NP * c;
}

// Element offsets (within a row) of the two 8-element groups of chunk c < D/16:
// half-split [8c, 8c+8) and [D/2 + 8c, +8); interleaved [16c, 16c+8) and
// [16c+8, 16c+16). Both use the table entries [8c, 8c+8) of the row's position.
__device__ __forceinline__ int rope_off_a(int c, bool inter) { return inter ? 16 * c : 8 * c; }
__device__ __forceinline__ int rope_off_b(int c, int D, bool inter) {
  return inter ? 16 * c + 8 : D / 2 + 8 * c;
}
