// The RoPE rotation of 8 (value, partner) pairs, shared by every kernel that
// rotates rows (the pre-passes, the forward's in-kernel rotation of its Q tiles,
// decode, the dq finalisation), so that a row rotated in two places rounds
// identically. The products and the fused add are spelled out: a contraction
// chosen differently by the compiler in two kernels would change the last bit.
//
// Half-split ("Picotron模型实现解析Llama架构与Flash Attention集成", §1 嵌入层与位置编码;
// "ColossalAI 中的 PaLM 教学实现…", §2.3 RotaryEmbedding): pair i is (a_i, b_i) at
// frequency i, x*cos + rotate_half(x)*sin. Interleaved ("深度学习系统设计llama3-from-
// scratch：并行计算架构", §RoPE): pairs (a_2j, a_2j+1) at frequency j and
// (b_2j, b_2j+1) at 4 + j, the complex product by e^(i angle). cs / sn hold the 8
// table entries of the frequencies; sgn = 1 rotates by +angle, -1 by -angle.
#pragma once

// One pair (a, b) rotated by the angle with cosine c and sine s.
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

// Element offsets (within a row) of the two 8-element groups of chunk c < D/16:
// half-split [8c, 8c+8) and [D/2 + 8c, +8); interleaved [16c, 16c+8) and
// [16c+8, 16c+16). Both use the table entries [8c, 8c+8) of the row's position.
__device__ __forceinline__ int rope_off_a(int c, bool inter) { return inter ? 16 * c : 8 * c; }
__device__ __forceinline__ int rope_off_b(int c, int D, bool inter) {
  return inter ? 16 * c + 8 : D / 2 + 8 * c;
}
