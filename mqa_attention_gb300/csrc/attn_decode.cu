// Decode-shape attention for sm_103a: a few new queries per sequence (Sq rows
// per query head) against a long key/value cache.
//
// What it computes is the forward of attn_fwd restricted to those rows: query i
// of a head sits at position q_pos0 + i and sees the cached keys at positions
// j <= q_pos0 + i (j < Skv); scores q~.k~ scale, softmax with the row maximum
// subtracted, P v ("ColossalAI 中的 PaLM 教学实现…", §2.5 Attention, where one
// shared K/V head is what makes such decoding cheap; "深度学习系统设计llama3-
// from-scratch：并行计算架构", §键值（Key-Value）共享机制).
//
// GB300 design. The work is bound by reading the cache once, so the G query
// heads that share a K/V head are packed into the rows of one 128-row MMA tile
// (G * Sq <= 128 real rows: one CTA serves the whole group and each K/V tile is
// read once), and the cache of each (batch, KV head) is split into chunks of
// key tiles spread over the SMs. Per chunk a CTA loads the group's query rows,
// rotates them in shared memory (RoPE at their positions, rounded to bf16 as the
// pre-pass of attn_fwd does), streams K~/V tiles through a TMA ring; S = Q~ K~ᵀ
// (tcgen05, two TMEM buffers so that the next score MMA runs while the softmax
// works), P (bf16, over S) and O += P V (TS MMA) as in the forward kernel, and
// writes its rows' partial out (fp32, already divided by the chunk's row sum) and
// lse. decode_merge_kernel then combines the chunks of each row by their
// log-sum-exp weights, spread over the whole GPU (merging in the last CTA of a
// K/V head instead put up to a megabyte of partial rows on one SM).
// Warp roles: 0-3 softmax (thread = tile row), 4 TMA producer, 5 MMA issuer (whole
// warp, one elected lane issues) and TMEM owner.
// TMEM: S_0 [0,128), S_1 [128,256), O [256, 256 + D).
#include "kernels.h"
#include "ptx.cuh"
#include "rope_math.cuh"

namespace gbattn {
namespace {

using namespace gb;

constexpr float kLn2 = 0.6931471805599453f;
constexpr int kThreads = 192;
constexpr int kWarpLoad = 4;
constexpr int kWarpMma = 5;

enum : int {
  kSiteQ = 41, kSiteKvFull = 42, kSiteKvEmpty = 43, kSiteSFull = 44, kSitePFull = 45,
  kSiteODone = 46, kSiteQRot = 47,
  // index checks of the debug build (a tile may end past the last row: TMA fills it)
  kChkQ = 53, kChkKv = 54, kChkTab = 55, kChkPart = 56
};

template <int D>
struct DecCfg {
  static constexpr int kRegionBytes = 128 * 128;  // 128 rows x 128 B (64 bf16)
  static constexpr int kRegions = D / 64;
  static constexpr int kTileBytes = kRegions * kRegionBytes;
  static constexpr int kSlots = D == 128 ? 6 : 12;  // K/V ring depth (tiles)
  static constexpr int kKvOff = kTileBytes;         // after the Q tile
  static constexpr int kSmemBytes = kKvOff + kSlots * kTileBytes + 1024;
  static_assert(kSmemBytes + 1024 <= 232448, "shared memory budget");
  static constexpr uint32_t kColO = 256;
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs / 4) return;
  }
}

// kExact: the Q rows are rotated with the exactly rounded rotation (ATTN_ROPE_EXACT);
// a separate instantiation, so that the default kernel's code holds none of it.
template <int D, bool kExact>
__global__ void __launch_bounds__(kThreads, 1) attn_decode_kernel(const __grid_constant__ DecParams p) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_q_rot, bar_drain, bar_o_done;
  __shared__ __align__(8) uint64_t bar_kv_full[C::kSlots], bar_kv_empty[C::kSlots];
  __shared__ __align__(8) uint64_t bar_s_full[2], bar_p_full[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;

  // ---- work item: chunk c of the cache of (batch, KV head) bhk
  const int nu = p.B * p.Hkv;
  const int c = static_cast<int>(blockIdx.x) / nu;
  const int bhk = static_cast<int>(blockIdx.x) % nu;
  const int b = bhk / p.Hkv;
  const int hkv = bhk % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int m_real = G * p.Sq;                               // real rows of the tile
  const int q_row0 = (b * p.Hq + hkv * G) * p.Sq;            // first row of the group
  const int kv_row0 = bhk * p.Skv;
  const int ntiles = (p.Skv + kTile - 1) / kTile;
  const int last_q = p.q_pos0 + p.Sq - 1;                    // largest query position
  int kt0 = c * p.tiles_per_chunk;
  int kt1 = kt0 + p.tiles_per_chunk;
  kt1 = kt1 < ntiles ? kt1 : ntiles;
  const int kt_vis = last_q / kTile + 1;                     // tiles with a visible key
  kt1 = kt1 < kt_vis ? kt1 : kt_vis;
  const int n = kt1 > kt0 ? kt1 - kt0 : 0;

  // ---- setup
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q), 1);
    mbar_init(smem_u32(&bar_q_rot), 128);
    mbar_init(smem_u32(&bar_drain), 1);
    mbar_init(smem_u32(&bar_o_done), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(smem_u32(&bar_kv_full[s]), 1);
      mbar_init(smem_u32(&bar_kv_empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bar_s_full[t]), 1);
      mbar_init(smem_u32(&bar_p_full[t]), 128);
    }
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_ptr = &abort_flag;
  // Up to here nothing touched global memory, so this prologue may overlap the grid
  // before it in the stream; the merge of this call may be scheduled from now on (it
  // waits for this grid to complete before it reads the partial results).
  pdl_wait();
  pdl_launch_dependents();

  if (warp == kWarpLoad) {
    // ================================================================ producer
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&p.map_q);
      tma_prefetch_desc(&p.map_k);
      tma_prefetch_desc(&p.map_v);
      mbar_arrive_expect_tx(smem_u32(&bar_q), C::kTileBytes);
      if (bounds_ok(q_row0 >= 0 && q_row0 < p.rows, p.status, kChkQ))
        for (int r = 0; r < C::kRegions; ++r)
          tma_load_2d(sbase + r * C::kRegionBytes, &p.map_q, r * 64, q_row0, smem_u32(&bar_q));
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        for (int w = 0; w < 2; ++w) {  // K_j, then V_j
          const int slot = issued % C::kSlots;
          const uint32_t ph = ((issued / C::kSlots) & 1) ^ 1;
          if (!bounded_wait(smem_u32(&bar_kv_empty[slot]), ph, abort_ptr, p.status, kSiteKvEmpty)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&bar_kv_full[slot]);
          mbar_arrive_expect_tx(full, C::kTileBytes);
          const CUtensorMap* map = w == 0 ? &p.map_k : &p.map_v;
          const uint32_t dst = sbase + C::kKvOff + slot * C::kTileBytes;
          const long long krow = kv_row0 + static_cast<long long>(kt0 + j) * kTile;
          if (bounds_ok(krow < static_cast<long long>(p.B) * p.Hkv * p.Skv, p.status, kChkKv))
            for (int r = 0; r < C::kRegions; ++r)
              tma_load_2d(dst + r * C::kRegionBytes, map, r * 64, kv_row0 + (kt0 + j) * kTile, full);
          ++issued;
        }
      }
      // Loads already issued land before the CTA releases its shared memory.
      drain_wait(smem_u32(&bar_q), 0);
      for (int i = issued - C::kSlots > 0 ? issued - C::kSlots : 0; i < issued; ++i)
        drain_wait(smem_u32(&bar_kv_full[i % C::kSlots]), (i / C::kSlots) & 1);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ================================================================ MMA issuer
    constexpr uint32_t idesc_qk = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16(128, D, 0, 1);
    constexpr uint64_t kKmaj = sdesc_hi(16, 1024);
    constexpr uint64_t kMnV = sdesc_hi(C::kRegionBytes, 1024);
    auto desc = [](uint64_t hi, uint32_t addr) { return hi | static_cast<uint64_t>(addr >> 4); };
    auto wait = [&](uint32_t bar, uint32_t parity, int site) {
      return __all_sync(0xffffffffu, bounded_wait(bar, parity, abort_ptr, p.status, site));
    };
    auto slot_addr = [&](int i) { return sbase + C::kKvOff + (i % C::kSlots) * C::kTileBytes; };
    auto wait_kv = [&](int i) {
      return wait(smem_u32(&bar_kv_full[i % C::kSlots]), (i / C::kSlots) & 1, kSiteKvFull);
    };
    // S_(j&1) = Q~ K_jᵀ (K_j at ring index 2j)
    auto issue_qk = [&](int j) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * C::kRegionBytes + (kk & 3) * 32;
        mma_ss_w(tmem + (j & 1) * 128, desc(kKmaj, sbase + off), desc(kKmaj, slot_addr(2 * j) + off),
                 idesc_qk, kk > 0);
      }
      mma_commit_w(smem_u32(&bar_s_full[j & 1]));
      mma_commit_w(smem_u32(&bar_kv_empty[(2 * j) % C::kSlots]));
    };
    bool ok = n > 0;
    ok = ok && wait(smem_u32(&bar_q_rot), 0, kSiteQRot);  // loaded and rotated
    for (int j = 0; j < 2 && j < n && ok; ++j) {
      ok = wait_kv(2 * j);
      if (!ok) break;
      tc_fence_after();
      issue_qk(j);
    }
    for (int j = 0; j < n && ok; ++j) {
      ok = wait(smem_u32(&bar_p_full[j & 1]), (j >> 1) & 1, kSitePFull) && wait_kv(2 * j + 1);
      if (!ok) break;
      tc_fence_after();
      const uint32_t vaddr = slot_addr(2 * j + 1);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)  // O += P_j V_j, P packed over S_(j&1)
        mma_ts_w(tmem + C::kColO, tmem + (j & 1) * 128 + kk * 8,
                 desc(kMnV, vaddr + kk * 16 * 128), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
      mma_commit_w(smem_u32(&bar_o_done));
      mma_commit_w(smem_u32(&bar_kv_empty[(2 * j + 1) % C::kSlots]));
      if (j + 2 < n) {  // after P V(j) in issue order: P_j is read before S_(j&1) is rewritten
        ok = wait_kv(2 * (j + 2));
        if (!ok) break;
        issue_qk(j + 2);
      }
    }
    // Every MMA issued above completes before the tensor memory is released.
    mma_commit_w(smem_u32(&bar_drain));
    drain_wait(smem_u32(&bar_drain), 0);
    __syncwarp();
  } else {
    // ================================================================ softmax (rows)
    const int r = tid;  // tile row == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const bool row_real = r < m_real;
    const int qpos = p.q_pos0 + (row_real ? r % p.Sq : 0);  // this row's query position
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running maximum (base 2); -inf while no key was seen
    float l = 0.f;
    bool ok = true;
    if (n > 0) {
      // ---- RoPE of this row of the Q tile, in place (128-byte swizzled rows). The
      // row's cos / sin values are loaded while the tile is in flight.
      float cv[D / 2], sv[D / 2];
      const long long trow = static_cast<long long>(qpos) * (D / 2);
      if (row_real && bounds_ok(qpos < p.tab_rows, p.status, kChkTab)) {
        const float4* cs = reinterpret_cast<const float4*>(p.cos_tab + trow);
        const float4* sn = reinterpret_cast<const float4*>(p.sin_tab + trow);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
          const float4 a = __ldg(cs + i), bq = __ldg(sn + i);
          cv[4 * i] = a.x; cv[4 * i + 1] = a.y; cv[4 * i + 2] = a.z; cv[4 * i + 3] = a.w;
          sv[4 * i] = bq.x; sv[4 * i + 1] = bq.y; sv[4 * i + 2] = bq.z; sv[4 * i + 3] = bq.w;
        }
        // exact rounding reads the lo parts group by group below: bring their lines to
        // L1 now
        if constexpr (kExact) {
#pragma unroll
          for (int i = 0; i < D / 2; i += 32) {
            asm volatile("prefetch.global.L1 [%0];" ::"l"(p.cos_lo + trow + i));
            asm volatile("prefetch.global.L1 [%0];" ::"l"(p.sin_lo + trow + i));
          }
        }
      }
      ok = __all_sync(0xffffffffu, bounded_wait(smem_u32(&bar_q), 0, abort_ptr, p.status, kSiteQ));
      if (ok && row_real) {
        uint8_t* qs = smem_raw + (sbase - smem_u32(smem_raw));
        auto chunk = [&](int col) {  // 16-byte chunk holding columns col..col+7 of row r
          return reinterpret_cast<uint4*>(qs + (col / 64) * C::kRegionBytes +
                                          sw128_offset(r, (col % 64) / 8));
        };
        auto unpack = [](uint4 v, float (&f)[8]) {
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
          }
        };
        auto pack = [](const float (&f)[8]) {
          return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                            pack_bf16(f[6], f[7]));
        };
#pragma unroll
        for (int g = 0; g < D / 16; ++g) {
          // half-split: columns [8g, +8) pair with [D/2 + 8g, +8), frequencies 8g + k;
          // interleaved: columns [16g, +16) hold the pairs of frequencies 8g + k
          uint4* pa = chunk(rope_off_a(g, p.rope_interleaved != 0));
          uint4* pb = chunk(rope_off_b(g, D, p.rope_interleaved != 0));
          float a[8], bb[8], c8[8], s8[8];
          unpack(*pa, a);
          unpack(*pb, bb);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            c8[k] = cv[8 * g + k];
            s8[k] = sv[8 * g + k];
          }
          float ya[8], yb[8];
          if constexpr (kExact) {
            float cl8[8], sl8[8];
            const float4* clo = reinterpret_cast<const float4*>(p.cos_lo + trow + 8 * g);
            const float4* slo = reinterpret_cast<const float4*>(p.sin_lo + trow + 8 * g);
            const float4 c0 = __ldg(clo), c1 = __ldg(clo + 1), s0 = __ldg(slo), s1 = __ldg(slo + 1);
            cl8[0] = c0.x; cl8[1] = c0.y; cl8[2] = c0.z; cl8[3] = c0.w;
            cl8[4] = c1.x; cl8[5] = c1.y; cl8[6] = c1.z; cl8[7] = c1.w;
            sl8[0] = s0.x; sl8[1] = s0.y; sl8[2] = s0.z; sl8[3] = s0.w;
            sl8[4] = s1.x; sl8[5] = s1.y; sl8[6] = s1.z; sl8[7] = s1.w;
            rope_rotate16_exact(a, bb, c8, cl8, s8, sl8, p.rope_interleaved != 0, ya, yb);
          } else {
            rope_rotate16(a, bb, c8, s8, p.rope_interleaved != 0, 1.f, ya, yb);
          }
          *pa = pack(ya);
          *pb = pack(yb);
        }
      }
      fence_async_smem();  // the rotated rows are read by the tensor core
      mbar_arrive(smem_u32(&bar_q_rot));
    }
    for (int j = 0; j < n && ok; ++j) {
      const uint32_t tS = tmem + lane_base + (j & 1) * 128;
      ok = __all_sync(0xffffffffu, bounded_wait(smem_u32(&bar_s_full[j & 1]), (j >> 1) & 1,
                                                abort_ptr, p.status, kSiteSFull));
      if (!ok) break;
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t u[32], w[32];
        tmem_ld32x2(tS + cc * 64, tS + cc * 64 + 32, u, w);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[cc * 64 + i] = __uint_as_float(u[i]);
          s[cc * 64 + 32 + i] = __uint_as_float(w[i]);
        }
      }
      // keys after the row's position, or past the end of the cache, are masked
      const int k0 = (kt0 + j) * kTile;
      const int lim_c = qpos - k0 + 1;   // keys k0 + i with i < lim_c are visible
      const int lim_e = p.Skv - k0;      // ... and exist
      const int lim = lim_c < lim_e ? lim_c : lim_e;
      if (lim < 128) {
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = i >= lim ? -INFINITY : s[i];
      }
      float mp[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mp[k] = s[k];
#pragma unroll
      for (int i = 8; i < 128; i += 8)
#pragma unroll
        for (int k = 0; k < 8; ++k) mp[k] = fmaxf(mp[k], s[i + k]);
      const float mx2 = sl2 * fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                                    fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      float alpha = 1.f;
      bool grew = false;
      if (mx2 > m + 8.f) {  // lazy rescaling, as in the forward kernel
        alpha = m == -INFINITY ? 0.f : ex2(m - mx2);
        grew = true;
        m = mx2;
      }
      const float msub = m == -INFINITY ? 0.f : m;  // a row with no key yet: P = 0
      float rp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float a0 = ex2(fmaf(s[hh * 64 + 2 * i], sl2, -msub));
          const float a1 = ex2(fmaf(s[hh * 64 + 2 * i + 1], sl2, -msub));
          rp[i & 7] += a0 + a1;
          pk[i] = pack_bf16(a0, a1);
        }
        tmem_st32(tS + hh * 32, pk);
      }
      l = l * alpha + (((rp[0] + rp[1]) + (rp[2] + rp[3])) + ((rp[4] + rp[5]) + (rp[6] + rp[7])));
      // O of the previous step is complete before it is rescaled (and the softmax
      // stays in step with the barrier's phases)
      if (j > 0) {
        ok = __all_sync(0xffffffffu, bounded_wait(smem_u32(&bar_o_done), (j - 1) & 1, abort_ptr,
                                                  p.status, kSiteODone));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, grew)) {
          const float f = grew ? alpha : 1.f;
          const uint32_t tO = tmem + lane_base + C::kColO;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t u[32];
            tmem_ld32(tO + cc * 32, u);
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * f);
            tmem_st32(tO + cc * 32, u);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_p_full[j & 1]));
    }
    // ------------------------------------------------------------ partial result
    if (ok && n > 0)
      ok = __all_sync(0xffffffffu, bounded_wait(smem_u32(&bar_o_done), (n - 1) & 1, abort_ptr,
                                                p.status, kSiteODone));
    const long long grow = q_row0 + r;  // the row's index among the B*Hq*Sq rows
    if (ok) {
      tc_fence_after();
      const long long prow = static_cast<long long>(c) * p.rows + grow;
      const bool part_ok = bounds_ok(!row_real || prow < p.nchunks * p.rows, p.status, kChkPart);
      float* dst = p.part_out + prow * D;
      const bool seen = n > 0 && l > 0.f;
      const float inv_l = seen ? 1.f / l : 0.f;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t u[32];
        if (n > 0) tmem_ld32(tmem + lane_base + C::kColO + cc * 32, u);
        if (row_real && part_ok) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(dst + cc * 32)[i] =
                n > 0 ? make_float4(__uint_as_float(u[4 * i]) * inv_l,
                                    __uint_as_float(u[4 * i + 1]) * inv_l,
                                    __uint_as_float(u[4 * i + 2]) * inv_l,
                                    __uint_as_float(u[4 * i + 3]) * inv_l)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (row_real && part_ok) p.part_lse[prow] = seen ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// out_i = sum_c exp(lse_c - lse) out_c, lse = ln sum_c exp(lse_c) over the chunks c.
// A row is served by T = D/8 element lanes (8 elements each) times L chunk lanes;
// chunk lane l takes the chunks l, l + L, ... four at a time (their loads in flight
// together), keeping a running maximum, weight sum and weighted sum, and the L lanes
// of an element lane (adjacent lanes of a warp) combine theirs with shuffles.
constexpr int kMergeL = 8;
constexpr int kMergeThreads = 256;

struct MergeAcc {
  float m, ws, acc[8];
};

// Combines (m2, ws2, acc2) into a: both rescaled to the larger maximum.
__device__ __forceinline__ void merge_combine(MergeAcc& a, float m2, float ws2, const float (&acc2)[8]) {
  const float M = fmaxf(a.m, m2);
  if (M == -INFINITY) return;  // neither side has seen a key
  const float s1 = a.m == -INFINITY ? 0.f : expf(a.m - M);
  const float s2 = m2 == -INFINITY ? 0.f : expf(m2 - M);
  a.ws = a.ws * s1 + ws2 * s2;
#pragma unroll
  for (int i = 0; i < 8; ++i) a.acc[i] = a.acc[i] * s1 + acc2[i] * s2;
  a.m = M;
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecParams p) {
  constexpr int T = D / 8;
  constexpr int L = kMergeL;
  constexpr int U = 4;
  static_assert((T * L) % 32 == 0, "the lanes of a row fill whole warps");
  pdl_wait();  // the chunk grid has completed and its partial results are visible
  const long long t = blockIdx.x * static_cast<long long>(kMergeThreads) + threadIdx.x;
  const long long row = t / (T * L);
  if (row >= p.rows) return;  // a row's T * L lanes fill whole warps: a warp leaves together
  const int e = static_cast<int>(t / L % T) * 8;
  const int l = static_cast<int>(t % L);
  const float* lse_c = p.part_lse + row;
  const float* out_c = p.part_out + row * D + e;
  const long long ostride = p.rows * D;
  MergeAcc a{-INFINITY, 0.f, {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}};
  for (int c0 = l; c0 < p.nchunks; c0 += U * L) {
    float lv[U];
    float4 x[U], y[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * L;
      lv[u] = -INFINITY;
      x[u] = y[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < p.nchunks) {
        lv[u] = __ldcg(lse_c + c * p.rows);
        const float4* src = reinterpret_cast<const float4*>(out_c + c * ostride);
        x[u] = __ldcg(src);
        y[u] = __ldcg(src + 1);
      }
    }
    float acc2[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float m2 = -INFINITY, ws2 = 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) m2 = fmaxf(m2, lv[u]);
    if (m2 != -INFINITY) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float w = expf(lv[u] - m2);  // 0: a chunk without keys, or past the last
        ws2 += w;
        acc2[0] += w * x[u].x; acc2[1] += w * x[u].y; acc2[2] += w * x[u].z; acc2[3] += w * x[u].w;
        acc2[4] += w * y[u].x; acc2[5] += w * y[u].y; acc2[6] += w * y[u].z; acc2[7] += w * y[u].w;
      }
    }
    merge_combine(a, m2, ws2, acc2);
  }
#pragma unroll
  for (int off = 1; off < L; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, a.m, off);
    const float ws2 = __shfl_xor_sync(0xffffffffu, a.ws, off);
    float acc2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc2[i] = __shfl_xor_sync(0xffffffffu, a.acc[i], off);
    merge_combine(a, m2, ws2, acc2);
  }
  if (l != 0) return;
  const float inv = a.ws > 0.f ? 1.f / a.ws : 0.f;
  *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + row * D + e) =
      make_uint4(pack_bf16(a.acc[0] * inv, a.acc[1] * inv), pack_bf16(a.acc[2] * inv, a.acc[3] * inv),
                 pack_bf16(a.acc[4] * inv, a.acc[5] * inv), pack_bf16(a.acc[6] * inv, a.acc[7] * inv));
  if (e == 0) p.lse[row] = a.ws > 0.f ? a.m + logf(a.ws) : -INFINITY;
}

template <int D, bool kExact>
cudaError_t launch_decode_chunks(const DecParams& p, cudaStream_t stream) {
  using C = DecCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<D, kExact>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_decode_kernel<D, kExact>,
                    dim3(static_cast<unsigned>(p.nchunks * p.B * p.Hkv)), dim3(kThreads),
                    C::kSmemBytes, stream, p);
}

template <int D>
cudaError_t launch_decode_d(const DecParams& p, cudaStream_t stream) {
  cudaError_t e = p.exact ? launch_decode_chunks<D, true>(p, stream)
                          : launch_decode_chunks<D, false>(p, stream);
  if (e != cudaSuccess) return e;
  const long long mthreads = p.rows * (D / 8) * kMergeL;
  return launch_pdl(decode_merge_kernel<D>,
                    dim3(static_cast<unsigned>((mthreads + kMergeThreads - 1) / kMergeThreads)),
                    dim3(kMergeThreads), 0, stream, p);
}

}  // namespace

cudaError_t launch_decode(const DecParams& p, cudaStream_t stream) {
  return p.D == 128 ? launch_decode_d<128>(p, stream) : launch_decode_d<64>(p, stream);
}

}  // namespace gbattn
