// Exact delta pass of the backward, for sm_103a:
//   delta_i = sum_j P_ij dP_ij,  P_ij = exp(s_ij - lse_i),  dP_ij = dout_i . v_j,
// the row sums of P o dP over every visible key. In exact arithmetic this equals
// dout_i . out_i, but the `out` a backward call receives is rounded to bf16, and the
// rounding of each out element enters delta_i, every dS_ij of the row and, through the
// sums over a group's query heads, dk ("深度学习系统设计llama3-from-scratch：并行计算架构",
// §键值（Key-Value）共享机制; "ColossalAI 中的 PaLM 教学实现…", §2.5 multi-query); with
// sharply peaked rows (the row maximum subtracted before the softmax, PaLM §2.5) it is
// the largest error of dq and dk. This pass forms delta from the scores themselves.
//
// GB300 design (the forward's): one CTA owns two 128-row query tiles of one head and
// streams the key tiles of its KV head through a TMA ring (K_j, V_j alternating).
// Per key tile and query tile, two tcgen05 products into TMEM:
//   S_t  = Q~_t K~_jᵀ  [128 queries x 128 keys]
//   dP_t = dO_t V_jᵀ   [128 queries x 128 keys]
// and the query tile's four softmax warps (one thread per query row) add
// P o dP along their row in registers. The operands are the backward pre-pass's fp16
// copies (q~, k~ scaled by 2^(eq+ek), dO and v by 2^(edo+ev)), so S and dP equal the
// main kernel's, and delta leaves scaled by 2^(edo+ev) as the main kernel reads it.
// Warp roles: 0-3 / 4-7 rows of query tile 0 / 1, 8 TMA producer, 9 MMA issuer.
// TMEM: S_0 [0,128), S_1 [128,256), dP_0 [256,384), dP_1 [384,512).
#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

using namespace gb;

constexpr int kThreads = 320;
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;

enum : int {
  kSiteQ = 40, kSiteKvFull = 41, kSiteKvEmpty = 42, kSiteSFull = 43, kSitePFree = 44,
  kSiteInject = 45,
  // index checks of the debug build
  kChkKv = 50, kChkQ = 51, kChkRow = 52
};

template <int D>
struct DeltaCfg {
  static constexpr int kRegionBytes = 128 * 128;  // 128 rows x 128 B (64 fp16)
  static constexpr int kRegions = D / 64;
  static constexpr int kTileBytes = kRegions * kRegionBytes;
  static constexpr int kKvOff = 4 * kTileBytes;  // after Q~_0, Q~_1, dO_0, dO_1
  static constexpr int kSlots = D == 128 ? 3 : 10;
  static constexpr int kSmemBytes = kKvOff + kSlots * kTileBytes + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
  __device__ static constexpr uint32_t col_dp(int t) { return t ? 384u : 256u; }
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs / 4) return;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_delta_kernel(const __grid_constant__ DeltaParams p) {
  using C = DeltaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_drain, bar_never;
  __shared__ __align__(8) uint64_t bar_kv_full[C::kSlots], bar_kv_empty[C::kSlots];
  __shared__ __align__(8) uint64_t bar_s_full[2], bar_p_free[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;

  // ---- work item: heaviest query-tile pairs first (self-attention, S rows per head)
  const int nq = p.S / kTile;
  const int npairs = (nq + 1) / 2;
  const int BH = p.B * p.Hq;
  const int c = npairs - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int b = bh / p.Hq;
  const int h = bh % p.Hq;
  const int hkv = h / (p.Hq / p.Hkv);
  auto tiles_of = [&](int t) {
    const int qt = 2 * c + t;
    if (qt >= nq) return 0;
    return p.causal ? qt + 1 : nq;
  };
  const int n_0 = tiles_of(0);
  const int n_1 = tiles_of(1);
  const int n = n_0 > n_1 ? n_0 : n_1;
  const int q_row0 = bh * p.S;
  const int kv_row0 = (b * p.Hkv + hkv) * p.S;
  const long long rows_q = static_cast<long long>(p.B) * p.Hq * p.S;
  const long long rows_kv = static_cast<long long>(p.B) * p.Hkv * p.S;

  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  const bool producer = warp == kWarpLoad && lane == 0;
  int issued = 0;
  // ring load i: K_(i/2) or V_(i/2) into slot i % kSlots, once that slot is free
  auto issue_kv = [&](int i) {
    const int slot = i % C::kSlots;
    const uint32_t ph = ((i / C::kSlots) & 1) ^ 1;
    if (!bounded_wait(smem_u32(&bar_kv_empty[slot]), ph, &abort_flag, p.status, kSiteKvEmpty))
      return false;
    const uint32_t full = smem_u32(&bar_kv_full[slot]);
    mbar_arrive_expect_tx(full, C::kTileBytes);
    const CUtensorMap* map = (i & 1) == 0 ? &p.map_k : &p.map_v;
    const uint32_t dst = sbase + C::kKvOff + slot * C::kTileBytes;
    if (bounds_ok(kv_row0 + ((i >> 1) + 1LL) * kTile <= rows_kv, p.status, kChkKv))
      for (int r = 0; r < C::kRegions; ++r)
        tma_load_2d(dst + r * C::kRegionBytes, map, r * 64, kv_row0 + (i >> 1) * kTile, full);
    return true;
  };
  if (producer) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_q), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    mbar_init(smem_u32(&bar_never), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(smem_u32(&bar_kv_full[s]), 1);
      mbar_init(smem_u32(&bar_kv_empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bar_s_full[t]), 1);
      mbar_init(smem_u32(&bar_p_free[t]), 128);
    }
    fence_mbar_init();
    pdl_wait();  // the operands come from the pre-pass before this kernel
    tma_prefetch_desc(&p.map_q);
    tma_prefetch_desc(&p.map_do);
    tma_prefetch_desc(&p.map_k);
    tma_prefetch_desc(&p.map_v);
    const int nvalid = (n_0 > 0) + (n_1 > 0);
    mbar_arrive_expect_tx(smem_u32(&bar_q), 2 * nvalid * C::kTileBytes);
    for (int t = 0; t < 2; ++t) {
      if ((t ? n_1 : n_0) == 0) continue;
      if (!bounds_ok(q_row0 + (2LL * c + t + 1) * kTile <= rows_q, p.status, kChkQ)) continue;
      for (int r = 0; r < C::kRegions; ++r) {
        tma_load_2d(sbase + t * C::kTileBytes + r * C::kRegionBytes, &p.map_q, r * 64,
                    q_row0 + (2 * c + t) * kTile, smem_u32(&bar_q));
        tma_load_2d(sbase + (2 + t) * C::kTileBytes + r * C::kRegionBytes, &p.map_do, r * 64,
                    q_row0 + (2 * c + t) * kTile, smem_u32(&bar_q));
      }
    }
    while (issued < 2 * n && issued < C::kSlots && issue_kv(issued)) ++issued;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_ptr = &abort_flag;
  pdl_wait();
  pdl_launch_dependents();

  if (warp == kWarpLoad) {
    // ================================================================ producer
    if (lane == 0) {
      while (issued < 2 * n && issue_kv(issued)) ++issued;
      drain_wait(smem_u32(&bar_q), 0);
      for (int i = issued - C::kSlots > 0 ? issued - C::kSlots : 0; i < issued; ++i)
        drain_wait(smem_u32(&bar_kv_full[i % C::kSlots]), (i / C::kSlots) & 1);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ================================================================ MMA issuer
    constexpr uint32_t idesc = idesc_fp16(128, 128, 0, 0);
    constexpr uint64_t kKmaj = sdesc_hi(16, 1024);
    auto desc = [](uint64_t hi, uint32_t addr) { return hi | static_cast<uint64_t>(addr >> 4); };
    auto wait = [&](uint32_t bar, uint32_t parity, int site) {
      return __all_sync(0xffffffffu, bounded_wait(bar, parity, abort_ptr, p.status, site));
    };
    auto slot_addr = [&](int i) { return sbase + C::kKvOff + (i % C::kSlots) * C::kTileBytes; };
    auto wait_kv = [&](int i) {
      return wait(smem_u32(&bar_kv_full[i % C::kSlots]), (i / C::kSlots) & 1, kSiteKvFull);
    };
    // D (tmem col) = A (smem tile, rows = queries) x B (smem tile, rows = keys)ᵀ
    auto issue = [&](uint32_t col, uint32_t aaddr, uint32_t baddr) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * C::kRegionBytes + (kk & 3) * 32;
        mma_ss_w(tmem + col, desc(kKmaj, aaddr + off), desc(kKmaj, baddr + off), idesc, kk > 0);
      }
    };
    bool ok = true;
    if (p.inject_timeout) ok = wait(smem_u32(&bar_never), 0, kSiteInject);
    ok = ok && wait(smem_u32(&bar_q), 0, kSiteQ);
    for (int j = 0; j < n && ok; ++j) {
      const int ik = 2 * j, iv = 2 * j + 1;
      ok = wait_kv(ik) && wait_kv(iv);
      if (!ok) break;
      tc_fence_after();
      for (int t = 0; t < 2 && ok; ++t) {
        if (j >= (t ? n_1 : n_0)) continue;
        if (j > 0) {
          ok = wait(smem_u32(&bar_p_free[t]), (j - 1) & 1, kSitePFree);
          if (!ok) break;
          tc_fence_after();
        }
        issue(C::col_s(t), sbase + t * C::kTileBytes, slot_addr(ik));
        issue(C::col_dp(t), sbase + (2 + t) * C::kTileBytes, slot_addr(iv));
        mma_commit_w(smem_u32(&bar_s_full[t]));
      }
      if (!ok) break;
      mma_commit_w(smem_u32(&bar_kv_empty[ik % C::kSlots]));
      mma_commit_w(smem_u32(&bar_kv_empty[iv % C::kSlots]));
    }
    mma_commit_w(smem_u32(&bar_drain));
    drain_wait(smem_u32(&bar_drain), 0);
    __syncwarp();
  } else {
    // ================================================================ rows
    const int t = warp >> 2;
    const int r = tid & 127;  // query row in the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::col_s(t);
    const uint32_t tP = tmem + lane_base + C::col_dp(t);
    const int nt = t ? n_1 : n_0;
    const int qt = 2 * c + t;
    const long long row = static_cast<long long>(q_row0) + qt * kTile + r;
    const BwdExponents ex = bwd_exponents(p.maxes);
    // S arrives multiplied by 2^(eq+ek); lse2 = lse log2 e (+inf on padding rows)
    const float sl2 = p.scale_log2 * exp2i(-(ex.q + ex.k));
    const bool row_ok = bounds_ok(qt >= nq || row < rows_q, p.status, kChkRow);
    const float lse2 = nt > 0 && row_ok ? p.lse2[row] : 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < nt; ++j) {
      const bool got = bounded_wait(smem_u32(&bar_s_full[t]), j & 1, abort_ptr, p.status, kSiteSFull);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const bool diag = p.causal && j == qt;  // keys after the query are masked
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t sv[32], dv[32];
        tmem_ld32x2(tS + cc * 32, tP + cc * 32, sv, dv);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float pr = ex2(__fmaf_rn(__uint_as_float(sv[i]), sl2, -lse2));
          const float pm = (diag && cc * 32 + i > r) ? 0.f : pr;
          acc[i & 3] = __fmaf_rn(pm, __uint_as_float(dv[i]), acc[i & 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_p_free[t]));
    }
    if (qt < nq && row_ok) p.delta[row] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_delta_d(const DeltaParams& p, cudaStream_t stream) {
  using C = DeltaCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_delta_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int nq = p.S / kTile;
  const unsigned grid = static_cast<unsigned>(((nq + 1) / 2) * p.B * p.Hq);
  return launch_pdl(attn_delta_kernel<D>, dim3(grid), dim3(kThreads), C::kSmemBytes, stream, p);
}

}  // namespace

cudaError_t launch_delta(const DeltaParams& p, cudaStream_t stream) {
  return p.D == 128 ? launch_delta_d<128>(p, stream) : launch_delta_d<64>(p, stream);
}

}  // namespace gbattn
