// Backward attention main kernel for sm_103a: dK, dV and the dQ partial sums.
//
// The gradients are the chain rule through the forward definition (scores
// q~.k~ scale with keys after the query masked, softmax, P v; see attn_fwd.cu for
// the pages it follows). With P recomputed from the saved lse:
//   dP_ij = dout_i . v_j,  dS_ij = P_ij (dP_ij - delta_i),  delta_i = dout_i . out_i
//   dv_j  = sum_{h in group} sum_i P_ij dout_i
//   dk~_j = scale sum_{h in group} sum_i dS_ij q~_i      (rotated back here: dk = R_jᵀ dk~)
//   dq~_i = scale sum_j dS_ij k~_j                      (summed into an fp32 buffer)
// Query heads sharing one K/V head ("深度学习系统设计llama3-from-scratch：并行计算架构",
// §键值（Key-Value）共享机制; "ColossalAI 中的 PaLM 教学实现…", §2.5 multi-query) are
// reduced inside the CTA: dK and dV accumulate in tensor memory across every
// query head of the group.
//
// GB300 design: one CTA per (batch, KV head, 128-key tile) keeps K~ and V in
// shared memory and walks the (query head, 64-query tile) steps that see its
// keys (only tiles on or below the diagonal when causal). The CTAs run heaviest
// first, from a work-order table the host fills: when a few long CTAs would finish
// last (or one CTA per key tile would leave SMs idle) and the group has an even
// number of query heads, the heaviest key tiles get two CTAs, each taking half of
// the heads and adding its dK/dV partials into zeroed rows. The epilogue stages
// dK / dV in shared memory and writes (or adds) them as TMA tiles.
//
// Per step s (buffer b = s & 1), in TMEM:
//   Sᵀ_b  = K~ Q~ᵀ  [128 keys x 64 queries]   (SS MMA; D = 64: TS, K~ from TMEM)
//   dPᵀ_b = V dOᵀ   [128 keys x 64 queries]   (SS MMA; D = 64: TS, V from TMEM)
//   softmax warps: Pᵀ = 2^(Sᵀ scale log2e - lse2), dSᵀ = Pᵀ (dPᵀ - delta), packed as
//     fp16 back over the step's own Sᵀ columns (softmax half h: Pᵀ at
//     [128b+32h, +16), dSᵀ at [128b+32h+16, +16)); dSᵀ also to shared memory
//   dV += Pᵀ dO, dK += dSᵀ Q~                 (TS MMAs, A from TMEM)
//   D = 128: dQᵀ = K~ᵀ dSᵀ [128 d x 64 queries] over the step's dPᵀ columns;
//   D = 64:  dQ = dS K~ [128 queries x 64 d] once per pair of steps (the two
//            64-query tiles of one head that follow each other), in its own
//            64 columns, A taken from the pair's two adjacent dSᵀ buffers.
// The dQ drain warps add the partials into an fp32 buffer: at D = 128 with global
// reductions (a lane holds one d of 64 query rows); at D = 64, where a lane holds a
// whole query row, by staging the pair's 128 rows in shared memory and issuing one
// TMA reduction per 32-column box. Two (Sᵀ, dPᵀ) buffers let the score MMAs of
// step s+2 run while the softmax of step s+1 works.
// TMEM columns: Sᵀ_0 [0,64) dPᵀ_0 [64,128) Sᵀ_1 [128,192) dPᵀ_1 [192,256), then
//   D = 128: dV [256,384) dK [384,512);
//   D = 64:  dQ [256,320) dV [320,384) dK [384,448), K~ [448,480) V [480,512) (fp16
//            pairs, copied from shared memory by the softmax warps at the start).
// Q~/dO tiles (with lse2 and delta) arrive through a TMA ring of 3 stages (5 at D = 64).
// All products run in fp16 (kind::f16 with fp16 A and B): the operands q~, k~,
// v, dO arrive from the pre-pass multiplied by exact powers of two (q~ and k~
// hold their bf16-rounded values, so the recomputed scores equal the
// forward's), and Pᵀ, dSᵀ are rounded to fp16 (2^-11) instead of bf16 (2^-9);
// the scales are undone in the epilogues.
// Warp roles: 0-7 softmax (two 32-query halves), 8-11 dQ drain, 12 TMA
// producer, 13 MMA issuer (whole warp, one elected lane issues) and TMEM owner.
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

using namespace gb;

constexpr int kThreads = 448;
constexpr int kWarpLoad = 12;
constexpr int kWarpMma = 13;

enum : int {
  kSiteKv = 17, kSiteStageFull = 18, kSiteStageEmpty = 19, kSiteSFull = 20, kSiteDsFull = 21,
  kSiteDqFull = 22, kSiteDqFree = 23, kSiteDone = 24, kSiteInject = 25, kSiteTab = 26,
  kSiteKvTmem = 33, kSiteDqStg = 34,
  // index checks of the debug build
  kChkStage = 27, kChkKv = 28, kChkDq = 29, kChkDkdv = 30, kChkTab = 31
};

template <int D>
struct BwdCfg {
  static constexpr int BQ = 64;                    // query rows per step
  static constexpr bool kDqPair = D == 64;         // dQ once per pair of steps
  static constexpr int kRegions = D / 64;          // 64-column swizzle regions per row
  static constexpr int kKRegionBytes = 128 * 128;  // 128 key rows x 128 B
  static constexpr int kQRegionBytes = BQ * 128;   // 64 query rows x 128 B
  static constexpr int kKTileBytes = kRegions * kKRegionBytes;
  static constexpr int kQTileBytes = kRegions * kQRegionBytes;
  // D = 64: K~ and V also sit in tensor memory (packed fp16, the free 64 columns), so
  // that the score products Sᵀ = K~ Q~ᵀ and dPᵀ = V dOᵀ read their A operand from
  // there rather than from shared memory, whose bandwidth the N = 64 products
  // otherwise spend on re-reading K~ and V every step; the freed bandwidth also buys a
  // fourth and a fifth Q~/dO stage.
  static constexpr bool kKvTmem = D == 64;
  static constexpr int kStages = kKvTmem ? 5 : 3;
  static constexpr int kStageBytes = ((2 * kQTileBytes + 2 * BQ * 4) + 1023) / 1024 * 1024;
  static constexpr int kDsBufs = kDqPair ? 4 : 2;  // dSᵀ buffers (pairs stay adjacent)
  static constexpr int kDsBytes = 16384;           // dSᵀ: 128 key rows x 64 queries fp16
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKTileBytes;
  static constexpr int kStageOff = 2 * kKTileBytes;
  static constexpr int kDsOff = kStageOff + kStages * kStageBytes;
  // D = 64: a dQ pair's 128 rows staged for the TMA reduction into the accumulator,
  // two 128-byte swizzled boxes of 32 fp32 columns x 128 rows
  static constexpr int kDqStgOff = kDsOff + kDsBufs * kDsBytes;
  static constexpr int kSmemBytes = kDqStgOff + (kDqPair ? 2 * 128 * 128 : 0) + 1024;
  __device__ static constexpr uint32_t col_st(int buf) { return buf ? 128u : 0u; }
  __device__ static constexpr uint32_t col_dpt(int buf) { return buf ? 192u : 64u; }
  static constexpr uint32_t kColDQ = 256;  // D = 64 only
  static constexpr uint32_t kColDV = kDqPair ? 320 : 256;
  static constexpr uint32_t kColDK = 384;
  static constexpr uint32_t kColKt = 448;  // D = 64: K~ rows, 32 columns of fp16 pairs
  static constexpr uint32_t kColVt = 480;  // D = 64: V rows
  static_assert(kColDK + D <= (kKvTmem ? kColKt : 512u), "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // Epilogue staging, in the shared memory the main loop used: the cos and sin rows
  // of the tile's keys, then dV and dK, as 128-byte swizzled boxes of 32 fp32
  // columns x 128 rows (the TMA layout).
  static constexpr int kBoxBytes = 128 * 128;
  static constexpr int kTabBoxes = D / 64;  // boxes per table row set (D/2 floats)
  static constexpr int kEpiCos = 0;
  static constexpr int kEpiSin = kTabBoxes * kBoxBytes;
  static constexpr int kEpiDv = 2 * kTabBoxes * kBoxBytes;
  static constexpr int kEpiDk = kEpiDv + (D / 32) * kBoxBytes;
  static_assert(kEpiDk + (D / 32) * kBoxBytes <= kDsOff + kDsBufs * kDsBytes, "epilogue staging");
};

// Packed fp32 pairs: one instruction for two lanes' worth of the same operation,
// each rounded as the scalar form.
__device__ __forceinline__ uint64_t pack2(float2 a) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
  return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t r) {
  float2 a;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
  return a;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)), "l"(pack2(c)));
  return unpack2(d);
}
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)));
  return unpack2(d);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)));
  return unpack2(d);
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs / 4) return;
  }
}


template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int BQ = C::BQ;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_kv, bar_done, bar_drain, bar_never, bar_tab, bar_kvt;
  __shared__ __align__(8) uint64_t bar_stg_full, bar_stg_free;
  __shared__ __align__(8) uint64_t bar_stage_full[C::kStages], bar_stage_empty[C::kStages];
  __shared__ __align__(8) uint64_t bar_s_full[2], bar_ds_full[2], bar_dq_full[2], bar_dq_free[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const sgen = smem_raw + (sbase - smem_u32(smem_raw));

  // ---- work item: key tile kt of KV head (b, hkv), query heads of part `part`
  // of the group (nparts parts), heaviest first
  int kt, nparts, idx;
  if (p.nplan > 0) {
    const int per = p.B * p.Hkv;
    int start = 0, e = 0;
    for (; e < p.nplan - 1; ++e) {
      const int cnt = p.plan_parts[e] * per;
      if (static_cast<int>(blockIdx.x) < start + cnt) break;
      start += cnt;
    }
    kt = p.plan_kt[e];
    nparts = p.plan_parts[e];
    idx = static_cast<int>(blockIdx.x) - start;
  } else {
    const int units = p.B * p.Hkv * p.hsplit;
    kt = static_cast<int>(blockIdx.x) / units;
    nparts = p.hsplit;
    idx = static_cast<int>(blockIdx.x) % units;
  }
  const int bhk = idx / nparts;
  const int part = idx % nparts;
  const int b = bhk / p.Hkv;
  const int hkv = bhk % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int Gc = G / nparts;  // query heads of this CTA
  const int h_first = hkv * G + part * Gc;
  const int k0 = kt * kTile;                  // first key row of the tile in the block
  const int k0p = (p.kv_tile0 + kt) * kTile;  // its position
  const int q0p = p.q_tile0 * kTile;          // position of the query block's first row
  const int kv_row = bhk * p.Skv + k0;
  const int nqt = p.Sq / BQ;
  const long long rows_q = static_cast<long long>(p.B) * p.Hq * p.Sq;  // rows of q~, dO, dqacc
  const long long rows_kv = static_cast<long long>(p.B) * p.Hkv * p.Skv;
  // causal: the query tiles at or after the key tile's position
  int qt_begin = p.causal ? (k0p - q0p) / BQ : 0;
  qt_begin = qt_begin < 0 ? 0 : (qt_begin > nqt ? nqt : qt_begin);
  const int per_head = nqt - qt_begin;  // even: Sq and the offsets are multiples of 128
  const int n = Gc * per_head;          // 0: no query of the block sees these keys
  auto step_qt = [&](int s) { return qt_begin + s % per_head; };
  auto step_row = [&](int s) {
    const int h = h_first + s / per_head;
    return (b * p.Hq + h) * p.Sq + step_qt(s) * BQ;
  };

  // ---- setup. The producer's lane initialises the barriers and, as soon as the
  // previous kernel's writes are visible, starts the K~/V and first Q~/dO loads while
  // the MMA warp allocates tensor memory.
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  const bool producer = warp == kWarpLoad && lane == 0;
  auto stage_addr = [&](int s) { return sbase + C::kStageOff + (s % C::kStages) * C::kStageBytes; };
  auto ds_addr = [&](int s) { return sbase + C::kDsOff + (s % C::kDsBufs) * C::kDsBytes; };
  int issued = 0;  // Q~/dO stage loads issued (producer lane)
  // stage load of step s, once the stage is free
  auto issue_stage = [&](int s) {
    const int st = s % C::kStages;
    if (!bounded_wait(smem_u32(&bar_stage_empty[st]), ((s / C::kStages) & 1) ^ 1, &abort_flag,
                      p.status, kSiteStageEmpty))
      return false;
    const uint32_t full = smem_u32(&bar_stage_full[st]);
    const uint32_t dst = stage_addr(s);
    const int row = step_row(s);
    mbar_arrive_expect_tx(full, 2 * C::kQTileBytes + 2 * BQ * 4);
    if (bounds_ok(row >= 0 && row + BQ <= rows_q, p.status, kChkStage)) {
      for (int r = 0; r < C::kRegions; ++r) {
        tma_load_2d(dst + r * C::kQRegionBytes, &p.map_q, r * 64, row, full);
        tma_load_2d(dst + C::kQTileBytes + r * C::kQRegionBytes, &p.map_do, r * 64, row, full);
      }
      bulk_load(dst + 2 * C::kQTileBytes, p.lse2 + row, BQ * 4, full);
      bulk_load(dst + 2 * C::kQTileBytes + BQ * 4, p.delta + row, BQ * 4, full);
    }
    return true;
  };
  if (producer) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_kv), 1);
    mbar_init(smem_u32(&bar_done), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    mbar_init(smem_u32(&bar_never), 1);
    mbar_init(smem_u32(&bar_tab), 1);
    mbar_init(smem_u32(&bar_kvt), 256);
    mbar_init(smem_u32(&bar_stg_full), 128);
    mbar_init(smem_u32(&bar_stg_free), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&bar_stage_full[s]), 1);
      mbar_init(smem_u32(&bar_stage_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_s_full[i]), 1);
      mbar_init(smem_u32(&bar_ds_full[i]), 256);
      mbar_init(smem_u32(&bar_dq_full[i]), 1);
      mbar_init(smem_u32(&bar_dq_free[i]), 128);
    }
    fence_mbar_init();
    pdl_wait();  // the operands come from the pre-pass before this kernel
    tma_prefetch_desc(&p.map_q);
    tma_prefetch_desc(&p.map_do);
    const uint32_t kvb = smem_u32(&bar_kv);
    mbar_arrive_expect_tx(kvb, 2 * C::kKTileBytes);
    if (bounds_ok(kv_row + kTile <= rows_kv, p.status, kChkKv))
      for (int r = 0; r < C::kRegions; ++r) {
        tma_load_2d(sbase + C::kKOff + r * C::kKRegionBytes, &p.map_k, r * 64, kv_row, kvb);
        tma_load_2d(sbase + C::kVOff + r * C::kKRegionBytes, &p.map_v, r * 64, kv_row, kvb);
      }
    while (issued < n && issued < C::kStages && issue_stage(issued)) ++issued;  // free stages
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_ptr = &abort_flag;
  // Nothing above except the producer's loads (after its own wait) touched global
  // memory: this prologue may overlap the kernel before it in the stream.
  pdl_wait();
  pdl_launch_dependents();
  const BwdExponents ex = bwd_exponents(p.maxes);  // fp16 operand scales

  if (warp == kWarpLoad) {
    // ================================================================ producer
    if (lane == 0) {
      while (issued < n && issue_stage(issued)) ++issued;
      // Copies already issued land before the CTA releases its shared memory
      // (at most one in flight per stage: a stage is refilled only once consumed).
      drain_wait(smem_u32(&bar_kv), 0);
      for (int i = issued - C::kStages > 0 ? issued - C::kStages : 0; i < issued; ++i)
        drain_wait(smem_u32(&bar_stage_full[i % C::kStages]), (i / C::kStages) & 1);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ================================================================ MMA issuer (whole warp)
    constexpr uint32_t idesc_st = idesc_fp16(128, BQ, 0, 0);
    constexpr uint32_t idesc_acc = idesc_fp16(128, D, 0, 1);
    constexpr uint32_t idesc_dq = C::kDqPair ? idesc_fp16(128, D, 1, 1) : idesc_fp16(128, BQ, 1, 1);
    constexpr uint64_t kKmaj = sdesc_hi(16, 1024);
    constexpr uint64_t kMnQ = sdesc_hi(C::kQRegionBytes, 1024);
    constexpr uint64_t kMnK = sdesc_hi(C::kKRegionBytes, 1024);
    constexpr uint64_t kMnDs = sdesc_hi(C::kDsBytes, 1024);
    auto desc = [](uint64_t hi, uint32_t addr) { return hi | static_cast<uint64_t>(addr >> 4); };
    auto wait = [&](uint32_t bar, uint32_t parity, int site) {
      return __all_sync(0xffffffffu, bounded_wait(bar, parity, abort_ptr, p.status, site));
    };
    const uint32_t kaddr = sbase + C::kKOff;
    const uint32_t vaddr = sbase + C::kVOff;
    // Sᵀ_b = K~ Q~ᵀ and dPᵀ_b = V dOᵀ of step s (b = s & 1)
    auto issue_s = [&](int s) {
      const uint32_t qaddr = stage_addr(s);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ok_ = (kk >> 2) * C::kKRegionBytes + (kk & 3) * 32;
        const uint32_t oq = (kk >> 2) * C::kQRegionBytes + (kk & 3) * 32;
        if constexpr (C::kKvTmem)  // 16 d per product: 8 columns of fp16 pairs
          mma_ts_w(tmem + C::col_st(s & 1), tmem + C::kColKt + kk * 8, desc(kKmaj, qaddr + oq),
                   idesc_st, kk > 0);
        else
          mma_ss_w(tmem + C::col_st(s & 1), desc(kKmaj, kaddr + ok_), desc(kKmaj, qaddr + oq),
                   idesc_st, kk > 0);
      }
    };
    auto issue_dp = [&](int s) {
      const uint32_t doaddr = stage_addr(s) + C::kQTileBytes;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ok_ = (kk >> 2) * C::kKRegionBytes + (kk & 3) * 32;
        const uint32_t oq = (kk >> 2) * C::kQRegionBytes + (kk & 3) * 32;
        if constexpr (C::kKvTmem)
          mma_ts_w(tmem + C::col_dpt(s & 1), tmem + C::kColVt + kk * 8, desc(kKmaj, doaddr + oq),
                   idesc_st, kk > 0);
        else
          mma_ss_w(tmem + C::col_dpt(s & 1), desc(kKmaj, vaddr + ok_), desc(kKmaj, doaddr + oq),
                   idesc_st, kk > 0);
      }
    };
    auto issue_dvdk = [&](int s, bool first) {
      const uint32_t qaddr = stage_addr(s);
      const uint32_t doaddr = qaddr + C::kQTileBytes;
      const uint32_t pt = tmem + C::col_st(s & 1);
#pragma unroll
      for (int kk = 0; kk < BQ / 16; ++kk)  // queries 16kk.. sit at (kk/2)*32 + (kk%2)*8
        mma_ts_w(tmem + C::kColDV, pt + (kk >> 1) * 32 + (kk & 1) * 8,
                 desc(kMnQ, doaddr + kk * 2048), idesc_acc, (!first || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < BQ / 16; ++kk)  // dSᵀ sits 16 columns after Pᵀ
        mma_ts_w(tmem + C::kColDK, pt + (kk >> 1) * 32 + 16 + (kk & 1) * 8,
                 desc(kMnQ, qaddr + kk * 2048), idesc_acc, (!first || kk > 0) ? 1u : 0u);
    };
    // D = 128: dQᵀ [D x 64] = K~ᵀ dSᵀ of step s, over the step's dPᵀ columns.
    // D = 64 : dQ [128 x D] = dS K~ of steps s-1, s (A: the pair's dSᵀ buffers).
    auto issue_dq = [&](int s) {
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        if constexpr (C::kDqPair) {
          mma_ss_w(tmem + C::kColDQ, desc(kMnDs, ds_addr(s - 1) + kk * 2048),
                   desc(kMnK, kaddr + kk * 2048), idesc_dq, kk > 0);
        } else {
          mma_ss_w(tmem + C::col_dpt(s & 1), desc(kMnK, kaddr + kk * 2048),
                   desc(kMnDs, ds_addr(s) + kk * 2048), idesc_dq, kk > 0);
        }
      }
    };

    bool ok = true;
    if (p.inject_timeout)  // nothing ever arrives on bar_never
      ok = wait(smem_u32(&bar_never), 0, kSiteInject);
    ok = ok && wait(smem_u32(&bar_kv), 0, kSiteKv);
    if constexpr (C::kKvTmem) ok = ok && wait(smem_u32(&bar_kvt), 0, kSiteKvTmem);
    for (int s = 0; s < 2 && s < n && ok; ++s) {
      ok = wait(smem_u32(&bar_stage_full[s]), 0, kSiteStageFull);
      if (!ok) break;
      tc_fence_after();
      issue_s(s);
      issue_dp(s);
      mma_commit_w(smem_u32(&bar_s_full[s]));
    }
    for (int s = 0; s < n && ok; ++s) {
      const int buf = s & 1;
      ok = wait(smem_u32(&bar_ds_full[buf]), (s >> 1) & 1, kSiteDsFull);
      if (!ok) break;
      tc_fence_after();
      if constexpr (!C::kDqPair) {
        // dQᵀ(s) first: its drain then overlaps dV/dK(s) and Sᵀ(s+2), and is done
        // before dPᵀ(s+2) needs the columns (dPᵀ(s) was consumed by the softmax)
        issue_dq(s);
        mma_commit_w(smem_u32(&bar_dq_full[buf]));
      }
      issue_dvdk(s, s == 0);
      mma_commit_w(smem_u32(&bar_stage_empty[s % C::kStages]));
      if constexpr (C::kDqPair) {
        if (s & 1) {
          const int m = s >> 1;  // pair index; its drain frees the single dQ buffer
          ok = wait(smem_u32(&bar_dq_free[0]), (m & 1) ^ 1, kSiteDqFree);
          if (!ok) break;
          tc_fence_after();
          issue_dq(s);
          mma_commit_w(smem_u32(&bar_dq_full[0]));
        }
      }
      if (s + 2 < n) {
        ok = wait(smem_u32(&bar_stage_full[(s + 2) % C::kStages]), ((s + 2) / C::kStages) & 1,
                  kSiteStageFull);
        if (!ok) break;
        issue_s(s + 2);  // after dV(s) in issue order: Pᵀ(s) is read before it is overwritten
        if constexpr (!C::kDqPair) {
          ok = wait(smem_u32(&bar_dq_free[buf]), (s >> 1) & 1, kSiteDqFree);
          if (!ok) break;
          tc_fence_after();
        }
        issue_dp(s + 2);  // D = 128: the drain has read dQᵀ(s) from these columns
        mma_commit_w(smem_u32(&bar_s_full[buf]));
      }
    }
    if (ok) mma_commit_w(smem_u32(&bar_done));
    // Every MMA issued above completes before the tensor memory is released.
    mma_commit_w(smem_u32(&bar_drain));
    drain_wait(smem_u32(&bar_drain), 0);
    __syncwarp();
  } else if (warp >= 8) {
    // ================================================================ dQ drain
    const int r = tid & 127;  // TMEM lane: d (D = 128) or query row of the pair (D = 64)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    if constexpr (C::kDqPair) {
      // A pair's 128 dQ rows (one per lane) go to shared memory as two 128-byte swizzled
      // boxes of 32 fp32 columns, which the drain's first thread adds into the
      // accumulator rows with one TMA reduction each. The boxes are rewritten once the
      // previous pair's reductions have read them; the first thread checks that only
      // after it has read the next pair's partials, so that the check never holds back
      // the release of the dQ columns.
      const uint32_t stg = sbase + C::kDqStgOff;
      const bool issuer = tid == 8 * 32;
      for (int m = 0; m < n / 2; ++m) {
        const bool got =
            bounded_wait(smem_u32(&bar_dq_full[0]), m & 1, abort_ptr, p.status, kSiteDqFull);
        if (!__all_sync(0xffffffffu, got)) break;
        tc_fence_after();
        uint32_t u0[32], u1[32];
        tmem_ld32x2(tmem + lane_base + C::kColDQ, tmem + lane_base + C::kColDQ + 32, u0, u1);
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_dq_free[0]));
        if (m > 0) {
          if (issuer) {
            bulk_wait_read_all();
            mbar_arrive(smem_u32(&bar_stg_free));
          }
          const bool free_ok = bounded_wait(smem_u32(&bar_stg_free), (m - 1) & 1, abort_ptr,
                                            p.status, kSiteDqStg);
          if (!__all_sync(0xffffffffu, free_ok)) break;
        }
        // columns 4i..4i+3 sit in 16-byte chunk i ^ (r & 7) of the row's 128 bytes
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t off = static_cast<uint32_t>(r * 128 + ((i ^ (r & 7)) << 4));
          st_shared_v4(stg + off, u0[4 * i], u0[4 * i + 1], u0[4 * i + 2], u0[4 * i + 3]);
          st_shared_v4(stg + C::kBoxBytes + off, u1[4 * i], u1[4 * i + 1], u1[4 * i + 2],
                       u1[4 * i + 3]);
        }
        fence_async_smem();
        mbar_arrive(smem_u32(&bar_stg_full));
        if (issuer && bounded_wait(smem_u32(&bar_stg_full), m & 1, abort_ptr, p.status,
                                   kSiteDqStg)) {
          // query rows of steps 2m, 2m+1: consecutive rows of one head
          const int row0 = step_row(2 * m);
          if (bounds_ok(row0 >= 0 && row0 + 128LL <= rows_q, p.status, kChkDq)) {
            tma_reduce_add_2d(&p.map_dqacc, 0, row0, stg);
            tma_reduce_add_2d(&p.map_dqacc, 32, row0, stg + C::kBoxBytes);
          }
          bulk_commit();
        }
      }
      // the last reductions have read the boxes before the CTA releases its shared memory
      if (issuer) bulk_wait_read_all();
    } else {
      for (int s = 0; s < n; ++s) {
        const int buf = s & 1;
        const bool got = bounded_wait(smem_u32(&bar_dq_full[buf]), (s >> 1) & 1, abort_ptr,
                                      p.status, kSiteDqFull);
        if (!__all_sync(0xffffffffu, got)) break;
        tc_fence_after();
        uint32_t u0[32], u1[32];
        tmem_ld32x2(tmem + lane_base + C::col_dpt(buf), tmem + lane_base + C::col_dpt(buf) + 32,
                    u0, u1);
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_dq_free[buf]));
        // lane r = d; columns = the 64 query rows of the step
        const long long srow = step_row(s);
        if (bounds_ok(srow + BQ <= rows_q, p.status, kChkDq)) {
          float* base = p.dqacc + srow * D + r;
#pragma unroll
          for (int q = 0; q < 32; ++q) red_add_f32(base + (long long)q * D, __uint_as_float(u0[q]));
#pragma unroll
          for (int q = 0; q < 32; ++q)
            red_add_f32(base + (long long)(q + 32) * D, __uint_as_float(u1[q]));
        }
      }
    }
  } else {
    // ================================================================ softmax
    const int half = warp >> 2;
    const int r = tid & 127;  // key row in the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // Sᵀ arrives multiplied by 2^(eq+ek), dPᵀ and delta by 2^(edo+ev)
    const float sl2 = p.scale_log2 * exp2i(-(ex.q + ex.k));
    const int key = k0p + r;  // this thread's key position
    const int qb = half * 32;  // this half's first query column
    if constexpr (C::kKvTmem) {
      // row r of K~ (warps 0-3) or V (warps 4-7) from its swizzled tile into this
      // thread's tensor-memory lane: 64 fp16 values as 32 columns of pairs
      if (bounded_wait(smem_u32(&bar_kv), 0, abort_ptr, p.status, kSiteKv)) {
        const uint32_t src = sbase + (half == 0 ? C::kKOff : C::kVOff);
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          ld_shared_v4(src + sw128_offset(r, c), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        tmem_st32(tmem + lane_base + (half == 0 ? C::kColKt : C::kColVt), w);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_kvt));
    }
    for (int s = 0; s < n; ++s) {
      const int buf = s & 1;
      const bool got = bounded_wait(smem_u32(&bar_s_full[buf]), (s >> 1) & 1, abort_ptr, p.status,
                                    kSiteSFull);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const uint32_t st = stage_addr(s);
      const float4* lse4 =
          reinterpret_cast<const float4*>(sgen + (st - sbase) + 2 * C::kQTileBytes) + qb / 4;
      const float4* del4 = lse4 + BQ / 4;
      const int q0 = q0p + step_qt(s) * BQ;  // position of the step's first query
      uint32_t sv[32], dpv[32];
      tmem_ld32x2(tmem + lane_base + C::col_st(buf) + qb, tmem + lane_base + C::col_dpt(buf) + qb,
                  sv, dpv);
      uint32_t pk[16], dk[16];
      // keys after the query are masked on the diagonal steps only: query columns
      // below lim; the other steps take the loop without the selects
      const int lim = (p.causal && q0 < k0p + kTile) ? key - q0 - qb : -1;
      auto columns = [&](auto masked) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float4 l4 = lse4[g];
          const float4 d4 = del4[g];
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
          const float dl[4] = {d4.x, d4.y, d4.z, d4.w};
          float pr[4], dsv[4];
#pragma unroll
          for (int e = 0; e < 4; e += 2) {  // two query columns per packed f32x2 operation
            const float2 x = ffma2(make_float2(__uint_as_float(sv[4 * g + e]),
                                               __uint_as_float(sv[4 * g + e + 1])),
                                   make_float2(sl2, sl2), make_float2(-lv[e], -lv[e + 1]));
            float2 pv = make_float2(ex2(x.x), ex2(x.y));
            if constexpr (decltype(masked)::value) {
              pv.x = (4 * g + e < lim) ? 0.f : pv.x;
              pv.y = (4 * g + e + 1 < lim) ? 0.f : pv.y;
            }
            const float2 dp = fsub2(make_float2(__uint_as_float(dpv[4 * g + e]),
                                                __uint_as_float(dpv[4 * g + e + 1])),
                                    make_float2(dl[e], dl[e + 1]));
            const float2 ds = fmul2(pv, dp);
            pr[e] = pv.x;
            pr[e + 1] = pv.y;
            dsv[e] = ds.x;
            dsv[e + 1] = ds.y;
          }
          pk[2 * g] = pack_fp16(pr[0], pr[1]);
          pk[2 * g + 1] = pack_fp16(pr[2], pr[3]);
          dk[2 * g] = pack_fp16(dsv[0], dsv[1]);
          dk[2 * g + 1] = pack_fp16(dsv[2], dsv[3]);
        }
      };
      if (__any_sync(0xffffffffu, lim > 0)) columns(std::true_type{});
      else columns(std::false_type{});
      // Pᵀ and dSᵀ over this half's own (already read) Sᵀ columns. The previous
      // readers of these TMEM columns and of this step's dSᵀ shared-memory buffer
      // belong to earlier steps whose MMAs were issued before Sᵀ(s), so they had
      // completed when s_full(s) arrived.
      tmem_st32(tmem + lane_base + C::col_st(buf) + qb, pk, dk);
      // dSᵀ row r, query columns qb..qb+31 (chunks 4*half ..), swizzled K-major
      const uint32_t dsb = ds_addr(s);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        st_shared_v4(dsb + sw128_offset(r, half * 4 + q4), dk[4 * q4], dk[4 * q4 + 1],
                     dk[4 * q4 + 2], dk[4 * q4 + 3]);
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_ds_full[buf]));
    }
    // ------------------------------------------------------------ dK / dV epilogue
    bounded_wait(smem_u32(&bar_done), 0, abort_ptr, p.status, kSiteDone);
    __syncwarp();
    tc_fence_after();
    const long long grow = kv_row + r;
    const bool sum_parts = nparts > 1;  // another CTA adds into the same dk/dv rows
    if (n == 0) {
      // no query of the block sees these keys: dk = dv = 0 (summed rows start at 0)
      if (!sum_parts && bounds_ok(grow < rows_kv, p.status, kChkDkdv)) {
        float4* dst = reinterpret_cast<float4*>((half == 0 ? p.dv : p.dk) + grow * D);
#pragma unroll
        for (int i = 0; i < D / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else {
      // Rows go to shared memory (conflict-free swizzled 16-byte chunks) and leave in
      // 128-row TMA tiles (added into the rows when two CTAs share the key tile), so
      // that no warp issues scattered row-per-thread stores.
      auto at = [&](uint32_t base, int col) {  // fp32 column col of this thread's row
        return base + static_cast<uint32_t>((col / 32) * C::kBoxBytes + r * 128 +
                                            ((((col % 32) / 4) ^ (r & 7)) << 4));
      };
      const uint32_t tcos = sbase + C::kEpiCos, tsin = sbase + C::kEpiSin;
      const uint32_t stage = sbase + (half == 0 ? C::kEpiDv : C::kEpiDk);
      if (half == 0) {
        // dV accumulated Pᵀ (dO 2^edo)
        const float f = exp2i(-ex.dout);
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t u[32];
          tmem_ld32(tmem + lane_base + C::kColDV + cc * 32, u);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_shared_v4(at(stage, cc * 32 + 4 * i), __float_as_uint(f * __uint_as_float(u[4 * i])),
                         __float_as_uint(f * __uint_as_float(u[4 * i + 1])),
                         __float_as_uint(f * __uint_as_float(u[4 * i + 2])),
                         __float_as_uint(f * __uint_as_float(u[4 * i + 3])));
        }
      } else {
        // dk = scale * R_keyᵀ dk~ (rotation by -angle); dK accumulated
        // (dS 2^(edo+ev)) (q~ 2^eq). The cos / sin rows of the tile's keys arrive by TMA.
        if (r == 0) {
          mbar_arrive_expect_tx(smem_u32(&bar_tab), 2 * C::kTabBoxes * C::kBoxBytes);
          if (bounds_ok(k0p + kTile <= p.tab_rows, p.status, kChkTab))
          for (int bx = 0; bx < C::kTabBoxes; ++bx) {
            tma_load_2d(tcos + bx * C::kBoxBytes, &p.map_cos, bx * 32, k0p, smem_u32(&bar_tab));
            tma_load_2d(tsin + bx * C::kBoxBytes, &p.map_sin, bx * 32, k0p, smem_u32(&bar_tab));
          }
        }
        const float f = p.scale * exp2i(-(ex.dout + ex.v + ex.q));
        const bool got = bounded_wait(smem_u32(&bar_tab), 0, abort_ptr, p.status, kSiteTab);
        if (got) {
          auto tab4 = [&](uint32_t base, int fq, float (&o)[4]) {  // frequencies fq..fq+3
            uint32_t w0, w1, w2, w3;
            ld_shared_v4(at(base, fq), w0, w1, w2, w3);
            o[0] = __uint_as_float(w0); o[1] = __uint_as_float(w1);
            o[2] = __uint_as_float(w2); o[3] = __uint_as_float(w3);
          };
          auto put = [&](int col, float a, float b, float c, float d) {
            st_shared_v4(at(stage, col), __float_as_uint(a), __float_as_uint(b), __float_as_uint(c),
                         __float_as_uint(d));
          };
          if (p.rope_interleaved) {
            // complex pairs (2j, 2j+1) at frequency j: columns [64 ch, 64 ch + 64) hold
            // the frequencies [32 ch, 32 ch + 32)
#pragma unroll 1
            for (int ch = 0; ch < D / 64; ++ch) {
              uint32_t x1[32], x2[32];
              tmem_ld32x2(tmem + lane_base + C::kColDK + ch * 64,
                          tmem + lane_base + C::kColDK + ch * 64 + 32, x1, x2);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                float cc[4], ss[4];
                tab4(tcos, ch * 32 + 4 * i, cc);
                tab4(tsin, ch * 32 + 4 * i, ss);
                float y[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int k = 8 * (i & 3) + 2 * e;
                  const float xe = __uint_as_float(i < 4 ? x1[k] : x2[k]);
                  const float xo = __uint_as_float(i < 4 ? x1[k + 1] : x2[k + 1]);
                  y[2 * e] = f * (xe * cc[e] + xo * ss[e]);
                  y[2 * e + 1] = f * (xo * cc[e] - xe * ss[e]);
                }
                put(ch * 64 + 8 * i, y[0], y[1], y[2], y[3]);
                put(ch * 64 + 8 * i + 4, y[4], y[5], y[6], y[7]);
              }
            }
          } else {
#pragma unroll 1
            for (int ch = 0; ch < D / 64; ++ch) {
              uint32_t x1[32], x2[32];
              tmem_ld32x2(tmem + lane_base + C::kColDK + ch * 32,
                          tmem + lane_base + C::kColDK + D / 2 + ch * 32, x1, x2);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                float cc[4], ss[4];
                tab4(tcos, ch * 32 + 4 * i, cc);
                tab4(tsin, ch * 32 + 4 * i, ss);
                float y1[4], y2[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float a = __uint_as_float(x1[4 * i + e]);
                  const float bb = __uint_as_float(x2[4 * i + e]);
                  y1[e] = f * (a * cc[e] + bb * ss[e]);
                  y2[e] = f * (bb * cc[e] - a * ss[e]);
                }
                put(ch * 32 + 4 * i, y1[0], y1[1], y1[2], y1[3]);
                put(D / 2 + ch * 32 + 4 * i, y2[0], y2[1], y2[2], y2[3]);
              }
            }
          }
        }
      }
      // this half's 128 rows are staged: one thread stores (or adds) the tiles
      fence_async_smem();
      named_bar_sync(1 + half, 128);
      if (r == 0) {
        const CUtensorMap* map = half == 0 ? &p.map_dv : &p.map_dk;
        if (bounds_ok(kv_row + kTile <= rows_kv, p.status, kChkDkdv))
        for (int bx = 0; bx < D / 32; ++bx) {
          if (sum_parts) tma_reduce_add_2d(map, bx * 32, kv_row, stage + bx * C::kBoxBytes);
          else tma_store_2d(map, bx * 32, kv_row, stage + bx * C::kBoxBytes);
        }
        bulk_commit();
        bulk_wait_read_all();  // the tiles have left shared memory before the CTA ends
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_bwd_d(const BwdParams& p, cudaStream_t stream) {
  using C = BwdCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  long long ctas = 0;
  if (p.nplan > 0) {
    for (int e = 0; e < p.nplan; ++e) ctas += p.plan_parts[e];
    ctas *= static_cast<long long>(p.B) * p.Hkv;
  } else {
    ctas = static_cast<long long>(p.Skv / kTile) * p.B * p.Hkv * p.hsplit;
  }
  const unsigned grid = static_cast<unsigned>(ctas);
  return launch_pdl(attn_bwd_kernel<D>, dim3(grid), dim3(kThreads), C::kSmemBytes, stream, p);
}

}  // namespace

cudaError_t launch_bwd_main(const BwdParams& p, cudaStream_t stream) {
  return p.D == 128 ? launch_bwd_d<128>(p, stream) : launch_bwd_d<64>(p, stream);
}

}  // namespace gbattn
