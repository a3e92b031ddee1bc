// Forward attention kernel for sm_103a: out = softmax(scale q~ k~ᵀ + mask) v and lse.
//
// The method (pages cited by title and section):
//   scores q~_i . k~_j / sqrt(D) with keys after the query masked
//     ("深度学习系统设计llama3-from-scratch：并行计算架构", §注意力得分矩阵计算, §因果掩码的并行应用);
//   row maximum subtracted before the softmax, then P v
//     ("ColossalAI 中的 PaLM 教学实现…", §2.5 Attention);
//   IO-aware tiling that never writes the S x S score matrix to memory
//     ("Picotron模型实现解析Llama架构与Flash Attention集成", §Flash Attention的优势).
// The tiled softmax keeps, per query row, a running maximum m and sum l and
// rescales the partial output when m grows; the final out = O / l and
// lse = m + ln l equal the plain definition up to rounding.
//
// GB300 design: at D = 128 one CTA owns two 128-row query tiles (2c, 2c+1) of one
// head and streams the 128-key K/V tiles of its KV head through a TMA ring. Warp
// roles:
//   warps 0-3 / 4-7  softmax for query tile 0 / 1 (one thread per row),
//   warp 8           TMA producer (Q once, then K_j, V_j into the ring),
//   warp 9           tcgen05 MMA issuer (one thread) and TMEM owner.
// TMEM (512 columns): S_0, S_1 (128 fp32 columns each), O_0, O_1 (D columns
// each). P_t is written back as packed bf16 into the first 64 columns of S_t
// and consumed from TMEM by the P.V MMA. While one tile's softmax runs, the
// tensor core works on the other tile's MMAs. KV tiles above the diagonal are
// never loaded; only the diagonal tile is masked.
// At D = 64 a CTA works on one query tile at a time (warps 0-3 softmax, 4 producer, 5
// MMA; 256 TMEM columns) and two CTAs share an SM: the tensor core alternates between
// their tiles as it does between the two tiles of one CTA at D = 128, and one CTA's
// fixed parts (Q landing, first scores, epilogue) overlap the other's steps. At the
// D = 64 shapes measured (S = 1024, 2048) a query tile sees 4.5-8.5 K/V tiles on
// average, so those fixed parts would otherwise be a large share of a tile's time.
// The persistent form below (attn_fwd_persist_kernel) also keeps the CTAs resident
// across tiles; the one-tile-per-CTA form remains for blocks where a query tile may
// see no key.
#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

using namespace gb;

constexpr float kLn2 = 0.6931471805599453f;

// Wait-site codes reported in the status word.
enum : int {
  kSiteQ = 1, kSiteKvFull = 2, kSiteKvEmpty = 3, kSiteSFull = 4, kSitePFull = 5,
  kSiteODone = 6, kSiteInject = 7,
  // index checks of the debug build
  kChkKv = 8, kChkQ = 9, kChkOut = 10, kChkLse = 11
};

template <int D>
struct FwdCfg {
  static constexpr int kTiles = D == 128 ? 2 : 1;      // query tiles per CTA
  static constexpr int kThreads = 128 * kTiles + 64;   // softmax warps, producer, MMA
  static constexpr int kWarpLoad = 4 * kTiles;
  static constexpr int kWarpMma = 4 * kTiles + 1;
  static constexpr int kMinBlocks = 3 - kTiles;        // CTAs per SM the launch asks for
  static constexpr uint32_t kTmemCols = 256u * kTiles;
  static constexpr int kRegionBytes = 128 * 128;       // 128 rows x 128 B (64 bf16)
  static constexpr int kRegions = D / 64;
  static constexpr int kTileBytes = kRegions * kRegionBytes;
  static constexpr int kSlots = 5;                     // K/V ring depth (tiles)
  static constexpr int kKvOff = kTiles * kTileBytes;   // after the Q tiles
  static constexpr int kSmemBytes = kKvOff + kSlots * kTileBytes + 1024;
  __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __device__ static constexpr uint32_t col_o(int t) { return 128u * kTiles + D * t; }
  static_assert(col_o(kTiles - 1) + D <= kTmemCols, "TMEM budget");
  static_assert(kMinBlocks * (kSmemBytes + 1024) <= 233472, "shared memory per SM");
};

// Packed fp32 pairs (fma.rn.f32x2 / add.rn.f32x2: one instruction for two lanes'
// worth of the same operation, each rounded as the scalar form) and the
// three-input maximum.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  uint64_t ra, rb, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}


// 128 consecutive 32-bit TMEM columns of this thread's lane in one load, one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}

// Waits for a phase without looking at the abort flag (used to drain copies
// and MMAs that were already issued before the CTA releases its resources).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs / 4) return;
  }
}

template <int D>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, FwdCfg<D>::kMinBlocks)
    attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int kTiles = C::kTiles;
  constexpr int kWarpLoad = C::kWarpLoad;
  constexpr int kWarpMma = C::kWarpMma;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_drain, bar_never;
  __shared__ __align__(8) uint64_t bar_kv_full[C::kSlots], bar_kv_empty[C::kSlots];
  __shared__ __align__(8) uint64_t bar_s_full[kTiles], bar_p_full[kTiles], bar_o_done[kTiles];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;

  // ---- work item: the query tiles kTiles c .. kTiles c + kTiles - 1 of one head,
  // heaviest first
  const int nq = p.Sq / kTile;
  const int nkv = p.Skv / kTile;
  const int nitems = (nq + kTiles - 1) / kTiles;
  const int BH = p.B * p.Hq;
  const int c = nitems - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int b = bh / p.Hq;
  const int h = bh % p.Hq;
  const int hkv = h / (p.Hq / p.Hkv);
  // KV tiles seen by query tile kTiles c + t: those at or before its position when
  // causal (0 when that tile is past the end, or precedes the whole K/V block)
  auto tiles_of = [&](int t) {
    if (t >= kTiles) return 0;
    const int qt = kTiles * c + t;
    if (qt >= nq) return 0;
    if (!p.causal) return nkv;
    const int vis = p.q_tile0 + qt - p.kv_tile0 + 1;
    return vis < 0 ? 0 : (vis > nkv ? nkv : vis);
  };
  const int n_0 = tiles_of(0);
  const int n_1 = tiles_of(1);
  const int n = n_0 > n_1 ? n_0 : n_1;
  // The K/V tiles stream from the last visible one down to tile 0: stream position j
  // holds K/V tile n - 1 - j, and query tile t (which sees tiles 0 .. n_t - 1) joins at
  // position n - n_t with its diagonal tile. Tile 2c+1 sees one tile more than 2c, so
  // its extra step comes first and both tiles end on tile 0 together: the CTA's two
  // epilogues run side by side instead of one waiting for the other's last step.
  auto start_of = [&](int t) { return n - (t ? n_1 : n_0); };
  const int kv_valid = p.kv_valid > 0 ? p.kv_valid : p.Skv;  // keys that exist per head
  const int q_row0 = bh * p.Sq;
  const int kv_row0 = (b * p.Hkv + hkv) * p.Skv;
  const long long rows_q = static_cast<long long>(p.B) * p.Hq * p.Sq;  // rows of q~, out, lse
  const long long rows_kv = static_cast<long long>(p.B) * p.Hkv * p.Skv;

  // ---- setup. The producer's lane initialises the barriers and, as soon as the
  // previous kernel's writes are visible, starts the Q loads and fills the K/V ring
  // while the MMA warp allocates tensor memory.
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  const bool producer = warp == kWarpLoad && lane == 0;
  int issued = 0;  // K/V ring loads issued (producer lane)
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
    const long long row = kv_row0 + static_cast<long long>(n - 1 - (i >> 1)) * kTile;
    if (bounds_ok(row + kTile <= rows_kv, p.status, kChkKv))
      for (int r = 0; r < C::kRegions; ++r)
        tma_load_2d(dst + r * C::kRegionBytes, map, r * 64, static_cast<int>(row), full);
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
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(smem_u32(&bar_s_full[t]), 1);
      mbar_init(smem_u32(&bar_p_full[t]), 128);
      mbar_init(smem_u32(&bar_o_done[t]), 1);
    }
    fence_mbar_init();
    pdl_wait();  // q~, k~ come from the pre-pass before this kernel
    tma_prefetch_desc(&p.map_q);
    tma_prefetch_desc(&p.map_k);
    tma_prefetch_desc(&p.map_v);
    const int nvalid = (n_0 > 0) + (n_1 > 0);
    mbar_arrive_expect_tx(smem_u32(&bar_q), nvalid * C::kTileBytes);
    for (int t = 0; t < kTiles; ++t) {
      if ((t ? n_1 : n_0) == 0) continue;
      if (!bounds_ok(q_row0 + (static_cast<long long>(kTiles) * c + t + 1) * kTile <= rows_q,
                     p.status, kChkQ))
        continue;
      for (int r = 0; r < C::kRegions; ++r)
        tma_load_2d(sbase + t * C::kTileBytes + r * C::kRegionBytes, &p.map_q, r * 64,
                    q_row0 + (kTiles * c + t) * kTile, smem_u32(&bar_q));
    }
    while (issued < 2 * n && issued < C::kSlots && issue_kv(issued)) ++issued;  // free slots
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

  if (warp == kWarpLoad) {
    // ================================================================ producer
    if (lane == 0) {
      while (issued < 2 * n && issue_kv(issued)) ++issued;
      // Loads already issued land before the CTA releases its shared memory (a
      // no-op in a healthy run). Each slot has at most one load in flight: a load
      // is issued only after the previous one in its slot was consumed.
      drain_wait(smem_u32(&bar_q), 0);
      for (int i = issued - C::kSlots > 0 ? issued - C::kSlots : 0; i < issued; ++i)
        drain_wait(smem_u32(&bar_kv_full[i % C::kSlots]), (i / C::kSlots) & 1);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ================================================================ MMA issuer
    // The whole warp runs this loop with warp-uniform operands; elect.sync inside
    // the MMA / commit wrappers lets one lane issue.
    constexpr uint32_t idesc_qk = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16(128, D, 0, 1);
    constexpr uint64_t kKmaj = sdesc_hi(16, 1024);                 // K-major operand
    constexpr uint64_t kMnV = sdesc_hi(C::kRegionBytes, 1024);     // MN-major V
    auto desc = [](uint64_t hi, uint32_t addr) { return hi | static_cast<uint64_t>(addr >> 4); };
    auto wait = [&](uint32_t bar, uint32_t parity, int site) {
      return __all_sync(0xffffffffu, bounded_wait(bar, parity, abort_ptr, p.status, site));
    };
    auto slot_addr = [&](int i) { return sbase + C::kKvOff + (i % C::kSlots) * C::kTileBytes; };
    auto wait_kv = [&](int i) {
      return wait(smem_u32(&bar_kv_full[i % C::kSlots]), (i / C::kSlots) & 1, kSiteKvFull);
    };
    auto issue_qk = [&](int t, uint32_t kaddr) {
      const uint32_t qaddr = sbase + t * C::kTileBytes;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * C::kRegionBytes + (kk & 3) * 32;
        mma_ss_w(tmem + C::col_s(t), desc(kKmaj, qaddr + off), desc(kKmaj, kaddr + off), idesc_qk,
                 kk > 0);
      }
    };
    auto issue_pv = [&](int t, uint32_t vaddr, bool acc) {
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_ts_w(tmem + C::col_o(t), tmem + C::col_s(t) + kk * 8, desc(kMnV, vaddr + kk * 16 * 128),
                 idesc_pv, (acc || kk > 0) ? 1u : 0u);
    };

    bool ok = true;
    if (p.inject_timeout)  // nothing ever arrives on bar_never
      ok = wait(smem_u32(&bar_never), 0, kSiteInject);
    ok = ok && wait(smem_u32(&bar_q), 0, kSiteQ);
    ok = ok && n > 0 && wait_kv(0);  // n = 0: both query tiles see no key of the block
    if (ok) {
      tc_fence_after();
      for (int t = 0; t < kTiles; ++t) {
        if ((t ? n_1 : n_0) == 0 || start_of(t) > 0) continue;
        issue_qk(t, slot_addr(0));
        mma_commit_w(smem_u32(&bar_s_full[t]));
      }
      mma_commit_w(smem_u32(&bar_kv_empty[0]));
    }
    for (int j = 0; j < n && ok; ++j) {
      const int iv = 2 * j + 1;  // ring index of V_j
      const int ik = 2 * j + 2;  // ring index of K_{j+1}
      const bool next = j + 1 < n;
      ok = wait_kv(iv) && (!next || wait_kv(ik));
      if (!ok) break;
      for (int t = 0; t < kTiles && ok; ++t) {
        const int nt = t ? n_1 : n_0;
        const int jt = j - start_of(t);  // the tile's own step
        if (nt > 0 && jt >= 0) {
          ok = wait(smem_u32(&bar_p_full[t]), jt & 1, kSitePFull);
          if (!ok) break;
          tc_fence_after();
          issue_pv(t, slot_addr(iv), jt > 0);
          if (jt == nt - 1) mma_commit_w(smem_u32(&bar_o_done[t]));
        }
        if (next && nt > 0 && jt + 1 >= 0) {  // the tile's next step, maybe its first
          issue_qk(t, slot_addr(ik));
          mma_commit_w(smem_u32(&bar_s_full[t]));
        }
      }
      if (!ok) break;
      mma_commit_w(smem_u32(&bar_kv_empty[iv % C::kSlots]));
      if (next) mma_commit_w(smem_u32(&bar_kv_empty[ik % C::kSlots]));
    }
    // Every MMA issued above completes before the tensor memory is released.
    mma_commit_w(smem_u32(&bar_drain));
    drain_wait(smem_u32(&bar_drain), 0);
    __syncwarp();
  } else {
    // ================================================================ softmax
    const int t = warp >> 2;
    const int r = tid & 127;  // row in the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::col_s(t);
    const uint32_t tO = tmem + lane_base + C::col_o(t);
    const int nt = t ? n_1 : n_0;
    const int qt = kTiles * c + t;
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running maximum, base-2 units (scores * scale * log2 e)
    float l = 0.f;        // running sum of 2^(score2 - m)
    for (int j = 0; j < nt; ++j) {
      const bool got = bounded_wait(smem_u32(&bar_s_full[t]), j & 1, abort_ptr, p.status, kSiteSFull);
      if (!__all_sync(0xffffffffu, got)) break;
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
      const int kvj = nt - 1 - j;  // the K/V tile of this step (see start_of)
      if (p.causal && p.kv_tile0 + kvj == p.q_tile0 + qt) {  // diagonal tile: keys after the query are masked
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = i > r ? -INFINITY : s[i];
      }
      if (!p.causal && (kvj + 1) * kTile > kv_valid) {  // padding keys of the last tile
        const int lim = kv_valid - kvj * kTile;
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = i >= lim ? -INFINITY : s[i];
      }
      // Row maximum as 4 independent chains of three-input maxima (the softmax warps'
      // instruction issue, not the tensor core, is what a step waits for).
      float mp[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) mp[k] = fmaxf(s[k], s[k + 4]);
#pragma unroll
      for (int i = 8; i < 128; i += 8)
#pragma unroll
        for (int k = 0; k < 4; ++k) mp[k] = fmax3(mp[k], s[i + k], s[i + 4 + k]);
      const float mx = fmax3(fmax3(mp[0], mp[1], mp[2]), mp[3], mp[3]);
      const float mx2 = mx * sl2;
      float alpha = 1.f;
      bool grew = false;
      // Lazy rescaling: keep the old maximum unless the row maximum grew by more
      // than 2^8; probabilities then stay below 256, well inside fp32 / bf16.
      if (mx2 > m + 8.f) {
        alpha = ex2(m - mx2);  // 0 on the first tile (m = -inf)
        grew = true;
        m = mx2;
      }
      // exponent arguments and partial row sums two columns at a time (packed f32x2)
      float2 rp[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
      const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(-m, -m);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 x =
              ffma2(make_float2(s[hh * 64 + 2 * i], s[hh * 64 + 2 * i + 1]), sl2x2, negm);
          const float2 a = make_float2(ex2(x.x), ex2(x.y));
          rp[i & 3] = fadd2(rp[i & 3], a);
          pk[i] = pack_bf16(a.x, a.y);
        }
        tmem_st32(tS + hh * 32, pk);
      }
      const float2 r2 = fadd2(fadd2(rp[0], rp[1]), fadd2(rp[2], rp[3]));
      const float rs = r2.x + r2.y;
      l = l * alpha + rs;
      if (j > 0 && __any_sync(0xffffffffu, grew)) {
        const float f = grew ? alpha : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t u[32];
          tmem_ld32(tO + cc * 32, u);
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * f);
          tmem_st32(tO + cc * 32, u);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_p_full[t]));
    }
    if (nt > 0) {
      // ------------------------------------------------------------ epilogue
      bounded_wait(smem_u32(&bar_o_done[t]), 0, abort_ptr, p.status, kSiteODone);
      __syncwarp();
      tc_fence_after();
      const float inv_l = 1.f / l;
      const uint32_t obuf = sbase + t * C::kTileBytes;  // Q_t is no longer read
#pragma unroll
      for (int c2 = 0; c2 < D / 64; ++c2) {  // 64 columns (one swizzle region) per wait
        uint32_t u[2][32];
        tmem_ld32x2(tO + c2 * 64, tO + c2 * 64 + 32, u[0], u[1]);
        const uint32_t region = obuf + c2 * C::kRegionBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16(__uint_as_float(u[h][8 * q4 + 2 * e]) * inv_l,
                               __uint_as_float(u[h][8 * q4 + 2 * e + 1]) * inv_l);
            st_shared_v4(region + sw128_offset(r, 4 * h + q4), w[0], w[1], w[2], w[3]);
          }
      }
      fence_async_smem();
      named_bar_sync(1 + t, 128);
      if (r == 0) {
        if (bounds_ok(q_row0 + (qt + 1LL) * kTile <= rows_q, p.status, kChkOut))
          for (int rg = 0; rg < C::kRegions; ++rg)
            tma_store_2d(&p.map_out, rg * 64, q_row0 + qt * kTile, obuf + rg * C::kRegionBytes);
        bulk_commit();
        bulk_wait_read_all();
      }
      const long long lrow = static_cast<long long>(q_row0) + qt * kTile + r;
      if (bounds_ok(lrow < rows_q, p.status, kChkLse)) p.lse[lrow] = (m + log2f(l)) * kLn2;
    } else if (qt < nq) {
      // a query tile that sees no key of the block: out = 0, lse = -inf
      const long long row = static_cast<long long>(q_row0) + qt * kTile + r;
      if (bounds_ok(row < rows_q, p.status, kChkOut)) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + row * D);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
        p.lse[row] = -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- D = 64, persistent
// At D = 64 a CTA's own start (the Q tile landing, ~1 µs) and the gap before the next
// CTA takes its place (~1.2 µs) are as long as a query tile's loop of a few K/V tiles.
// This form keeps two CTAs per SM for the whole launch. Each takes query tiles, heaviest
// first, from a counter (its first tile is blockIdx.x) and runs them back to back.
// The producer loads a tile's Q into one of two buffers while the previous tile still
// streams its K/V. P has tensor-memory columns of its own (S [0,128), P [128,192), O
// [192,256)), so the scores of the next K/V tile are computed as soon as the softmax
// has read the current ones into registers, beside its exponentials, instead of after
// the P.V product. A tile's Q buffer holds its output for the store.
// Every query tile must see at least one K/V tile (the host checks that).
struct PersistCfg {
  static constexpr int kThreads = 192;  // warps 0-3 softmax, 4 producer, 5 MMA
  static constexpr int kWarpLoad = 4;
  static constexpr int kWarpMma = 5;
  static constexpr uint32_t kTmemCols = 256;  // S [0,128), P [128,192) (bf16), O [192,256)
  static constexpr int kTileBytes = 128 * 128;  // 128 rows x 64 bf16
  static constexpr int kSlots = 4;              // K/V ring depth (tiles)
  static constexpr int kKvOff = 2 * kTileBytes;  // after the two Q buffers
  static constexpr int kSmemBytes = kKvOff + kSlots * kTileBytes + 1024;
  static constexpr uint32_t kColP = 128;
  static constexpr uint32_t kColO = 192;
  static_assert(2 * (kSmemBytes + 1024 + 1024) <= 233472, "two CTAs per SM");
};
enum : int { kSiteUnit = 12, kSiteUnitEmpty = 13, kSiteQEmpty = 14, kSiteOEmpty = 15, kSiteStg = 16 };

__global__ void __launch_bounds__(PersistCfg::kThreads, 2)
    attn_fwd_persist_kernel(const __grid_constant__ FwdParams p) {
  using C = PersistCfg;
  constexpr int D = 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_unit_full[2], bar_unit_empty[2], bar_q_full[2], bar_q_empty[2];
  __shared__ __align__(8) uint64_t bar_kv_full[C::kSlots], bar_kv_empty[C::kSlots];
  __shared__ __align__(8) uint64_t bar_s_full, bar_s_free, bar_p_full, bar_p_free;
  __shared__ __align__(8) uint64_t bar_o_done, bar_o_empty, bar_stg;
  __shared__ __align__(8) uint64_t bar_drain, bar_never;
  __shared__ int unit_rec[2][2];  // (query tile unit, its K/V tiles); unit -1: none left
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int nq = p.Sq / kTile;
  const int nkv = p.Skv / kTile;
  const int BH = p.B * p.Hq;
  const int units = nq * BH;
  const int kv_valid = p.kv_valid > 0 ? p.kv_valid : p.Skv;
  const long long rows_q = static_cast<long long>(p.B) * p.Hq * p.Sq;
  const long long rows_kv = static_cast<long long>(p.B) * p.Hkv * p.Skv;
  // unit u: query tile nq - 1 - u / BH of head u % BH (causal: heaviest first)
  auto unit_qt = [&](int u) { return nq - 1 - u / BH; };
  auto unit_bh = [&](int u) { return u % BH; };
  auto tiles_of = [&](int u) {
    if (!p.causal) return nkv;
    const int vis = p.q_tile0 + unit_qt(u) - p.kv_tile0 + 1;
    return vis < 0 ? 0 : (vis > nkv ? nkv : vis);
  };
  auto qbuf = [&](int k) { return sbase + (k & 1) * C::kTileBytes; };
  auto slot_addr = [&](int i) { return sbase + C::kKvOff + (i % C::kSlots) * C::kTileBytes; };

  if (warp == C::kWarpMma) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == C::kWarpLoad && lane == 0) {
    abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bar_unit_full[s]), 1);
      mbar_init(smem_u32(&bar_unit_empty[s]), 5);  // the MMA warp and the 4 softmax warps
      mbar_init(smem_u32(&bar_q_full[s]), 1);
      mbar_init(smem_u32(&bar_q_empty[s]), 1);
    }
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(smem_u32(&bar_kv_full[s]), 1);
      mbar_init(smem_u32(&bar_kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar_s_full), 1);
    mbar_init(smem_u32(&bar_s_free), 128);
    mbar_init(smem_u32(&bar_p_full), 128);
    mbar_init(smem_u32(&bar_p_free), 1);
    mbar_init(smem_u32(&bar_o_done), 1);
    mbar_init(smem_u32(&bar_o_empty), 128);
    mbar_init(smem_u32(&bar_stg), 128);
    mbar_init(smem_u32(&bar_drain), 1);
    mbar_init(smem_u32(&bar_never), 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_ptr = &abort_flag;
  // Nothing above touched global memory: this prologue may overlap the kernel before
  // it in the stream (the RoPE pre-pass, which also zeroes the unit counter).
  pdl_wait();
  pdl_launch_dependents();

  if (warp == C::kWarpLoad) {
    // ================================================================ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.map_q);
      tma_prefetch_desc(&p.map_k);
      tma_prefetch_desc(&p.map_v);
      int issued = 0;    // K/V ring loads issued
      int q_issued = 0;  // Q loads issued
      for (int k = 0;; ++k) {
        const int s = k & 1;
        int u = k == 0 ? static_cast<int>(blockIdx.x)
                       : static_cast<int>(gridDim.x) + atomicAdd(p.unit_counter, 1);
        if (u >= units) u = -1;
        const int n = u >= 0 ? tiles_of(u) : 0;
        if (k >= 2 && !bounded_wait(smem_u32(&bar_unit_empty[s]), ((k >> 1) - 1) & 1, &abort_flag,
                                    p.status, kSiteUnitEmpty))
          break;
        unit_rec[s][0] = u;
        unit_rec[s][1] = n;
        mbar_arrive(smem_u32(&bar_unit_full[s]));
        if (u < 0) break;
        // Q into buffer s once the store of unit k-2's output (staged there) has read it
        if (k >= 2 && !bounded_wait(smem_u32(&bar_q_empty[s]), ((k >> 1) - 1) & 1, &abort_flag,
                                    p.status, kSiteQEmpty))
          break;
        const int bh = unit_bh(u);
        const long long qrow = static_cast<long long>(bh) * p.Sq + unit_qt(u) * kTile;
        mbar_arrive_expect_tx(smem_u32(&bar_q_full[s]), C::kTileBytes);
        if (bounds_ok(qrow + kTile <= rows_q, p.status, kChkQ))
          tma_load_2d(qbuf(k), &p.map_q, 0, static_cast<int>(qrow), smem_u32(&bar_q_full[s]));
        ++q_issued;
        // its K/V tiles through the ring, the diagonal one first
        const int b = bh / p.Hq;
        const int hkv = (bh % p.Hq) / (p.Hq / p.Hkv);
        const long long kv_row0 = static_cast<long long>(b * p.Hkv + hkv) * p.Skv;
        bool ok = true;
        for (int i = 0; i < 2 * n && ok; ++i, ++issued) {
          const int slot = issued % C::kSlots;
          ok = bounded_wait(smem_u32(&bar_kv_empty[slot]), ((issued / C::kSlots) & 1) ^ 1,
                            &abort_flag, p.status, kSiteKvEmpty);
          if (!ok) break;
          const uint32_t full = smem_u32(&bar_kv_full[slot]);
          mbar_arrive_expect_tx(full, C::kTileBytes);
          const long long row = kv_row0 + static_cast<long long>(n - 1 - (i >> 1)) * kTile;
          if (bounds_ok(row + kTile <= rows_kv, p.status, kChkKv))
            tma_load_2d(slot_addr(issued), (i & 1) == 0 ? &p.map_k : &p.map_v, 0,
                        static_cast<int>(row), full);
        }
        if (!ok) break;
      }
      // Loads already issued land before the CTA releases its shared memory (a no-op in
      // a healthy run): at most one per ring slot and one per Q buffer is in flight.
      for (int i = issued - C::kSlots > 0 ? issued - C::kSlots : 0; i < issued; ++i)
        drain_wait(smem_u32(&bar_kv_full[i % C::kSlots]), (i / C::kSlots) & 1);
      for (int k = q_issued - 2 > 0 ? q_issued - 2 : 0; k < q_issued; ++k)
        drain_wait(smem_u32(&bar_q_full[k & 1]), (k >> 1) & 1);
    }
    __syncwarp();
  } else if (warp == C::kWarpMma) {
    // ================================================================ MMA issuer
    constexpr uint32_t idesc_qk = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16(128, D, 0, 1);
    constexpr uint64_t kKmaj = sdesc_hi(16, 1024);
    constexpr uint64_t kMnV = sdesc_hi(C::kTileBytes, 1024);
    auto desc = [](uint64_t hi, uint32_t addr) { return hi | static_cast<uint64_t>(addr >> 4); };
    auto wait = [&](uint32_t bar, uint32_t parity, int site) {
      return __all_sync(0xffffffffu, bounded_wait(bar, parity, abort_ptr, p.status, site));
    };
    auto wait_kv = [&](int i) {
      return wait(smem_u32(&bar_kv_full[i % C::kSlots]), (i / C::kSlots) & 1, kSiteKvFull);
    };
    auto issue_qk = [&](uint32_t qaddr, uint32_t kaddr) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss_w(tmem, desc(kKmaj, qaddr + kk * 32), desc(kKmaj, kaddr + kk * 32), idesc_qk, kk > 0);
    };
    auto issue_pv = [&](uint32_t vaddr, bool acc) {
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_ts_w(tmem + C::kColO, tmem + C::kColP + kk * 8, desc(kMnV, vaddr + kk * 16 * 128),
                 idesc_pv, (acc || kk > 0) ? 1u : 0u);
    };
    bool ok = true;
    if (p.inject_timeout)  // nothing ever arrives on bar_never
      ok = wait(smem_u32(&bar_never), 0, kSiteInject);
    int base = 0;  // ring load of the unit's first K tile (K_j at base + 2j, V_j at base + 2j + 1)
    int g = 0;     // K/V tiles of all units so far (barrier phases of S and P)
    // scores of step g into S once the softmax has read step g - 1's
    auto issue_s = [&](uint32_t qaddr, int ring) {
      bool w = g == 0 || wait(smem_u32(&bar_s_free), (g - 1) & 1, kSiteSFull);
      w = w && wait_kv(ring);
      if (!w) return false;
      tc_fence_after();
      issue_qk(qaddr, slot_addr(ring));
      mma_commit_w(smem_u32(&bar_s_full));
      mma_commit_w(smem_u32(&bar_kv_empty[ring % C::kSlots]));
      return true;
    };
    for (int k = 0; ok; ++k) {
      const int s = k & 1;
      ok = wait(smem_u32(&bar_unit_full[s]), (k >> 1) & 1, kSiteUnit);
      if (!ok) break;
      const int u = unit_rec[s][0];
      const int n = unit_rec[s][1];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_unit_empty[s]));
      if (u < 0) break;
      ok = wait(smem_u32(&bar_q_full[s]), (k >> 1) & 1, kSiteQ) && issue_s(qbuf(k), base);
      if (!ok) break;
      for (int j = 0; j < n; ++j) {
        // the next tile's scores first: they need only the softmax's read of these
        if (j + 1 < n) {
          ++g;
          ok = issue_s(qbuf(k), base + 2 * j + 2);
          --g;
          if (!ok) break;
        }
        const int iv = base + 2 * j + 1;
        ok = wait_kv(iv) && wait(smem_u32(&bar_p_full), g & 1, kSitePFull);
        // O is free once the previous unit's epilogue has read it
        if (ok && j == 0 && k > 0) ok = wait(smem_u32(&bar_o_empty), (k - 1) & 1, kSiteOEmpty);
        if (!ok) break;
        tc_fence_after();
        issue_pv(slot_addr(iv), j > 0);
        mma_commit_w(smem_u32(&bar_p_free));
        if (j + 1 == n) mma_commit_w(smem_u32(&bar_o_done));
        mma_commit_w(smem_u32(&bar_kv_empty[iv % C::kSlots]));
        ++g;
      }
      base += 2 * n;
    }
    // Every MMA issued above completes before the tensor memory is released.
    mma_commit_w(smem_u32(&bar_drain));
    drain_wait(smem_u32(&bar_drain), 0);
    __syncwarp();
  } else {
    // ================================================================ softmax
    const int r = tid;  // row in the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_base;
    const float sl2 = p.scale_log2;
    int g = 0;
    // thread 0: 1 + the buffer of a store whose shared-memory reads may be in flight, or 0;
    // once they are done the buffer may take a Q tile
    int pending = 0;
    auto release = [&]() {
      if (pending) {
        bulk_wait_read_all();
        mbar_arrive(smem_u32(&bar_q_empty[pending - 1]));
        pending = 0;
      }
    };
    for (int k = 0;; ++k) {
      const int s = k & 1;
      const bool have = bounded_wait(smem_u32(&bar_unit_full[s]), (k >> 1) & 1, abort_ptr, p.status,
                                     kSiteUnit);
      if (!__all_sync(0xffffffffu, have)) break;
      const int u = unit_rec[s][0];
      const int n = unit_rec[s][1];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_unit_empty[s]));
      if (u < 0) break;
      const int qt = unit_qt(u);
      const uint32_t tO = tmem + lane_base + C::kColO;
      const uint32_t tP = tmem + lane_base + C::kColP;
      float m = -INFINITY;  // running maximum, base-2 units (scores * scale * log2 e)
      float l = 0.f;        // running sum of 2^(score2 - m)
      bool ok = true;
      for (int j = 0; j < n; ++j, ++g) {
        const bool got = bounded_wait(smem_u32(&bar_s_full), g & 1, abort_ptr, p.status, kSiteSFull);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sc[128];
        {
          uint32_t a[128];
          tmem_ld128(tS, a);
#pragma unroll
          for (int e = 0; e < 128; ++e) sc[e] = __uint_as_float(a[e]);
        }
        // the scores are in registers: the MMA warp may compute the next ones into S
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_s_free));
        const int kvj = n - 1 - j;  // the K/V tile of this step (diagonal first)
        if (p.causal && p.kv_tile0 + kvj == p.q_tile0 + qt) {
#pragma unroll
          for (int e = 0; e < 128; ++e) sc[e] = e > r ? -INFINITY : sc[e];
        }
        if (!p.causal && (kvj + 1) * kTile > kv_valid) {  // padding keys of the last tile
          const int lim = kv_valid - kvj * kTile;
#pragma unroll
          for (int e = 0; e < 128; ++e) sc[e] = e >= lim ? -INFINITY : sc[e];
        }
        float mp[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) mp[q] = fmaxf(sc[q], sc[q + 4]);
#pragma unroll
        for (int e = 8; e < 128; e += 8)
#pragma unroll
          for (int q = 0; q < 4; ++q) mp[q] = fmax3(mp[q], sc[e + q], sc[e + 4 + q]);
        const float mx = fmax3(fmax3(mp[0], mp[1], mp[2]), mp[3], mp[3]);
        const float mx2 = mx * sl2;
        float alpha = 1.f;
        bool grew = false;
        // lazy rescaling, as in the kernel above (threshold 2^8)
        if (mx2 > m + 8.f) {
          alpha = ex2(m - mx2);
          grew = true;
          m = mx2;
        }
        float2 rp[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
        const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(-m, -m);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 x =
                ffma2(make_float2(sc[hh * 64 + 2 * e], sc[hh * 64 + 2 * e + 1]), sl2x2, negm);
            const float2 a = make_float2(ex2(x.x), ex2(x.y));
            rp[e & 3] = fadd2(rp[e & 3], a);
            pk[e] = pack_bf16(a.x, a.y);
          }
          // P and O are free once the previous step's P.V product has completed
          if (hh == 0 && g > 0) {
            const bool pf =
                bounded_wait(smem_u32(&bar_p_free), (g - 1) & 1, abort_ptr, p.status, kSitePFull);
            if (!__all_sync(0xffffffffu, pf)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          tmem_st32(tP + hh * 32, pk);
        }
        if (!ok) break;
        const float2 r2 = fadd2(fadd2(rp[0], rp[1]), fadd2(rp[2], rp[3]));
        l = l * alpha + (r2.x + r2.y);
        if (j > 0 && __any_sync(0xffffffffu, grew)) {
          const float f = grew ? alpha : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(tO + cc * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_p_full));
        if (j == 0 && tid == 0) release();  // the previous unit's store, behind this step
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      const bool done = bounded_wait(smem_u32(&bar_o_done), k & 1, abort_ptr, p.status, kSiteODone);
      if (!__all_sync(0xffffffffu, done)) break;
      tc_fence_after();
      uint32_t o[2][32];
      tmem_ld32x2(tO, tO + 32, o[0], o[1]);
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_o_empty));
      const float inv_l = 1.f / l;
      const uint32_t obuf = qbuf(k);  // the unit's Q tile: its last score product is done
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16(__uint_as_float(o[h][8 * q4 + 2 * e]) * inv_l,
                             __uint_as_float(o[h][8 * q4 + 2 * e + 1]) * inv_l);
          st_shared_v4(obuf + sw128_offset(r, 4 * h + q4), w[0], w[1], w[2], w[3]);
        }
      fence_async_smem();
      mbar_arrive(smem_u32(&bar_stg));
      const long long qrow = static_cast<long long>(unit_bh(u)) * p.Sq + qt * kTile;
      if (tid == 0) {
        release();
        if (bounded_wait(smem_u32(&bar_stg), k & 1, abort_ptr, p.status, kSiteStg)) {
          if (bounds_ok(qrow + kTile <= rows_q, p.status, kChkOut))
            tma_store_2d(&p.map_out, 0, static_cast<int>(qrow), obuf);
          bulk_commit();
          pending = 1 + s;
        }
      }
      if (bounds_ok(qrow + r < rows_q, p.status, kChkLse)) p.lse[qrow + r] = (m + log2f(l)) * kLn2;
    }
    // the last store has read its buffer before the CTA releases its shared memory
    if (tid == 0 && pending) bulk_wait_read_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_fwd_d(const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int nq = p.Sq / kTile;
  const unsigned grid = static_cast<unsigned>(((nq + C::kTiles - 1) / C::kTiles) * p.B * p.Hq);
  return launch_pdl(attn_fwd_kernel<D>, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, p);
}

}  // namespace

cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream) {
  if (p.D == 128) return launch_fwd_d<128>(p, stream);
  // the persistent form needs the unit counter and a key tile for every query tile
  if (p.unit_counter != nullptr && (!p.causal || p.q_tile0 >= p.kv_tile0) && p.Skv >= kTile) {
    using C = PersistCfg;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_persist_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    const long long units = static_cast<long long>(p.Sq / kTile) * p.B * p.Hq;
    const unsigned grid = static_cast<unsigned>(units < 2LL * nsm ? units : 2LL * nsm);
    return launch_pdl(attn_fwd_persist_kernel, dim3(grid), dim3(C::kThreads), C::kSmemBytes,
                      stream, p);
  }
  return launch_fwd_d<64>(p, stream);
}

}  // namespace gbattn
