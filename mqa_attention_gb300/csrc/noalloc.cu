// attn_fwd_noalloc: the forward pass for callers that cannot allocate GPU
// memory. Some callers are not allowed to call cudaMalloc or any allocating
// routine: code that runs where an allocation could block, fail or be
// forbidden (a real-time or fixed-memory service that reserves all device
// memory up front, an embedding runtime that owns the allocator, a tool that
// must not perturb the memory pool it is observing). attn_fwd takes its
// workspace from a stream-ordered pool and caches its RoPE tables with
// cudaMalloc; this entry point instead uses a fixed array in device memory
// that the CUDA runtime reserves on each GPU where this code is loaded and
// keeps until the process exits. The first call on a device looks up the
// array's device address (cudaGetSymbolAddress, with that device current), so
// that first call belongs before any stream capture.
//
// The array holds, for one call: the RoPE cos/sin table and the rotated q and k.
// Every call on a device uses the same array and leaves its contents behind;
// everything in it is fully rewritten before it is read. Two calls whose work
// overlaps on the GPU (different streams, or different host threads) race on
// the array and produce undefined results: serialise them. A kernel wait that
// expires is recorded in the library's status word (a static device variable,
// found without allocating), which attn_sync_status reads.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // ATTN_FWD_NOALLOC_SCRATCH_BYTES
static_assert(kScratchBytes == ATTN_FWD_NOALLOC_SCRATCH_BYTES, "header and library disagree");

static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};  // device address of g_fwd_scratch, per device

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Device address of the array for the current device; looked up once per
// device (with that device current) and remembered.
int scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || p == nullptr)
      return ATTN_ERR_CUDA;
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return ATTN_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool map_bf16(CUtensorMap* m, const void* ptr, long long rows, int D) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(gbattn::kTile)};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out,
                                float* lse, int B, int Hq, int Hkv, int S, int D,
                                float rope_theta, float scale, int causal, attn_stream_t stream_) {
  // Argument rules are those of attn_fwd.
  const void* ptrs[] = {q, k, v, out, lse};
  for (const void* p : ptrs)
    if (!aligned16(p)) return ATTN_ERR_INVALID;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || D <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID;
  if (!std::isfinite(rope_theta) || rope_theta <= 0.f || !std::isfinite(scale) || scale <= 0.f)
    return ATTN_ERR_INVALID;
  if (static_cast<long long>(B) * Hq * S >= (1LL << 31)) return ATTN_ERR_INVALID;
  if ((D != 64 && D != 128) || S % gbattn::kTile != 0) return ATTN_ERR_UNSUPPORTED;

  // Scratch layout: table (cos hi | sin hi | cos lo | sin lo) | rotated q | rotated k |
  // the forward's unit counter (256 bytes).
  const long long qrows = static_cast<long long>(B) * Hq * S;
  const long long krows = static_cast<long long>(B) * Hkv * S;
  const long long tab_n = (static_cast<long long>(S) * (D / 2) + 63) / 64 * 64;  // floats per array
  const size_t tab = static_cast<size_t>(tab_n) * sizeof(float);
  const size_t qbytes = round256(static_cast<size_t>(qrows) * D * 2);
  const size_t kbytes = round256(static_cast<size_t>(krows) * D * 2);
  const size_t need = 4 * tab + qbytes + kbytes + 256;
  if (need > kScratchBytes) return ATTN_ERR_UNSUPPORTED;  // beyond the fixed array

  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;
  void* base = nullptr;
  int st = scratch_address(dev, &base);
  if (st != ATTN_OK) return st;
  int* status = nullptr;
  if ((st = gbattn::device_status_word(&status)) != ATTN_OK) return st;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t* w = static_cast<uint8_t*>(base);
  float* tabp = reinterpret_cast<float*>(w);
  void* qr = w + 4 * tab;
  void* kr = w + 4 * tab + qbytes;
  int* counter = reinterpret_cast<int*>(w + 4 * tab + qbytes + kbytes);

  bool ok = gbattn::launch_rope_table(tabp, tab_n, S, D, static_cast<double>(rope_theta),
                                      stream) == cudaSuccess;
  gbattn::RowPrepParams rp{};
  rp.status = status;
  rp.bwd = 0;
  rp.D = D;
  rp.cos_tab = tabp;
  rp.sin_tab = tabp + tab_n;
  rp.cos_lo = tabp + 2 * tab_n;
  rp.sin_lo = tabp + 3 * tab_n;
  rp.tab_rows = S;
  rp.seg[0] = {q, qr, nullptr, nullptr, qrows, S, S, 0};
  rp.seg[1] = {k, kr, nullptr, nullptr, krows, S, S, 0};
  rp.zero_word = counter;
  ok = ok && gbattn::launch_row_prep(rp, stream) == cudaSuccess;
  gbattn::FwdParams fp{};
  ok = ok && map_bf16(&fp.map_q, qr, qrows, D) && map_bf16(&fp.map_k, kr, krows, D) &&
       map_bf16(&fp.map_v, v, krows, D) && map_bf16(&fp.map_out, out, qrows, D);
  if (!ok) return ATTN_ERR_CUDA;
  fp.lse = lse;
  fp.status = status;
  fp.B = B; fp.Hq = Hq; fp.Hkv = Hkv; fp.Sq = S; fp.Skv = S; fp.D = D;
  fp.out = out;
  fp.kv_valid = S;
  fp.scale_log2 = scale * 1.4426950408889634f;
  fp.causal = causal ? 1 : 0;
  fp.inject_timeout = 0;
  fp.unit_counter = counter;
  return gbattn::launch_fwd(fp, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
