// Host side of the C ABI declared in include/attn.h: argument validation,
// per-device state (status word, workspace pool, RoPE table cache), TMA tensor
// maps, kernel launches and optional per-kernel event timing.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <functional>
#include <queue>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <tuple>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "kernels.h"

using gbattn::kTile;

namespace {

constexpr int kMaxDevices = 64;
constexpr int gb_status_bounds = 0x200;  // the kernels' kStatusBounds bit

// One RoPE table (see launch_rope_table): positions [0, npos) of one (D, theta), four
// fp32 arrays n floats apart, built on the stream of the call that first needed it.
struct RopeTable {
  float* buf = nullptr;
  int npos = 0;
  long long n = 0;
  cudaEvent_t ready = nullptr;  // recorded after the build
  bool known_ready = false;     // the build was seen complete (no wait needed any more)
  // Streams that read the table outside stream capture (at most kRopeStreams tracked;
  // many_streams beyond that). A retired table is freed in stream order on the stream
  // that retires it only when that stream is the only one that read it.
  std::vector<cudaStream_t> uses;
  bool many_streams = false;
  bool pinned = false;   // read under stream capture: a graph may hold its address
  bool retired = false;  // replaced or evicted: freed when the last holder releases it
  int active = 0;        // calls between rope_acquire and rope_release
  uint64_t tick = 0;     // last acquisition (least recently used is evicted first)
};
using RopePtr = std::shared_ptr<RopeTable>;

struct DeviceState {
  bool init = false;
  bool supported = false;
  int* status = nullptr;            // device status word (a static device variable)
  cudaMemPool_t pool = nullptr;     // library-owned stream-ordered pool
  std::map<std::pair<int, uint32_t>, RopePtr> rope;  // (D, theta bits)
  std::vector<RopePtr> to_free;     // retired under capture: freed by the next plain call
  uint64_t tick = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// RoPE tables kept per device (distinct (D, theta) pairs), and streams tracked per table.
constexpr int kRopeKeys = 8;
constexpr int kRopeStreams = 8;
bool g_inject_timeout = false;

// Groups larger than this take the exact delta pass by default (see bwd_common).
constexpr int kExactDeltaGroup = 8;

// ------------------------------------------------------------------ profiling
struct Profile {
  bool on = false;
  int cap = 0;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> rec[ATTN_NUM_KERNELS];
  std::vector<cudaEvent_t> spare;
};
Profile g_prof;

cudaEvent_t take_event() {
  if (!g_prof.spare.empty()) {
    cudaEvent_t e = g_prof.spare.back();
    g_prof.spare.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Records events around one launch when profiling is on.
struct LaunchTimer {
  int kind;
  cudaStream_t stream;
  cudaEvent_t start = nullptr, stop = nullptr;
  LaunchTimer(int k, cudaStream_t s) : kind(k), stream(s) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_prof.on || static_cast<int>(g_prof.rec[kind].size()) >= g_prof.cap) return;
    start = take_event();
    stop = take_event();
    if (start && stop) cudaEventRecord(start, stream);
  }
  void done() {
    if (!start || !stop) return;
    cudaEventRecord(stop, stream);
    std::lock_guard<std::mutex> lk(g_mu);
    g_prof.rec[kind].emplace_back(start, stop);
  }
};

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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
  return fn;
}

// 16-bit (bf16 or fp16) matrix [rows][D], 128-byte swizzled boxes of
// {64 columns, box_rows rows}.
bool make_map(CUtensorMap* m, const void* ptr, long long rows, int D, int box_rows,
              bool fp16 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  const CUtensorMapDataType dt =
      fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 matrix [rows][cols], 128-byte swizzled boxes of {32 columns, 128 rows}.
bool make_map_f32(CUtensorMap* m, const void* ptr, long long rows, int cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kTile)};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ validation
bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate(const void* const* ptrs, int nptr, int B, int Hq, int Hkv, int S, int D, float theta,
             float scale) {
  for (int i = 0; i < nptr; ++i)
    if (!aligned16(ptrs[i])) return ATTN_ERR_INVALID;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || D <= 0) return ATTN_ERR_INVALID;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID;
  if (!std::isfinite(theta) || theta <= 0.f || !std::isfinite(scale) || scale <= 0.f)
    return ATTN_ERR_INVALID;
  if (static_cast<long long>(B) * Hq * S >= (1LL << 31)) return ATTN_ERR_INVALID;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

int round_tile(int S) { return (S + kTile - 1) / kTile * kTile; }

// rope_mode of an entry point: one ATTN_ROPE_* layout, optionally with ATTN_ROPE_EXACT,
// plus the flags in `allowed`. Returns false for anything else.
bool parse_rope_mode(int rope_mode, int allowed, int* layout, bool* exact) {
  *layout = rope_mode & 0xf;
  *exact = (rope_mode & ATTN_ROPE_EXACT) != 0;
  if (*layout != ATTN_ROPE_HALF && *layout != ATTN_ROPE_INTERLEAVED) return false;
  return (rope_mode & ~(0xf | ATTN_ROPE_EXACT | allowed)) == 0;
}

// Query / K-V block arguments of the partial entry points: Sq, Skv multiples of
// 128 (checked with the other sizes by validate), positions non-negative
// multiples of 128, the last position below 2^30.
int validate_blocks(int Sq, int Skv, int q_pos0, int kv_pos0) {
  if (Sq <= 0 || Skv <= 0 || q_pos0 < 0 || kv_pos0 < 0) return ATTN_ERR_INVALID;
  if (static_cast<long long>(q_pos0) + Sq > (1LL << 30) ||
      static_cast<long long>(kv_pos0) + Skv > (1LL << 30))
    return ATTN_ERR_INVALID;
  if (Sq % kTile != 0 || Skv % kTile != 0 || q_pos0 % kTile != 0 || kv_pos0 % kTile != 0)
    return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// The device status word: a static device variable, zero when the library is loaded
// on a device, so that no call allocates it. Kernels record an expired wait in it;
// attn_sync_status reads and clears it.
__device__ int g_status_word;
int* g_status_ptr[kMaxDevices] = {};

// Device address of the status word on device `dev` (the current device), looked up
// once per device. Caller holds g_mu.
int status_word_locked(int dev, int** out) {
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_status_ptr[dev];
  return ATTN_OK;
}

// Current device's state, initialised on first use. Returns an ATTN_* code.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    d.supported = major == 10 && minor == 3;
    if (d.supported) {
      if (status_word_locked(dev, &d.status) != ATTN_OK) return ATTN_ERR_CUDA;
      cudaMemPoolProps props;
      std::memset(&props, 0, sizeof(props));
      props.allocType = cudaMemAllocationTypePinned;
      props.handleTypes = cudaMemHandleTypeNone;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) return ATTN_ERR_CUDA;
      uint64_t keep = UINT64_MAX;  // keep freed blocks for reuse by later calls
      cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    }
    d.init = true;
  }
  if (!d.supported) return ATTN_ERR_UNSUPPORTED;
  *out = &d;
  return ATTN_OK;
}

}  // namespace

namespace gbattn {
// The status word of the current device, for entry points that must not create the
// library's pool (it allocates nothing).
int device_status_word(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  return status_word_locked(dev, out);
}
}  // namespace gbattn

namespace {

bool stream_capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone;
}

// Releases a retired table in stream order on `stream` (alive and not capturing) when
// every read of it was enqueued on `stream`: the free then follows them. A table read
// by another stream, or under stream capture (a graph may still read it), stays
// allocated until the process exits; recording an event after every call to order a
// free after other streams' reads would cost each call its overlap with the next
// kernel (an event between two launches holds back the second's early start).
void rope_free_locked(RopeTable& t, cudaStream_t stream) {
  bool only_here = !t.pinned && !t.many_streams;
  for (cudaStream_t u : t.uses) only_here = only_here && u == stream;
  if (only_here && t.buf) cudaFreeAsync(t.buf, stream);
  if (t.ready) cudaEventDestroy(t.ready);
  t.uses.clear();
  t.ready = nullptr;
  t.buf = nullptr;
}

// Marks a table retired; frees it now when no call holds it. Caller holds g_mu.
void rope_retire_locked(DeviceState* d, const RopePtr& t, cudaStream_t stream, bool capturing) {
  t->retired = true;
  if (t->active > 0) return;  // the last rope_release frees it
  if (capturing) d->to_free.push_back(t);
  else rope_free_locked(*t, stream);
}

// The RoPE table of one call: the four arrays for positions [0, npos).
struct RopeUse {
  RopePtr t;
  const float *ch = nullptr, *sh = nullptr, *cl = nullptr, *sl = nullptr;
  int npos = 0;  // positions the table holds (>= the ones asked for)
};

// Table covering positions [0, npos) for (D, theta), built when missing or too short:
// memory from the library pool and the build kernel, both in stream order on `stream`,
// with no host synchronisation; another stream that reads the table before the build
// has completed waits for it on the device. A longer table replaces a shorter one (at
// least doubling its length); at most kRopeKeys (D, theta) pairs are kept, the least
// recently used evicted first. A build cannot be recorded into a stream capture
// (ATTN_ERR_UNSUPPORTED): the first call for a (D, theta), or for a longer sequence than
// before, belongs outside capture, and so does one more call after the build has
// completed. Pair with rope_release after the call's launches.
int rope_acquire(DeviceState* d, int npos, int D, float theta, cudaStream_t stream,
                 bool capturing, RopeUse* out) {
  uint32_t tb;
  std::memcpy(&tb, &theta, 4);
  const auto key = std::make_pair(D, tb);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!capturing && !d->to_free.empty()) {
    for (auto& t : d->to_free) rope_free_locked(*t, stream);
    d->to_free.clear();
  }
  auto it = d->rope.find(key);
  RopePtr t = it != d->rope.end() ? it->second : nullptr;
  if (!t || t->npos < npos) {
    if (capturing) return ATTN_ERR_UNSUPPORTED;
    long long want = (static_cast<long long>(npos) + kTile - 1) / kTile * kTile;
    if (t) want = std::max(want, std::min(2LL * t->npos, 1LL << 30));
    auto nt = std::make_shared<RopeTable>();
    nt->npos = static_cast<int>(want);
    nt->n = (want * (D / 2) + 63) / 64 * 64;  // arrays 256-byte aligned
    void* buf = nullptr;
    if (cudaMallocFromPoolAsync(&buf, static_cast<size_t>(4 * nt->n) * sizeof(float), d->pool,
                                stream) != cudaSuccess)
      return ATTN_ERR_CUDA;
    nt->buf = static_cast<float*>(buf);
    if (gbattn::launch_rope_table(nt->buf, nt->n, nt->npos, D, static_cast<double>(theta),
                                  stream) != cudaSuccess ||
        cudaEventCreateWithFlags(&nt->ready, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventRecord(nt->ready, stream) != cudaSuccess) {
      if (nt->ready) cudaEventDestroy(nt->ready);
      cudaFreeAsync(nt->buf, stream);
      return ATTN_ERR_CUDA;
    }
    if (t) {
      rope_retire_locked(d, t, stream, false);
    } else if (static_cast<int>(d->rope.size()) >= kRopeKeys) {
      auto lru = d->rope.begin();
      for (auto i = d->rope.begin(); i != d->rope.end(); ++i)
        if (i->second->tick < lru->second->tick) lru = i;
      rope_retire_locked(d, lru->second, stream, false);
      d->rope.erase(lru);
    }
    d->rope[key] = nt;
    t = nt;
  } else if (!t->known_ready) {
    // Built by a call whose stream may not have finished the build yet. Outside
    // capture this stream waits for it on the device; a capture cannot take that
    // dependency, so the build must already have been seen complete by an earlier call.
    if (capturing) return ATTN_ERR_UNSUPPORTED;
    if (cudaEventQuery(t->ready) == cudaSuccess) t->known_ready = true;
    else if (cudaStreamWaitEvent(stream, t->ready, 0) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  t->active += 1;
  t->tick = ++d->tick;
  if (capturing) t->pinned = true;
  out->t = t;
  out->ch = t->buf;
  out->sh = t->buf + t->n;
  out->cl = t->buf + 2 * t->n;
  out->sl = t->buf + 3 * t->n;
  out->npos = t->npos;
  return ATTN_OK;
}

// Ends a call's use of its table: notes the stream that read it (outside capture) and
// frees the table if it was retired meanwhile and nothing else holds it.
void rope_release(DeviceState* d, RopeUse& u, cudaStream_t stream, bool capturing) {
  if (!u.t) return;
  std::lock_guard<std::mutex> lk(g_mu);
  RopeTable& t = *u.t;
  t.active -= 1;
  if (!capturing && !t.many_streams) {
    bool seen = false;
    for (cudaStream_t s : t.uses) seen = seen || s == stream;
    if (!seen) {
      if (static_cast<int>(t.uses.size()) >= kRopeStreams) t.many_streams = true;
      else t.uses.push_back(stream);
    }
  }
  if (t.retired && t.active == 0) {
    if (capturing) d->to_free.push_back(u.t);
    else rope_free_locked(t, stream);
  }
  u.t.reset();
}

// Holds a call's RoPE table from acquisition to the end of the call (every launch that
// reads it has been enqueued by then).
struct RopeGuard {
  DeviceState* d;
  cudaStream_t stream;
  bool capturing;
  RopeUse u;
  RopeGuard(DeviceState* d_, cudaStream_t s_) : d(d_), stream(s_), capturing(stream_capturing(s_)) {}
  int acquire(int npos, int D, float theta) {
    return rope_acquire(d, npos, D, theta, stream, capturing, &u);
  }
  ~RopeGuard() { rope_release(d, u, stream, capturing); }
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" {

const char* attn_version(void) { return "mqa_attention_gb300 0.1.0 (sm_103a)"; }

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported size or device";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
    case ATTN_ERR_BOUNDS: return "device index check failed";
    default: return "unknown status";
  }
}

// Forward pass of a query block (Sq rows per head at positions q_pos0..) against
// a K/V block (Skv rows at kv_pos0..); self-attention is Sq = Skv, both 0.
// A self-attention call (ragged = true: Sq = Skv = S, offsets 0) may have any S:
// the main kernels then work on copies padded to whole 128-row tiles, and the
// valid rows of out / lse are copied into the caller's buffers at the end.
static int fwd_common(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                      int Hq, int Hkv, int Sq, int Skv, int D, int q_pos0, int kv_pos0,
                      float rope_theta, int rope_mode, float scale, int causal,
                      attn_stream_t stream_, bool ragged) {
  const void* ptrs[] = {q, k, v, out, lse};
  int st = validate(ptrs, 5, B, Hq, Hkv, Sq > Skv ? Sq : Skv, D, rope_theta, scale);
  if (st != ATTN_OK) return st;
  if (!ragged && (st = validate_blocks(Sq, Skv, q_pos0, kv_pos0)) != ATTN_OK) return st;
  int layout = 0;
  bool exact_rope = false;
  if (!parse_rope_mode(rope_mode, 0, &layout, &exact_rope)) return ATTN_ERR_INVALID;
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != ATTN_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // Table rows for every position a kernel reads, the padding rows of a ragged
  // sequence included (they are rotated like any row, and then ignored).
  const int npos = q_pos0 + round_tile(Sq) > kv_pos0 + round_tile(Skv) ? q_pos0 + round_tile(Sq)
                                                                        : kv_pos0 + round_tile(Skv);
  RopeGuard rope(d, stream);
  if ((st = rope.acquire(npos, D, rope_theta)) != ATTN_OK) return st;

  const int Sqp = round_tile(Sq), Skvp = round_tile(Skv);  // rows per head the kernels see
  const bool padded = Sqp != Sq || Skvp != Skv;
  if (static_cast<long long>(B) * Hq * Sqp >= (1LL << 31) ||
      static_cast<long long>(B) * Hkv * Skvp >= (1LL << 31))
    return ATTN_ERR_INVALID;
  const long long qrows = static_cast<long long>(B) * Hq * Sq;
  const long long qrows_p = static_cast<long long>(B) * Hq * Sqp;
  const long long krows_p = static_cast<long long>(B) * Hkv * Skvp;
  const size_t qbytes = round256(static_cast<size_t>(qrows_p) * D * 2);
  const size_t kbytes = round256(static_cast<size_t>(krows_p) * D * 2);
  const size_t lbytes = padded ? round256(static_cast<size_t>(qrows_p) * 4) : 0;
  const size_t cbytes = 256;  // the forward's unit counter
  uint8_t* ws = nullptr;
  if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws),
                              qbytes + kbytes + (padded ? kbytes + qbytes : 0) + lbytes + cbytes,
                              d->pool, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  void* qr = ws;
  void* kr = ws + qbytes;
  // padded: v, out and lse in whole tiles
  void* vk = padded ? static_cast<void*>(ws + qbytes + kbytes) : const_cast<void*>(v);
  void* ok_out = padded ? static_cast<void*>(ws + qbytes + 2 * kbytes) : out;
  float* ok_lse = padded ? reinterpret_cast<float*>(ws + 2 * qbytes + 2 * kbytes) : lse;
  int* counter = reinterpret_cast<int*>(ws + qbytes + kbytes + (padded ? kbytes + qbytes : 0) + lbytes);

  bool ok = true;
  {
    gbattn::RowPrepParams rp{};
    rp.status = d->status;
    rp.bwd = 0;
    rp.rope_interleaved = layout == ATTN_ROPE_INTERLEAVED;
    rp.exact = exact_rope ? 1 : 0;
    rp.D = D;
    rp.cos_tab = rope.u.ch;
    rp.sin_tab = rope.u.sh;
    rp.cos_lo = rope.u.cl;
    rp.sin_lo = rope.u.sl;
    rp.tab_rows = rope.u.npos;
    rp.seg[0] = {q, qr, nullptr, nullptr, qrows_p, Sq, Sqp, q_pos0};
    rp.seg[1] = {k, kr, padded ? v : nullptr, padded ? vk : nullptr, krows_p, Skv, Skvp, kv_pos0};
    rp.zero_word = counter;
    LaunchTimer tm(ATTN_KERNEL_ROPE, stream);
    ok = gbattn::launch_row_prep(rp, stream) == cudaSuccess;
    tm.done();
  }
  gbattn::FwdParams fp{};
  ok = ok && make_map(&fp.map_q, qr, qrows_p, D, kTile) &&
       make_map(&fp.map_k, kr, krows_p, D, kTile) && make_map(&fp.map_v, vk, krows_p, D, kTile) &&
       make_map(&fp.map_out, ok_out, qrows_p, D, kTile);
  if (ok) {
    fp.out = ok_out;
    fp.lse = ok_lse;
    fp.status = d->status;
    fp.B = B; fp.Hq = Hq; fp.Hkv = Hkv; fp.Sq = Sqp; fp.Skv = Skvp; fp.D = D;
    fp.kv_valid = Skv;
    fp.q_tile0 = q_pos0 / kTile;
    fp.kv_tile0 = kv_pos0 / kTile;
    fp.scale_log2 = scale * 1.4426950408889634f;
    fp.causal = causal ? 1 : 0;
    fp.inject_timeout = g_inject_timeout ? 1 : 0;
    fp.unit_counter = counter;
    LaunchTimer tm(ATTN_KERNEL_FWD, stream);
    ok = gbattn::launch_fwd(fp, stream) == cudaSuccess;
    tm.done();
  }
  if (ok && padded)
    ok = gbattn::launch_unpad_rows(ok_out, out, qrows, Sq, Sqp, D / 2, false, stream) ==
             cudaSuccess &&
         gbattn::launch_unpad_rows(ok_lse, lse, qrows, Sq, Sqp, 1, false, stream) == cudaSuccess;
  cudaFreeAsync(ws, stream);
  return ok ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_fwd_ex(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                int Hq, int Hkv, int S, int D, float rope_theta, int rope_mode, float scale,
                int causal, attn_stream_t stream) {
  return fwd_common(q, k, v, out, lse, B, Hq, Hkv, S, S, D, 0, 0, rope_theta, rope_mode, scale,
                    causal, stream, true);
}

int attn_fwd_partial(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                     int Hq, int Hkv, int Sq, int Skv, int D, int q_pos0, int kv_pos0,
                     float rope_theta, int rope_mode, float scale, int causal,
                     attn_stream_t stream) {
  return fwd_common(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, D, q_pos0, kv_pos0, rope_theta,
                    rope_mode, scale, causal, stream, false);
}

int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
             int Hkv, int S, int D, float rope_theta, float scale, int causal,
             attn_stream_t stream) {
  return attn_fwd_ex(q, k, v, out, lse, B, Hq, Hkv, S, D, rope_theta, ATTN_ROPE_HALF, scale,
                     causal, stream);
}

// Work order of the backward main kernel. A CTA owns one key tile of one (batch, KV
// head) and walks the group's query heads over the query tiles that see it, so
// under causal masking the first key tiles carry the most steps. The CTAs run
// heaviest first; when that leaves a few long CTAs finishing last, the heaviest
// key tiles are split between two CTAs (half of the group's query heads each, dK/dV
// added). The number of tiles to split is chosen by simulating the greedy schedule
// on the SMs (about three steps of start-up per CTA), once per shape.
struct BwdPlan {
  int nplan = 0;  // 0: no table (one CTA per key tile, or `uniform` each)
  int uniform = 1;
  int split = 0;  // key tiles [0, split) have two CTAs
  short kt[gbattn::kMaxBwdPlan];
  signed char parts[gbattn::kMaxBwdPlan];
};

static BwdPlan choose_bwd_plan(int nkt, int per, int G, int causal, int q_tile0, int kv_tile0,
                               int nqt, int nsm) {
  BwdPlan pl;
  const long long key_tiles = static_cast<long long>(per) * nkt;
  const bool even = G % 2 == 0;
  // Many waves (or nothing to split): the greedy schedule is already balanced.
  if (!even || nkt > gbattn::kMaxBwdPlan || key_tiles > 4LL * nsm) {
    pl.uniform = (even && key_tiles < nsm) ? 2 : 1;
    pl.split = pl.uniform == 2 ? nkt : 0;
    return pl;
  }
  std::vector<int> sph(nkt);  // steps per query head of each key tile
  for (int kt = 0; kt < nkt; ++kt) {
    int begin = 0;
    if (causal) {
      const int d = ((kv_tile0 + kt) * kTile - q_tile0 * kTile) / 64;
      begin = d < 0 ? 0 : (d > nqt ? nqt : d);
    }
    sph[kt] = nqt - begin;
  }
  const double ovh = 3.0;
  auto makespan = [&](int split) {
    std::vector<double> u;
    u.reserve(static_cast<size_t>(2 * key_tiles));
    for (int kt = 0; kt < nkt; ++kt) {
      const int parts = kt < split ? 2 : 1;
      const double size = static_cast<double>(G / parts) * sph[kt] + ovh;
      for (int i = 0; i < parts * per; ++i) u.push_back(size);
    }
    std::sort(u.begin(), u.end(), std::greater<double>());
    std::priority_queue<double, std::vector<double>, std::greater<double>> sm;
    for (int i = 0; i < nsm; ++i) sm.push(0.0);
    for (double x : u) {
      const double l = sm.top();
      sm.pop();
      sm.push(l + x);
    }
    double m = 0.0;
    while (!sm.empty()) {
      m = std::max(m, sm.top());
      sm.pop();
    }
    return m;
  };
  double best = makespan(0);
  for (int split = 1; split <= nkt; ++split) {
    const double m = makespan(split);
    if (m < best - 1e-9) {
      best = m;
      pl.split = split;
    }
  }
  // the table: key tiles by unit size, heaviest first (ties by key tile)
  std::vector<int> order(nkt);
  for (int kt = 0; kt < nkt; ++kt) order[kt] = kt;
  auto unit = [&](int kt) { return (kt < pl.split ? G / 2 : G) * sph[kt]; };
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return unit(a) > unit(b); });
  pl.nplan = nkt;
  for (int e = 0; e < nkt; ++e) {
    pl.kt[e] = static_cast<short>(order[e]);
    pl.parts[e] = static_cast<signed char>(order[e] < pl.split ? 2 : 1);
  }
  return pl;
}

static const BwdPlan& bwd_plan_cached(int nkt, int per, int G, int causal, int q_tile0,
                                      int kv_tile0, int nqt, int nsm) {
  static std::map<std::tuple<int, int, int, int, int, int, int, int>, BwdPlan> cache;
  const auto key = std::make_tuple(nkt, per, G, causal, q_tile0, kv_tile0, nqt, nsm);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  BwdPlan pl = choose_bwd_plan(nkt, per, G, causal, q_tile0, kv_tile0, nqt, nsm);
  std::lock_guard<std::mutex> lk(g_mu);
  return cache.emplace(key, pl).first->second;  // std::map references stay valid
}

// The backward pass with fp32 gradients, or (bf16_grads) with gradients rounded
// to bf16 at the end: dq by the finalisation, dk and dv by a conversion pass over
// fp32 copies kept in the workspace, so that every gradient is the fp32 result
// rounded to nearest even.
static int bwd_common(const void* q, const void* k, const void* v, const void* out,
                      const float* lse, const void* dout, void* dq_out, void* dk_out, void* dv_out,
                      int B, int Hq, int Hkv, int Sq, int Skv, int D, int q_pos0, int kv_pos0,
                      float rope_theta, int rope_mode, float scale, int causal,
                      attn_stream_t stream_, bool bf16_grads, bool ragged) {
  const void* ptrs[] = {q, k, v, out, lse, dout, dq_out, dk_out, dv_out};
  int st = validate(ptrs, 9, B, Hq, Hkv, Sq > Skv ? Sq : Skv, D, rope_theta, scale);
  if (st != ATTN_OK) return st;
  if (!ragged && (st = validate_blocks(Sq, Skv, q_pos0, kv_pos0)) != ATTN_OK) return st;
  // rope_mode: the RoPE pair layout and rounding, optionally with one delta flag
  // (self-attention only)
  int layout = 0;
  bool exact_rope = false;
  if (!parse_rope_mode(rope_mode, ATTN_DELTA_EXACT | ATTN_DELTA_FROM_OUT, &layout, &exact_rope))
    return ATTN_ERR_INVALID;
  const int dflags = rope_mode & (ATTN_DELTA_EXACT | ATTN_DELTA_FROM_OUT);
  if (dflags == (ATTN_DELTA_EXACT | ATTN_DELTA_FROM_OUT)) return ATTN_ERR_INVALID;
  if (!ragged && dflags == ATTN_DELTA_EXACT) return ATTN_ERR_INVALID;
  const int inter = layout == ATTN_ROPE_INTERLEAVED;
  // delta from the scores (the exact pass) or from the bf16 `out` (one HBM read): by
  // default exact when more than 8 query heads share a K/V head, whose dk sums the
  // rounding of out over the whole group
  const bool exact_delta =
      ragged && (dflags == ATTN_DELTA_EXACT || (dflags == 0 && Hq / Hkv > kExactDeltaGroup));
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != ATTN_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // Table rows for every position a kernel reads, the padding rows of a ragged
  // sequence included (they are rotated like any row, and then ignored).
  const int npos = q_pos0 + round_tile(Sq) > kv_pos0 + round_tile(Skv) ? q_pos0 + round_tile(Sq)
                                                                        : kv_pos0 + round_tile(Skv);
  RopeGuard rope(d, stream);
  if ((st = rope.acquire(npos, D, rope_theta)) != ATTN_OK) return st;
  const float* cs = rope.u.ch;
  const float* sn = rope.u.sh;

  // The main kernel's work order (bwd_plan_cached) depends on the number of SMs.
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  // rows per head the kernels see (padded to whole tiles for a ragged S)
  const int Sqp = round_tile(Sq), Skvp = round_tile(Skv);
  const bool padded = Sqp != Sq || Skvp != Skv;
  if (static_cast<long long>(B) * Hq * Sqp >= (1LL << 31) ||
      static_cast<long long>(B) * Hkv * Skvp >= (1LL << 31))
    return ATTN_ERR_INVALID;
  const long long qrows = static_cast<long long>(B) * Hq * Sq;
  const long long krows = static_cast<long long>(B) * Hkv * Skv;
  const long long qrows_p = static_cast<long long>(B) * Hq * Sqp;
  const long long krows_p = static_cast<long long>(B) * Hkv * Skvp;
  const BwdPlan& plan = bwd_plan_cached(Skvp / kTile, B * Hkv, Hq / Hkv, causal ? 1 : 0,
                                        q_pos0 / kTile, kv_pos0 / kTile, Sqp / 64, nsm);
  const size_t qbytes = round256(static_cast<size_t>(qrows_p) * D * 2);
  const size_t kbytes = round256(static_cast<size_t>(krows_p) * D * 2);
  const size_t accbytes = round256(static_cast<size_t>(qrows_p) * D * 4);
  const size_t rowbytes = round256(static_cast<size_t>(qrows_p) * 4);
  const size_t maxbytes = 256;
  const bool own_dkdv = bf16_grads || padded;  // dk, dv go through workspace copies
  const size_t gradbytes = own_dkdv ? round256(static_cast<size_t>(krows_p) * D * 4) : 0;
  uint8_t* ws = nullptr;
  if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws),
                              2 * qbytes + 2 * kbytes + accbytes + 2 * rowbytes + maxbytes +
                                  2 * gradbytes,
                              d->pool,
                              stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  uint8_t* w = ws;
  void* qr = w; w += qbytes;        // fp16, scaled rotated q
  void* dos = w; w += qbytes;       // fp16, scaled dout
  void* kr = w; w += kbytes;        // fp16, scaled rotated k
  void* vs = w; w += kbytes;        // fp16, scaled v
  float* dqacc = reinterpret_cast<float*>(w); w += accbytes;
  float* delta = reinterpret_cast<float*>(w); w += rowbytes;
  float* lse2 = reinterpret_cast<float*>(w); w += rowbytes;
  float* maxes = reinterpret_cast<float*>(w); w += maxbytes;
  // fp32 dk, dv: the caller's buffers, or workspace copies (padded rows, and/or
  // rounded to bf16) copied into the caller's buffers at the end
  float* dk = own_dkdv ? reinterpret_cast<float*>(w) : static_cast<float*>(dk_out);
  float* dv = own_dkdv ? reinterpret_cast<float*>(w + gradbytes) : static_cast<float*>(dv_out);
  bool ok = true;
  {
    LaunchTimer tm(ATTN_KERNEL_BWD_PREP, stream);
    gbattn::AbsMaxParams ap{};
    ap.x[gbattn::kMaxQ] = q; ap.n[gbattn::kMaxQ] = qrows * D;
    ap.x[gbattn::kMaxK] = k; ap.n[gbattn::kMaxK] = krows * D;
    ap.x[gbattn::kMaxV] = v; ap.n[gbattn::kMaxV] = krows * D;
    ap.x[gbattn::kMaxDO] = dout; ap.n[gbattn::kMaxDO] = qrows * D;
    ap.maxes = maxes;
    ok = gbattn::launch_zero_words(maxes, 4, stream) == cudaSuccess &&
         gbattn::launch_absmax(ap, stream) == cudaSuccess;
    gbattn::RowPrepParams rp{};
    rp.status = d->status;
    rp.bwd = 1;
    rp.rope_interleaved = inter;
    rp.exact = exact_rope ? 1 : 0;
    rp.D = D;
    rp.cos_tab = cs;
    rp.sin_tab = sn;
    rp.cos_lo = rope.u.cl;
    rp.sin_lo = rope.u.sl;
    rp.tab_rows = rope.u.npos;
    rp.maxes = maxes;
    rp.seg[0] = {q, qr, dout, dos, qrows_p, Sq, Sqp, q_pos0};
    rp.seg[1] = {k, kr, v, vs, krows_p, Skv, Skvp, kv_pos0};
    rp.out = exact_delta ? nullptr : out;
    rp.delta = delta; rp.lse = lse; rp.lse2 = lse2; rp.dqacc = dqacc;
    if (plan.split > 0) {  // the main kernel adds dK/dV partials of two CTAs there
      rp.dk_zero = dk;
      rp.dv_zero = dv;
      rp.dk_zero_rows = plan.split * kTile;
    }
    ok = ok && gbattn::launch_row_prep(rp, stream) == cudaSuccess;
    tm.done();
  }
  if (ok && exact_delta) {
    gbattn::DeltaParams xp{};
    ok = make_map(&xp.map_q, qr, qrows_p, D, kTile, true) &&
         make_map(&xp.map_do, dos, qrows_p, D, kTile, true) &&
         make_map(&xp.map_k, kr, krows_p, D, kTile, true) &&
         make_map(&xp.map_v, vs, krows_p, D, kTile, true);
    if (ok) {
      xp.lse2 = lse2;
      xp.maxes = maxes;
      xp.delta = delta;
      xp.status = d->status;
      xp.B = B; xp.Hq = Hq; xp.Hkv = Hkv; xp.S = Sqp; xp.D = D;
      xp.scale_log2 = scale * 1.4426950408889634f;
      xp.causal = causal ? 1 : 0;
      xp.inject_timeout = g_inject_timeout ? 1 : 0;
      LaunchTimer tm(ATTN_KERNEL_DELTA, stream);
      ok = gbattn::launch_delta(xp, stream) == cudaSuccess;
      tm.done();
    }
  }
  gbattn::BwdParams bp{};
  const int bq = gbattn::bwd_query_tile(D);
  ok = ok && make_map(&bp.map_q, qr, qrows_p, D, bq, true) &&
       make_map(&bp.map_do, dos, qrows_p, D, bq, true) &&
       make_map(&bp.map_k, kr, krows_p, D, kTile, true) &&
       make_map(&bp.map_v, vs, krows_p, D, kTile, true) &&
       make_map_f32(&bp.map_dk, dk, krows_p, D) && make_map_f32(&bp.map_dv, dv, krows_p, D) &&
       make_map_f32(&bp.map_dqacc, dqacc, qrows_p, D) &&
       make_map_f32(&bp.map_cos, cs, rope.u.npos, D / 2) &&
       make_map_f32(&bp.map_sin, sn, rope.u.npos, D / 2);
  if (ok) {
    bp.lse2 = lse2;
    bp.delta = delta;
    bp.maxes = maxes;
    bp.dqacc = dqacc;
    bp.dk = dk;
    bp.dv = dv;
    bp.cos_tab = cs;
    bp.sin_tab = sn;
    bp.tab_rows = rope.u.npos;
    bp.status = d->status;
    bp.B = B; bp.Hq = Hq; bp.Hkv = Hkv; bp.Sq = Sqp; bp.Skv = Skvp; bp.D = D;
    bp.q_tile0 = q_pos0 / kTile;
    bp.kv_tile0 = kv_pos0 / kTile;
    bp.scale = scale;
    bp.scale_log2 = scale * 1.4426950408889634f;
    bp.causal = causal ? 1 : 0;
    bp.inject_timeout = g_inject_timeout ? 1 : 0;
    bp.hsplit = plan.uniform;
    bp.nplan = plan.nplan;
    for (int e = 0; e < plan.nplan; ++e) {
      bp.plan_kt[e] = plan.kt[e];
      bp.plan_parts[e] = plan.parts[e];
    }
    bp.rope_interleaved = inter;
    LaunchTimer tm(ATTN_KERNEL_BWD_MAIN, stream);
    ok = gbattn::launch_bwd_main(bp, stream) == cudaSuccess;
    tm.done();
  }
  if (ok) {
    LaunchTimer tm(ATTN_KERNEL_DQ_FINAL, stream);
    ok = gbattn::launch_dq_finalize(dqacc, dq_out, bf16_grads, qrows, Sq, Sqp, q_pos0, D, scale,
                                    maxes, cs, sn, rope.u.npos, inter, d->status,
                                    stream) == cudaSuccess;
    if (padded)
      ok = ok &&
           gbattn::launch_unpad_rows(dk, dk_out, krows, Skv, Skvp, D, bf16_grads, stream) ==
               cudaSuccess &&
           gbattn::launch_unpad_rows(dv, dv_out, krows, Skv, Skvp, D, bf16_grads, stream) ==
               cudaSuccess;
    else if (bf16_grads)
      ok = ok && gbattn::launch_f32_to_bf16(dk, dk_out, krows * D, stream) == cudaSuccess &&
           gbattn::launch_f32_to_bf16(dv, dv_out, krows * D, stream) == cudaSuccess;
    tm.done();
  }
  cudaFreeAsync(ws, stream);
  return ok ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_bwd_ex(const void* q, const void* k, const void* v, const void* out, const float* lse,
                const void* dout, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int S,
                int D, float rope_theta, int rope_mode, float scale, int causal,
                attn_stream_t stream) {
  return bwd_common(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, S, D, 0, 0, rope_theta,
                    rope_mode, scale, causal, stream, false, true);
}

int attn_bwd_partial(const void* q, const void* k, const void* v, const void* out,
                     const float* lse, const void* dout, float* dq, float* dk, float* dv, int B,
                     int Hq, int Hkv, int Sq, int Skv, int D, int q_pos0, int kv_pos0,
                     float rope_theta, int rope_mode, float scale, int causal,
                     attn_stream_t stream) {
  return bwd_common(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Skv, D, q_pos0, kv_pos0,
                    rope_theta, rope_mode, scale, causal, stream, false, false);
}

int attn_bwd_bf16(const void* q, const void* k, const void* v, const void* out, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S,
                  int D, float rope_theta, int rope_mode, float scale, int causal,
                  attn_stream_t stream) {
  return bwd_common(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, S, D, 0, 0, rope_theta,
                    rope_mode, scale, causal, stream, true, true);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
             const void* dout, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int S,
             int D, float rope_theta, float scale, int causal, attn_stream_t stream) {
  return attn_bwd_ex(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, D, rope_theta,
                     ATTN_ROPE_HALF, scale, causal, stream);
}

int attn_rope(const void* x, void* y, long long heads, int S, int pos0, int D, float rope_theta,
              int rope_mode, attn_stream_t stream_) {
  if (!aligned16(x) || !aligned16(y)) return ATTN_ERR_INVALID;
  if (heads <= 0 || S <= 0 || pos0 < 0 || heads * S >= (1LL << 31) ||
      static_cast<long long>(pos0) + S > (1LL << 30))
    return ATTN_ERR_INVALID;
  if (!std::isfinite(rope_theta) || rope_theta <= 0.f) return ATTN_ERR_INVALID;
  int layout = 0;
  bool exact_rope = false;
  if (!parse_rope_mode(rope_mode, 0, &layout, &exact_rope)) return ATTN_ERR_INVALID;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  int st = device_state(&d);
  if (st != ATTN_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  RopeGuard rope(d, stream);
  if ((st = rope.acquire(pos0 + S, D, rope_theta)) != ATTN_OK) return st;
  gbattn::RowPrepParams rp{};
    rp.status = d->status;
  rp.bwd = 0;
  rp.rope_interleaved = layout == ATTN_ROPE_INTERLEAVED;
  rp.exact = exact_rope ? 1 : 0;
  rp.D = D;
  rp.cos_tab = rope.u.ch;
  rp.sin_tab = rope.u.sh;
  rp.cos_lo = rope.u.cl;
  rp.sin_lo = rope.u.sl;
  rp.tab_rows = rope.u.npos;
  rp.seg[0] = {x, y, nullptr, nullptr, heads * S, S, S, pos0};
  rp.seg[1] = {x, y, nullptr, nullptr, 0, S, S, pos0};
  return gbattn::launch_row_prep(rp, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_decode(const void* q, const void* k_rot, const void* v, void* out, float* lse, int B,
                int Hq, int Hkv, int Sq, int Skv, int D, int q_pos0, float rope_theta,
                int rope_mode, float scale, attn_stream_t stream_) {
  const void* ptrs[] = {q, k_rot, v, out, lse};
  int st = validate(ptrs, 5, B, Hq, Hkv, Sq > Skv ? Sq : Skv, D, rope_theta, scale);
  if (st != ATTN_OK) return st;
  int layout = 0;
  bool exact_rope = false;
  if (!parse_rope_mode(rope_mode, 0, &layout, &exact_rope)) return ATTN_ERR_INVALID;
  if (q_pos0 < 0 || static_cast<long long>(q_pos0) + Sq > (1LL << 30) ||
      static_cast<long long>(B) * Hkv * Skv >= (1LL << 31))
    return ATTN_ERR_INVALID;
  if ((Hq / Hkv) * Sq > kTile) return ATTN_ERR_UNSUPPORTED;  // one tile holds a group's rows
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != ATTN_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  RopeGuard rope(d, stream);
  if ((st = rope.acquire(q_pos0 + Sq, D, rope_theta)) != ATTN_OK) return st;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;

  // Chunks: about one CTA per SM over all (batch, KV head) caches (a CTA holds a
  // whole SM's shared memory, so more would run in a second wave).
  gbattn::DecParams dp{};
  const long long nu = static_cast<long long>(B) * Hkv;
  const int last_q = q_pos0 + Sq - 1;
  const int ntiles_all = (Skv + kTile - 1) / kTile;
  const int vis = last_q / kTile + 1;
  const int ntiles = vis < ntiles_all ? vis : ntiles_all;  // tiles with a visible key
  long long tpc = (static_cast<long long>(ntiles) * nu + nsm - 1) / nsm;
  tpc = tpc < 1 ? 1 : tpc;
  dp.tiles_per_chunk = static_cast<int>(tpc);
  dp.nchunks = static_cast<int>((ntiles + tpc - 1) / tpc);
  if (dp.nchunks < 1) dp.nchunks = 1;
  dp.rows = static_cast<long long>(B) * Hq * Sq;

  const size_t obytes = round256(static_cast<size_t>(dp.nchunks) * dp.rows * D * 4);
  const size_t lbytes = round256(static_cast<size_t>(dp.nchunks) * dp.rows * 4);
  uint8_t* ws = nullptr;
  if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws), obytes + lbytes, d->pool, stream) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  dp.part_out = reinterpret_cast<float*>(ws);
  dp.part_lse = reinterpret_cast<float*>(ws + obytes);
  const long long krows = static_cast<long long>(B) * Hkv * Skv;
  bool ok = make_map(&dp.map_q, q, dp.rows, D, kTile) &&
            make_map(&dp.map_k, k_rot, krows, D, kTile) && make_map(&dp.map_v, v, krows, D, kTile);
  if (ok) {
    dp.out = out;
    dp.lse = lse;
    dp.cos_tab = rope.u.ch;
    dp.sin_tab = rope.u.sh;
    dp.cos_lo = rope.u.cl;
    dp.sin_lo = rope.u.sl;
    dp.tab_rows = rope.u.npos;
    dp.rope_interleaved = layout == ATTN_ROPE_INTERLEAVED;
    dp.exact = exact_rope ? 1 : 0;
    dp.status = d->status;
    dp.B = B; dp.Hq = Hq; dp.Hkv = Hkv; dp.Sq = Sq; dp.Skv = Skv; dp.D = D;
    dp.q_pos0 = q_pos0;
    dp.scale_log2 = scale * 1.4426950408889634f;
    LaunchTimer tm(ATTN_KERNEL_FWD, stream);
    ok = gbattn::launch_decode(dp, stream) == cudaSuccess;
    tm.done();
  }
  cudaFreeAsync(ws, stream);
  return ok ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_merge(const void* out_a, const float* lse_a, const void* out_b, const float* lse_b,
               void* out, float* lse, long long rows, int D, attn_stream_t stream_) {
  const void* ptrs[] = {out_a, lse_a, out_b, lse_b, out, lse};
  for (const void* p : ptrs)
    if (!aligned16(p)) return ATTN_ERR_INVALID;
  if (rows <= 0 || rows >= (1LL << 31)) return ATTN_ERR_INVALID;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  DeviceState* d = nullptr;
  int st = device_state(&d);
  if (st != ATTN_OK) return st;
  return gbattn::launch_merge(out_a, lse_a, out_b, lse_b, out, lse, rows, D,
                              reinterpret_cast<cudaStream_t>(stream_)) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

int attn_sync_status(attn_stream_t stream_) {
  DeviceState* d = nullptr;
  int st = device_state(&d);
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream_)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return (word & gb_status_bounds) ? ATTN_ERR_BOUNDS : ATTN_ERR_TIMEOUT;
  }
  return ATTN_OK;
}

int attn_profile_begin(int max_launches) {
  if (max_launches <= 0) return ATTN_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& r : g_prof.rec) {
    for (auto& pr : r) {
      g_prof.spare.push_back(pr.first);
      g_prof.spare.push_back(pr.second);
    }
    r.clear();
  }
  g_prof.cap = max_launches;
  g_prof.on = true;
  return ATTN_OK;
}

int attn_profile_end(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof.on = false;
  return ATTN_OK;
}

int attn_profile_query(int kernel, int* launches, float* total_ms) {
  if (kernel < 0 || kernel >= ATTN_NUM_KERNELS || !launches || !total_ms) return ATTN_ERR_INVALID;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> rec;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    rec = g_prof.rec[kernel];
  }
  float sum = 0.f;
  for (auto& pr : rec) {
    if (cudaEventSynchronize(pr.second) != cudaSuccess) return ATTN_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, pr.first, pr.second) != cudaSuccess) return ATTN_ERR_CUDA;
    sum += ms;
  }
  *launches = static_cast<int>(rec.size());
  *total_ms = sum;
  return ATTN_OK;
}

int attn_debug_inject_timeout(int enable) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_inject_timeout = enable != 0;
  return ATTN_OK;
}

int attn_debug_bwd_plan(int B, int Hq, int Hkv, int Sq, int Skv, int q_pos0, int kv_pos0,
                        int causal, int nsm, int* split_key_tiles, int* ctas) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Sq <= 0 || Skv <= 0 || nsm <= 0 ||
      q_pos0 < 0 || kv_pos0 < 0 || q_pos0 % kTile != 0 || kv_pos0 % kTile != 0 ||
      !split_key_tiles || !ctas)
    return ATTN_ERR_INVALID;
  const int nkt = round_tile(Skv) / kTile;
  const BwdPlan& pl = bwd_plan_cached(nkt, B * Hkv, Hq / Hkv, causal ? 1 : 0, q_pos0 / kTile,
                                      kv_pos0 / kTile, round_tile(Sq) / 64, nsm);
  *split_key_tiles = pl.split;
  long long n = 0;
  if (pl.nplan > 0) {
    for (int e = 0; e < pl.nplan; ++e) n += pl.parts[e];
  } else {
    n = static_cast<long long>(nkt) * pl.uniform;
  }
  *ctas = static_cast<int>(n * B * Hkv);
  return ATTN_OK;
}

}  // extern "C"
