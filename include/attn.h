/*
 * mqa_attention_gb300 — C ABI of a CUDA library for NVIDIA GB300 (sm_103a).
 *
 * The library computes causal self-attention with rotary position embedding
 * (RoPE) applied to Q and K, grouped-query / multi-query K/V sharing and a
 * numerically stable (online) softmax, forward and backward:
 *
 *   q~_i = R_i q_i,  k~_j = R_j k_j                  (half-split RoPE)
 *   s_ij = scale * q~_i . k~_j,  j <= i when causal
 *   lse_i = ln sum_j exp(s_ij),  P_ij = exp(s_ij - lse_i)
 *   out_i = sum_j P_ij v_j
 *
 * Sources (web pages, cited by title and section):
 *   "Picotron模型实现解析Llama架构与Flash Attention集成", §1 嵌入层与位置编码
 *     (apply_rotary_pos_emb: x*cos + rotate_half(x)*sin, rotate_half = cat(-x2, x1)),
 *     §2 注意力机制实现 (flash_attn_func(q, k, v, causal)), §Flash Attention的优势
 *     (IO-aware tiling that never stores the S x S score matrix);
 *   "深度学习系统设计llama3-from-scratch：并行计算架构", §键值（Key-Value）共享机制
 *     (32 query heads share 8 key/value heads), §RoPE位置编码的并行实现,
 *     §注意力得分矩阵计算 (q.kᵀ / sqrt(head_dim)), §因果掩码的并行应用, §Softmax的并行计算;
 *   "ColossalAI 中的 PaLM 教学实现不到 200 行核心代码与 Booster 分布式训练实战",
 *     §2.3 RotaryEmbedding (inv_freq = 1/theta^(2i/dim), cat(freqs, freqs), both q and k
 *     rotated), §2.5 Attention (multi-query: one K/V head for all query heads; upper
 *     triangle masked; row maximum subtracted before the softmax).
 *
 * Conventions shared by every entry point
 *   Layout   q, out, dq: [B, Hq, S, D]; k, v, dk, dv: [B, Hkv, S, D]; lse: [B, Hq, S];
 *            all contiguous row-major, D innermost.
 *   Heads    query head h reads K/V head h / (Hq / Hkv) (contiguous groups).
 *   RoPE     half-split: for i < D/2, angle = p * theta^(-2i/D) at position p = 0..S-1;
 *            y_i = x_i cos - x_{i+D/2} sin, y_{i+D/2} = x_{i+D/2} cos + x_i sin.
 *            The rotated q and k are rounded to bf16 before the score product (see
 *            ATTN_ROPE_EXACT for how).
 *   Sizes    D in {64, 128}; S > 0 (the kernels work in 128-row tiles: for an S that is
 *            not a multiple of 128 they run on copies padded to whole tiles, with the
 *            padding rows contributing nothing, and copy the valid rows out, at the
 *            cost of those extra passes); Hq a multiple of Hkv;
 *            B * Hq * S < 2^31 (with S rounded up to a multiple of 128).
 *   Pointers device pointers, 16-byte aligned, not aliasing one another. The caller owns
 *            every buffer; the library never frees or keeps them.
 *   Stream   all work is enqueued on `stream` (a cudaStream_t, or 0); no call
 *            synchronises with the host except attn_sync_status and
 *            attn_profile_query. Temporary workspace is taken from a library-owned
 *            stream-ordered pool on the current device and released in stream order.
 *   RoPE     the cos/sin table of a (D, rope_theta) is built on the device the first
 *   table    time a call needs it (and rebuilt, at least twice as long, when a later
 *            call needs more positions), in stream order on that call's stream: memory
 *            from the pool, no host synchronisation; a call on another stream waits
 *            for the build on the device. At most 8 (D, rope_theta) tables are kept per
 *            device (least recently used dropped first); a dropped table is freed in
 *            stream order on the stream that drops it when only that stream read it,
 *            and otherwise (read by other streams, or under stream capture, where a
 *            graph may still read it) stays allocated until the process exits. A call
 *            under stream capture needs its table built and already seen complete by
 *            an earlier call outside capture (else ATTN_ERR_UNSUPPORTED): run a call
 *            for the same (D, rope_theta) and length, and one more after it has
 *            finished, before capturing (the usual warm-up does both).
 *   Device   the current CUDA device must be an sm_103 GPU (GB300).
 *   Errors   every entry point returns ATTN_OK (0) or one of the codes below and writes
 *            nothing when it rejects its arguments. Device-side failures of a launched
 *            kernel (a wait that exceeded its time limit) are reported by
 *            attn_sync_status().
 */
#ifndef MQA_ATTENTION_GB300_ATTN_H_
#define MQA_ATTENTION_GB300_ATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t; /* same type as cudaStream_t */

enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID = 1,     /* null / misaligned pointer, non-positive size, Hq % Hkv != 0,
                               non-finite or non-positive scale or theta, size overflow */
  ATTN_ERR_UNSUPPORTED = 2, /* D not in {64,128}, a partial block or position not a multiple
                               of 128, or device is not sm_103 */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  ATTN_ERR_TIMEOUT = 4,     /* a kernel's bounded wait expired (see attn_sync_status) */
  ATTN_ERR_BOUNDS = 5       /* debug build only: a kernel's index check failed and the access
                               was skipped (see attn_sync_status) */
};

/* Forward pass.
 *   q    [B,Hq,S,D]  bf16, read
 *   k, v [B,Hkv,S,D] bf16, read
 *   out  [B,Hq,S,D]  bf16, written: softmax(scale * q~ k~ᵀ + mask) v
 *   lse  [B,Hq,S]    fp32, written: natural-log log-sum-exp of each score row
 *   rope_theta > 0 (RoPE base), scale > 0 (score multiplier, usually 1/sqrt(D)),
 *   causal != 0 masks keys after the query (j > i); causal == 0 attends to all keys.
 * Sources: Picotron §1, §2; llama3-from-scratch §注意力得分矩阵计算, §因果掩码的并行应用,
 *   §Softmax的并行计算; PaLM §2.3, §2.5 (see the file header). */
int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
             int Hkv, int S, int D, float rope_theta, float scale, int causal,
             attn_stream_t stream);

/* Backward pass of attn_fwd with respect to q, k and v, for L = sum(dout * out).
 *   q, k, v, out (bf16) and lse (fp32) as produced by / given to attn_fwd;
 *   dout [B,Hq,S,D] bf16, read;
 *   dq [B,Hq,S,D], dk, dv [B,Hkv,S,D]: fp32, written (fully overwritten).
 *   dk and dv sum the contributions of all Hq/Hkv query heads of each group.
 * With dP_ij = dout_i.v_j, delta_i = dout_i.out_i, dS_ij = P_ij (dP_ij - delta_i):
 *   dq_i = scale R_iᵀ sum_j dS_ij k~_j,  dk_j = scale R_jᵀ sum_{h,i} dS_ij q~_i,
 *   dv_j = sum_{h,i} P_ij dout_i.
 * lse is treated as an input that is not differentiated. The gradient formulas are the
 * chain rule through the forward definition above (no page writes them out).
 * delta_i: in exact arithmetic dout_i.out_i = sum_j P_ij dP_ij. The `out` received is
 * rounded to bf16, and that rounding enters every dS_ij of the row and, summed over a
 * group's query heads, dk. attn_bwd takes delta from `out` (one read of it) when
 * Hq/Hkv <= 8, and otherwise runs an extra tensor-core pass over the scores that forms
 * sum_j P_ij dP_ij itself (about the cost of a forward pass); attn_bwd_ex can choose
 * either (ATTN_DELTA_* below). */
int attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
             const void* dout, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int S,
             int D, float rope_theta, float scale, int causal, attn_stream_t stream);

/* RoPE pair layouts of attn_fwd_ex / attn_bwd_ex. Both rotate pair i of a row at
 * position p by the angle p * rope_theta^(-2i/D), i < D/2:
 *   ATTN_ROPE_HALF        pairs (x_i, x_{i+D/2}): x*cos + rotate_half(x)*sin with
 *                         rotate_half(x) = cat(-x2, x1) (Picotron §1; PaLM §2.3);
 *                         the layout of attn_fwd / attn_bwd.
 *   ATTN_ROPE_INTERLEAVED pairs (x_{2i}, x_{2i+1}) read as the complex number
 *                         x_2i + j x_2i+1 and multiplied by polar(1, angle)
 *                         (llama3-from-scratch §RoPE). */
enum { ATTN_ROPE_HALF = 0, ATTN_ROPE_INTERLEAVED = 1 };

/* Rounding of the rotated q and k, OR-ed into the rope_mode argument of any entry point
 * that takes one. By default the rotation runs in fp32 (the table's cosines and sines
 * rounded to fp32) and is rounded once to bf16; in about 1 element of 40,000 that bf16
 * value differs from the value nearest the exact rotation, by one ulp or (where the
 * rotation cancels to far below its inputs) by up to 2^-22 (|x_i| + |x_(i+D/2)|). With
 * ATTN_ROPE_EXACT every rotated element is the bf16 value nearest the exact rotation
 * (cos/sin in fp64; evaluated with error-free products and sums, slower pre-passes).
 * A backward call must use the same rounding as the forward call whose out and lse it
 * receives (its recomputed scores are then the forward's). */
enum { ATTN_ROPE_EXACT = 0x10 };

/* Delta flags, OR-ed into the rope_mode argument of attn_bwd_ex and attn_bwd_bf16 (not
 * attn_bwd_partial, whose out is the merged result of every K/V block):
 *   ATTN_DELTA_EXACT     always form delta_i = sum_j P_ij dP_ij with the extra pass:
 *                        gradients free of the rounding of `out` (which dominates their
 *                        error when the softmax rows are sharply peaked or many query
 *                        heads share a K/V head); `out` is then not read;
 *   ATTN_DELTA_FROM_OUT  always take delta_i = dout_i.out_i from the bf16 `out`.
 * Neither: the default of attn_bwd (exact when Hq/Hkv > 8). Both: ATTN_ERR_INVALID. */
enum { ATTN_DELTA_EXACT = 0x100, ATTN_DELTA_FROM_OUT = 0x200 };

/* attn_fwd / attn_bwd with the RoPE pair layout chosen by rope_mode (one of the
 * ATTN_ROPE_* layouts, optionally OR-ed with ATTN_ROPE_EXACT, and for attn_bwd_ex with one
 * ATTN_DELTA_* flag; anything else returns ATTN_ERR_INVALID). Arguments, layouts,
 * ownership and errors are otherwise those of attn_fwd / attn_bwd; attn_fwd(...) is
 * attn_fwd_ex(..., rope_theta, ATTN_ROPE_HALF, scale, ...). */
int attn_fwd_ex(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                int Hq, int Hkv, int S, int D, float rope_theta, int rope_mode, float scale,
                int causal, attn_stream_t stream);
int attn_bwd_ex(const void* q, const void* k, const void* v, const void* out, const float* lse,
                const void* dout, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int S,
                int D, float rope_theta, int rope_mode, float scale, int causal,
                attn_stream_t stream);

/* Blocks of queries and keys: the pieces a context-parallel (ring) schedule computes
 * when the sequence is split across devices or passes (Picotron §上下文并行, with the
 * 32K-token sequences of Megatron-SP). The query block holds Sq rows per head at
 * positions q_pos0 + i, the K/V block Skv rows at kv_pos0 + j; RoPE rotates every row
 * by its own position and the causal mask compares positions. Sq, Skv, q_pos0 and
 * kv_pos0 are multiples of 128 (else ATTN_ERR_UNSUPPORTED; negative: ATTN_ERR_INVALID).
 *
 * attn_fwd_partial: out [B,Hq,Sq,D] bf16 and lse [B,Hq,Sq] fp32 of the attention over
 *   this K/V block alone; a row that sees none of its keys gets out = 0, lse = -inf.
 *   attn_fwd_ex(...) is attn_fwd_partial with Sq = Skv = S, q_pos0 = kv_pos0 = 0.
 * attn_bwd_partial: the contributions of this K/V block to the gradients, given the
 *   out and lse of the query block's whole attention (merged over every K/V block):
 *   P_ij = exp(s_ij - lse_i) for this block's keys, delta_i = dout_i . out_i. dq
 *   [B,Hq,Sq,D] (summed over the K/V blocks by the caller), dk, dv [B,Hkv,Skv,D]
 *   (summed over the query blocks) are fp32, fully overwritten.
 * attn_merge: out, lse of the union of two disjoint key sets of the same `rows` query
 *   rows (B*Hq*Sq) from their partial results: lse = ln(e^lse_a + e^lse_b),
 *   out = e^(lse_a - lse) out_a + e^(lse_b - lse) out_b (bf16 out, fp32 lse); out and
 *   lse may be out_a and lse_a. */
int attn_fwd_partial(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                     int Hq, int Hkv, int Sq, int Skv, int D, int q_pos0, int kv_pos0,
                     float rope_theta, int rope_mode, float scale, int causal,
                     attn_stream_t stream);
int attn_bwd_partial(const void* q, const void* k, const void* v, const void* out,
                     const float* lse, const void* dout, float* dq, float* dk, float* dv, int B,
                     int Hq, int Hkv, int Sq, int Skv, int D, int q_pos0, int kv_pos0,
                     float rope_theta, int rope_mode, float scale, int causal,
                     attn_stream_t stream);
int attn_merge(const void* out_a, const float* lse_a, const void* out_b, const float* lse_b,
               void* out, float* lse, long long rows, int D, attn_stream_t stream);

/* y = RoPE(x) rounded to bf16: x, y [heads, S, D] bf16 (may be the same buffer), row i
 * of every head rotated by the angle of position pos0 + i in the layout rope_mode (the
 * rotation attn_fwd applies to q and k). Fills the rotated key cache attn_decode
 * reads. */
int attn_rope(const void* x, void* y, long long heads, int S, int pos0, int D,
              float rope_theta, int rope_mode, attn_stream_t stream);

/* Decode-shape forward: Sq new query rows per head (q [B,Hq,Sq,D] bf16, not rotated;
 * row i at position q_pos0 + i) against a cache of Skv keys and values:
 * k_rot [B,Hkv,Skv,D] bf16 holding the keys already rotated by their positions
 * 0..Skv-1 (as attn_rope writes them), v [B,Hkv,Skv,D] bf16. Key j is seen by query i
 * when j <= q_pos0 + i (and j < Skv); out [B,Hq,Sq,D] bf16, lse [B,Hq,Sq] fp32 as in
 * attn_fwd (a row that sees no key: out = 0, lse = -inf). The Hq/Hkv query heads of a
 * K/V head share each pass over its cache (PaLM §2.5: one shared K/V head is what
 * makes decoding cheap), so (Hq/Hkv) * Sq <= 128 (else ATTN_ERR_UNSUPPORTED). Any
 * Skv >= 1. */
int attn_decode(const void* q, const void* k_rot, const void* v, void* out, float* lse, int B,
                int Hq, int Hkv, int Sq, int Skv, int D, int q_pos0, float rope_theta,
                int rope_mode, float scale, attn_stream_t stream);

/* attn_bwd_ex writing bf16 gradients: dq [B,Hq,S,D], dk, dv [B,Hkv,S,D] bf16, each the
 * value attn_bwd_ex writes in fp32 rounded to nearest even (dk and dv bit for bit;
 * dq's fp32 value sums its partial products in a run-dependent order, so it may
 * differ from another run's by one bf16 ulp). The rounding alone can exceed the
 * fp32 path's error by half a bf16 ulp of the gradient (|dv| ~ 11 at the PaLM-MQA
 * shape gives ~0.03), which is why fp32 is the primary output. Uses
 * 2 * B*Hkv*S*D*4 bytes more workspace than attn_bwd_ex. */
int attn_bwd_bf16(const void* q, const void* k, const void* v, const void* out, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S,
                  int D, float rope_theta, int rope_mode, float scale, int causal,
                  attn_stream_t stream);

/* Waits for all work on `stream`, then reads and clears the device status word of the
 * current device: ATTN_OK, or ATTN_ERR_TIMEOUT if a kernel gave up on a wait since the
 * last call, or (in the library built with GB_BOUNDS_CHECK, which checks every global
 * index and TMA coordinate before using it) ATTN_ERR_BOUNDS if a check failed; the
 * outputs are then undefined. The first failure since the last call is the one kept.
 * Synchronises the host with `stream`. */
int attn_sync_status(attn_stream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* attn_status_string(int status);

/* Kernel timing with CUDA events recorded on the launching stream around every kernel
 * the library launches. attn_profile_begin clears previous records and enables
 * recording (at most `max_launches` launches per kernel kind are kept);
 * attn_profile_end disables it. attn_profile_query synchronises the recorded events and
 * returns the number of recorded launches of `kernel` and their summed duration in ms.
 * Kernel kinds: 0 rope (forward RoPE pre-pass), 1 forward attention, 2 backward
 * pre-pass, 3 backward dK/dV/dQ main kernel, 4 dQ finalisation, 5 the exact delta pass. */
enum {
  ATTN_KERNEL_ROPE = 0,
  ATTN_KERNEL_FWD = 1,
  ATTN_KERNEL_BWD_PREP = 2,
  ATTN_KERNEL_BWD_MAIN = 3,
  ATTN_KERNEL_DQ_FINAL = 4,
  ATTN_KERNEL_DELTA = 5,
  ATTN_NUM_KERNELS = 6
};
int attn_profile_begin(int max_launches);
int attn_profile_end(void);
int attn_profile_query(int kernel, int* launches, float* total_ms);

/* Fault-path testing: while `enable` is non-zero, the main kernels of subsequent
 * attn_fwd / attn_bwd calls wait on a barrier that nothing signals, so the wait expires
 * after its time limit (about two seconds), the kernel unwinds, releases its tensor
 * memory and reports ATTN_ERR_TIMEOUT through attn_sync_status(). Outputs of such a
 * call are undefined. Not for production use. */
int attn_debug_inject_timeout(int enable);

/* The backward main kernel's work plan for these sizes on a GPU with `nsm` SMs, as
 * attn_bwd / attn_bwd_partial would choose it (host computation only; touches no
 * device): *split_key_tiles = how many of the heaviest key tiles get two CTAs (each
 * half of the group's query heads, dK/dV added), *ctas = CTAs launched. Sizes as in
 * attn_bwd_partial (self-attention: Sq = Skv, positions 0). Returns ATTN_OK, or
 * ATTN_ERR_INVALID for invalid sizes or null outputs. */
int attn_debug_bwd_plan(int B, int Hq, int Hkv, int Sq, int Skv, int q_pos0, int kv_pos0,
                        int causal, int nsm, int* split_key_tiles, int* ctas);

/* Library version string. */
const char* attn_version(void);

/* Forward pass that allocates nothing (no counterpart on the source pages: it exists
 * for callers of this library that may not allocate GPU memory, e.g. services that
 * reserve all device memory up front or runtimes that own the allocator).
 * Arguments, layouts, results and argument errors are those of attn_fwd, except that
 * S must be a multiple of 128 (else ATTN_ERR_UNSUPPORTED). Instead of
 * attn_fwd's pooled workspace and cached RoPE tables it uses one fixed array of
 * ATTN_FWD_NOALLOC_SCRATCH_BYTES in device memory that the CUDA runtime reserves on
 * every GPU where the library's code is loaded and keeps until the process exits.
 * Limit: 16*ceil64(S*D/2) + round256(2*B*Hq*S*D) + round256(2*B*Hkv*S*D) + 256 bytes
 * (ceil64: rounded up to a multiple of 64) must fit in that array (e.g. B=1, Hq=32,
 * Hkv=8, S=4096, D=128 needs 46 MB); larger problems return ATTN_ERR_UNSUPPORTED.
 * The first call on each device looks up the array's device address (with that
 * device current); make that first call before any stream capture.
 * All calls on a device share the array and leave their contents in it: calls whose
 * GPU work overlaps (other streams, other host threads) race and give undefined
 * results. A kernel wait that expires here leaves out/lse undefined and is reported
 * by attn_sync_status like any other (the status word is a static device variable, so
 * finding it allocates nothing). The device address of that array and of the status
 * word may not outlive the CUDA context they were looked up in: do not keep using the
 * library across cudaDeviceReset. No cudaMalloc, cudaFree or allocating routine. */
#define ATTN_FWD_NOALLOC_SCRATCH_BYTES (64u << 20)
int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                     int Hq, int Hkv, int S, int D, float rope_theta, float scale, int causal,
                     attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MQA_ATTENTION_GB300_ATTN_H_ */
