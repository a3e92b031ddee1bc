"""Python binding of the mqa_attention_gb300 C ABI (include/attn.h).

Argument marshalling only: every step of the attention computation runs in
the CUDA kernels of ``libmqa_attention_gb300.so``. There is no CPU fallback;
calling into the library without the built shared library raises.

Tensors are passed as ``torch.Tensor`` (their device pointer is used) or as
raw integer device pointers. The stream defaults to torch's current stream.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = [
    "AttnError",
    "lib",
    "attn_fwd",
    "attn_bwd",
    "attn_fwd_noalloc",
    "attn_fwd_ex",
    "attn_bwd_ex",
    "attn_bwd_bf16",
    "attn_fwd_partial",
    "attn_bwd_partial",
    "attn_merge",
    "attn_rope",
    "attn_decode",
    "rope",
    "decode",
    "forward",
    "forward_partial",
    "backward_partial",
    "merge",
    "backward",
    "sync_status",
    "status_string",
    "profile_begin",
    "profile_end",
    "profile_query",
    "debug_inject_timeout",
    "debug_bwd_plan",
    "version",
    "EXPORTED_SYMBOLS",
    "KERNEL_ROPE",
    "KERNEL_FWD",
    "KERNEL_BWD_PREP",
    "KERNEL_BWD_MAIN",
    "KERNEL_DQ_FINAL",
    "KERNEL_DELTA",
    "DELTA_MODES",
    "ROPE_EXACT",
]

LIB_NAME = "libmqa_attention_gb300.so"
# MQA_ATTENTION_GB300_LIB selects another build of the library (for example the
# bounds-checking one, libmqa_attention_gb300_debug.so) for the whole process.
LIB_PATH = os.environ.get("MQA_ATTENTION_GB300_LIB") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), LIB_NAME)

ATTN_OK, ATTN_ERR_INVALID, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = range(5)
ATTN_ERR_BOUNDS = 5
KERNEL_ROPE, KERNEL_FWD, KERNEL_BWD_PREP, KERNEL_BWD_MAIN, KERNEL_DQ_FINAL, KERNEL_DELTA = range(6)
# delta flags OR-ed into the rope_mode of attn_bwd_ex / attn_bwd_bf16 (ATTN_DELTA_*)
DELTA_MODES = {"auto": 0, "exact": 0x100, "from_out": 0x200}
ROPE_EXACT = 0x10  # ATTN_ROPE_EXACT: rotated q, k rounded as the exact rotation rounds

EXPORTED_SYMBOLS = (
    "attn_fwd",
    "attn_bwd",
    "attn_fwd_ex",
    "attn_bwd_ex",
    "attn_bwd_bf16",
    "attn_fwd_partial",
    "attn_bwd_partial",
    "attn_merge",
    "attn_rope",
    "attn_decode",
    "attn_sync_status",
    "attn_status_string",
    "attn_profile_begin",
    "attn_profile_end",
    "attn_profile_query",
    "attn_debug_inject_timeout",
    "attn_debug_bwd_plan",
    "attn_version",
    "attn_fwd_noalloc",
)


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (status {code})")


_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float


def lib() -> ctypes.CDLL:
    """The loaded shared library (loaded on first use; raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_NAME} is not built; run `python -m mqa_attention_gb300.build` "
                    "(or __graft_entry__.build())"
                )
            L = ctypes.CDLL(LIB_PATH)
            L.attn_fwd.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _I, _P]
            L.attn_fwd.restype = _I
            L.attn_bwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _I, _I, _I, _I, _I, _F, _F, _I, _P]
            L.attn_bwd.restype = _I
            L.attn_sync_status.argtypes = [_P]
            L.attn_sync_status.restype = _I
            L.attn_status_string.argtypes = [_I]
            L.attn_status_string.restype = ctypes.c_char_p
            L.attn_profile_begin.argtypes = [_I]
            L.attn_profile_begin.restype = _I
            L.attn_profile_end.argtypes = []
            L.attn_profile_end.restype = _I
            L.attn_profile_query.argtypes = [_I, ctypes.POINTER(_I), ctypes.POINTER(_F)]
            L.attn_profile_query.restype = _I
            L.attn_debug_inject_timeout.argtypes = [_I]
            L.attn_debug_inject_timeout.restype = _I
            L.attn_debug_bwd_plan.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, _I,
                                              ctypes.POINTER(_I), ctypes.POINTER(_I)]
            L.attn_debug_bwd_plan.restype = _I
            L.attn_version.argtypes = []
            L.attn_version.restype = ctypes.c_char_p
            L.attn_fwd_noalloc.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _I, _P]
            L.attn_fwd_noalloc.restype = _I
            L.attn_fwd_ex.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _F, _I, _P]
            L.attn_fwd_ex.restype = _I
            L.attn_bwd_ex.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P,
                                      _I, _I, _I, _I, _I, _F, _I, _F, _I, _P]
            L.attn_bwd_ex.restype = _I
            L.attn_bwd_bf16.argtypes = L.attn_bwd_ex.argtypes
            L.attn_bwd_bf16.restype = _I
            L.attn_fwd_partial.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                           _F, _I, _F, _I, _P]
            L.attn_fwd_partial.restype = _I
            L.attn_bwd_partial.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                           _I, _I, _I, _F, _I, _F, _I, _P]
            L.attn_bwd_partial.restype = _I
            L.attn_merge.argtypes = [_P, _P, _P, _P, _P, _P, ctypes.c_longlong, _I, _P]
            L.attn_merge.restype = _I
            L.attn_rope.argtypes = [_P, _P, ctypes.c_longlong, _I, _I, _I, _F, _I, _P]
            L.attn_rope.restype = _I
            L.attn_decode.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _F,
                                      _P]
            L.attn_decode.restype = _I
            _lib = L
        return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, what: str):
    if code != ATTN_OK:
        raise AttnError(code, what)


def attn_fwd(q, k, v, out, lse, B, Hq, Hkv, S, D, rope_theta, scale, causal, stream=None):
    """C ABI attn_fwd: out (bf16) and lse (fp32) from q, k, v (bf16)."""
    _check(lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(B), int(Hq),
                          int(Hkv), int(S), int(D), float(rope_theta), float(scale),
                          1 if causal else 0, _stream(stream)), "attn_fwd")


def attn_fwd_noalloc(q, k, v, out, lse, B, Hq, Hkv, S, D, rope_theta, scale, causal,
                     stream=None):
    """C ABI attn_fwd_noalloc: attn_fwd for callers that may not allocate GPU memory
    (it works in a fixed array the library reserves on each GPU; see attn.h for the
    size limit and the rule that overlapping calls race)."""
    _check(lib().attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(B),
                                  int(Hq), int(Hkv), int(S), int(D), float(rope_theta),
                                  float(scale), 1 if causal else 0, _stream(stream)),
           "attn_fwd_noalloc")


def attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, D, rope_theta, scale, causal,
             stream=None):
    """C ABI attn_bwd: dq, dk, dv (fp32) from q, k, v, out, dout (bf16) and lse (fp32)."""
    _check(lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                          _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv), int(S), int(D),
                          float(rope_theta), float(scale), 1 if causal else 0,
                          _stream(stream)), "attn_bwd")


ROPE_MODES = {"half": 0, "interleaved": 1}  # ATTN_ROPE_HALF, ATTN_ROPE_INTERLEAVED


def attn_fwd_ex(q, k, v, out, lse, B, Hq, Hkv, S, D, rope_theta, rope_mode, scale, causal,
                stream=None):
    """C ABI attn_fwd_ex: attn_fwd with the RoPE pair layout rope_mode (0 half-split,
    1 interleaved complex pairs)."""
    _check(lib().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(B), int(Hq),
                             int(Hkv), int(S), int(D), float(rope_theta), int(rope_mode),
                             float(scale), 1 if causal else 0, _stream(stream)), "attn_fwd_ex")


def attn_bwd_ex(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, D, rope_theta, rope_mode,
                scale, causal, stream=None):
    """C ABI attn_bwd_ex: attn_bwd with the RoPE pair layout rope_mode."""
    _check(lib().attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                             _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv), int(S),
                             int(D), float(rope_theta), int(rope_mode), float(scale),
                             1 if causal else 0, _stream(stream)), "attn_bwd_ex")


def attn_bwd_bf16(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, D, rope_theta, rope_mode,
                  scale, causal, stream=None):
    """C ABI attn_bwd_bf16: attn_bwd_ex writing bf16 dq, dk, dv (the fp32 values
    rounded to nearest even)."""
    _check(lib().attn_bwd_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                               _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv), int(S),
                               int(D), float(rope_theta), int(rope_mode), float(scale),
                               1 if causal else 0, _stream(stream)), "attn_bwd_bf16")


def attn_fwd_partial(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, D, q_pos0, kv_pos0, rope_theta,
                     rope_mode, scale, causal, stream=None):
    """C ABI attn_fwd_partial: attention of a query block over one K/V block."""
    _check(lib().attn_fwd_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(B),
                                  int(Hq), int(Hkv), int(Sq), int(Skv), int(D), int(q_pos0),
                                  int(kv_pos0), float(rope_theta), int(rope_mode), float(scale),
                                  1 if causal else 0, _stream(stream)), "attn_fwd_partial")


def attn_bwd_partial(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Skv, D, q_pos0,
                     kv_pos0, rope_theta, rope_mode, scale, causal, stream=None):
    """C ABI attn_bwd_partial: one K/V block's gradient contributions."""
    _check(lib().attn_bwd_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                  _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv),
                                  int(Sq), int(Skv), int(D), int(q_pos0), int(kv_pos0),
                                  float(rope_theta), int(rope_mode), float(scale),
                                  1 if causal else 0, _stream(stream)), "attn_bwd_partial")


def attn_merge(out_a, lse_a, out_b, lse_b, out, lse, rows, D, stream=None):
    """C ABI attn_merge: combine two partial results of the same query rows."""
    _check(lib().attn_merge(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), _ptr(out),
                            _ptr(lse), int(rows), int(D), _stream(stream)), "attn_merge")


def attn_rope(x, y, heads, S, pos0, D, rope_theta, rope_mode, stream=None):
    """C ABI attn_rope: y = bf16(RoPE(x)) for rows at positions pos0 + i."""
    _check(lib().attn_rope(_ptr(x), _ptr(y), int(heads), int(S), int(pos0), int(D),
                           float(rope_theta), int(rope_mode), _stream(stream)), "attn_rope")


def attn_decode(q, k_rot, v, out, lse, B, Hq, Hkv, Sq, Skv, D, q_pos0, rope_theta, rope_mode,
                scale, stream=None):
    """C ABI attn_decode: Sq new queries per head against a rotated K/V cache."""
    _check(lib().attn_decode(_ptr(q), _ptr(k_rot), _ptr(v), _ptr(out), _ptr(lse), int(B),
                             int(Hq), int(Hkv), int(Sq), int(Skv), int(D), int(q_pos0),
                             float(rope_theta), int(rope_mode), float(scale), _stream(stream)),
           "attn_decode")


def rope(x, rope_theta, pos0=0, out=None, stream=None, rope="half", exact=False):
    """bf16 RoPE(x) of x [..., S, D] (rows at positions pos0..pos0+S-1); exact=True
    rounds as the exact rotation rounds (ATTN_ROPE_EXACT)."""
    import torch

    S, D = x.shape[-2], x.shape[-1]
    y = torch.empty_like(x) if out is None else out
    attn_rope(x, y, x.numel() // (S * D), S, pos0, D, rope_theta,
              ROPE_MODES[rope] | (ROPE_EXACT if exact else 0), stream)
    return y


def decode(q, k_rot, v, rope_theta, q_pos0=None, scale=None, stream=None, rope="half"):
    """Allocates out / lse and runs attn_decode; q: [B,Hq,Sq,D], caches [B,Hkv,Skv,D].
    q_pos0 defaults to Skv - Sq (the new tokens are the cache's last positions)."""
    import torch

    B, Hq, Sq, D = q.shape
    Hkv, Skv = k_rot.shape[1], k_rot.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    q_pos0 = Skv - Sq if q_pos0 is None else q_pos0
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    attn_decode(q, k_rot, v, out, lse, B, Hq, Hkv, Sq, Skv, D, q_pos0, rope_theta,
                ROPE_MODES[rope], scale, stream)
    return out, lse


def forward_partial(q, k, v, rope_theta, q_pos0, kv_pos0, scale=None, causal=True, stream=None,
                    rope="half"):
    """Allocates out / lse and runs attn_fwd_partial. q: [B,Hq,Sq,D], k, v: [B,Hkv,Skv,D]."""
    import torch

    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    attn_fwd_partial(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, D, q_pos0, kv_pos0, rope_theta,
                     ROPE_MODES[rope], scale, causal, stream)
    return out, lse


def backward_partial(q, k, v, out, lse, dout, rope_theta, q_pos0, kv_pos0, scale=None,
                     causal=True, stream=None, rope="half"):
    """Allocates fp32 dq, dk, dv and runs attn_bwd_partial (out, lse: the query
    block's merged attention)."""
    import torch

    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    dv = torch.empty(v.shape, dtype=torch.float32, device=q.device)
    attn_bwd_partial(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Skv, D, q_pos0,
                     kv_pos0, rope_theta, ROPE_MODES[rope], scale, causal, stream)
    return dq, dk, dv


def merge(out_a, lse_a, out_b, lse_b, out=None, lse=None, stream=None):
    """attn_merge into new tensors, or in place when out / lse are given (they may
    be out_a / lse_a)."""
    import torch

    out = torch.empty_like(out_a) if out is None else out
    lse = torch.empty_like(lse_a) if lse is None else lse
    attn_merge(out_a, lse_a, out_b, lse_b, out, lse, lse_a.numel(), out_a.shape[-1], stream)
    return out, lse


def _shapes(q, k):
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    return B, Hq, Hkv, S, D


def forward(q, k, v, rope_theta, scale=None, causal=True, stream=None, rope="half",
            exact_rope=False):
    """Allocates out / lse like q and runs attn_fwd (attn_fwd_ex for rope="interleaved" or
    exact_rope=True, ATTN_ROPE_EXACT). q: [B,Hq,S,D], k, v: [B,Hkv,S,D]."""
    import torch

    B, Hq, Hkv, S, D = _shapes(q, k)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    mode = ROPE_MODES[rope] | (ROPE_EXACT if exact_rope else 0)
    if mode == 0:
        attn_fwd(q, k, v, out, lse, B, Hq, Hkv, S, D, rope_theta, scale, causal, stream)
    else:
        attn_fwd_ex(q, k, v, out, lse, B, Hq, Hkv, S, D, rope_theta, mode, scale, causal, stream)
    return out, lse


def backward(q, k, v, out, lse, dout, rope_theta, scale=None, causal=True, stream=None,
             rope="half", grad_dtype=None, delta="auto", exact_rope=False):
    """Allocates dq, dk, dv and runs attn_bwd (attn_bwd_ex for rope="interleaved" or a
    delta mode other than "auto", attn_bwd_bf16 for grad_dtype=torch.bfloat16; fp32
    gradients otherwise). delta: "auto" (attn_bwd's choice), "exact" (the extra pass over
    the scores) or "from_out" (dout . out). exact_rope: as the forward call's."""
    import torch

    B, Hq, Hkv, S, D = _shapes(q, k)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    gd = torch.bfloat16 if grad_dtype == torch.bfloat16 else torch.float32
    dq = torch.empty(q.shape, dtype=gd, device=q.device)
    dk = torch.empty(k.shape, dtype=gd, device=q.device)
    dv = torch.empty(v.shape, dtype=gd, device=q.device)
    mode = ROPE_MODES[rope] | DELTA_MODES[delta] | (ROPE_EXACT if exact_rope else 0)
    if gd == torch.bfloat16:
        attn_bwd_bf16(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, D, rope_theta, mode,
                      scale, causal, stream)
    elif mode == 0:
        attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, D, rope_theta, scale, causal,
                 stream)
    else:
        attn_bwd_ex(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, D, rope_theta, mode,
                    scale, causal, stream)
    return dq, dk, dv


def sync_status(stream=None) -> int:
    """Synchronises `stream` and returns (and clears) the device status code."""
    return lib().attn_sync_status(_stream(stream))


def status_string(code: int) -> str:
    try:
        return lib().attn_status_string(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


def profile_begin(max_launches: int = 4096):
    _check(lib().attn_profile_begin(int(max_launches)), "attn_profile_begin")


def profile_end():
    _check(lib().attn_profile_end(), "attn_profile_end")


def profile_query(kernel: int):
    """(launches, total_ms) recorded for one kernel kind since profile_begin."""
    n = _I(0)
    ms = _F(0.0)
    _check(lib().attn_profile_query(int(kernel), ctypes.byref(n), ctypes.byref(ms)),
           "attn_profile_query")
    return n.value, ms.value


def debug_inject_timeout(enable: bool):
    _check(lib().attn_debug_inject_timeout(1 if enable else 0), "attn_debug_inject_timeout")


def debug_bwd_plan(B, Hq, Hkv, Sq, Skv, nsm, q_pos0=0, kv_pos0=0, causal=True):
    """The backward main kernel's work plan on a GPU with `nsm` SMs (host only):
    (number of heaviest key tiles split between two CTAs, CTAs launched)."""
    split, ctas = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().attn_debug_bwd_plan(B, Hq, Hkv, Sq, Skv, q_pos0, kv_pos0, 1 if causal else 0,
                                     nsm, ctypes.byref(split), ctypes.byref(ctas)),
           "attn_debug_bwd_plan")
    return split.value, ctas.value


def version() -> str:
    return lib().attn_version().decode()
