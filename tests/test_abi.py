"""The C-ABI library loads, exports every symbol include/attn.h declares, and
rejects bad arguments before touching the GPU (so these run without one)."""
import ctypes
import os
import re

import pytest

import mqa_attention_gb300 as M

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "attn.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_\w+)\s*\(", src)))


def test_header_matches_binding_list():
    assert declared_functions() == sorted(M.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(built_lib):
    for name in declared_functions():
        assert hasattr(built_lib, name), name


def test_version_and_status_strings(built_lib):
    assert "sm_103a" in M.version()
    assert M.status_string(0) == "ok"
    assert M.status_string(M.ATTN_ERR_TIMEOUT) == "device wait timed out"
    assert M.status_string(99) == "unknown status"


FAKE = 0x10000  # aligned, never dereferenced: validation rejects first


def fwd_code(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=FAKE, B=1, Hq=4, Hkv=1, S=128, D=64,
             theta=10000.0, scale=0.125):
    return lib.attn_fwd(q, k, v, out, lse, B, Hq, Hkv, S, D, theta, scale, 1, None)


def bwd_code(lib, ptr=FAKE, B=1, Hq=4, Hkv=1, S=128, D=64, theta=10000.0, scale=0.125, **over):
    p = dict(q=ptr, k=ptr, v=ptr, out=ptr, lse=ptr, dout=ptr, dq=ptr, dk=ptr, dv=ptr)
    p.update(over)
    return lib.attn_bwd(p["q"], p["k"], p["v"], p["out"], p["lse"], p["dout"], p["dq"], p["dk"],
                        p["dv"], B, Hq, Hkv, S, D, theta, scale, 1, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), M.ATTN_ERR_INVALID),
    (dict(lse=FAKE + 4), M.ATTN_ERR_INVALID),
    (dict(B=0), M.ATTN_ERR_INVALID),
    (dict(Hq=6, Hkv=4), M.ATTN_ERR_INVALID),
    (dict(scale=float("nan")), M.ATTN_ERR_INVALID),
    (dict(scale=-1.0), M.ATTN_ERR_INVALID),
    (dict(theta=0.0), M.ATTN_ERR_INVALID),
    (dict(theta=float("inf")), M.ATTN_ERR_INVALID),
    (dict(B=1 << 12, Hq=1 << 12, S=1 << 8), M.ATTN_ERR_INVALID),
    (dict(D=96), M.ATTN_ERR_UNSUPPORTED),
    (dict(D=256), M.ATTN_ERR_UNSUPPORTED),
])
def test_fwd_rejects_bad_arguments(built_lib, kw, code):
    assert fwd_code(built_lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(dv=None), M.ATTN_ERR_INVALID),
    (dict(dq=FAKE + 8), M.ATTN_ERR_INVALID),
    (dict(Hq=3, Hkv=2), M.ATTN_ERR_INVALID),
    (dict(S=-128), M.ATTN_ERR_INVALID),
    (dict(D=32), M.ATTN_ERR_UNSUPPORTED),
])
def test_bwd_rejects_bad_arguments(built_lib, kw, code):
    assert bwd_code(built_lib, **kw) == code


@pytest.mark.parametrize("mode", [-1, 2, 7])
def test_ex_entry_points_reject_unknown_rope_modes(built_lib, mode):
    """attn_fwd_ex / attn_bwd_ex take ATTN_ROPE_HALF (0) or ATTN_ROPE_INTERLEAVED (1)."""
    lib = built_lib
    assert lib.attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 128, 64, 10000.0, mode, 0.125,
                           1, None) == M.ATTN_ERR_INVALID
    assert lib.attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 128, 64,
                           10000.0, mode, 0.125, 1, None) == M.ATTN_ERR_INVALID


@pytest.mark.parametrize("mode", [0x100 | 0x200, 0x400, 0x100 | 2])
def test_bwd_rejects_bad_delta_flags(built_lib, mode):
    """ATTN_DELTA_EXACT (0x100) and ATTN_DELTA_FROM_OUT (0x200) exclude each other; no
    other flag exists; the layout must still be valid."""
    assert built_lib.attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1,
                                 128, 64, 10000.0, mode, 0.125, 1, None) == M.ATTN_ERR_INVALID
    assert built_lib.attn_bwd_bf16(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1,
                                   128, 64, 10000.0, mode, 0.125, 1, None) == M.ATTN_ERR_INVALID


def test_exact_rope_flag_is_accepted_where_rope_mode_is(built_lib):
    """ATTN_ROPE_EXACT (0x10) combines with either layout; with a bad layout, or on an
    entry point that takes no flags besides it, the call is still rejected first."""
    lib = built_lib
    ex = M.ROPE_EXACT
    assert lib.attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 128, 96, 10000.0, ex | 1, 0.125,
                           1, None) == M.ATTN_ERR_UNSUPPORTED  # flag accepted, D rejected
    assert lib.attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 128, 64, 10000.0, ex | 2, 0.125,
                           1, None) == M.ATTN_ERR_INVALID
    assert lib.attn_rope(FAKE, FAKE, 4, 100, 0, 64, 10000.0, ex | 0x100, None) == \
        M.ATTN_ERR_INVALID


def test_delta_flags_only_where_they_apply(built_lib):
    """The exact delta pass needs the whole attention of each query row: a partial
    block's backward and every forward entry point refuse the flag."""
    lib = built_lib
    exact = M.DELTA_MODES["exact"]
    assert lib.attn_bwd_partial(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1,
                                128, 128, 64, 0, 0, 10000.0, exact, 0.125, 1,
                                None) == M.ATTN_ERR_INVALID
    assert lib.attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 128, 64, 10000.0, exact, 0.125,
                           1, None) == M.ATTN_ERR_INVALID


def test_profile_arguments(built_lib):
    assert built_lib.attn_profile_begin(0) == M.ATTN_ERR_INVALID
    n, ms = ctypes.c_int(), ctypes.c_float()
    assert built_lib.attn_profile_query(7, ctypes.byref(n), ctypes.byref(ms)) == M.ATTN_ERR_INVALID
    assert built_lib.attn_profile_query(0, None, None) == M.ATTN_ERR_INVALID
    assert built_lib.attn_profile_begin(16) == 0
    assert built_lib.attn_profile_query(1, ctypes.byref(n), ctypes.byref(ms)) == 0
    assert n.value == 0 and ms.value == 0.0
    assert built_lib.attn_profile_end() == 0


def test_missing_library_fails_loudly(monkeypatch):
    """Without the shared library the binding raises; there is no fallback."""
    monkeypatch.setattr(M, "_lib", None)
    monkeypatch.setattr(M, "LIB_PATH", "/nonexistent/libmqa_attention_gb300.so")
    with pytest.raises(RuntimeError, match="not built"):
        M.lib()


def test_partial_entry_points_reject_unaligned_blocks(built_lib):
    """Blocks and their positions are multiples of 128; negative positions are invalid."""
    lib = built_lib
    f = lambda sq, skv, qp, kp: lib.attn_fwd_partial(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, sq,
                                                     skv, 64, qp, kp, 10000.0, 0, 0.125, 1, None)
    assert f(128, 256, 64, 0) == M.ATTN_ERR_UNSUPPORTED
    assert f(128, 200, 0, 0) == M.ATTN_ERR_UNSUPPORTED
    assert f(128, 128, -128, 0) == M.ATTN_ERR_INVALID
    assert lib.attn_merge(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 64, None) == M.ATTN_ERR_INVALID
    assert lib.attn_merge(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 96, None) == \
        M.ATTN_ERR_UNSUPPORTED


def test_decode_rejects_groups_beyond_one_tile(built_lib):
    """A K/V head's query rows (Hq/Hkv * Sq) must fit one 128-row tile."""
    lib = built_lib
    assert lib.attn_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 1, 17, 256, 64, 239, 10000.0, 0,
                           0.125, None) == M.ATTN_ERR_UNSUPPORTED
    assert lib.attn_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 1, 1, 256, 64, -1, 10000.0, 0,
                           0.125, None) == M.ATTN_ERR_INVALID
    assert lib.attn_rope(FAKE, FAKE, 4, 100, 0, 96, 10000.0, 0, None) == M.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("shape,want", [
    # (B, Hq, Hkv, Sq, Skv, SMs) -> (key tiles split in two, CTAs)
    ((1, 32, 8, 4096, 4096, 152), (6, 304)),       # Llama-3-8B: the 6 heaviest key tiles
    ((8, 8, 1, 2048, 2048, 152), (12, 224)),       # PaLM-MQA: 128 key tiles < 152 SMs
    ((4, 32, 32, 1024, 1024, 152), (0, 1024)),     # SmolLM (MHA): one head per group, no split
    ((1, 32, 8, 32768, 32768, 152), (0, 2048)),    # 13 waves: balanced as it is
    ((1, 8, 1, 16384, 16384, 152), (128, 256)),    # beyond the table: every tile split
])
def test_backward_work_plan(shape, want):
    """The host's choice of which heavy key tiles to split (a simulated greedy
    schedule of the CTAs on the SMs; no GPU needed)."""
    assert M.debug_bwd_plan(*shape) == want


def test_backward_work_plan_counts_ctas():
    for B, Hq, Hkv, S in [(1, 32, 8, 4096), (2, 16, 4, 2048), (8, 8, 1, 2048), (1, 4, 1, 300)]:
        nkt = -(-S // 128)
        split, ctas = M.debug_bwd_plan(B, Hq, Hkv, S, S, 152)
        assert 0 <= split <= nkt
        if (Hq // Hkv) % 2:
            assert split == 0
        assert ctas == B * Hkv * (nkt + split)
    with pytest.raises(M.AttnError):
        M.debug_bwd_plan(1, 6, 4, 128, 128, 152)  # Hq not a multiple of Hkv
