"""The boundary's stream contract: every call is enqueued on the caller's stream with no
host synchronisation, including the first call for a (D, rope_theta) that builds the
RoPE table; another stream that reads a table built on a busy stream waits for it on
the device; a captured call needs its table built beforehand, and its graph replays to
the same result."""
import numpy as np
import pytest
import torch

import mqa_attention_gb300 as M
import oracle as O
from mqa_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _inputs(seed, B, Hq, Hkv, S, D):
    sh = {"q": (B, Hq, S, D), "k": (B, Hkv, S, D), "v": (B, Hkv, S, D)}
    bits = {n: I.normal_bf16_bits(seed + i, s) for i, (n, s) in enumerate(sh.items())}
    dev = {n: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
           for n, b in bits.items()}
    return dev, {n: torch.from_numpy(I.bf16_bits_to_f64(b)) for n, b in bits.items()}


def _busy(stream, ms=200.0):
    """Enqueues about `ms` of bf16 matmuls on `stream` (sized from a timed sample)."""
    a = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(4):
            a @ a
        e1.record(stream)
    torch.cuda.synchronize()
    n = max(8, int(ms / (e0.elapsed_time(e1) / 4)))
    with torch.cuda.stream(stream):
        for _ in range(n):
            a @ a
    return a


def test_first_call_for_a_new_table_does_not_wait_for_the_stream(built_lib):
    torch.cuda.set_device(0)
    B, Hq, Hkv, S, D, theta = 1, 4, 2, 384, 128, 123457.0  # a theta no other test uses
    x, f = _inputs(8100, B, Hq, Hkv, S, D)
    out = torch.empty_like(x["q"])
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    keep = _busy(s1)
    M.attn_fwd(x["q"], x["k"], x["v"], out, lse, B, Hq, Hkv, S, D, theta, D ** -0.5, True,
               stream=s1)
    assert not s1.query(), "the call waited for the work queued before it"
    # a second stream reads the table s1 is still building: it waits on the device
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    M.attn_fwd(x["q"], x["k"], x["v"], out2, lse2, B, Hq, Hkv, S, D, theta, D ** -0.5, True,
               stream=s2)
    torch.cuda.synchronize()
    assert M.sync_status() == 0
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    o, l = O.attention_forward(f["q"], f["k"], f["v"], D ** -0.5, theta, True, round_rotated=True)
    eo = (out.double().cpu() - o).abs()
    assert eo.max().item() <= 2e-2 and eo.mean().item() <= 2e-3
    assert (lse.double().cpu() - l).abs().max().item() <= 1e-3
    del keep


def test_capture_needs_a_built_table_and_replays(built_lib):
    torch.cuda.set_device(0)
    B, Hq, Hkv, S, D = 1, 4, 1, 256, 64
    x, _ = _inputs(8200, B, Hq, Hkv, S, D)
    out = torch.empty_like(x["q"])
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    # no table yet for this theta: refused inside the capture, nothing enqueued
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            with pytest.raises(M.AttnError) as e:
                M.attn_fwd(x["q"], x["k"], x["v"], out, lse, B, Hq, Hkv, S, D, 77777.0,
                           D ** -0.5, True, stream=side)
    assert e.value.code == M.ATTN_ERR_UNSUPPORTED
    # warm up outside capture (builds the table, then sees it complete), then capture
    for _ in range(2):
        M.attn_fwd(x["q"], x["k"], x["v"], out, lse, B, Hq, Hkv, S, D, 77777.0, D ** -0.5, True)
        torch.cuda.synchronize()
    ref = out.clone(), lse.clone()
    out.zero_()
    lse.zero_()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g2, stream=side):
            M.attn_fwd(x["q"], x["k"], x["v"], out, lse, B, Hq, Hkv, S, D, 77777.0, D ** -0.5,
                       True, stream=side)
    g2.replay()
    torch.cuda.synchronize()
    assert M.sync_status() == 0
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])
