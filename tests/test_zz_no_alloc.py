"""attn_fwd_noalloc: the forward pass for callers that may not allocate GPU memory
(for example a service that reserves all device memory up front, or a runtime
that owns the allocator). It works in a fixed device array the library reserves
on each GPU instead of a memory pool. It runs the same kernels as attn_fwd on the
same data, so its outputs must equal attn_fwd's bit for bit, on calls in a row
(each reusing the array the previous one left behind, with other sizes); and,
in a fresh process where attn_fwd never ran, repeated calls must not change the
device memory in use."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import mqa_attention_gb300 as M
import oracle as O
from mqa_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(seed_base, B, Hq, Hkv, S, D):
    shapes = {"q": (B, Hq, S, D), "k": (B, Hkv, S, D), "v": (B, Hkv, S, D)}
    bits = {n: I.normal_bf16_bits(seed_base + i, s) for i, (n, s) in enumerate(shapes.items())}
    dev = {n: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
           for n, b in bits.items()}
    return dev, {n: torch.from_numpy(I.bf16_bits_to_f64(b)) for n, b in bits.items()}


CALLS = [
    # (B, Hq, Hkv, S, D, theta, causal): in this order, each reusing the array
    (1, 4, 1, 128, 64, 10000.0, 1),
    (1, 8, 2, 512, 128, 500000.0, 1),
    (2, 8, 2, 256, 64, 10000.0, 1),
    (1, 4, 2, 384, 128, 500000.0, 0),
]


def test_noalloc_equals_attn_fwd_on_calls_in_a_row(built_lib):
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream
    for i, (B, Hq, Hkv, S, D, theta, causal) in enumerate(CALLS):
        x, _ = _inputs(7000 + 10 * i, B, Hq, Hkv, S, D)
        scale = 1.0 / D ** 0.5
        ref_out = torch.empty_like(x["q"])
        ref_lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
        out = torch.full_like(x["q"], float("nan"))
        lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
        assert built_lib.attn_fwd(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                                  ref_out.data_ptr(), ref_lse.data_ptr(), B, Hq, Hkv, S, D, theta,
                                  scale, causal, stream) == 0
        assert built_lib.attn_fwd_noalloc(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                                          out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, S, D, theta,
                                          scale, causal, stream) == 0
        torch.cuda.synchronize()
        assert M.sync_status() == 0
        assert torch.equal(out, ref_out), (i, "out")
        assert torch.equal(lse, ref_lse), (i, "lse")


def test_noalloc_matches_the_oracle(built_lib):
    """One small multi-query shape against the fp64 oracle at the stated bounds."""
    torch.cuda.set_device(0)
    B, Hq, Hkv, S, D, theta = 1, 8, 2, 384, 64, 10000.0
    x, f = _inputs(7100, B, Hq, Hkv, S, D)
    scale = 1.0 / D ** 0.5
    out = torch.empty_like(x["q"])
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    M.attn_fwd_noalloc(x["q"], x["k"], x["v"], out, lse, B, Hq, Hkv, S, D, theta, scale, True)
    torch.cuda.synchronize()
    assert M.sync_status() == 0
    o, l = O.attention_forward(f["q"], f["k"], f["v"], scale, theta, True, round_rotated=True)
    eo = (out.double().cpu() - o).abs()
    assert eo.max().item() <= 2e-2 and eo.mean().item() <= 2e-3
    assert (lse.double().cpu() - l).abs().max().item() <= 1e-3


_FRESH = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
import mqa_attention_gb300 as M
from mqa_attention_gb300 import inputs as I

torch.cuda.set_device(0)
torch.cuda.init()
def make(seed, B, Hq, Hkv, S, D):
    t = lambda i, s: torch.from_numpy(I.normal_bf16_bits(seed + i, s).view(np.int16)).view(
        torch.bfloat16).cuda()
    q, k, v = t(0, (B, Hq, S, D)), t(1, (B, Hkv, S, D)), t(2, (B, Hkv, S, D))
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    return q, k, v, out, lse
shapes = [(1, 4, 1, 128, 64), (1, 8, 2, 512, 128), (2, 8, 2, 256, 64)]
bufs = [make(7200 + 10 * i, *s) for i, s in enumerate(shapes)]
torch.cuda.synchronize()
def call(i):
    B, Hq, Hkv, S, D = shapes[i]
    q, k, v, out, lse = bufs[i]
    M.attn_fwd_noalloc(q, k, v, out, lse, B, Hq, Hkv, S, D, 10000.0, D ** -0.5, True)
call(0)  # the first call loads the module and finds the fixed array
torch.cuda.synchronize()
free0, _ = torch.cuda.mem_get_info()
for r in range(3):
    for i in range(len(shapes)):
        call(i)
torch.cuda.synchronize()
free1, _ = torch.cuda.mem_get_info()
assert M.sync_status() == 0
print("FREE", free0, free1)
"""


def test_noalloc_allocates_nothing_in_a_fresh_process(built_lib):
    """In a process where attn_fwd never ran (no library pool, no cached RoPE table),
    nine more calls of three sizes leave the device's free memory unchanged."""
    res = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + _FRESH],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-3000:]
    line = [l for l in res.stdout.splitlines() if l.startswith("FREE")][-1]
    free0, free1 = (int(x) for x in line.split()[1:])
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"


def test_noalloc_rejects_problems_beyond_its_array(built_lib):
    """Sizes whose RoPE table and rotated q and k do not fit in the fixed array are
    refused before any GPU work (the pointers are never touched)."""
    fake = 0x10000
    # B=1, Hq=32, Hkv=8, S=32768, D=128 needs about 335 MB of rotated q and k.
    code = built_lib.attn_fwd_noalloc(fake, fake, fake, fake, fake, 1, 32, 8, 32768, 128,
                                      500000.0, 0.088, 1, None)
    assert code == M.ATTN_ERR_UNSUPPORTED
