"""The bounds-checking build (GB_BOUNDS_CHECK): every kernel checks each global index
and TMA coordinate before using it and records a failed check in the device status
word (attn_sync_status then returns ATTN_ERR_BOUNDS). It stands in for a memory
checker here: the small-shape and ragged parity lists, both RoPE roundings, the
exact delta pass, partial blocks with their merge, decode and the RoPE entry point
all run through it with a clean status, and a few results are checked against the
oracle."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SCRIPT = r"""
import sys
sys.path.insert(0, ROOT)
import numpy as np
import torch
import mqa_attention_gb300 as M
import oracle as O
from mqa_attention_gb300 import inputs as I

assert M.LIB_PATH.endswith("_debug.so"), M.LIB_PATH
torch.cuda.set_device(0)

def gen(seed, B, Hq, Hkv, S, D):
    sh = {"q": (B, Hq, S, D), "k": (B, Hkv, S, D), "v": (B, Hkv, S, D), "dout": (B, Hq, S, D)}
    bits = {n: I.normal_bf16_bits(seed + i, s) for i, (n, s) in enumerate(sh.items())}
    dev = {n: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda() for n, b in bits.items()}
    return dev, {n: torch.from_numpy(I.bf16_bits_to_f64(b)) for n, b in bits.items()}

def clean(what):
    torch.cuda.synchronize()
    st = M.sync_status()
    assert st == 0, f"{what}: status {st} ({M.status_string(st)})"

CASES = [
    (1, 4, 1, 128, 64, True), (1, 2, 1, 256, 128, True), (2, 4, 2, 384, 64, True),
    (1, 6, 2, 640, 128, True), (1, 8, 1, 256, 64, True), (1, 4, 4, 256, 128, True),
    (1, 32, 1, 128, 64, True), (2, 2, 1, 256, 64, False), (1, 4, 2, 384, 128, False),
    (2, 8, 2, 1024, 64, True), (1, 8, 8, 1536, 128, True),
    (1, 4, 1, 1, 64, True), (1, 2, 1, 100, 128, True), (2, 4, 2, 300, 64, True),
    (1, 4, 4, 200, 128, False), (2, 2, 1, 77, 64, False),
]
n = 0
for i, (B, Hq, Hkv, S, D, causal) in enumerate(CASES):
    theta = 10000.0 if D == 64 else 500000.0
    dev, f = gen(1000 * (i + 1), B, Hq, Hkv, S, D)
    for exact in (False, True):
        out, lse = M.forward(dev["q"], dev["k"], dev["v"], theta, None, causal, exact_rope=exact)
        g = M.backward(dev["q"], dev["k"], dev["v"], out, lse, dev["dout"], theta, None, causal,
                       exact_rope=exact, delta="exact" if exact else "auto")
        clean(f"case {i} exact={exact}")
        n += 1
    if i in (0, 3, 13):  # a few against the oracle (rotated operands rounded to bf16)
        scale = D ** -0.5
        o, l = O.attention_forward(f["q"], f["k"], f["v"], scale, theta, causal, round_rotated=True)
        want = O.attention_backward(f["q"], f["k"], f["v"], f["dout"], scale, theta, causal,
                                    round_rotated=True)
        assert (out.double().cpu() - o).abs().max().item() <= 2e-2
        assert (lse.double().cpu() - l).abs().max().item() <= 1e-3
        for got, ref in zip(g, want):
            assert (got.double().cpu() - ref).abs().max().item() <= 2e-2

# partial blocks (a 2 x 2 schedule) and their merge
dev, _ = gen(90000, 1, 4, 2, 512, 128)
cut = lambda t, j: t[:, :, 256 * j:256 * (j + 1)].contiguous()
for i in range(2):
    for j in range(i + 1):
        o, l = M.forward_partial(cut(dev["q"], i), cut(dev["k"], j), cut(dev["v"], j), 500000.0,
                                 256 * i, 256 * j)
        M.backward_partial(cut(dev["q"], i), cut(dev["k"], j), cut(dev["v"], j), o, l,
                           cut(dev["dout"], i), 500000.0, 256 * i, 256 * j)
        M.merge(o, l, o, l)
clean("partial")
# decode against a rotated cache, and the RoPE entry point on an odd length
dev, _ = gen(91000, 2, 8, 2, 333, 64)
k_rot = M.rope(dev["k"], 10000.0)
M.decode(dev["q"][:, :, -3:].contiguous(), k_rot, dev["v"], 10000.0, q_pos0=330)
M.rope(dev["q"], 10000.0, pos0=5, exact=True)
clean("decode / rope")
print("OK", n)
"""


def test_bounds_checked_build_runs_clean(built_lib):
    from mqa_attention_gb300 import build as B

    path = B.build(debug=True)
    env = dict(os.environ, MQA_ATTENTION_GB300_LIB=path)
    res = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + _SCRIPT], env=env,
                         capture_output=True, text=True, timeout=1200, cwd=ROOT)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-3000:]
    assert "OK" in res.stdout
