"""Decode shapes (attn_decode) and the rotation entry point (attn_rope) against
the fp64 oracle. Decode is the forward of a block of Sq query rows at positions
q_pos0.. against the whole key/value cache, so the oracle is its block attention
(attention_forward_partial with the cache at position 0); bounds as for the full
forward: out max-abs 2e-2, mean-abs 2e-3, lse 1e-3."""
import numpy as np
import pytest
import torch

import mqa_attention_gb300 as M
import oracle as O
from mqa_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return built_lib


def tensors(seed, shapes):
    host = {n: I.normal_bf16_bits(seed * 10 + i, s) for i, (n, s) in enumerate(shapes.items())}
    dev = {n: torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).cuda()
           for n, h in host.items()}
    return dev, {n: torch.from_numpy(I.bf16_bits_to_f64(h)) for n, h in host.items()}


@pytest.mark.parametrize("rope", ["half", "interleaved"])
def test_rope_rows(rope):
    """attn_rope rounds the fp32 rotation to bf16; the oracle rotates in fp64 and
    rounds, so the two agree within one bf16 ulp."""
    dev, f = tensors(400, {"x": (2, 3, 200, 128)})
    y = M.rope(dev["x"], 500000.0, pos0=37, rope=rope)
    torch.cuda.synchronize()
    ang = O.rope_angles(200, 128, 500000.0, 37)
    want = O.round_to_bf16(O.rope_half_split(f["x"], ang) if rope == "half"
                           else O.rope_interleaved(f["x"], ang))
    got = y.double().cpu()
    assert ((got - want).abs() <= want.abs() * 2.0 ** -7 + 1e-30).all()


DECODE = [
    # (B, Hq, Hkv, Sq, Skv, D, q_pos0, rope)
    (2, 32, 8, 1, 4096, 128, 4095, "half"),    # Llama-3-8B decode
    (4, 8, 1, 4, 2048, 64, 2044, "half"),      # PaLM MQA, four new tokens
    (1, 8, 1, 16, 1000, 128, 984, "half"),     # a full 128-row tile, ragged cache
    (1, 4, 4, 2, 300, 64, 298, "half"),        # MHA
    (1, 8, 2, 3, 777, 128, 500, "interleaved"),  # queries mid-cache: later keys masked
    (1, 2, 1, 1, 1, 64, 0, "half"),            # a single cached key
    (1, 8, 1, 8, 256, 64, 124, "half"),        # rows 124..127 see no key of the second chunk
    (1, 8, 1, 1, 65536, 64, 65535, "half"),    # one cache over 128 chunks: a long merge
    (1, 32, 8, 4, 32768, 128, 32764, "half"),  # the S = 32768 decode line, four new tokens
    (8, 8, 1, 16, 2048, 64, 2032, "half"),     # PaLM MQA, 16 new tokens: 128 rows per tile
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,qp,rope", DECODE)
def test_decode(B, Hq, Hkv, Sq, Skv, D, qp, rope):
    theta = 10000.0 if D == 64 else 500000.0
    scale = D ** -0.5
    dev, f = tensors(410 + Sq + D + Skv % 89,
                     {"q": (B, Hq, Sq, D), "k": (B, Hkv, Skv, D), "v": (B, Hkv, Skv, D)})
    k_rot = M.rope(dev["k"], theta, rope=rope)
    out, lse = M.decode(dev["q"], k_rot, dev["v"], theta, q_pos0=qp, scale=scale, rope=rope)
    torch.cuda.synchronize()
    assert M.sync_status() == 0
    wo, wl = O.attention_forward_partial(f["q"], f["k"], f["v"], scale, theta, qp, 0, True,
                                         rope=rope, round_rotated=True)
    e = (out.double().cpu() - wo).abs()
    assert e.max().item() <= 2e-2 and e.mean().item() <= 2e-3, (e.max().item(), e.mean().item())
    assert (lse.double().cpu() - wl).abs().max().item() <= 1e-3
