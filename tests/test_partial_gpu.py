"""Blocks of queries and keys (attn_fwd_partial, attn_bwd_partial, attn_merge)
against the fp64 oracle: the pieces a context-parallel (ring) schedule computes
("Picotron模型实现解析Llama架构与Flash Attention集成", §上下文并行).

Bounds as for the full passes: out, dq, dk, dv max-abs 2e-2 and mean-abs 2e-3,
lse 1e-3 (oracle with bf16-rounded RoPE(q), RoPE(k)); rows that see no key must
give exactly out = 0 and lse = -inf."""
import numpy as np
import pytest
import torch

import mqa_attention_gb300 as M
import oracle as O
from mqa_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 2e-2, 2e-3, 1e-3


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


def close(name, got, want, mx=MAX_ABS, mn=MEAN_ABS):
    got = got.double().cpu()
    assert got.shape == want.shape, name
    e = (got - want).abs()
    assert e.max().item() <= mx and e.mean().item() <= mn, \
        f"{name}: max {e.max().item():.3e} mean {e.mean().item():.3e}"


def check_lse(got, want):
    got = got.double().cpu()
    none = torch.isneginf(want)
    assert torch.equal(torch.isneginf(got), none), "rows without keys"
    if (~none).any():
        assert (got[~none] - want[~none]).abs().max().item() <= LSE_ABS


FWD_CASES = [
    # (B, Hq, Hkv, Sq, Skv, D, q_pos0, kv_pos0, causal)
    (1, 4, 2, 256, 384, 128, 384, 0, True),    # keys all before the queries: no mask
    (1, 4, 2, 256, 384, 64, 384, 0, True),     # the same at D = 64 (persistent forward)
    (1, 4, 1, 256, 256, 64, 256, 256, True),   # the diagonal block
    (1, 2, 2, 384, 256, 128, 0, 128, True),    # keys partly after: query tile 0 sees none
    (1, 2, 2, 384, 256, 64, 0, 128, True),     # the same at D = 64 (one query tile per CTA)
    (2, 8, 1, 128, 512, 64, 1024, 256, False),  # non-causal, offset positions
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,qp,kp,causal", FWD_CASES)
def test_forward_partial(B, Hq, Hkv, Sq, Skv, D, qp, kp, causal):
    theta = 10000.0 if D == 64 else 500000.0
    dev, f = tensors(300 + Sq // 128 + D + qp // 128,
                     {"q": (B, Hq, Sq, D), "k": (B, Hkv, Skv, D), "v": (B, Hkv, Skv, D)})
    scale = D ** -0.5
    out, lse = M.forward_partial(dev["q"], dev["k"], dev["v"], theta, qp, kp, scale, causal)
    torch.cuda.synchronize()
    assert M.sync_status() == 0
    wo, wl = O.attention_forward_partial(f["q"], f["k"], f["v"], scale, theta, qp, kp, causal,
                                         round_rotated=True)
    check_lse(lse, wl)
    close("out", out, wo)
    empty = torch.isneginf(wl)
    assert (out.double().cpu()[empty] == 0).all()


@pytest.mark.parametrize("D", [64, 128])
def test_backward_partial_with_empty_tiles(D):
    """A key block partly after the query block, given the oracle's out and lse."""
    B, Hq, Hkv, Sq, Skv, qp, kp = 1, 4, 2, 384, 256, 0, 128
    theta, scale = (10000.0 if D == 64 else 500000.0), D ** -0.5
    dev, f = tensors(321 + D, {"q": (B, Hq, Sq, D), "k": (B, Hkv, Skv, D), "v": (B, Hkv, Skv, D),
                           "dout": (B, Hq, Sq, D)})
    wo, wl = O.attention_forward_partial(f["q"], f["k"], f["v"], scale, theta, qp, kp, True,
                                         round_rotated=True)
    out16 = wo.to(torch.bfloat16).cuda()
    lse32 = wl.to(torch.float32).cuda()
    g = M.backward_partial(dev["q"], dev["k"], dev["v"], out16, lse32, dev["dout"], theta, qp, kp,
                           scale, True)
    torch.cuda.synchronize()
    assert M.sync_status() == 0
    want = O.attention_backward_partial(f["q"], f["k"], f["v"], f["dout"],
                                        out16.double().cpu(), lse32.double().cpu(), scale, theta,
                                        qp, kp, True, round_rotated=True)
    for name, a, b in zip(("dq", "dk", "dv"), g, want):
        close(name, a, b)


@pytest.mark.parametrize("D", [64, 128])
def test_ring_of_blocks_equals_full_attention(D):
    """Causal self-attention at S = 512 cut into 2 query x 2 key blocks: partial
    forwards merged in place, then partial backwards with the merged out / lse,
    summed over the other blocks, match the oracle's full attention."""
    B, Hq, Hkv, S, blk = 1, 4, 2, 512, 256
    theta, scale = (10000.0 if D == 64 else 500000.0), D ** -0.5
    dev, f = tensors(340 + D, {"q": (B, Hq, S, D), "k": (B, Hkv, S, D), "v": (B, Hkv, S, D),
                               "dout": (B, Hq, S, D)})
    out = torch.empty_like(dev["q"])
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    dq = torch.zeros((B, Hq, S, D), dtype=torch.float32, device="cuda")
    dk = torch.zeros((B, Hkv, S, D), dtype=torch.float32, device="cuda")
    dv = torch.zeros((B, Hkv, S, D), dtype=torch.float32, device="cuda")
    cuts = [(0, blk), (blk, S)]
    for q0, q1 in cuts:
        qb = dev["q"][:, :, q0:q1].contiguous()
        acc = None
        for k0, k1 in cuts:
            kb, vb = dev["k"][:, :, k0:k1].contiguous(), dev["v"][:, :, k0:k1].contiguous()
            po, pl = M.forward_partial(qb, kb, vb, theta, q0, k0, scale, True)
            if acc is None:
                acc = (po, pl)
            else:
                M.merge(acc[0], acc[1], po, pl, out=acc[0], lse=acc[1])  # in place
        out[:, :, q0:q1] = acc[0]
        lse[:, :, q0:q1] = acc[1]
    for q0, q1 in cuts:
        qb, dob = dev["q"][:, :, q0:q1].contiguous(), dev["dout"][:, :, q0:q1].contiguous()
        ob, lb = out[:, :, q0:q1].contiguous(), lse[:, :, q0:q1].contiguous()
        for k0, k1 in cuts:
            kb, vb = dev["k"][:, :, k0:k1].contiguous(), dev["v"][:, :, k0:k1].contiguous()
            g = M.backward_partial(qb, kb, vb, ob, lb, dob, theta, q0, k0, scale, True)
            dq[:, :, q0:q1] += g[0]
            dk[:, :, k0:k1] += g[1]
            dv[:, :, k0:k1] += g[2]
    torch.cuda.synchronize()
    assert M.sync_status() == 0
    wo, wl = O.attention_forward(f["q"], f["k"], f["v"], scale, theta, True, round_rotated=True)
    check_lse(lse, wl)
    close("out", out, wo)
    want = O.attention_backward(f["q"], f["k"], f["v"], f["dout"], scale, theta, True,
                                round_rotated=True)
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
        close(name, a, b)
