"""Failure detection without a GPU fault: a debug switch makes the main
kernels wait on a barrier that nothing signals; the bounded wait expires after
about two seconds, the kernel unwinds (draining its copies and MMAs, freeing
its tensor memory) and the host reads ATTN_ERR_TIMEOUT. The context stays
usable: the next call succeeds and matches the oracle."""
import numpy as np
import pytest
import torch

import mqa_attention_gb300 as M
import oracle as O
from mqa_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _inputs(D):
    B, Hq, Hkv, S = 1, 1, 1, 128
    host = {n: I.normal_bf16_bits(I.seed_for(170 + D, n), (B, h, S, D))
            for n, h in (("q", Hq), ("k", Hkv), ("v", Hkv), ("dout", Hq))}
    dev = {n: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
           for n, x in host.items()}
    f = {n: torch.from_numpy(I.bf16_bits_to_f64(x)) for n, x in host.items()}
    return dev, f


@pytest.mark.parametrize("D", [64, 128])
def test_injected_wait_timeout_is_reported_and_recoverable(built_lib, D):
    dev, f = _inputs(D)
    theta = 10000.0
    assert M.sync_status() == M.ATTN_OK
    M.debug_inject_timeout(True)
    try:
        out, lse = M.forward(dev["q"], dev["k"], dev["v"], theta)
        assert M.sync_status() == M.ATTN_ERR_TIMEOUT
        M.backward(dev["q"], dev["k"], dev["v"], out, lse, dev["dout"], theta)
        assert M.sync_status() == M.ATTN_ERR_TIMEOUT
    finally:
        M.debug_inject_timeout(False)
    assert M.sync_status() == M.ATTN_OK
    out, lse = M.forward(dev["q"], dev["k"], dev["v"], theta)
    dq, dk, dv = M.backward(dev["q"], dev["k"], dev["v"], out, lse, dev["dout"], theta)
    assert M.sync_status() == M.ATTN_OK
    scale = 1.0 / D ** 0.5
    o_ref, l_ref = O.attention_forward(f["q"], f["k"], f["v"], scale, theta, round_rotated=True)
    g_ref = O.attention_backward(f["q"], f["k"], f["v"], f["dout"], scale, theta,
                                 round_rotated=True)
    assert (out.double().cpu() - o_ref).abs().max() < 2e-2
    assert (lse.double().cpu() - l_ref).abs().max() < 1e-3
    for got, want in zip((dq, dk, dv), g_ref):
        assert (got.double().cpu() - want).abs().max() < 2e-2
