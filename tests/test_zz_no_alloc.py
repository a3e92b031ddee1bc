"""attn_fwd_noalloc: the forward pass for callers that may not allocate GPU memory
(for example a service that reserves all device memory up front, or a runtime
that owns the allocator). It works in a fixed device array the library reserves
on each GPU instead of a memory pool. Its outputs must match attn_fwd's on the
same inputs, on two calls in a row (the second call reuses the array the first
one left behind, with different sizes)."""
import numpy as np
import pytest
import torch

import mqa_attention_gb300 as M
from mqa_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

OUT_MAX_ABS, LSE_MAX_ABS = 2e-2, 1e-3


def _inputs(seed_base, B, Hq, Hkv, S, D):
    shapes = {"q": (B, Hq, S, D), "k": (B, Hkv, S, D), "v": (B, Hkv, S, D)}
    return {n: torch.from_numpy(I.normal_bf16_bits(seed_base + i, s).view(np.int16))
            .view(torch.bfloat16).cuda() for i, (n, s) in enumerate(shapes.items())}


@pytest.mark.parametrize("calls", [[(1, 4, 1, 128, 64, 10000.0), (1, 8, 2, 512, 128, 500000.0)]])
def test_noalloc_matches_attn_fwd_on_two_calls(built_lib, calls):
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream
    for i, (B, Hq, Hkv, S, D, theta) in enumerate(calls):
        x = _inputs(7000 + 10 * i, B, Hq, Hkv, S, D)
        scale = 1.0 / D ** 0.5
        ref_out = torch.empty_like(x["q"])
        ref_lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
        out = torch.full_like(x["q"], float("nan"))
        lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
        assert built_lib.attn_fwd(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                                  ref_out.data_ptr(), ref_lse.data_ptr(), B, Hq, Hkv, S, D, theta,
                                  scale, 1, stream) == 0
        assert built_lib.attn_fwd_noalloc(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                                          out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, S, D, theta,
                                          scale, 1, stream) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        assert (out.float() - ref_out.float()).abs().max().item() <= OUT_MAX_ABS
        assert (lse - ref_lse).abs().max().item() <= LSE_MAX_ABS


def test_noalloc_rejects_problems_beyond_its_array(built_lib):
    """Sizes whose rotated q and k do not fit in the fixed array are refused
    before any GPU work (the pointers are never touched)."""
    fake = 0x10000
    # B=1, Hq=32, Hkv=8, S=32768, D=128 needs about 335 MB of rotated q and k.
    code = built_lib.attn_fwd_noalloc(fake, fake, fake, fake, fake, 1, 32, 8, 32768, 128,
                                      500000.0, 0.088, 1, None)
    assert code == M.ATTN_ERR_UNSUPPORTED
