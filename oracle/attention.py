"""fp64 CPU oracle for causal RoPE attention with grouped / multi-query K/V.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module;
only the tests, the package smoke check and the benchmark's CPU-baseline leg
call it. It shares no code with the CUDA library: it is the plain
definition, written out densely with PyTorch CPU tensors in float64 (a matmul
is the only library primitive used as a step), so that each line can be
checked by eye against the pages it cites.

Sources (web pages, cited by title and section):
  [Picotron]  "Picotron模型实现解析Llama架构与Flash Attention集成",
              §1 嵌入层与位置编码 (apply_rotary_pos_emb / rotate_half),
              §2 注意力机制实现 (flash_attn_func(q, k, v, causal)).
  [llama3]    "深度学习系统设计llama3-from-scratch：并行计算架构",
              §键值（Key-Value）共享机制 (32 query heads over 8 KV heads),
              §RoPE位置编码的并行实现 (frequencies, complex-pair rotation),
              §注意力得分矩阵计算 (q·kᵀ / sqrt(head_dim)),
              §因果掩码的并行应用 (triu(-inf, diagonal=1)),
              §Softmax的并行计算.
  [PaLM]      "ColossalAI 中的 PaLM 教学实现不到 200 行核心代码与 Booster
              分布式训练实战", §2.3 RotaryEmbedding (1/10000^(2i/dim),
              cat(freqs, freqs), rotation of both q and k), §2.5 Attention
              (multi-query: one shared K/V head; upper-triangle mask; row-max
              subtraction before softmax; P·V).

Readings where the pages leave a step open (each is also listed with the
design notes of the library):
  * RoPE is the half-split form (rotate_half = cat(-x2, x1)); the
    interleaved complex-pair form of [llama3] is kept here as a second
    function because it is the same rotation up to a fixed permutation of
    the head dimensions, which one of the pins checks.
  * Query head h reads K/V head h // (Hq // Hkv) (contiguous groups).
  * Positions are 0..S-1 (an offset exists only for the shift pin).
  * LSE uses the natural logarithm; masked scores are excluded (-inf).
  * The backward pass is textbook softmax calculus (no page writes it); lse
    is not differentiated. Gradients are returned in float64.
  * ``round_rotated=True`` rounds RoPE(q) and RoPE(k) to bf16 (round to
    nearest even) before the scores, the precision in which a bf16 training
    stack feeds them to the score product; the gradient passes straight
    through that rounding.

Arrays may be given as numpy arrays or torch tensors; results are float64
torch tensors on the CPU.
"""
from __future__ import annotations

import torch

__all__ = [
    "rope_inv_freq",
    "rope_angles",
    "rope_half_split",
    "rope_interleaved",
    "round_to_bf16",
    "attention_forward",
    "attention_backward",
    "forward_rows",
    "backward_dq_rows",
    "attention_forward_partial",
    "attention_backward_partial",
    "merge_partials",
    "backward_dkdv_keys",
]

F64 = torch.float64


def _t(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=F64, device="cpu")


# --------------------------------------------------------------------- RoPE
def rope_inv_freq(D: int, theta: float) -> torch.Tensor:
    """inv_freq_i = theta^(-2i/D), i = 0..D/2-1 ([PaLM] §2.3; [llama3] §RoPE)."""
    i = torch.arange(D // 2, dtype=F64)
    return torch.pow(torch.tensor(float(theta), dtype=F64), -(2.0 * i) / D)


def rope_angles(S: int, D: int, theta: float, offset: int = 0) -> torch.Tensor:
    """Angle p * inv_freq_i for positions p = offset..offset+S-1: shape [S, D/2]
    ([PaLM] §2.3: outer product of positions and inverse frequencies)."""
    pos = torch.arange(S, dtype=F64) + float(offset)
    return torch.outer(pos, rope_inv_freq(D, theta))


def rope_half_split(x, ang, inverse: bool = False) -> torch.Tensor:
    """x * cos + rotate_half(x) * sin with rotate_half(x) = cat(-x2, x1) and
    cos/sin = cat(freqs, freqs) over the last axis ([Picotron] §1;
    [PaLM] §2.3). ``inverse`` applies the transpose (rotation by -angle).

    x: [..., S, D]; ang: [S, D/2]."""
    x, ang = _t(x), _t(ang)
    h = x.shape[-1] // 2
    c = torch.cos(ang)
    s = torch.sin(ang)
    if inverse:
        s = -s
    x1 = x[..., :h]
    x2 = x[..., h:]
    return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)


def rope_interleaved(x, ang, inverse: bool = False) -> torch.Tensor:
    """Pairs (2i, 2i+1) read as the complex number x_2i + j x_2i+1 and
    multiplied by polar(1, angle_i) ([llama3] §RoPE: view_as_complex,
    freqs_cis = polar(ones, freqs))."""
    x, ang = _t(x), _t(ang)
    z = torch.complex(x[..., 0::2], x[..., 1::2])
    rot = torch.polar(torch.ones_like(ang), -ang if inverse else ang)
    y = z * rot
    out = torch.empty_like(x)
    out[..., 0::2] = y.real
    out[..., 1::2] = y.imag
    return out


def round_to_bf16(x) -> torch.Tensor:
    """Round float64 values to the nearest bf16 value (ties to even), returned as
    float64. bf16 keeps 8 significant bits."""
    x = _t(x)
    m, e = torch.frexp(x)  # x = m * 2^e, 0.5 <= |m| < 1
    return torch.ldexp(torch.round(m * 256.0), (e - 8).to(F64))


def _rotate(x, ang, rope, inverse=False):
    if rope == "half":
        return rope_half_split(x, ang, inverse)
    if rope == "interleaved":
        return rope_interleaved(x, ang, inverse)
    raise ValueError(rope)


def _scores(qr_rows, kr, scale, rows, causal):
    """s_ij = scale * q~_i . k~_j ([llama3] §注意力得分矩阵计算), with keys j > i
    excluded when causal ([llama3] §因果掩码: triu(-inf, diagonal=1);
    [PaLM] §2.5 upper-triangle mask)."""
    s = scale * (qr_rows @ kr.T)
    if causal:
        j = torch.arange(kr.shape[0])
        i = torch.as_tensor(rows)
        s = s.masked_fill(j[None, :] > i[:, None], float("-inf"))
    return s


def _softmax_rows(s):
    """Row max subtracted before exponentiation ([PaLM] §2.5); returns
    (P, lse) with lse = m + ln sum exp(s - m)."""
    m = s.max(dim=1).values
    e = torch.exp(s - m[:, None])
    lse = m + torch.log(e.sum(dim=1))
    return torch.exp(s - lse[:, None]), lse


def _check_shapes(q, k, v):
    B, Hq, S, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if (Bk, Sk, Dk) != (B, S, D) or tuple(v.shape) != tuple(k.shape) or Hq % Hkv:
        raise ValueError("shape mismatch")
    return B, Hq, Hkv, S, D, Hq // Hkv


def _maybe_round(x, round_rotated):
    return round_to_bf16(x) if round_rotated else x


# --------------------------------------------------------------- full passes
def attention_forward(q, k, v, scale, theta, causal=True, rope="half", pos_offset=0,
                      round_rotated=False):
    """out = softmax(RoPE(q) RoPE(k)ᵀ scale + mask) v, per query head, with
    query head h using K/V head h // G ([llama3] §键值共享机制; [PaLM] §2.5).

    q: [B, Hq, S, D]; k, v: [B, Hkv, S, D]. Returns out [B,Hq,S,D] and
    lse [B,Hq,S]."""
    q, k, v = _t(q), _t(k), _t(v)
    B, Hq, Hkv, S, D, G = _check_shapes(q, k, v)
    ang = rope_angles(S, D, theta, pos_offset)
    qr = _maybe_round(_rotate(q, ang, rope), round_rotated)
    kr = _maybe_round(_rotate(k, ang, rope), round_rotated)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=F64)
    rows = torch.arange(S)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            p, lse[b, h] = _softmax_rows(_scores(qr[b, h], kr[b, g], scale, rows, causal))
            out[b, h] = p @ v[b, g]
    return out, lse


def attention_backward(q, k, v, dout, scale, theta, causal=True, rope="half", pos_offset=0,
                       round_rotated=False, return_delta=False):
    """Gradients of L = sum(dout * out) with respect to q, k, v (lse treated as
    not differentiated). With P the softmax of the scores:
        dP_ij = dO_i . v_j,   delta_i = sum_j P_ij dP_ij,
        dS_ij = P_ij (dP_ij - delta_i),
        dq~_i = scale sum_j dS_ij k~_j,   dk~_j = scale sum_{h in group} sum_i dS_ij q~_i,
        dv_j  = sum_{h in group} sum_i P_ij dO_i,
        dq = R_iᵀ dq~, dk = R_jᵀ dk~ (transpose of the rotation).
    Returns (dq, dk, dv) [, delta]."""
    q, k, v, dout = _t(q), _t(k), _t(v), _t(dout)
    B, Hq, Hkv, S, D, G = _check_shapes(q, k, v)
    ang = rope_angles(S, D, theta, pos_offset)
    qr = _maybe_round(_rotate(q, ang, rope), round_rotated)
    kr = _maybe_round(_rotate(k, ang, rope), round_rotated)
    dqr = torch.empty_like(q)
    dkr = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    delta = torch.empty((B, Hq, S), dtype=F64)
    rows = torch.arange(S)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            p, _ = _softmax_rows(_scores(qr[b, h], kr[b, g], scale, rows, causal))
            dp = dout[b, h] @ v[b, g].T
            delta[b, h] = (p * dp).sum(dim=1)
            ds = p * (dp - delta[b, h][:, None])
            dqr[b, h] = scale * (ds @ kr[b, g])
            dkr[b, g] += scale * (ds.T @ qr[b, h])
            dv[b, g] += p.T @ dout[b, h]
    dq = _rotate(dqr, ang, rope, inverse=True)
    dk = _rotate(dkr, ang, rope, inverse=True)
    if return_delta:
        return dq, dk, dv, delta
    return dq, dk, dv


# ------------------------------------------------- sampled rows (large S)
def forward_rows(q, k, v, rows, scale, theta, causal=True, round_rotated=False):
    """out and lse of the given query rows only (every head); each row needs
    only its own scores. Returns out [B,Hq,R,D], lse [B,Hq,R]."""
    q, k, v = _t(q), _t(k), _t(v)
    B, Hq, Hkv, S, D, G = _check_shapes(q, k, v)
    rows = torch.as_tensor(rows)
    ang = rope_angles(S, D, theta)
    qr = _maybe_round(rope_half_split(q[:, :, rows, :], ang[rows]), round_rotated)
    kr = _maybe_round(rope_half_split(k, ang), round_rotated)
    out = torch.empty((B, Hq, rows.numel(), D), dtype=F64)
    lse = torch.empty((B, Hq, rows.numel()), dtype=F64)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            p, lse[b, h] = _softmax_rows(_scores(qr[b, h], kr[b, g], scale, rows, causal))
            out[b, h] = p @ v[b, g]
    return out, lse


def backward_dq_rows(q, k, v, dout, rows, scale, theta, causal=True, round_rotated=False):
    """dq of the given query rows only; row i needs only its own P and dP."""
    q, k, v, dout = _t(q), _t(k), _t(v), _t(dout)
    B, Hq, Hkv, S, D, G = _check_shapes(q, k, v)
    rows = torch.as_tensor(rows)
    ang = rope_angles(S, D, theta)
    qr = _maybe_round(rope_half_split(q[:, :, rows, :], ang[rows]), round_rotated)
    kr = _maybe_round(rope_half_split(k, ang), round_rotated)
    dqr = torch.empty((B, Hq, rows.numel(), D), dtype=F64)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            p, _ = _softmax_rows(_scores(qr[b, h], kr[b, g], scale, rows, causal))
            dp = dout[b, h][rows] @ v[b, g].T
            delta = (p * dp).sum(dim=1)
            ds = p * (dp - delta[:, None])
            dqr[b, h] = scale * (ds @ kr[b, g])
    return rope_half_split(dqr, ang[rows], inverse=True)


def backward_dkdv_keys(q, k, v, dout, keys, scale, theta, causal=True, round_rotated=False,
                       batches=None, kv_heads=None, row_block=1024):
    """dk and dv of the given key rows, for the given batches and KV heads.
    Every query row's lse and delta enter, so all rows of the group's query
    heads are processed, in blocks of ``row_block`` rows (a memory bound, not
    a reordering of the arithmetic: each block's rows are independent).
    Returns dk, dv of shape [len(batches), len(kv_heads), len(keys), D]."""
    q, k, v, dout = _t(q), _t(k), _t(v), _t(dout)
    B, Hq, Hkv, S, D, G = _check_shapes(q, k, v)
    keys = torch.as_tensor(keys)
    batches = list(range(B)) if batches is None else list(batches)
    kv_heads = list(range(Hkv)) if kv_heads is None else list(kv_heads)
    ang = rope_angles(S, D, theta)
    dkr = torch.zeros((len(batches), len(kv_heads), keys.numel(), D), dtype=F64)
    dv = torch.zeros((len(batches), len(kv_heads), keys.numel(), D), dtype=F64)
    for bi, b in enumerate(batches):
        for gi, g in enumerate(kv_heads):
            kr = _maybe_round(rope_half_split(k[b, g], ang), round_rotated)
            for h in range(g * G, (g + 1) * G):
                for r0 in range(0, S, row_block):
                    r1 = min(S, r0 + row_block)
                    rows = torch.arange(r0, r1)
                    # With the causal mask, keys after the block's last row are
                    # excluded for every row of the block: only keys < r1 enter.
                    ncol = r1 if causal else S
                    qr = _maybe_round(rope_half_split(q[b, h, rows], ang[rows]), round_rotated)
                    p, _ = _softmax_rows(_scores(qr, kr[:ncol], scale, rows, causal))
                    dp = dout[b, h, rows] @ v[b, g, :ncol].T
                    delta = (p * dp).sum(dim=1)
                    ds = p * (dp - delta[:, None])
                    sel = keys < ncol
                    ks = keys[sel]
                    dkr[bi, gi, sel] += scale * (ds[:, ks].T @ qr)
                    dv[bi, gi, sel] += p[:, ks].T @ dout[b, h, rows]
    dk = rope_half_split(dkr, ang[keys], inverse=True)
    return dk, dv


# ------------------------------------- a query block against one key/value block
def attention_forward_partial(q, k, v, scale, theta, q_pos0, kv_pos0, causal=True, rope="half",
                              round_rotated=False):
    """Attention of a query block over one key/value block, the piece a
    context-parallel / ring schedule computes per block ([Picotron] §上下文并行).
    Query row i sits at position q_pos0 + i, key row j at kv_pos0 + j; RoPE
    rotates each row by its own position and the causal mask excludes keys
    after the query's position. Over the visible keys of row i:
        lse_i = ln sum_j exp(s_ij),   out_i = sum_j exp(s_ij - lse_i) v_j;
    a row with no visible key has lse_i = -inf and out_i = 0.

    q: [B, Hq, Sq, D]; k, v: [B, Hkv, Skv, D]."""
    q, k, v = _t(q), _t(k), _t(v)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    qr = _maybe_round(_rotate(q, rope_angles(Sq, D, theta, q_pos0), rope), round_rotated)
    kr = _maybe_round(_rotate(k, rope_angles(Skv, D, theta, kv_pos0), rope), round_rotated)
    qpos = q_pos0 + torch.arange(Sq)
    kpos = kv_pos0 + torch.arange(Skv)
    out = torch.zeros((B, Hq, Sq, D), dtype=F64)
    lse = torch.full((B, Hq, Sq), float("-inf"), dtype=F64)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            s = scale * (qr[b, h] @ kr[b, g].T)
            if causal:
                s = s.masked_fill(kpos[None, :] > qpos[:, None], float("-inf"))
            vis = torch.isfinite(s).any(dim=1)
            if vis.any():
                p, lse[b, h, vis] = _softmax_rows(s[vis])
                out[b, h, vis] = p @ v[b, g]
    return out, lse


def attention_backward_partial(q, k, v, dout, out, lse, scale, theta, q_pos0, kv_pos0,
                               causal=True, rope="half", round_rotated=False):
    """Contributions of one key/value block to the gradients of the whole
    attention of a query block, given that attention's out and lse (over all
    key blocks): for this block's keys P_ij = exp(s_ij - lse_i), and with
    delta_i = dO_i . out_i the steps of attention_backward follow. Summed over
    the key blocks, dq is the full dq; a block's dk and dv, summed over the
    query blocks, are its rows of the full dk and dv.
    Returns (dq [B,Hq,Sq,D], dk, dv [B,Hkv,Skv,D])."""
    q, k, v, dout, out, lse = _t(q), _t(k), _t(v), _t(dout), _t(out), _t(lse)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    qang = rope_angles(Sq, D, theta, q_pos0)
    kang = rope_angles(Skv, D, theta, kv_pos0)
    qr = _maybe_round(_rotate(q, qang, rope), round_rotated)
    kr = _maybe_round(_rotate(k, kang, rope), round_rotated)
    qpos = q_pos0 + torch.arange(Sq)
    kpos = kv_pos0 + torch.arange(Skv)
    dqr = torch.zeros_like(q)
    dkr = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            s = scale * (qr[b, h] @ kr[b, g].T)
            if causal:
                s = s.masked_fill(kpos[None, :] > qpos[:, None], float("-inf"))
            p = torch.exp(s - lse[b, h][:, None])
            p = torch.nan_to_num(p, nan=0.0)  # rows with lse = -inf see no key
            dp = dout[b, h] @ v[b, g].T
            delta = (dout[b, h] * out[b, h]).sum(dim=1)
            ds = p * (dp - delta[:, None])
            dqr[b, h] = scale * (ds @ kr[b, g])
            dkr[b, g] += scale * (ds.T @ qr[b, h])
            dv[b, g] += p.T @ dout[b, h]
    return _rotate(dqr, qang, rope, inverse=True), _rotate(dkr, kang, rope, inverse=True), dv


def merge_partials(out_a, lse_a, out_b, lse_b):
    """The attention over the union of two disjoint key sets from the two
    partial results: with lse = ln(exp(lse_a) + exp(lse_b)),
        out = exp(lse_a - lse) out_a + exp(lse_b - lse) out_b
    (rows that see no key in either: lse = -inf, out = 0)."""
    out_a, lse_a, out_b, lse_b = _t(out_a), _t(lse_a), _t(out_b), _t(lse_b)
    lse = torch.logaddexp(lse_a, lse_b)
    wa = torch.nan_to_num(torch.exp(lse_a - lse), nan=0.0)
    wb = torch.nan_to_num(torch.exp(lse_b - lse), nan=0.0)
    return wa[..., None] * out_a + wb[..., None] * out_b, lse
