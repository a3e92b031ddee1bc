"""Pins of the fp64 oracle to facts that do not come from the oracle itself:
closed forms, exact invariants, special cases, page-printed expressions, brute
force on tiny inputs and finite differences. CPU only."""
import json
import math
import os

import pytest
import torch

import oracle as O

F64 = torch.float64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")


def rnd(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return scale * torch.randn(shape, generator=g, dtype=F64)


def qkvd(B, Hq, Hkv, S, D, seed=0, scale=1.0):
    return (rnd((B, Hq, S, D), seed, scale), rnd((B, Hkv, S, D), seed + 1, scale),
            rnd((B, Hkv, S, D), seed + 2), rnd((B, Hq, S, D), seed + 3))


@pytest.fixture(scope="module")
def facts():
    with open(GOLDEN) as f:
        return json.load(f)


# ----------------------------------------------------------------- page facts
def test_llama3_frequency_expression(facts):
    """The llama3-from-scratch page writes the frequencies as
    1/(rope_theta ** (arange(64)/64)) for head_dim 128; the PaLM page writes
    1/(10000 ** (arange(0, dim, 2)/dim)). Both must equal rope_inv_freq."""
    f = facts["llama3_rope_frequencies"]
    n, D = f["count"], f["head_dim"]
    for theta in (500000.0, 10000.0):
        page = 1.0 / (theta ** (torch.arange(n, dtype=F64) / n))
        assert torch.allclose(O.rope_inv_freq(D, theta), page, rtol=1e-15, atol=0)
    for dim in (64, 128, 2):
        page = 1.0 / (10000.0 ** (torch.arange(0, dim, 2, dtype=F64) / dim))
        assert torch.allclose(O.rope_inv_freq(dim, 10000.0), page, rtol=1e-15, atol=0)


def test_picotron_rotate_half_expression():
    """Picotron's apply_rotary_pos_emb: rotate_half = cat([-x2, x1]) and
    x*cos + rotate_half*sin with cos/sin built from cat((freqs, freqs))
    (PaLM §2.3)."""
    S, D = 7, 8
    x = rnd((2, S, D), 5)
    freqs = torch.outer(torch.arange(S, dtype=F64),
                        1.0 / (10000.0 ** (torch.arange(0, D, 2, dtype=F64) / D)))
    emb = torch.cat((freqs, freqs), dim=-1)
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    page = x * emb.cos() + torch.cat([-x2, x1], dim=-1) * emb.sin()
    got = O.rope_half_split(x, O.rope_angles(S, D, 10000.0))
    assert torch.allclose(got, page, rtol=0, atol=1e-14)


def test_causal_mask_matches_page(facts):
    """P is zero exactly where triu(full(-inf), diagonal=1) is -inf."""
    q, k, v, _ = qkvd(1, 1, 1, 6, 4, seed=3)
    S = 6
    page_mask = torch.triu(torch.full((S, S), float("-inf"), dtype=F64), diagonal=1)
    # recover P from out with v = identity columns (S x S one-hot values)
    eye = torch.eye(S, dtype=F64).reshape(1, 1, S, S)
    qq = torch.cat([q, torch.zeros(1, 1, S, S - 4, dtype=F64)], dim=-1)[..., :S]
    kk = torch.cat([k, torch.zeros(1, 1, S, S - 4, dtype=F64)], dim=-1)[..., :S]
    out, _ = O.attention_forward(qq, kk, eye, 0.5, 10000.0, causal=True)
    P = out[0, 0]
    assert torch.all(P[torch.isinf(page_mask)] == 0)
    assert torch.all(P[~torch.isinf(page_mask)] > 0)


def test_workload_shapes_from_pages(facts):
    c = facts["llama3_config"]
    v = facts["llama3_head_views"]
    assert c["dim"] // c["n_heads"] == v["wq_view"][1] == 128
    assert c["n_heads"] // c["n_kv_heads"] == v["query_heads_per_kv_head"] == 4
    assert v["wk_view"][0] == c["n_kv_heads"]
    p = facts["palm_defaults"]
    assert (p["heads"], p["dim_head"]) == (8, 64)


# ----------------------------------------------------------------- closed forms
def test_gqa_equals_mha_with_repeated_kv():
    """Query head h reads K/V head h // G: repeating each K/V head G times gives an
    MHA problem with identical out/lse/dq, and dk/dv are its group sums."""
    B, Hq, Hkv, S, D = 2, 6, 2, 9, 8
    G = Hq // Hkv
    q, k, v, do = qkvd(B, Hq, Hkv, S, D, seed=11)
    km, vm = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    for causal in (True, False):
        o1, l1 = O.attention_forward(q, k, v, 0.35, 10000.0, causal)
        o2, l2 = O.attention_forward(q, km, vm, 0.35, 10000.0, causal)
        assert torch.allclose(o1, o2, atol=1e-13) and torch.allclose(l1, l2, atol=1e-13)
        g1 = O.attention_backward(q, k, v, do, 0.35, 10000.0, causal)
        g2 = O.attention_backward(q, km, vm, do, 0.35, 10000.0, causal)
        assert torch.allclose(g1[0], g2[0], atol=1e-12)
        assert torch.allclose(g1[1], g2[1].reshape(B, Hkv, G, S, D).sum(2), atol=1e-12)
        assert torch.allclose(g1[2], g2[2].reshape(B, Hkv, G, S, D).sum(2), atol=1e-12)


def test_zero_query_prefix_mean():
    """q = 0 makes every score 0: out_i = mean(v_0..v_i), lse_i = ln(i+1),
    dk = 0 and dv_j = sum_{h in group} sum_{i>=j} dO_i / (i+1)."""
    B, Hq, Hkv, S, D = 1, 4, 2, 11, 8
    G = Hq // Hkv
    _, k, v, do = qkvd(B, Hq, Hkv, S, D, seed=21)
    q = torch.zeros(B, Hq, S, D, dtype=F64)
    out, lse = O.attention_forward(q, k, v, 0.3, 500000.0)
    dq, dk, dv = O.attention_backward(q, k, v, do, 0.3, 500000.0)
    for h in range(Hq):
        for i in range(S):
            mean = sum(v[0, h // G, j] for j in range(i + 1)) / (i + 1)
            assert torch.allclose(out[0, h, i], mean, atol=1e-14)
            assert abs(lse[0, h, i].item() - math.log(i + 1)) < 1e-14
    assert torch.all(dk.abs() < 1e-15)
    for g in range(Hkv):
        for j in range(S):
            want = sum(do[0, h, i] / (i + 1) for h in range(g * G, (g + 1) * G)
                       for i in range(j, S))
            assert torch.allclose(dv[0, g, j], want, atol=1e-13)


def test_first_row():
    """Row 0 sees only key 0 (R_0 = I): out_0 = v_0, lse_0 = scale q_0.k_0, dq_0 = 0."""
    B, Hq, Hkv, S, D = 2, 4, 1, 6, 8
    q, k, v, do = qkvd(B, Hq, Hkv, S, D, seed=31)
    out, lse = O.attention_forward(q, k, v, 0.4, 10000.0)
    dq, _, _ = O.attention_backward(q, k, v, do, 0.4, 10000.0)
    for b in range(B):
        for h in range(Hq):
            assert torch.allclose(out[b, h, 0], v[b, 0, 0], atol=1e-15)
            assert abs(lse[b, h, 0].item() - 0.4 * float(q[b, h, 0] @ k[b, 0, 0])) < 1e-13
            assert torch.all(dq[b, h, 0].abs() < 1e-15)


def test_d2_closed_form():
    """D = 2 has one frequency (theta^0 = 1), so s_ij = scale |q_i||k_j|
    cos(phi_q_i + i - phi_k_j - j); lse and out follow in closed form."""
    S, scale = 7, 0.9
    q, k, v, _ = qkvd(1, 1, 1, S, 2, seed=41)
    out, lse = O.attention_forward(q, k, v, scale, 12345.0)
    for i in range(S):
        rq, fq = math.hypot(q[0, 0, i, 0], q[0, 0, i, 1]), math.atan2(q[0, 0, i, 1], q[0, 0, i, 0])
        s = []
        for j in range(i + 1):
            rk = math.hypot(k[0, 0, j, 0], k[0, 0, j, 1])
            fk = math.atan2(k[0, 0, j, 1], k[0, 0, j, 0])
            s.append(scale * rq * rk * math.cos(fq + i - fk - j))
        m = max(s)
        want = m + math.log(sum(math.exp(x - m) for x in s))
        assert abs(lse[0, 0, i].item() - want) < 1e-12
        w = [math.exp(x - want) for x in s]
        o = [sum(w[j] * float(v[0, 0, j, d]) for j in range(i + 1)) for d in range(2)]
        assert abs(out[0, 0, i, 0].item() - o[0]) < 1e-12
        assert abs(out[0, 0, i, 1].item() - o[1]) < 1e-12


@pytest.mark.parametrize("c", [1, 1000])
def test_relative_position_shift(c):
    """RoPE encodes relative position in the dot product (PaLM §2.3): shifting
    every position by c leaves out, lse and the gradients dq, dk, dv unchanged
    (dq_i = scale sum_j dS_ij R_{j-i} k_j depends on j - i only)."""
    q, k, v, do = qkvd(1, 2, 1, 8, 8, seed=51)
    o0, l0 = O.attention_forward(q, k, v, 0.5, 10000.0)
    o1, l1 = O.attention_forward(q, k, v, 0.5, 10000.0, pos_offset=c)
    assert torch.allclose(o0, o1, atol=1e-10) and torch.allclose(l0, l1, atol=1e-10)
    g0 = O.attention_backward(q, k, v, do, 0.5, 10000.0)
    g1 = O.attention_backward(q, k, v, do, 0.5, 10000.0, pos_offset=c)
    for a, b in zip(g0, g1):
        assert torch.allclose(a, b, atol=1e-10)


def test_shift_detects_wrong_inverse_sign():
    """Planted mistake: undoing the rotation with +angle instead of -angle breaks
    the shift invariance of dq, so the pin above would catch it."""
    q, k, v, do = qkvd(1, 1, 1, 6, 4, seed=52)
    outs = []
    for c in (0, 7):
        ang = O.rope_angles(6, 4, 10000.0, c)
        dq = O.attention_backward(q, k, v, do, 0.5, 10000.0, pos_offset=c)[0]
        dq_t = O.rope_half_split(dq, ang)  # back to the rotated frame
        outs.append(O.rope_half_split(dq_t, ang))  # wrong "inverse"
    assert not torch.allclose(outs[0], outs[1], atol=1e-6)


def test_interleaved_equals_permuted_half_split():
    """llama3-from-scratch rotates complex pairs (2i, 2i+1); Picotron/PaLM rotate
    halves (i, i + D/2). With the permutation pairing them the results agree."""
    B, Hq, Hkv, S, D = 1, 2, 1, 9, 8
    q, k, v, do = qkvd(B, Hq, Hkv, S, D, seed=61)
    perm = torch.cat([torch.arange(0, D, 2), torch.arange(1, D, 2)])
    o_i, l_i = O.attention_forward(q, k, v, 0.5, 10000.0, rope="interleaved")
    o_h, l_h = O.attention_forward(q[..., perm], k[..., perm], v, 0.5, 10000.0, rope="half")
    assert torch.allclose(o_i, o_h, atol=1e-13) and torch.allclose(l_i, l_h, atol=1e-13)
    gi = O.attention_backward(q, k, v, do, 0.5, 10000.0, rope="interleaved")
    gh = O.attention_backward(q[..., perm], k[..., perm], v, do, 0.5, 10000.0, rope="half")
    assert torch.allclose(gi[0][..., perm], gh[0], atol=1e-12)
    assert torch.allclose(gi[1][..., perm], gh[1], atol=1e-12)
    assert torch.allclose(gi[2], gh[2], atol=1e-12)


def test_exact_invariants():
    B, Hq, Hkv, S, D = 2, 4, 2, 12, 8
    G = Hq // Hkv
    q, k, v, do = qkvd(B, Hq, Hkv, S, D, seed=71)
    out, lse = O.attention_forward(q, k, v, 0.3, 10000.0)
    dq, dk, dv, delta = O.attention_backward(q, k, v, do, 0.3, 10000.0, return_delta=True)
    # sum_j dv_j = sum over the group's heads and rows of dO (rows of P sum to 1)
    assert torch.allclose(dv.sum(2), do.reshape(B, Hkv, G, S, D).sum((2, 3)), atol=1e-12)
    # sum_j R_j dk_j = 0 because every row of dS sums to 0
    dkr = O.rope_half_split(dk, O.rope_angles(S, D, 10000.0))
    assert torch.all(dkr.sum(2).abs() < 1e-12)
    # delta two ways: sum_j P dP = dO . out
    assert torch.allclose(delta, (do * out).sum(-1), atol=1e-12)
    # softmax rows sum to one: v = 1 gives out = 1
    ones = torch.ones_like(v)
    o1, _ = O.attention_forward(q, k, ones, 0.3, 10000.0)
    assert torch.allclose(o1, torch.ones_like(o1), atol=1e-14)


def _brute_forward(q, k, v, scale, theta, causal):
    """Scalar loops with the math module only (tiny sizes)."""
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    half = D // 2

    def rot(x, p):
        y = [0.0] * D
        for i in range(half):
            a = p * theta ** (-2.0 * i / D)
            y[i] = x[i] * math.cos(a) - x[i + half] * math.sin(a)
            y[i + half] = x[i + half] * math.cos(a) + x[i] * math.sin(a)
        return y

    out = [[[[0.0] * D for _ in range(S)] for _ in range(Hq)] for _ in range(B)]
    lse = [[[0.0] * S for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i in range(S):
                qi = rot([float(x) for x in q[b, h, i]], i)
                js = range(i + 1) if causal else range(S)
                s = [scale * sum(a * c for a, c in zip(qi, rot([float(x) for x in k[b, g, j]], j)))
                     for j in js]
                m = max(s)
                z = sum(math.exp(x - m) for x in s)
                lse[b][h][i] = m + math.log(z)
                for d in range(D):
                    out[b][h][i][d] = sum(math.exp(x - m) / z * float(v[b, g, j, d])
                                          for x, j in zip(s, js))
    return torch.tensor(out, dtype=F64), torch.tensor(lse, dtype=F64)


@pytest.mark.parametrize("causal", [True, False])
def test_brute_force_tiny(causal):
    q, k, v, _ = qkvd(2, 4, 2, 5, 6, seed=81)
    o, l = O.attention_forward(q, k, v, 0.45, 777.0, causal)
    ob, lb = _brute_forward(q, k, v, 0.45, 777.0, causal)
    assert torch.allclose(o, ob, atol=1e-13) and torch.allclose(l, lb, atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_finite_differences(causal):
    """Central differences of L = sum(dO * out), step 1e-6, on every element of
    q, k, v (B=1, Hq=2, Hkv=1, S=5, D=4)."""
    q, k, v, do = qkvd(1, 2, 1, 5, 4, seed=91)
    scale, theta, eps = 0.6, 10000.0, 1e-6
    grads = O.attention_backward(q, k, v, do, scale, theta, causal)

    def loss(q_, k_, v_):
        o, _ = O.attention_forward(q_, k_, v_, scale, theta, causal)
        return float((do * o).sum())

    for which, x in enumerate((q, k, v)):
        g = grads[which]
        flat = x.reshape(-1)
        for n in range(flat.numel()):
            args = [q.clone(), k.clone(), v.clone()]
            args[which].view(-1)[n] += eps
            lp = loss(*args)
            args[which].view(-1)[n] -= 2 * eps
            lm = loss(*args)
            fd = (lp - lm) / (2 * eps)
            an = float(g.reshape(-1)[n])
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (which, n, fd, an)


def test_round_to_bf16_matches_torch():
    """Round-to-nearest-even to bf16 agrees with torch's conversion on values
    that are exact in fp32 (so torch rounds once)."""
    x = rnd((10000,), 101, 3.0).to(torch.float32).to(F64)
    x = torch.cat([x, torch.tensor([0.0, 1.0, -2.5, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8], dtype=F64)])
    want = x.to(torch.bfloat16).to(F64)
    assert torch.equal(O.round_to_bf16(x), want)


def test_round_rotated_mode_is_close():
    """Rounding RoPE(q), RoPE(k) to bf16 moves lse by about bf16 resolution."""
    q, k, v, _ = qkvd(1, 2, 1, 16, 8, seed=111)
    _, l0 = O.attention_forward(q, k, v, 0.35, 10000.0)
    _, l1 = O.attention_forward(q, k, v, 0.35, 10000.0, round_rotated=True)
    assert 0 < (l0 - l1).abs().max() < 0.05


def test_sampled_rows_match_full():
    B, Hq, Hkv, S, D = 1, 4, 2, 40, 8
    q, k, v, do = qkvd(B, Hq, Hkv, S, D, seed=121)
    out, lse = O.attention_forward(q, k, v, 0.3, 10000.0, round_rotated=True)
    dq, dk, dv = O.attention_backward(q, k, v, do, 0.3, 10000.0, round_rotated=True)
    rows = torch.tensor([0, 5, 17, 39])
    o_r, l_r = O.forward_rows(q, k, v, rows, 0.3, 10000.0, round_rotated=True)
    assert torch.allclose(o_r, out[:, :, rows], atol=1e-13)
    assert torch.allclose(l_r, lse[:, :, rows], atol=1e-13)
    dq_r = O.backward_dq_rows(q, k, v, do, rows, 0.3, 10000.0, round_rotated=True)
    assert torch.allclose(dq_r, dq[:, :, rows], atol=1e-12)
    keys = torch.tensor([0, 3, 20, 39])
    dk_k, dv_k = O.backward_dkdv_keys(q, k, v, do, keys, 0.3, 10000.0, round_rotated=True,
                                      kv_heads=[1], row_block=16)
    assert torch.allclose(dk_k[:, 0], dk[:, 1][:, keys], atol=1e-12)
    assert torch.allclose(dv_k[:, 0], dv[:, 1][:, keys], atol=1e-12)


# ------------------------------------------- query / key-value blocks (context parallel)
def test_partial_over_the_whole_range_is_the_full_attention():
    """One block holding every query and key (positions from 0) is the plain
    attention, forward and backward."""
    B, Hq, Hkv, S, D = 1, 4, 2, 10, 8
    q, k, v, do = qkvd(B, Hq, Hkv, S, D, seed=81)
    for causal in (True, False):
        out, lse = O.attention_forward(q, k, v, 0.4, 10000.0, causal)
        po, pl = O.attention_forward_partial(q, k, v, 0.4, 10000.0, 0, 0, causal)
        assert torch.allclose(po, out, atol=1e-13) and torch.allclose(pl, lse, atol=1e-13)
        full = O.attention_backward(q, k, v, do, 0.4, 10000.0, causal)
        part = O.attention_backward_partial(q, k, v, do, out, lse, 0.4, 10000.0, 0, 0, causal)
        for a, b in zip(part, full):
            assert torch.allclose(a, b, atol=1e-12)


@pytest.mark.parametrize("rope", ["half", "interleaved"])
def test_blocks_merge_to_the_full_attention(rope):
    """Queries and keys cut into two blocks each (a 2 x 2 ring schedule): merging
    each query block's partial results over the key blocks gives the full out and
    lse; the partial gradients, summed over the other blocks, give the full dq,
    dk, dv."""
    B, Hq, Hkv, S, D, cut = 1, 2, 1, 12, 8, 5
    q, k, v, do = qkvd(B, Hq, Hkv, S, D, seed=91)
    out, lse = O.attention_forward(q, k, v, 0.3, 10000.0, True, rope=rope)
    dq, dk, dv = O.attention_backward(q, k, v, do, 0.3, 10000.0, True, rope=rope)
    blocks = [(0, cut), (cut, S)]
    got_dq = torch.zeros_like(dq)
    got_dk = torch.zeros_like(dk)
    got_dv = torch.zeros_like(dv)
    for q0, q1 in blocks:
        merged = None
        for k0, k1 in blocks:
            po, pl = O.attention_forward_partial(q[:, :, q0:q1], k[:, :, k0:k1], v[:, :, k0:k1],
                                                 0.3, 10000.0, q0, k0, True, rope=rope)
            merged = (po, pl) if merged is None else O.merge_partials(*merged, po, pl)
            g = O.attention_backward_partial(q[:, :, q0:q1], k[:, :, k0:k1], v[:, :, k0:k1],
                                             do[:, :, q0:q1], out[:, :, q0:q1], lse[:, :, q0:q1],
                                             0.3, 10000.0, q0, k0, True, rope=rope)
            got_dq[:, :, q0:q1] += g[0]
            got_dk[:, :, k0:k1] += g[1]
            got_dv[:, :, k0:k1] += g[2]
        assert torch.allclose(merged[0], out[:, :, q0:q1], atol=1e-13)
        assert torch.allclose(merged[1], lse[:, :, q0:q1], atol=1e-13)
    for a, b in ((got_dq, dq), (got_dk, dk), (got_dv, dv)):
        assert torch.allclose(a, b, atol=1e-12)


def test_query_block_before_every_key_sees_nothing():
    """Under the causal mask, queries earlier than the whole key block attend to
    nothing: lse = -inf, out = 0, and the block contributes no gradient."""
    B, Hq, Hkv, D = 1, 2, 1, 4
    q, k, v, do = qkvd(B, Hq, Hkv, 3, D, seed=97)
    po, pl = O.attention_forward_partial(q, k, v, 0.5, 10000.0, 0, 3, True)
    assert torch.isneginf(pl).all() and (po == 0).all()
    g = O.attention_backward_partial(q, k, v, do, torch.zeros_like(po), pl, 0.5, 10000.0, 0, 3,
                                     True)
    assert all((t == 0).all() for t in g)
