"""Pins for the fp64 oracle (CPU only).

The oracle is checked against things other than itself: finite differences of
its own forward (which pin the explicit gradient formulas), closed forms,
invariants the method fixes (merging chunk partials equals the monolithic
softmax, DISTFLASHATTN §3.2; exactness of attention, §3.1/§3.3), and a library
special case (torch's scaled_dot_product_attention in fp64 with autograd).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def loss_and_grads(q, k, v, dO, **kw):
    O, _ = oracle.attn_fwd(q, k, v, **kw)
    return float(np.sum(O * dO))


# ---------------------------------------------------------------- finite differences
FD_CASES = [
    # (B, H, Hkv, Lq, Lkv, D, causal, q_offset, kv_offset)
    (1, 2, 1, 6, 6, 3, True, 0, 0),        # GQA, causal, self-attention
    (2, 1, 1, 5, 5, 4, False, 0, 0),       # batch, non-causal
    (1, 2, 2, 4, 7, 2, True, 5, 2),        # chunk pair with offsets: diagonal cuts the block
    (1, 3, 1, 8, 8, 4, True, 0, 0),        # G = 3
]


@pytest.mark.parametrize("case", FD_CASES)
def test_gradients_match_finite_differences(case):
    B, H, Hkv, Lq, Lkv, D, causal, qo, ko = case
    q, k, v = rnd((B, Lq, H, D), 1), rnd((B, Lkv, Hkv, D), 2), rnd((B, Lkv, Hkv, D), 3)
    dO = rnd((B, Lq, H, D), 4)
    kw = dict(causal=causal, scale=0.7, q_offset=qo, kv_offset=ko)
    dQ, dK, dV = oracle.attn_bwd(q, k, v, dO, **kw)
    h = 1e-6
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = loss_and_grads(args["q"], args["k"], args["v"], dO, **kw)
            args[name] = xm
            fm = loss_and_grads(args["q"], args["k"], args["v"], dO, **kw)
            fd[idx] = (fp - fm) / (2 * h)
        err = np.max(np.abs(fd - g) / np.maximum(1.0, np.abs(g)))
        assert err < 1e-7, (name, err)


# ---------------------------------------------------------------- closed forms
def test_row0_and_row1_closed_forms():
    B, H, S, D = 1, 1, 5, 4
    q, k, v = rnd((B, S, H, D), 10), rnd((B, S, H, D), 11), rnd((B, S, H, D), 12)
    scale = 0.5
    O, lse = oracle.attn_fwd(q, k, v, scale=scale)
    # Row 0 under causal attention sees only key 0.
    s00 = scale * q[0, 0, 0] @ k[0, 0, 0]
    np.testing.assert_allclose(O[0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-15)
    assert abs(lse[0, 0, 0] - s00) < 1e-14
    # Row 1: two-key softmax written out.
    s10 = scale * q[0, 1, 0] @ k[0, 0, 0]
    s11 = scale * q[0, 1, 0] @ k[0, 1, 0]
    w1 = 1.0 / (1.0 + math.exp(s10 - s11))
    np.testing.assert_allclose(O[0, 1, 0], (1 - w1) * v[0, 0, 0] + w1 * v[0, 1, 0], atol=1e-14)
    assert abs(lse[0, 0, 1] - math.log(math.exp(s10) + math.exp(s11))) < 1e-13


def test_identity_values_expose_probabilities():
    # With V = I (D = S) the output row is the probability row itself.
    S = 7
    q, k = rnd((1, S, 1, S), 20), rnd((1, S, 1, S), 21)
    v = np.eye(S).reshape(1, S, 1, S)
    P, lse = oracle.attn_fwd(q, k, v, scale=0.3)
    P = P[0, :, 0, :]
    np.testing.assert_allclose(P.sum(axis=1), np.ones(S), atol=1e-14)
    assert np.all(P[np.triu_indices(S, 1)] == 0.0)          # causal: nothing above the diagonal
    s = 0.3 * q[0, :, 0, :] @ k[0, :, 0, :].T
    for i in range(S):
        ratio = P[i, : i + 1] / np.exp(s[i, : i + 1] - s[i, 0])
        np.testing.assert_allclose(ratio, ratio[0], rtol=1e-13)   # P_ij proportional to exp(s_ij)


def test_constant_values_give_that_constant():
    B, H, Hkv, S, D = 2, 4, 2, 9, 3
    q, k = rnd((B, S, H, D), 30), rnd((B, S, Hkv, D), 31)
    c = np.array([1.5, -2.0, 0.25])
    v = np.broadcast_to(c, (B, S, Hkv, D)).copy()
    O, _ = oracle.attn_fwd(q, k, v)
    np.testing.assert_allclose(O, np.broadcast_to(c, O.shape), atol=1e-14)


def test_one_hot_dominant_key_selects_its_value():
    S, D = 6, 4
    q = rnd((1, S, 1, D), 40)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rnd((1, S, 1, D), 41) * 0.1
    v = rnd((1, S, 1, D), 42)
    # Row i = 5 gets a dominant key at j = 2.
    k[0, 2, 0] = 50.0 * q[0, 5, 0]
    O, _ = oracle.attn_fwd(q, k, v, scale=1.0)
    np.testing.assert_allclose(O[0, 5, 0], v[0, 2, 0], atol=1e-15 + 1e-12)


def test_key_shift_invariance():
    B, H, S, D = 1, 2, 8, 4
    q, k, v = rnd((B, S, H, D), 50), rnd((B, S, H, D), 51), rnd((B, S, H, D), 52)
    c = rnd((D,), 53)
    O1, lse1 = oracle.attn_fwd(q, k, v, scale=0.6)
    O2, lse2 = oracle.attn_fwd(q, k + c, v, scale=0.6)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    shift = 0.6 * np.einsum("bshd,d->bhs", q, c)
    np.testing.assert_allclose(lse2 - lse1, shift, atol=1e-12)


def test_empty_rows_of_a_chunk_pair():
    # kv block entirely in the future of the first query rows: O = 0, lse = -inf.
    q, k, v = rnd((1, 4, 1, 3), 60), rnd((1, 4, 1, 3), 61), rnd((1, 4, 1, 3), 62)
    O, lse = oracle.attn_fwd(q, k, v, q_offset=0, kv_offset=2)
    assert np.all(O[0, :2] == 0.0) and np.all(np.isneginf(lse[0, 0, :2]))
    assert np.all(np.isfinite(lse[0, 0, 2:]))


# ---------------------------------------------------------------- merge (online-softmax rule)
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_merging_chunk_partials_equals_monolithic(P):
    B, H, Hkv, S, D = 1, 2, 1, 24, 4
    C = S // P
    q, k, v = rnd((B, S, H, D), 70), rnd((B, S, Hkv, D), 71), rnd((B, S, Hkv, D), 72)
    O_ref, lse_ref = oracle.attn_fwd(q, k, v)
    for p in range(P):
        qs = q[:, p * C:(p + 1) * C]
        acc = None
        for t in range(p + 1):
            part = oracle.attn_fwd(qs, k[:, t * C:(t + 1) * C], v[:, t * C:(t + 1) * C],
                                   q_offset=p * C, kv_offset=t * C)
            acc = part if acc is None else oracle.merge(*acc, *part)
        np.testing.assert_allclose(acc[0], O_ref[:, p * C:(p + 1) * C], atol=1e-13)
        np.testing.assert_allclose(acc[1], lse_ref[:, :, p * C:(p + 1) * C], atol=1e-13)


# ---------------------------------------------------------------- chunk-pair backward (§3.3)
def chunk_bounds(S, cuts):
    edges = [0] + list(cuts) + [S]
    return list(zip(edges[:-1], edges[1:]))


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("cuts", [(), (12,), (5, 13), (4, 8, 16)])
def test_chunk_pair_backward_sums_to_full(cuts, causal):
    # Each worker's backward step gives partial dQ for its query chunk and partial
    # dK/dV for the key chunk it visits, from the rows' global lse and Delta; the
    # sum over the pairs must be the full gradient (pinned by finite differences).
    B, H, Hkv, S, D = 2, 4, 2, 21, 5
    q, k, v = rnd((B, S, H, D), 300), rnd((B, S, Hkv, D), 301), rnd((B, S, Hkv, D), 302)
    dO = rnd((B, S, H, D), 303)
    kw = dict(causal=causal, scale=0.6)
    _, lse = oracle.attn_fwd(q, k, v, **kw)
    dlt = oracle.delta(q, k, v, dO, **kw)
    dQ_ref, dK_ref, dV_ref = oracle.attn_bwd(q, k, v, dO, **kw)
    dQ, dK, dV = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    chunks = chunk_bounds(S, cuts)
    for qa, qb in chunks:
        for ka, kb in chunks:
            pq, pk, pv = oracle.chunk_bwd(q[:, qa:qb], k[:, ka:kb], v[:, ka:kb], dO[:, qa:qb],
                                          lse[:, :, qa:qb], dlt[:, :, qa:qb],
                                          q_offset=qa, kv_offset=ka, **kw)
            dQ[:, qa:qb] += pq
            dK[:, ka:kb] += pk
            dV[:, ka:kb] += pv
    np.testing.assert_allclose(dQ, dQ_ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(dK, dK_ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(dV, dV_ref, atol=1e-12, rtol=0)


def test_delta_equals_dO_dot_O():
    # sum_j P_ij <dO_i, v_j> = <dO_i, sum_j P_ij v_j> = <dO_i, O_i>
    B, H, Hkv, S, D = 1, 3, 1, 9, 4
    q, k, v, dO = rnd((B, S, H, D), 310), rnd((B, S, Hkv, D), 311), rnd((B, S, Hkv, D), 312), rnd((B, S, H, D), 313)
    O, _ = oracle.attn_fwd(q, k, v)
    np.testing.assert_allclose(oracle.delta(q, k, v, dO), np.einsum("bshd,bshd->bhs", O, dO), atol=1e-13)


def test_chunk_pair_above_the_diagonal_contributes_nothing():
    q, k, v, dO = rnd((1, 4, 2, 3), 320), rnd((1, 4, 1, 3), 321), rnd((1, 4, 1, 3), 322), rnd((1, 4, 2, 3), 323)
    lse, dlt = rnd((1, 2, 4), 324), rnd((1, 2, 4), 325)
    for out in oracle.chunk_bwd(q, k, v, dO, lse, dlt, q_offset=0, kv_offset=4):
        assert np.all(out == 0.0)
    # and a row whose global lse is -inf (no visible key anywhere) adds nothing
    lse[0, 1, 2] = -np.inf
    pq, _, _ = oracle.chunk_bwd(q, k, v, dO, lse, dlt, q_offset=4, kv_offset=0)
    assert np.all(pq[0, 2, 1] == 0.0)


# ---------------------------------------------------------------- local window (App. F)
def test_window_covering_every_chunk_is_plain_causal():
    B, H, Hkv, S, D = 1, 2, 1, 12, 3
    q, k, v, dO = rnd((B, S, H, D), 400), rnd((B, S, Hkv, D), 401), rnd((B, S, Hkv, D), 402), rnd((B, S, H, D), 403)
    for w in (3, 4, 7):
        a, b = oracle.attn_fwd_local(q, k, v, chunk=4, window=w), oracle.attn_fwd(q, k, v)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        for x, y in zip(oracle.attn_bwd_local(q, k, v, dO, chunk=4, window=w), oracle.attn_bwd(q, k, v, dO)):
            assert np.array_equal(x, y)


def test_window_of_one_chunk_is_independent_chunks():
    B, H, Hkv, S, D, C = 2, 2, 2, 15, 3, 5
    q, k, v, dO = rnd((B, S, H, D), 410), rnd((B, S, Hkv, D), 411), rnd((B, S, Hkv, D), 412), rnd((B, S, H, D), 413)
    O, lse = oracle.attn_fwd_local(q, k, v, chunk=C, window=1)
    dQ, dK, dV = oracle.attn_bwd_local(q, k, v, dO, chunk=C, window=1)
    for c in range(S // C):
        sl = slice(c * C, (c + 1) * C)
        Oc, lc = oracle.attn_fwd(q[:, sl], k[:, sl], v[:, sl])
        np.testing.assert_allclose(O[:, sl], Oc, atol=1e-14)
        np.testing.assert_allclose(lse[:, :, sl], lc, atol=1e-14)
        for g, r in zip((dQ[:, sl], dK[:, sl], dV[:, sl]), oracle.attn_bwd(q[:, sl], k[:, sl], v[:, sl], dO[:, sl])):
            np.testing.assert_allclose(g, r, atol=1e-13)


def test_window_of_two_chunks_merges_the_neighbour():
    # the pages' recipe: a worker fetches only the previous worker's key/value
    # block and merges that partial with its own chunk's (§3.2 merge rule)
    B, H, Hkv, S, D, C = 1, 2, 1, 18, 4, 6
    q, k, v = rnd((B, S, H, D), 420), rnd((B, S, Hkv, D), 421), rnd((B, S, Hkv, D), 422)
    O, lse = oracle.attn_fwd_local(q, k, v, chunk=C, window=2)
    for p in range(S // C):
        qs = slice(p * C, (p + 1) * C)
        acc = oracle.attn_fwd(q[:, qs], k[:, qs], v[:, qs], q_offset=p * C, kv_offset=p * C)
        if p > 0:
            ks = slice((p - 1) * C, p * C)
            acc = oracle.merge(*acc, *oracle.attn_fwd(q[:, qs], k[:, ks], v[:, ks], q_offset=p * C,
                                                      kv_offset=(p - 1) * C))
        np.testing.assert_allclose(O[:, qs], acc[0], atol=1e-13)
        np.testing.assert_allclose(lse[:, :, qs], acc[1], atol=1e-13)


def test_window_gradients_match_finite_differences():
    B, H, Hkv, S, D, C, w = 1, 2, 1, 9, 3, 3, 2
    q, k, v, dO = rnd((B, S, H, D), 430), rnd((B, S, Hkv, D), 431), rnd((B, S, Hkv, D), 432), rnd((B, S, H, D), 433)
    dQ, dK, dV = oracle.attn_bwd_local(q, k, v, dO, chunk=C, window=w, scale=0.8)
    loss = lambda q_, k_, v_: float(np.sum(oracle.attn_fwd_local(q_, k_, v_, chunk=C, window=w, scale=0.8)[0] * dO))
    h = 1e-6
    for idx, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            m = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[m] += h
            xm[m] -= h
            args_p = {"q": q, "k": k, "v": v}; args_p[idx] = xp
            args_m = {"q": q, "k": k, "v": v}; args_m[idx] = xm
            fd[m] = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        assert np.max(np.abs(fd - g) / np.maximum(1.0, np.abs(g))) < 1e-7, idx


@pytest.mark.parametrize("S,C,w", [(14, 4, 1), (14, 4, 2), (11, 3, 3), (9, 5, 1)])
def test_window_with_a_ragged_last_chunk_matches_torch_sdpa(S, C, w):
    # chunks of C tokens and a shorter last one (S = 14, C = 4: 4, 4, 4, 2);
    # the window mask written from its definition, attention by torch in fp64
    B, H, Hkv, D, scale = 1, 2, 1, 5, 0.6
    q, k, v, dO = rnd((B, S, H, D), 440), rnd((B, S, Hkv, D), 441), rnd((B, S, Hkv, D), 442), rnd((B, S, H, D), 443)
    O, lse = oracle.attn_fwd_local(q, k, v, chunk=C, window=w, scale=scale)
    dQ, dK, dV = oracle.attn_bwd_local(q, k, v, dO, chunk=C, window=w, scale=scale)
    i, j = np.arange(S)[:, None], np.arange(S)[None, :]
    allow = torch.tensor((j <= i) & (j // C >= i // C - (w - 1)))
    tq = torch.tensor(q).transpose(1, 2).requires_grad_()
    tk = torch.tensor(k).transpose(1, 2).requires_grad_()
    tv = torch.tensor(v).transpose(1, 2).requires_grad_()
    kk, vv = tk.repeat_interleave(H // Hkv, dim=1), tv.repeat_interleave(H // Hkv, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, attn_mask=allow, scale=scale)
    out.backward(torch.tensor(dO).transpose(1, 2))
    np.testing.assert_allclose(O, out.detach().transpose(1, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(dQ, tq.grad.transpose(1, 2).numpy(), atol=1e-11)
    np.testing.assert_allclose(dK, tk.grad.transpose(1, 2).numpy(), atol=1e-11)
    np.testing.assert_allclose(dV, tv.grad.transpose(1, 2).numpy(), atol=1e-11)
    s = scale * torch.einsum("bhid,bhjd->bhij", tq.detach(), kk.detach()).masked_fill(~allow, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


def test_merge_neutral_element_and_symmetry():
    O_a, O_b = rnd((1, 3, 2, 4), 80), rnd((1, 3, 2, 4), 81)
    la, lb = rnd((1, 2, 3), 82), rnd((1, 2, 3), 83)
    ninf = np.full_like(la, -np.inf)
    O, l = oracle.merge(O_a, la, np.zeros_like(O_b), ninf)
    np.testing.assert_allclose(O, O_a, atol=0)
    np.testing.assert_allclose(l, la, atol=0)
    O, l = oracle.merge(np.zeros_like(O_a), ninf, np.zeros_like(O_b), ninf)
    assert np.all(O == 0) and np.all(np.isneginf(l))
    O1, l1 = oracle.merge(O_a, la, O_b, lb)
    O2, l2 = oracle.merge(O_b, lb, O_a, la)
    np.testing.assert_allclose(O1, O2, atol=1e-15)
    np.testing.assert_allclose(l1, np.logaddexp(la, lb), atol=1e-14)


# ---------------------------------------------------------------- library special case
@pytest.mark.parametrize("H,Hkv,causal", [(4, 2, True), (2, 2, False), (3, 1, True)])
def test_matches_torch_sdpa_fp64(H, Hkv, causal):
    B, S, D = 2, 97, 16
    scale = 0.21
    q, k, v, dO = (rnd((B, S, H, D), 90)), rnd((B, S, Hkv, D), 91), rnd((B, S, Hkv, D), 92), rnd((B, S, H, D), 93)
    O, lse = oracle.attn_fwd(q, k, v, causal=causal, scale=scale)
    dQ, dK, dV = oracle.attn_bwd(q, k, v, dO, causal=causal, scale=scale)
    G = H // Hkv
    tq = torch.tensor(q).transpose(1, 2).requires_grad_()
    tk = torch.tensor(k).transpose(1, 2).requires_grad_()
    tv = torch.tensor(v).transpose(1, 2).requires_grad_()
    kk, vv = tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, is_causal=causal, scale=scale)
    out.backward(torch.tensor(dO).transpose(1, 2))
    np.testing.assert_allclose(O, out.detach().transpose(1, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(dQ, tq.grad.transpose(1, 2).numpy(), atol=1e-11)
    np.testing.assert_allclose(dK, tk.grad.transpose(1, 2).numpy(), atol=1e-11)
    np.testing.assert_allclose(dV, tv.grad.transpose(1, 2).numpy(), atol=1e-11)
    s = scale * torch.einsum("bhid,bhjd->bhij", tq.detach(), kk.detach())
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


# ---------------------------------------------------------------- gradient invariants
def test_gradient_invariants():
    B, H, Hkv, S, D = 1, 4, 2, 33, 8
    q, k, v, dO = rnd((B, S, H, D), 100), rnd((B, S, Hkv, D), 101), rnd((B, S, Hkv, D), 102), rnd((B, S, H, D), 103)
    O, _ = oracle.attn_fwd(q, k, v)
    dQ, dK, dV = oracle.attn_bwd(q, k, v, dO)
    G = H // Hkv
    for g in range(Hkv):
        heads = slice(g * G, (g + 1) * G)
        np.testing.assert_allclose(dV[:, :, g].sum(axis=(0, 1)), dO[:, :, heads].sum(axis=(0, 1, 2)), atol=1e-12)
        np.testing.assert_allclose(dK[:, :, g].sum(axis=(0, 1)), 0.0, atol=1e-12)
        assert abs(np.sum(q[:, :, heads] * dQ[:, :, heads]) - np.sum(k[:, :, g] * dK[:, :, g])) < 1e-11
        assert abs(np.sum(v[:, :, g] * dV[:, :, g]) - np.sum(O[:, :, heads] * dO[:, :, heads])) < 1e-11


# ---------------------------------------------------------------- sampled-row entry points
def test_row_entry_points_agree_with_full():
    B, H, Hkv, S, D = 2, 4, 2, 40, 8
    q, k, v, dO = rnd((B, S, H, D), 110), rnd((B, S, Hkv, D), 111), rnd((B, S, Hkv, D), 112), rnd((B, S, H, D), 113)
    O, lse = oracle.attn_fwd(q, k, v)
    dQ, dK, dV = oracle.attn_bwd(q, k, v, dO)
    rows = [(0, 0, 0), (1, 3, 39), (0, 2, 17), (1, 1, 5)]
    Or, lr = oracle.attn_fwd_rows(q, k, v, rows)
    dqr = oracle.attn_dq_rows(q, k, v, dO, rows)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(Or[n], O[b, i, h], atol=1e-14)
        assert abs(lr[n] - lse[b, h, i]) < 1e-14
        np.testing.assert_allclose(dqr[n], dQ[b, i, h], atol=1e-13)
    krows = [(0, 0, 0), (1, 1, 39), (0, 1, 20)]
    dkr, dvr = oracle.attn_dkv_rows(q, k, v, dO, krows)
    for n, (b, g, j) in enumerate(krows):
        np.testing.assert_allclose(dkr[n], dK[b, j, g], atol=1e-13)
        np.testing.assert_allclose(dvr[n], dV[b, j, g], atol=1e-13)


def test_bad_arguments_are_rejected():
    q = np.zeros((1, 4, 3, 2))
    k = np.zeros((1, 4, 2, 2))
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, k)             # H % H_kv != 0
    with pytest.raises(ValueError):
        oracle.attn_fwd_rows(q[:, :, :2], k, k, [(0, 0, 4)])   # row out of range


def test_golden_fixture_reproduces():
    """Regression fixture written by tests/golden/make_oracle_fixture.py (oracle only)."""
    with open(os.path.join(GOLDEN, "oracle_tiny_causal.json")) as f:
        fx = json.load(f)
    q, k, v, dO = (np.array(fx[n]) for n in ("q", "k", "v", "dO"))
    O, lse = oracle.attn_fwd(q, k, v, scale=fx["scale"])
    dQ, dK, dV = oracle.attn_bwd(q, k, v, dO, scale=fx["scale"])
    for name, got in (("O", O), ("lse", lse), ("dQ", dQ), ("dK", dK), ("dV", dV)):
        np.testing.assert_allclose(got, np.array(fx[name]), atol=1e-14, err_msg=name)


# ---------------------------------------------------------------- variable-length batches
def block_mask(cu, causal):
    """Allowed (query, key) pairs of a packed batch: same sequence, and key <= query when causal."""
    T = int(cu[-1])
    seq = np.searchsorted(np.asarray(cu), np.arange(T), side="right") - 1
    allow = seq[:, None] == seq[None, :]
    if causal:
        allow &= np.arange(T)[None, :] <= np.arange(T)[:, None]
    return allow


@pytest.mark.parametrize("lens,H,Hkv,causal", [([5, 0, 9, 1, 13], 4, 2, True), ([7, 7, 3], 2, 2, False),
                                               ([1], 3, 1, True), ([16, 2, 0], 2, 1, True)])
def test_varlen_matches_torch_sdpa_with_a_block_diagonal_mask(lens, H, Hkv, causal):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, D, scale = int(cu[-1]), 8, 0.37
    q, k, v, dO = rnd((T, H, D), 120), rnd((T, Hkv, D), 121), rnd((T, Hkv, D), 122), rnd((T, H, D), 123)
    O, lse = oracle.attn_fwd_varlen(q, k, v, cu, causal=causal, scale=scale)
    dQ, dK, dV = oracle.attn_bwd_varlen(q, k, v, dO, cu, causal=causal, scale=scale)
    G = H // Hkv
    tq = torch.tensor(q).transpose(0, 1)[None].requires_grad_()
    tk = torch.tensor(k).transpose(0, 1)[None].requires_grad_()
    tv = torch.tensor(v).transpose(0, 1)[None].requires_grad_()
    kk, vv = tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1)
    allow = torch.tensor(block_mask(cu, causal))
    out = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, attn_mask=allow, scale=scale)
    out.backward(torch.tensor(dO).transpose(0, 1)[None])
    np.testing.assert_allclose(O, out.detach()[0].transpose(0, 1).numpy(), atol=1e-12)
    np.testing.assert_allclose(dQ, tq.grad[0].transpose(0, 1).numpy(), atol=1e-11)
    np.testing.assert_allclose(dK, tk.grad[0].transpose(0, 1).numpy(), atol=1e-11)
    np.testing.assert_allclose(dV, tv.grad[0].transpose(0, 1).numpy(), atol=1e-11)
    s = scale * torch.einsum("hid,hjd->hij", tq.detach()[0], kk.detach()[0])
    s = s.masked_fill(~allow, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


def test_varlen_of_equal_lengths_is_the_dense_batch():
    n, L, H, Hkv, D = 3, 11, 4, 2, 6
    q, k, v, dO = rnd((n, L, H, D), 130), rnd((n, L, Hkv, D), 131), rnd((n, L, Hkv, D), 132), rnd((n, L, H, D), 133)
    cu = np.arange(n + 1) * L
    O, lse = oracle.attn_fwd_varlen(q.reshape(n * L, H, D), k.reshape(n * L, Hkv, D), v.reshape(n * L, Hkv, D), cu)
    Od, ld = oracle.attn_fwd(q, k, v)
    np.testing.assert_array_equal(O.reshape(n, L, H, D), Od)
    np.testing.assert_array_equal(lse.reshape(H, n, L).transpose(1, 0, 2), ld)
    g = oracle.attn_bwd_varlen(*(x.reshape(n * L, x.shape[2], D) for x in (q, k, v, dO)), cu)
    gd = oracle.attn_bwd(q, k, v, dO)
    for a, b in zip(g, gd):   # same sums, possibly another order across the batch
        np.testing.assert_allclose(a.reshape(b.shape), b, rtol=0, atol=1e-13)


def test_varlen_gradients_match_finite_differences():
    cu = np.array([0, 3, 3, 7])
    T, H, Hkv, D = 7, 2, 1, 2
    q, k, v, dO = rnd((T, H, D), 140), rnd((T, Hkv, D), 141), rnd((T, Hkv, D), 142), rnd((T, H, D), 143)
    dQ, dK, dV = oracle.attn_bwd_varlen(q, k, v, dO, cu, scale=0.9)
    h = 1e-6
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            vals = []
            for sgn in (1, -1):
                args = {"q": q, "k": k, "v": v}
                xx = x.copy()
                xx[idx] += sgn * h
                args[name] = xx
                O, _ = oracle.attn_fwd_varlen(args["q"], args["k"], args["v"], cu, scale=0.9)
                vals.append(float(np.sum(O * dO)))
            fd[idx] = (vals[0] - vals[1]) / (2 * h)
        assert np.max(np.abs(fd - g) / np.maximum(1.0, np.abs(g))) < 1e-7, name


def test_varlen_rejects_bad_offsets():
    q = rnd((4, 1, 2), 150)
    for cu in ([0, 3], [1, 4], [0, 3, 2, 4]):
        with pytest.raises(ValueError):
            oracle.attn_fwd_varlen(q, q, q, cu)


def test_local_window_slices_reproduce_the_whole_sequence():
    """With a window of two chunks, a query of chunk c sees chunks c - 1 and c
    and a key of chunk c - 1 is seen by the queries of chunks c - 1 and c, so
    the local window on the slice of chunks [c - 2, c] (offsets keeping the
    positions global) gives chunk c's O, lse and dQ and chunk c - 1's dK and
    dV exactly: the identity the full-size GPU check relies on."""
    rng = np.random.default_rng(0)
    S, D, C, W = 80, 8, 16, 2
    q, k, v, do = (rng.standard_normal((1, S, 1, D)) for _ in range(4))
    Of, lf = oracle.attn_fwd_local(q, k, v, chunk=C, window=W)
    dqf, dkf, dvf = oracle.attn_bwd_local(q, k, v, do, chunk=C, window=W)
    for c in range(1, S // C):
        a, m, b = max(c - 2, 0) * C, c * C, (c + 1) * C
        prev = m - C - a
        Or, lr = oracle.attn_fwd_local(q[:, a:b], k[:, a:b], v[:, a:b], chunk=C, window=W, q_offset=a, kv_offset=a)
        dqr, dkr, dvr = oracle.attn_bwd_local(q[:, a:b], k[:, a:b], v[:, a:b], do[:, a:b], chunk=C, window=W,
                                              q_offset=a, kv_offset=a)
        np.testing.assert_allclose(Or[:, m - a:], Of[:, m:b], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lr[:, :, m - a:], lf[:, :, m:b], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dqr[:, m - a:], dqf[:, m:b], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dkr[:, prev:prev + C], dkf[:, m - C:m], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dvr[:, prev:prev + C], dvf[:, m - C:m], rtol=0, atol=1e-12)
        if c >= 2:   # the two-chunk slice is not enough: chunk c - 1's own queries lose chunk c - 2
            _, dk2, _ = oracle.attn_bwd_local(q[:, m - C:b], k[:, m - C:b], v[:, m - C:b], do[:, m - C:b], chunk=C,
                                              window=W, q_offset=m - C, kv_offset=m - C)
            assert np.max(np.abs(dk2[:, :C] - dkf[:, m - C:m])) > 1e-3
