"""Pins for the fp64 oracle: facts fixed by the pages or by mathematics, not by
the oracle itself.  Each pin is a function of the oracle module, so the last
test can plant mistakes in a copy of the oracle and check that some pin fails.
"""

import json
import math
import os
import types

import numpy as np
import pytest
import torch

import oracle.attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(7)


def _rand(*shape, rng=None):
    rng = rng or RNG
    return rng.standard_normal(shape)


# ---------------------------------------------------------------------------
# Pins
# ---------------------------------------------------------------------------


def pin_rows_sum_to_one(o):
    """Softmax rows sum to 1, also when P is rebuilt from the saved LSE."""
    rng = np.random.default_rng(1)
    for causal, Lq, Lk in [(True, 9, 13), (False, 7, 5), (True, 16, 16)]:
        q, k, v = _rand(Lq, 8, rng=rng), _rand(Lk, 8, rng=rng), _rand(Lk, 8, rng=rng)
        P, _, lse = o.head_forward(q, k, v, 0.3, causal)
        assert np.allclose(P.sum(axis=1), 1.0, atol=1e-12)
        S = 0.3 * q @ k.T
        mask = o.visible(Lq, Lk, causal)
        P2 = np.where(mask, np.exp(S - lse[:, None]), 0.0)
        assert np.allclose(P2.sum(axis=1), 1.0, atol=1e-12)


def pin_zero_query(o):
    """Q = 0 makes every visible score equal: O_i is the mean of the visible V
    rows and the base-2 LSE is log2 of the number of visible keys."""
    rng = np.random.default_rng(2)
    B, Hq, Hkv, Lq, Lk, D = 1, 2, 1, 6, 10, 4
    q = np.zeros((B, Hq, Lq, D))
    k, v = _rand(B, Hkv, Lk, D, rng=rng), _rand(B, Hkv, Lk, D, rng=rng)
    out, lse2, _ = o.forward(q, k, v, 0.5, True)
    for i in range(Lq):
        n = i + (Lk - Lq) + 1  # bottom-right: keys 0 .. i + Lk - Lq
        for h in range(Hq):
            assert np.allclose(out[0, h, i], v[0, 0, :n].mean(axis=0), atol=1e-12)
            assert abs(lse2[0, h, i] - math.log2(n)) < 1e-12
    out, lse2, _ = o.forward(q, k, v, 0.5, False)
    assert np.allclose(out[0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (Lq, D)), atol=1e-12)
    assert np.allclose(lse2, math.log2(Lk), atol=1e-12)


def pin_causal_diagonal(o):
    """Keys beyond the diagonal get exactly zero probability; in a square causal
    problem row 0 sees only key 0, so O_0 = V_0 and lse2_0 = S_00 * log2(e)."""
    rng = np.random.default_rng(3)
    for Lq, Lk in [(8, 8), (5, 12)]:
        q, k, v = _rand(Lq, 4, rng=rng), _rand(Lk, 4, rng=rng), _rand(Lk, 4, rng=rng)
        P, O, lse = o.head_forward(q, k, v, 0.7, True)
        for i in range(Lq):
            for j in range(Lk):
                if j > i + (Lk - Lq):
                    assert P[i, j] == 0.0
                else:
                    assert P[i, j] > 0.0
    q, k, v = _rand(1, 1, 8, 4, rng=rng), _rand(1, 1, 8, 4, rng=rng), _rand(1, 1, 8, 4, rng=rng)
    out, lse2, _ = o.forward(q, k, v, 0.7, True)
    assert np.allclose(out[0, 0, 0], v[0, 0, 0], atol=1e-14)
    s00 = 0.7 * float(np.dot(q[0, 0, 0], k[0, 0, 0]))
    assert abs(lse2[0, 0, 0] - s00 / math.log(2.0)) < 1e-12


def pin_delta_identity(o):
    """delta_i = sum_d dO_id O_id equals rowsum(P * dP) when O is exact, since
    sum_j P_ij sum_d dO_id V_jd = sum_d dO_id O_id."""
    rng = np.random.default_rng(4)
    q, k, v, do = (_rand(1, 2, 7, 5, rng=rng), _rand(1, 1, 11, 5, rng=rng),
                   _rand(1, 1, 11, 5, rng=rng), _rand(1, 2, 7, 5, rng=rng))
    out, _, _ = o.forward(q, k, v, 0.4, True)
    d = o.delta(out, do)
    for h in range(2):
        P, _, _ = o.head_forward(q[0, h], k[0, 0], v[0, 0], 0.4, True)
        dP = do[0, h] @ v[0, 0].T
        assert np.allclose(d[0, h], (P * dP).sum(axis=1), atol=1e-12)


def pin_gqa_is_repeated_mha(o):
    """GQA equals MHA with each KV head repeated for its G consecutive query
    heads; the GQA dK/dV are the group sums of the MHA dK/dV."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, Lq, Lk, D = 2, 6, 2, 5, 7, 3
    G = Hq // Hkv
    q, k, v, do = (_rand(B, Hq, Lq, D, rng=rng), _rand(B, Hkv, Lk, D, rng=rng),
                   _rand(B, Hkv, Lk, D, rng=rng), _rand(B, Hq, Lq, D, rng=rng))
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    og, lg, _ = o.forward(q, k, v, 0.6, True)
    om, lm, _ = o.forward(q, kr, vr, 0.6, True)
    assert np.allclose(og, om, atol=1e-12) and np.allclose(lg, lm, atol=1e-12)
    dqg, dkg, dvg = o.backward(q, k, v, og, do, 0.6, True)
    dqm, dkm, dvm = o.backward(q, kr, vr, om, do, 0.6, True)
    assert np.allclose(dqg, dqm, atol=1e-12)
    assert np.allclose(dkg, dkm.reshape(B, Hkv, G, Lk, D).sum(axis=2), atol=1e-12)
    assert np.allclose(dvg, dvm.reshape(B, Hkv, G, Lk, D).sum(axis=2), atol=1e-12)


def pin_finite_differences(o):
    """Central differences of L = sum(dO * O) match dQ, dK, dV (fp64, tiny)."""
    rng = np.random.default_rng(6)
    h = 1e-6
    for causal, Lq, Lk in [(True, 5, 5), (True, 4, 7), (False, 6, 3)]:
        B, Hq, Hkv, D = 1, 2, 1, 4
        q, k, v, do = (_rand(B, Hq, Lq, D, rng=rng), _rand(B, Hkv, Lk, D, rng=rng),
                       _rand(B, Hkv, Lk, D, rng=rng), _rand(B, Hq, Lq, D, rng=rng))
        scale = 0.45
        out, _, _ = o.forward(q, k, v, scale, causal)
        grads = o.backward(q, k, v, out, do, scale, causal)

        def loss(q_, k_, v_):
            return float((o.forward(q_, k_, v_, scale, causal)[0] * do).sum())

        for which, x in enumerate((q, k, v)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p[which], args_m[which] = xp, xm
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert np.allclose(grads[which], num, atol=1e-7, rtol=1e-6), (which, causal, Lq, Lk)


def pin_torch_sdpa(o):
    """Cross-check against PyTorch's CPU fp64 scaled_dot_product_attention and
    autograd, with an explicit bottom-right boolean mask (torch's is_causal is
    top-left aligned when Lq != Lk)."""
    rng = np.random.default_rng(8)
    for causal, B, Hq, Hkv, Lq, Lk, D in [(True, 2, 4, 2, 6, 9, 8), (False, 1, 2, 2, 5, 4, 8),
                                          (True, 1, 4, 1, 12, 12, 16)]:
        G = Hq // Hkv
        q, k, v, do = (_rand(B, Hq, Lq, D, rng=rng), _rand(B, Hkv, Lk, D, rng=rng),
                       _rand(B, Hkv, Lk, D, rng=rng), _rand(B, Hq, Lq, D, rng=rng))
        scale = 1.0 / math.sqrt(D)
        tq = torch.tensor(q, requires_grad=True)
        tk = torch.tensor(k, requires_grad=True)
        tv = torch.tensor(v, requires_grad=True)
        kr = tk.repeat_interleave(G, dim=1)
        vr = tv.repeat_interleave(G, dim=1)
        if causal:
            mask = torch.ones(Lq, Lk, dtype=torch.bool).tril(diagonal=Lk - Lq)
        else:
            mask = None
        to = torch.nn.functional.scaled_dot_product_attention(tq, kr, vr, attn_mask=mask, scale=scale)
        to.backward(torch.tensor(do))
        scores = (tq.detach() @ kr.detach().transpose(-1, -2)) * scale
        if mask is not None:
            scores = scores.masked_fill(~mask, float("-inf"))
        tlse2 = torch.logsumexp(scores, dim=-1) / math.log(2.0)
        out, lse2, _ = o.forward(q, k, v, scale, causal)
        dq, dk, dv = o.backward(q, k, v, out, do, scale, causal)
        assert np.allclose(out, to.detach().numpy(), atol=1e-12)
        assert np.allclose(lse2, tlse2.numpy(), atol=1e-12)
        assert np.allclose(dq, tq.grad.numpy(), atol=1e-12)
        assert np.allclose(dk, tk.grad.numpy(), atol=1e-12)
        assert np.allclose(dv, tv.grad.numpy(), atol=1e-12)


def pin_brute_force_loops(o):
    """Pure-Python loops over the defining sums, on a tiny causal GQA case."""
    rng = np.random.default_rng(9)
    B, Hq, Hkv, Lq, Lk, D = 1, 2, 1, 3, 4, 2
    q, k, v, do = (_rand(B, Hq, Lq, D, rng=rng), _rand(B, Hkv, Lk, D, rng=rng),
                   _rand(B, Hkv, Lk, D, rng=rng), _rand(B, Hq, Lq, D, rng=rng))
    sc = 0.8
    out, lse2, _ = o.forward(q, k, v, sc, True)
    dq, dk, dv = o.backward(q, k, v, out, do, sc, True)
    dk_ref = [[0.0] * D for _ in range(Lk)]
    dv_ref = [[0.0] * D for _ in range(Lk)]
    for h in range(Hq):
        for i in range(Lq):
            vis = [j for j in range(Lk) if j <= i + Lk - Lq]
            s = {j: sc * sum(q[0, h, i, d] * k[0, 0, j, d] for d in range(D)) for j in vis}
            z = sum(math.exp(s[j]) for j in vis)
            p = {j: math.exp(s[j]) / z for j in vis}
            oi = [sum(p[j] * v[0, 0, j, d] for j in vis) for d in range(D)]
            assert np.allclose(out[0, h, i], oi, atol=1e-12)
            assert abs(lse2[0, h, i] - math.log(z) / math.log(2.0)) < 1e-12
            dl = sum(do[0, h, i, d] * oi[d] for d in range(D))
            dqi = [0.0] * D
            for j in vis:
                dp = sum(do[0, h, i, d] * v[0, 0, j, d] for d in range(D))
                ds = p[j] * (dp - dl)
                for d in range(D):
                    dqi[d] += sc * ds * k[0, 0, j, d]
                    dk_ref[j][d] += sc * ds * q[0, h, i, d]
                    dv_ref[j][d] += p[j] * do[0, h, i, d]
            assert np.allclose(dq[0, h, i], dqi, atol=1e-12)
    assert np.allclose(dk[0, 0], dk_ref, atol=1e-12)
    assert np.allclose(dv[0, 0], dv_ref, atol=1e-12)


def pin_sampled_helpers(o):
    """The row/head sampling helpers agree with the whole-problem functions."""
    rng = np.random.default_rng(10)
    B, Hq, Hkv, Lq, Lk, D = 2, 4, 2, 9, 11, 4
    q, k, v, do = (_rand(B, Hq, Lq, D, rng=rng), _rand(B, Hkv, Lk, D, rng=rng),
                   _rand(B, Hkv, Lk, D, rng=rng), _rand(B, Hq, Lq, D, rng=rng))
    out, lse2, _ = o.forward(q, k, v, 0.5, True)
    rows = [0, 4, 8]
    orow, lrow = o.forward_rows(q, k, v, 0.5, True, 1, 3, rows)
    assert np.allclose(orow, out[1, 3, rows], atol=1e-13)
    assert np.allclose(lrow, lse2[1, 3, rows], atol=1e-13)
    dq, dk, dv = o.backward(q, k, v, out, do, 0.5, True)
    dqs, dkh, dvh = o.backward_kv_head(q, k, v, out, do, 0.5, True, 1, 1)
    assert np.allclose(dqs, dq[1, 2:4], atol=1e-13)
    assert np.allclose(dkh, dk[1, 1], atol=1e-13) and np.allclose(dvh, dv[1, 1], atol=1e-13)
    for causal in (True, False):
        out, lse2, lse_nat = o.forward(q, k, v, 0.5, causal)
        dq, dk, dv = o.backward(q, k, v, out, do, 0.5, causal)
        assert np.allclose(o.lse_all_rows(q, k, 0.5, causal, 1, 2, block=4), lse_nat[1, 2], atol=1e-13)
        assert np.allclose(o.backward_query_rows(q, k, v, out, do, 0.5, causal, 0, 3, rows),
                           dq[0, 3, rows], atol=1e-13)
        keys = [0, 5, 10]
        dks, dvs = o.backward_key_rows(q, k, v, out, do, 0.5, causal, 1, 0, keys)
        assert np.allclose(dks, dk[1, 0, keys], atol=1e-13)
        assert np.allclose(dvs, dv[1, 0, keys], atol=1e-13)


def _rand_mask(rng, nqb, nkb, density=0.6):
    return (rng.random((nqb, nkb)) < density).astype(np.uint8)


def pin_block_mask_all_ones(o):
    """A block mask of ones changes nothing (page 1, "Sparse Block Masks":
    only zero entries skip a tile pair)."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, Lq, Lk, D = 1, 2, 1, 7, 9, 4
    q, k, v, do = (_rand(B, Hq, Lq, D, rng=rng), _rand(B, Hkv, Lk, D, rng=rng),
                   _rand(B, Hkv, Lk, D, rng=rng), _rand(B, Hq, Lq, D, rng=rng))
    for causal in (True, False):
        ones = np.ones((-(-Lq // 3), -(-Lk // 3)), dtype=np.uint8)
        out, lse2, _ = o.forward(q, k, v, 0.5, causal)
        outm, lse2m, _ = o.forward(q, k, v, 0.5, causal, ones, 3)
        assert np.array_equal(out, outm) and np.array_equal(lse2, lse2m)
        g = o.backward(q, k, v, out, do, 0.5, causal)
        gm = o.backward(q, k, v, out, do, 0.5, causal, ones, 3)
        assert all(np.array_equal(x, y) for x, y in zip(g, gm))


def pin_block_mask_block_diagonal(o):
    """With a block-diagonal mask every diagonal block is an attention problem
    of its own: its rows and keys match the unmasked definition on the block's
    sub-arrays (square blocks, so causal alignment is the same inside)."""
    rng = np.random.default_rng(12)
    B, Hq, Hkv, L, D, blk = 1, 2, 1, 6, 4, 2
    q, k, v, do = (_rand(B, Hq, L, D, rng=rng), _rand(B, Hkv, L, D, rng=rng),
                   _rand(B, Hkv, L, D, rng=rng), _rand(B, Hq, L, D, rng=rng))
    eye = np.eye(L // blk, dtype=np.uint8)
    for causal in (True, False):
        out, lse2, _ = o.forward(q, k, v, 0.7, causal, eye, blk)
        dq, dk, dv = o.backward(q, k, v, out, do, 0.7, causal, eye, blk)
        for t in range(L // blk):
            r = slice(t * blk, (t + 1) * blk)
            ob, lb, _ = o.forward(q[:, :, r], k[:, :, r], v[:, :, r], 0.7, causal)
            gb = o.backward(q[:, :, r], k[:, :, r], v[:, :, r], ob, do[:, :, r], 0.7, causal)
            assert np.allclose(out[:, :, r], ob, atol=1e-13) and np.allclose(lse2[:, :, r], lb, atol=1e-13)
            assert np.allclose(dq[:, :, r], gb[0], atol=1e-13)
            assert np.allclose(dk[:, :, r], gb[1], atol=1e-13) and np.allclose(dv[:, :, r], gb[2], atol=1e-13)


def pin_block_mask_torch_sdpa(o):
    """Against PyTorch's CPU fp64 attention and autograd with the explicit
    element mask causal AND block_mask[i // blk, j // blk] (every row keeps a
    visible key; non-square block grids catch a transposed mask)."""
    rng = np.random.default_rng(13)
    for causal, Lq, Lk, blk in [(True, 7, 11, 3), (False, 9, 5, 2), (True, 10, 10, 4)]:
        B, Hq, Hkv, D = 1, 4, 2, 8
        G = Hq // Hkv
        nqb, nkb = -(-Lq // blk), -(-Lk // blk)
        while True:
            bm = _rand_mask(rng, nqb, nkb)
            vis = o.visible(Lq, Lk, causal, bm, blk) if o is A else A.visible(Lq, Lk, causal, bm, blk)
            if vis.any(axis=1).all():
                break
        q, k, v, do = (_rand(B, Hq, Lq, D, rng=rng), _rand(B, Hkv, Lk, D, rng=rng),
                       _rand(B, Hkv, Lk, D, rng=rng), _rand(B, Hq, Lq, D, rng=rng))
        scale = 1.0 / math.sqrt(D)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        kr, vr = tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1)
        tmask = torch.tensor(vis)
        to = torch.nn.functional.scaled_dot_product_attention(tq, kr, vr, attn_mask=tmask, scale=scale)
        to.backward(torch.tensor(do))
        scores = ((tq.detach() @ kr.detach().transpose(-1, -2)) * scale).masked_fill(~tmask, float("-inf"))
        tlse2 = torch.logsumexp(scores, dim=-1) / math.log(2.0)
        out, lse2, _ = o.forward(q, k, v, scale, causal, bm, blk)
        dq, dk, dv = o.backward(q, k, v, out, do, scale, causal, bm, blk)
        assert np.allclose(out, to.detach().numpy(), atol=1e-12)
        assert np.allclose(lse2, tlse2.numpy(), atol=1e-12)
        assert np.allclose(dq, tq.grad.numpy(), atol=1e-12)
        assert np.allclose(dk, tk.grad.numpy(), atol=1e-12)
        assert np.allclose(dv, tv.grad.numpy(), atol=1e-12)


def pin_block_mask_empty_rows(o):
    """Query rows whose every key block is masked: O = 0, LSE = +inf, dQ = 0,
    and dK, dV equal the problem without those rows (non-causal, so dropping
    rows moves no causal offset)."""
    rng = np.random.default_rng(14)
    B, Hq, Hkv, Lq, Lk, D, blk = 1, 2, 1, 6, 6, 4, 2
    q, k, v, do = (_rand(B, Hq, Lq, D, rng=rng), _rand(B, Hkv, Lk, D, rng=rng),
                   _rand(B, Hkv, Lk, D, rng=rng), _rand(B, Hq, Lq, D, rng=rng))
    bm = np.ones((3, 3), dtype=np.uint8)
    bm[1] = 0  # query rows 2, 3 see nothing
    out, lse2, _ = o.forward(q, k, v, 0.6, False, bm, blk)
    dq, dk, dv = o.backward(q, k, v, out, do, 0.6, False, bm, blk)
    assert np.array_equal(out[:, :, 2:4], np.zeros_like(out[:, :, 2:4]))
    assert np.all(np.isposinf(lse2[:, :, 2:4]))
    assert np.array_equal(dq[:, :, 2:4], np.zeros_like(dq[:, :, 2:4]))
    keep = [0, 1, 4, 5]
    ok, lk, _ = o.forward(q[:, :, keep], k, v, 0.6, False)
    gk = o.backward(q[:, :, keep], k, v, ok, do[:, :, keep], 0.6, False)
    assert np.allclose(out[:, :, keep], ok, atol=1e-13) and np.allclose(lse2[:, :, keep], lk, atol=1e-13)
    assert np.allclose(dq[:, :, keep], gk[0], atol=1e-13)
    assert np.allclose(dk, gk[1], atol=1e-13) and np.allclose(dv, gk[2], atol=1e-13)


def pin_block_mask_finite_differences(o):
    """Central differences of L = sum(dO * O) match the gradients under a block
    mask that also empties a query block."""
    rng = np.random.default_rng(15)
    h = 1e-6
    B, Hq, Hkv, Lq, Lk, D, blk = 1, 2, 1, 6, 8, 3, 2
    bm = np.array([[1, 0, 1, 1], [0, 0, 0, 0], [1, 1, 0, 1]], dtype=np.uint8)
    for causal in (True, False):
        q, k, v, do = (_rand(B, Hq, Lq, D, rng=rng), _rand(B, Hkv, Lk, D, rng=rng),
                       _rand(B, Hkv, Lk, D, rng=rng), _rand(B, Hq, Lq, D, rng=rng))
        out, _, _ = o.forward(q, k, v, 0.5, causal, bm, blk)
        grads = o.backward(q, k, v, out, do, 0.5, causal, bm, blk)

        def loss(q_, k_, v_):
            return float((o.forward(q_, k_, v_, 0.5, causal, bm, blk)[0] * do).sum())

        for which, x in enumerate((q, k, v)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p, args_m = [q, k, v], [q, k, v]
                args_p[which], args_m[which] = xp, xm
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert np.allclose(grads[which], num, atol=1e-7, rtol=1e-6), (which, causal)


PINS = [pin_rows_sum_to_one, pin_zero_query, pin_causal_diagonal, pin_delta_identity,
        pin_gqa_is_repeated_mha, pin_finite_differences, pin_torch_sdpa, pin_brute_force_loops,
        pin_sampled_helpers, pin_block_mask_all_ones, pin_block_mask_block_diagonal,
        pin_block_mask_torch_sdpa, pin_block_mask_empty_rows, pin_block_mask_finite_differences]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(A)


# ---------------------------------------------------------------------------
# Pins fixed by numbers the pages print
# ---------------------------------------------------------------------------


def test_flop_convention_matches_printed_table():
    with open(os.path.join(GOLDEN, "flop_convention.json")) as f:
        g = json.load(f)
    for r in g["rows"]:
        f_fwd = A.flops_forward(r["B"], r["Hq"], r["Lq"], r["Lk"], r["D"], r["causal"])
        tf = f_fwd / (r["ms"] * 1e-3) / 1e12
        assert round(tf, 1) == r["tflops"], (r, tf)
    # backward credit is 2.5x the forward
    assert A.flops_fwd_bwd(1, 1, 8, 8, 4, True) == 3.5 * A.flops_forward(1, 1, 8, 8, 4, True)


def test_scale_constant_matches_printed_define():
    with open(os.path.join(GOLDEN, "scale_constant.json")) as f:
        g = json.load(f)
    s = float(np.float32(1.0 / math.sqrt(g["D"])))
    assert f"{s:.10f}" == g["printed_scale"]


# ---------------------------------------------------------------------------
# Planted mistakes: each mutant is the oracle with one plausible error; the
# pins above must reject every one of them.
# ---------------------------------------------------------------------------


def _mutant(**overrides):
    m = types.ModuleType("oracle_mutant")
    for name in dir(A):
        if not name.startswith("__"):
            setattr(m, name, getattr(A, name))
    for name, fn in overrides.items():
        setattr(m, name, fn)
    # rebind the module-level functions so they see the overrides
    import inspect

    for name in dir(A):
        obj = getattr(A, name)
        if inspect.isfunction(obj) and name not in overrides:
            setattr(m, name, types.FunctionType(obj.__code__, m.__dict__, name, obj.__defaults__))
    return m


def _top_left_visible(Lq, Lk, causal, block_mask=None, blk=A.MASK_BLOCK):
    vis = np.ones((Lq, Lk), dtype=bool) if not causal else np.arange(Lk)[None, :] <= np.arange(Lq)[:, None]
    if block_mask is not None:
        bm = np.asarray(block_mask) != 0
        vis = vis & bm[np.arange(Lq)[:, None] // blk, np.arange(Lk)[None, :] // blk]
    return vis


def _mask_transposed_visible(Lq, Lk, causal, block_mask=None, blk=A.MASK_BLOCK):
    # reads the block mask as [key block, query block]
    vis = A.visible(Lq, Lk, causal)
    if block_mask is not None:
        bm = np.asarray(block_mask) != 0
        kb, qb = np.arange(Lk)[None, :] // blk, np.arange(Lq)[:, None] // blk
        ok = (kb < bm.shape[0]) & (qb < bm.shape[1])
        vis = vis & ok & bm[np.minimum(kb, bm.shape[0] - 1), np.minimum(qb, bm.shape[1] - 1)]
    return vis


def _mask_ignored_visible(Lq, Lk, causal, block_mask=None, blk=A.MASK_BLOCK):
    return A.visible(Lq, Lk, causal)


def _mk_head_backward(change):
    def head_backward(qh, kh, vh, oh, doh, scale, causal, block_mask=None, blk=A.MASK_BLOCK):
        P, _, _ = A.head_forward(qh, kh, vh, scale, causal, block_mask, blk)
        dP = doh @ vh.T
        dlt = (oh * doh).sum(axis=-1)[:, None]
        if change == "drop_delta":
            dS = P * dP
        elif change == "sign":
            dS = P * (dlt - dP)
        else:
            dS = P * (dP - dlt)
        dq = (dS @ kh) if change == "no_scale_dq" else scale * (dS @ kh)
        dk = scale * (dS.T @ qh)
        dv = P.T @ doh
        if change == "swap_dk_dv":
            dk, dv = dv, dk
        if change == "dv_uses_dS":
            dv = dS.T @ doh
        return dq, dk, dv

    return head_backward


def _bad_forward_lse_natural(q, k, v, scale, causal, block_mask=None, blk=A.MASK_BLOCK):
    o, lse2, lse = A.forward(q, k, v, scale, causal, block_mask, blk)
    return o, lse, lse


def _bad_gqa_forward(q, k, v, scale, causal, block_mask=None, blk=A.MASK_BLOCK):
    # query head hq reads KV head hq % Hkv instead of hq // G
    Hq, Hkv = q.shape[1], k.shape[1]
    idx = [h % Hkv for h in range(Hq)]
    return A.forward(q, k[:, idx], v[:, idx], scale, causal, block_mask, blk)


def _bad_scale_forward(q, k, v, scale, causal, block_mask=None, blk=A.MASK_BLOCK):
    return A.forward(q, k, v, 1.0, causal, block_mask, blk)


def _masked_rows_uniform_softmax_rows(S, mask):
    # a row with no visible key spreads its probability over every key
    has = mask.any(axis=1, keepdims=True)
    mask = np.where(has, mask, True)
    return A._softmax_rows(S, mask)


MUTANTS = {
    "top_left_causal": dict(visible=_top_left_visible),
    "drop_delta": dict(head_backward=_mk_head_backward("drop_delta")),
    "dS_sign": dict(head_backward=_mk_head_backward("sign")),
    "dq_without_scale": dict(head_backward=_mk_head_backward("no_scale_dq")),
    "dk_dv_swapped": dict(head_backward=_mk_head_backward("swap_dk_dv")),
    "dv_from_dS": dict(head_backward=_mk_head_backward("dv_uses_dS")),
    "lse_natural_log": dict(forward=_bad_forward_lse_natural),
    "gqa_modulo_mapping": dict(forward=_bad_gqa_forward),
    "scale_ignored": dict(forward=_bad_scale_forward),
    "delta_zero": dict(delta=lambda o_, do_: np.zeros(o_.shape[:-1])),
    "block_mask_transposed": dict(visible=_mask_transposed_visible),
    "block_mask_ignored": dict(visible=_mask_ignored_visible),
    "masked_row_uniform": dict(_softmax_rows=_masked_rows_uniform_softmax_rows),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name):
    m = _mutant(**MUTANTS[name])
    failed = []
    for pin in PINS:
        try:
            pin(m)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_copy_passes_pins():
    m = _mutant()
    for pin in PINS:
        pin(m)
