"""Pins for the linear cross-entropy oracle (oracle/linear_ce.py) against
facts that do not come from the oracle itself: PyTorch's fp64 cross-entropy
with autograd (a library routine), the closed form at W = 0, the zero row sums
of the logit gradient, central finite differences, and a pure-Python loop on a
tiny case.  Planted mistakes in copies of the oracle must each fail a pin."""

import math

import numpy as np
import pytest
import torch

import oracle.linear_ce as L


def rand_case(N=7, Dm=5, V=11, seed=0, ignore=True):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((N, Dm))
    w = rng.standard_normal((V, Dm)) * 0.7
    t = rng.integers(0, V, N)
    if ignore:
        t[1] = -1
    dloss = rng.standard_normal(N)
    return h, w, t, dloss


def torch_reference(h, w, t, dloss):
    ht = torch.tensor(h, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    z = ht @ wt.T
    loss = torch.nn.functional.cross_entropy(z, torch.tensor(t), reduction="none", ignore_index=-1)
    (loss * torch.tensor(dloss)).sum().backward()
    return loss.detach().numpy(), torch.logsumexp(z, 1).detach().numpy(), ht.grad.numpy(), wt.grad.numpy()


def check_against_torch(fwd, bwd, seed=0):
    h, w, t, dloss = rand_case(seed=seed)
    loss, lse = fwd(h, w, t)
    dh, dw = bwd(h, w, t, lse, dloss)
    rl, rlse, rdh, rdw = torch_reference(h, w, t, dloss)
    np.testing.assert_allclose(loss, rl, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, rlse, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dh, rdh, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dw, rdw, rtol=1e-10, atol=1e-12)


def check_zero_weight_closed_form(fwd, bwd):
    h, w, t, dloss = rand_case(seed=1)
    w = np.zeros_like(w)
    V = w.shape[0]
    loss, lse = fwd(h, w, t)
    valid = t >= 0
    np.testing.assert_allclose(lse, math.log(V), rtol=0, atol=1e-14)
    np.testing.assert_allclose(loss[valid], math.log(V), rtol=0, atol=1e-14)
    assert np.all(loss[~valid] == 0)
    dh, dw = bwd(h, w, t, lse, dloss)
    np.testing.assert_allclose(dh, 0.0, atol=1e-14)
    g = np.zeros((h.shape[0], V))
    for i in np.nonzero(valid)[0]:
        g[i] = dloss[i] / V
        g[i, t[i]] -= dloss[i]
    np.testing.assert_allclose(dw, g.T @ h, rtol=1e-12, atol=1e-14)


def check_finite_differences(fwd, bwd, eps=1e-6):
    h, w, t, dloss = rand_case(N=4, Dm=3, V=6, seed=2)

    def objective(hh, ww):
        return float((fwd(hh, ww, t)[0] * dloss).sum())

    loss, lse = fwd(h, w, t)
    dh, dw = bwd(h, w, t, lse, dloss)
    for arr, grad in ((h, dh), (w, dw)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + eps
            fp = objective(h, w)
            arr[idx] = a0 - eps
            fm = objective(h, w)
            arr[idx] = a0
            num[idx] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8)


def check_python_loops(fwd, bwd):
    h, w, t, dloss = rand_case(N=3, Dm=2, V=4, seed=3, ignore=False)
    loss, lse = fwd(h, w, t)
    dh, dw = bwd(h, w, t, lse, dloss)
    N, Dm = h.shape
    V = w.shape[0]
    for i in range(N):
        z = [sum(h[i][d] * w[v][d] for d in range(Dm)) for v in range(V)]
        s = sum(math.exp(x) for x in z)
        assert abs(loss[i] - (math.log(s) - z[t[i]])) < 1e-12
        for d in range(Dm):
            ref = sum(dloss[i] * (math.exp(z[v]) / s - (v == t[i])) * w[v][d] for v in range(V))
            assert abs(dh[i][d] - ref) < 1e-12


PINS = [check_against_torch, check_zero_weight_closed_form, check_finite_differences, check_python_loops]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_passes_pin(pin):
    pin(L.forward, L.backward)


def test_gradient_rows_sum_to_zero():
    h, w, t, dloss = rand_case(seed=4)
    loss, lse = L.forward(h, w, t)
    g = L.grad_logits(h, w, t, lse, dloss)
    np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=1e-12)
    assert np.all(g[t < 0] == 0)


# ----- planted mistakes: each must fail at least one pin -----


def mut_onehot_sign(h, w, t, lse, dloss):
    g = L.grad_logits(h, w, t, lse, dloss)
    valid = t >= 0
    rows = np.arange(len(t))[valid]
    g[rows, t[valid]] += 2.0 * dloss[valid]  # p + onehot instead of p - onehot
    return g @ w, g.T @ h


def mut_no_dloss(h, w, t, lse, dloss):
    return L.backward(h, w, t, lse, np.ones_like(dloss))


def mut_dw_without_onehot(h, w, t, lse, dloss):
    dh, _ = L.backward(h, w, t, lse, dloss)
    p = np.exp(L.logits(h, w) - lse[:, None]) * dloss[:, None]
    return dh, p.T @ h


def mut_lse_is_max(h, w, t):
    z = L.logits(h, w)
    m = z.max(axis=1)
    rows = np.arange(len(t))
    return np.where(t >= 0, m - z[rows, np.maximum(t, 0)], 0.0), m


def mut_ignored_rows_count(h, w, t):
    loss, lse = L.forward(h, w, np.where(t >= 0, t, 0))
    return loss, lse


MUTANTS = [
    ("onehot_sign", L.forward, mut_onehot_sign),
    ("no_dloss", L.forward, mut_no_dloss),
    ("dw_without_onehot", L.forward, mut_dw_without_onehot),
    ("lse_is_max", mut_lse_is_max, L.backward),
    ("ignored_rows_count", mut_ignored_rows_count, L.backward),
]


@pytest.mark.parametrize("name,fwd,bwd", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, fwd, bwd):
    caught = False
    for pin in PINS:
        try:
            pin(fwd, bwd)
        except AssertionError:
            caught = True
    assert caught, name


def test_chunked_helpers_match_whole_problem():
    h, w, t, dloss = rand_case(N=9, Dm=4, V=37, seed=5)
    chunk = lambda v0, v1: w[v0:v1]  # noqa: E731
    loss, lse = L.forward(h, w, t)
    dh, dw = L.backward(h, w, t, lse, dloss)
    rows = np.array([0, 1, 5, 8])
    l2, lse2 = L.forward_rows(h[rows], t[rows], chunk, 37)
    np.testing.assert_allclose(l2, loss[rows], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse2, lse[rows], rtol=1e-13)
    np.testing.assert_allclose(L.dhidden_rows(h[rows], t[rows], dloss[rows], chunk, 37, chunk=10), dh[rows],
                               rtol=1e-12, atol=1e-13)
    ent = [0, 3, 36]
    np.testing.assert_allclose(L.dweight_entries(h, t, dloss, chunk, 37, ent), dw[ent], rtol=1e-12, atol=1e-13)
    g = L.grad_logits(h, w, t, lse, dloss)
    np.testing.assert_allclose(L.grad_logits_rows(h[rows], t[rows], dloss[rows], chunk, 37, chunk=10), g[rows],
                               rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(L.grad_logits_entries(h, t, dloss, chunk, 37, ent), g[:, ent], rtol=1e-12,
                               atol=1e-14)
    np.testing.assert_allclose(L.lse_rows(h, chunk, 37, block=4), lse, rtol=1e-13)
