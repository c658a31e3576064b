"""The bench's work accounting agrees with the oracle's FLOP convention (which
is pinned to the pages' printed table) and with brute-force pair counts."""

import numpy as np
import pytest

import oracle.attention as A
from bwd_flashattention_fwd_gb300 import flops as F


@pytest.mark.parametrize("Lq,Lk,causal", [(1, 1, True), (5, 9, True), (8, 8, True), (7, 3, False),
                                          (4064, 4112, True), (300, 300, True)])
def test_visible_pairs_brute_force(Lq, Lk, causal):
    assert F.visible_pairs(Lq, Lk, causal) == int(A.visible(Lq, Lk, causal).sum())


def test_visible_pairs_when_queries_outnumber_keys():
    assert F.visible_pairs(9, 4, True) == int(A.visible(9, 4, True).sum())


@pytest.mark.parametrize("shape", [(1, 16, 8192, 8192, 256, True), (2, 32, 2048, 2048, 128, True),
                                   (4, 16, 4064, 4112, 96, True), (1, 2, 100, 100, 64, False)])
def test_credit_matches_oracle_convention(shape):
    assert F.credited_forward(*shape) == A.flops_forward(*shape)
    assert F.credited_fwd_bwd(*shape) == A.flops_fwd_bwd(*shape)


def test_kernel_flops_and_delta_bytes():
    # square causal: pairs = L(L+1)/2; fwd = 2 matmuls of 2*D per pair
    assert F.kernel_flops("fwd", 1, 2, 4, 4, 8, True) == 2 * 8 * 2 * 2 * 10
    assert F.kernel_flops("bwd_dkv", 1, 1, 3, 3, 4, False) == 2 * 4 * 4 * 9
    assert F.delta_bytes(2, 3, 5, 64) == 2 * 30 * 64 * 2 + 4 * 30


@pytest.mark.parametrize("Lq,Lk,causal,seed", [(300, 300, True, 1), (300, 900, True, 2), (500, 260, False, 3),
                                               (1031, 1031, True, 4), (257, 129, False, 5)])
def test_visible_pairs_masked_brute_force(Lq, Lk, causal, seed):
    rng = np.random.default_rng(seed)
    bm = (rng.random((-(-Lq // 128), -(-Lk // 128))) < 0.5).astype(np.uint8)
    assert F.visible_pairs_masked(Lq, Lk, causal, bm) == int(A.visible(Lq, Lk, causal, bm).sum())
    ones = np.ones_like(bm)
    assert F.visible_pairs_masked(Lq, Lk, causal, ones) == F.visible_pairs(Lq, Lk, causal)
