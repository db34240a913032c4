"""CPU checks of the parity harness itself (no GPU)."""

import numpy as np

import layer_harness as H
import oracle_io as oio


def test_flip_bound_fast_matches_exact_on_tiny_shapes():
    """The batched single-decision bound equals (or, taking both rounding
    directions, exceeds) the one computed by recomputing each token."""
    work, Wn = H.prepare("tiny_layer", "cpu", T=6, ctx=40)
    ref = H.oracle_single_layer(work, Wn=Wn)
    exact = oio.flip_tolerance(work["cfgs"][0], Wn, ref)
    fast = oio.flip_tolerance_fast(work["cfgs"][0], Wn, ref)
    assert np.all(fast >= exact - 1e-12)
    assert np.all(fast > 0)


def test_ulp_floor_and_bound():
    ref = np.array([1.0, 5.0, 9.0, -12.0])
    assert np.array_equal(H.bf16_ulp(ref), [2 ** -7, 2 ** -5, 2 ** -4, 2 ** -4])
    got = ref + np.array([0.0, 0.0, 2 ** -4, 0.0])
    H.assert_close("x", got, ref)             # one ulp at |x| in [8, 16) is admissible


def test_router_check_accepts_reordered_ties_only():
    logits = np.zeros((1, 6), dtype=np.float32)
    logits[0, :4] = [3.0, 2.0, 2.0000002, 1.0]
    r_idx = np.array([[0, 2, 1]])                      # oracle order
    r_w = np.array([[0.5, 0.3, 0.2]])
    # sum |h w| = 0.01 per logit: slack = 2 (32 u 0.01 + u 2) = 2.6e-7
    abs_sum = np.full((1, 6), 0.01)
    # the two near-equal logits (2e-7 apart) swapped: admissible
    H.check_router(np.array([[0, 1, 2]]), np.array([[0.5, 0.2, 0.3]]), r_idx, r_w, logits, abs_sum)
    # with larger products the slack grows, but stays far below 1: still admissible
    H.check_router(np.array([[0, 1, 2]]), np.array([[0.5, 0.2, 0.3]]), r_idx, r_w, logits,
                   np.full((1, 6), 40.0))
    # a clearly larger logit placed after a smaller one: rejected
    try:
        H.check_router(np.array([[1, 0, 2]]), np.array([[0.2, 0.5, 0.3]]), r_idx, r_w, logits, abs_sum)
    except AssertionError:
        pass
    else:
        raise AssertionError("a reordering of clearly separated logits must be rejected")
    # a different set: rejected
    try:
        H.check_router(np.array([[0, 2, 3]]), np.array([[0.5, 0.3, 0.2]]), r_idx, r_w, logits, abs_sum)
    except AssertionError:
        return
    raise AssertionError("a different expert set must be rejected")
