"""The near-tie protocol used by the GPU parity tests accepts exactly the
valid alternatives: a different choice at a cut with key gap < 1e-5, or a
different order of two selected keys closer than 1e-5; anything else fails.
CPU only (the "GPU" ids here are hand-made)."""
import numpy as np
import pytest

import oracle
from parity import routing_force_mask, topk_choice_problems


def _route(logits, k, bias=None):
    return oracle.route(np.asarray(logits, np.float64), k, bias)


def test_identical_ids_force_nothing():
    r = _route([[3.0, 1.0, 0.0, -1.0], [0.0, 2.0, 1.0, 0.5]], 2)
    assert not routing_force_mask(r, r.ids.copy(), None).any()


def test_cut_tie_is_exempt():
    # experts 1 and 2 tie at the cut (k = 2): either choice is valid
    r = _route([[3.0, 1.0, 1.0 + 1e-9, -1.0]], 2)
    gpu = np.array([[0, 1]], np.int32)
    assert routing_force_mask(r, gpu, None).tolist() == [True]


def test_order_swap_inside_the_set_is_accepted_only_for_near_equal_keys():
    r = _route([[2.0, 2.0 + 1e-8, 0.0, -1.0]], 2)
    assert routing_force_mask(r, np.array([[0, 1]], np.int32), None).tolist() == [True]
    r2 = _route([[2.0, 3.0, 0.0, -1.0]], 2)
    with pytest.raises(AssertionError):
        routing_force_mask(r2, np.array([[0, 1]], np.int32), None)


def test_wrong_set_fails():
    r = _route([[3.0, 1.0, 0.0, -1.0]], 2)
    with pytest.raises(AssertionError):
        routing_force_mask(r, np.array([[0, 2]], np.int32), None)


def test_bias_enters_the_keys():
    # with a bias the selection keys are p + b; a swap is judged on those keys
    logits = [[1.0, 1.0, 0.0, 0.0]]
    bias = np.array([0.0, 0.0, 0.3, 0.3 + 1e-9], np.float32)
    r = _route(logits, 2, bias)
    gpu = r.ids[:, ::-1].copy()
    assert routing_force_mask(r, gpu, bias).tolist() == [True]


@pytest.mark.parametrize("gpu", [[0, 3],      # an expert far below the cut
                                 [0, 0],      # a repeated expert
                                 [0, 7],      # an expert that does not exist
                                 [1, 0],      # the set's keys out of order by far
                                 [2, 0]])
def test_near_tie_token_still_needs_a_valid_choice(gpu):
    # experts 1 and 2 tie at the cut, so the token is exempt from bit-exactness,
    # but the GPU's choice must still be a Top-2 of the keys within 1e-5
    r = _route([[3.0, 1.0, 1.0 + 1e-9, -1.0]], 2)
    assert r.gap[0] < 1e-5
    with pytest.raises(AssertionError):
        routing_force_mask(r, np.array([gpu], np.int32), None)


def test_topk_choice_problems_on_hand_keys():
    key = np.array([0.5, 0.2, 0.2 + 5e-6, 0.1])
    assert topk_choice_problems(key, [0, 2], 2) == []
    assert topk_choice_problems(key, [0, 1], 2) == []          # the tie at the cut
    assert topk_choice_problems(key, [0, 3], 2)                 # 0.1 < 0.2 - 1e-5
    assert topk_choice_problems(key, [2, 0], 2)                 # order reversed by 0.3
    assert topk_choice_problems(key, [0], 2)                    # too few
    assert topk_choice_problems(key, [0, 1, 2, 3], 4) == []     # k = E: every expert
