"""Pins of the oracle's next steps: bias routing ([P1] §4.3), masked P_i
([P2] §3.1) and the full backward through the gates."""

import pins
from oracle import router as R
from oracle import routing_ext as X


def test_biased_topk_bruteforce():
    pins.check_biased_topk_bruteforce(X)


def test_biased_topk_dominant_bias():
    pins.check_biased_topk_dominant(X)


def test_biased_selection_is_an_fp32_sum():
    pins.check_biased_sum_is_fp32(X)


def test_bias_update_hand_case():
    pins.check_bias_update_hand(X)


def test_bias_update_balances_a_skewed_batch():
    pins.check_bias_update_balances(X, R)


def test_masked_p_closed_forms():
    pins.check_masked_p_closed_forms(X, R)


def test_full_backward_finite_differences():
    pins.check_full_grad_finite_difference(X, R)


def test_full_backward_structure():
    pins.check_full_grad_structure(X, R)


def test_masked_p_hand_case():
    pins.check_masked_p_hand(X, R)


def test_softmax_backward_matches_autograd():
    pins.check_softmax_backward_autograd(X)


def test_grad_wrt_probs_finite_differences():
    pins.check_grad_wrt_probs_finite_difference(X, R)


def test_forward_ex_reduces_to_the_plain_forward():
    pins.check_forward_ex_reductions(X, R)
