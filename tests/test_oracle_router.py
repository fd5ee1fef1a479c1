"""Pins of the router oracle (softmax, top-k, gates, f, P, L_aux, CV, gradient)."""

import oracle
import synth
import pins


def test_softmax_matches_library():
    pins.check_softmax_library(oracle.router)


def test_topk_bruteforce_with_ties():
    pins.check_topk_bruteforce(oracle.router)


def test_top1_is_argmax():
    pins.check_top1_argmax(oracle.router)


def test_gate_hand_example():
    pins.check_gate_hand_example(oracle.router)


def test_counts_bruteforce_minlength():
    pins.check_counts_bruteforce(oracle.router)


def test_f_and_P_sum_to_one():
    pins.check_fp_sums(oracle.router, synth)


def test_balance_is_one_with_uniform_P():
    pins.check_balance_uniform_P(oracle.router)


def test_balance_is_one_with_uniform_f():
    pins.check_balance_uniform_f(oracle.router)


def test_switch_two_token_hand_example():
    pins.check_switch_hand_example(oracle.router)


def test_cv_closed_forms():
    pins.check_cv_closed_forms(oracle.router)


def test_tokens_per_expert_log_example():
    pins.check_log_example(oracle.router)


def test_rank_loads_contiguous_hand_case():
    pins.check_rank_loads_contiguous(oracle.router)


def test_batch_scalars_hand_case():
    pins.check_batch_scalars_hand(oracle.router)


def test_cv_grade_bands():
    pins.check_cv_grades(oracle.router)


def test_grad_matches_finite_differences():
    pins.check_grad_finite_difference(oracle.router)


def test_grad_rows_sum_to_zero_and_uniform_case():
    pins.check_grad_structure(oracle.router)


def test_widen_matches_torch_bf16():
    pins.check_widen_library(oracle.router)


def test_balance_degree_and_ratio_flag():
    pins.check_balance_degree_hand(oracle.router)
