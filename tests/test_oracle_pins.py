"""The CPU oracle against what the pages and the mathematics fix (no GPU needed)."""
import numpy as np
import pytest

import _pins


def test_worked_counter_example():
    _pins.check_worked_counter_example()


def test_p_equals_q_accepts_every_draft():
    _pins.check_p_equals_q_accepts_all()


def test_greedy_matches_brute_force():
    _pins.check_greedy_brute_force()


def test_grammar_invariants():
    _pins.check_grammar_invariants()


def test_softmax_matches_library():
    _pins.check_softmax_matches_library()


def test_chi_square_losslessness():
    res = _pins.check_chi_square()
    assert len(res) == 5


def test_strict_accept_comparison():
    _pins.check_strict_accept_comparison()


def test_edge_cases():
    _pins.check_edge_cases()


def test_residual_excludes_draft():
    _pins.check_residual_excludes_draft()


def test_telemetry_by_position():
    _pins.check_telemetry()


def test_ngram_proposer():
    _pins.check_ngram_proposer()


def test_bitmask_scatter():
    _pins.check_bitmask_scatter()


def test_top_k_top_p():
    res = _pins.check_top_k_top_p()
    assert len(res) == 4
