"""The acceptance rule the bench uses to check the config-4 step against
the kernel's own logits, pinned to the oracle's greedy verify."""
import numpy as np

import bench
from lossless_bit_weight_w12_gb300 import synth


def test_accept_rule_matches_oracle(oracle):
    for seed, (R, T, V) in enumerate([(1, 16, 500), (4, 16, 3000), (3, 5, 77), (2, 1, 40), (8, 16, 1000)]):
        rng = synth.streams(900 + seed, 2)
        lg = synth.logits(rng[0], R * T, V)
        g = np.argmax(lg, axis=1).reshape(R, T)
        draft = synth.draft_tokens(rng[1], g, R, T, V)
        acc, nxt = bench.accept_rule(g, draft)
        want = oracle.verify_greedy(lg, R, T, draft)
        assert acc.tolist() == want[0].tolist(), (R, T, V)
        assert nxt.tolist() == want[1].tolist(), (R, T, V)


def test_accept_rule_hand_cases():
    g = np.array([[5, 6, 7, 8]])
    assert [x.tolist() for x in bench.accept_rule(g, np.array([[5, 6, 7]]))] == [[3], [8]]  # all accepted
    assert [x.tolist() for x in bench.accept_rule(g, np.array([[5, 9, 7]]))] == [[1], [6]]  # first miss at 1
    assert [x.tolist() for x in bench.accept_rule(g, np.array([[0, 6, 7]]))] == [[0], [5]]  # immediate reject
