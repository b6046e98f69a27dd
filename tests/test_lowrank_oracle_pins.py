"""Pins of the low-rank bias oracle (``oracle/lowrank.py``) against things other than
itself: one-hot rows that select one coefficient row of the projection, a hand-worked
product, linearity on integers, and a planted transposition that must fail."""
import numpy as np
import pytest

import oracle.lowrank as lr


def bits(x):
    f = np.asarray(x, np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def test_one_hot_r_selects_a_projection_coefficient():
    rng = np.random.default_rng(0)
    for E, d in ((40, 16), (16, 16), (7, 32)):     # a square case catches a transposed use
        proj_t = bits(rng.standard_normal((E, d)))
        for j in (0, 3, d - 1):
            r = np.zeros((2, 3, d))
            r[1, 2, j] = 1.0
            rel = lr.rel_from_lowrank(bits(r), proj_t)
            assert rel.shape == (2, 3, E)
            assert np.array_equal(rel[1, 2], lr.bf16_bits_to_f64(proj_t[:, j]))
            assert not rel[0].any() and not rel[1, :2].any()


def test_hand_worked_product():
    # r = (1, 2), projection rows (c = 0: 1, 0, -1), (c = 1: 3, 0.5, 2):
    # rel = (1*1 + 2*3, 1*0 + 2*0.5, 1*-1 + 2*2) = (7, 1, 3)
    proj = np.array([[1, 0, -1], [3, 0.5, 2]])
    rel = lr.rel_from_lowrank(bits(np.array([[[1, 2]]])), bits(proj.T))
    assert np.array_equal(rel[0, 0], [7, 1, 3])
    rows = lr.rel_rows_from_lowrank(bits(np.array([[1, 2], [0, -1]])), bits(proj.T))
    assert np.array_equal(rows, [[7, 1, 3], [-3, -0.5, -2]])


def test_linear_in_r_exactly_on_integers():
    rng = np.random.default_rng(1)
    d, E = 64, 100
    a = rng.integers(-4, 5, (5, 2, d)).astype(float)
    b = rng.integers(-4, 5, (5, 2, d)).astype(float)
    p = bits(rng.integers(-3, 4, (E, d)).astype(float))
    lhs = lr.rel_from_lowrank(bits(a + b), p)
    rhs = lr.rel_from_lowrank(bits(a), p) + lr.rel_from_lowrank(bits(b), p)
    assert np.array_equal(lhs, rhs)
    # and matches the row form
    assert np.array_equal(lr.rel_rows_from_lowrank(bits(a).reshape(-1, d), p).reshape(5, 2, E),
                          lr.rel_from_lowrank(bits(a), p))


def test_planted_transposition_fails_a_pin():
    src = open(lr.__file__).read()
    mutant = src.replace("proj = bf16_bits_to_f64(proj_t_bits).T            # rel_logits_proj [d_rel, E]",
                         "proj = bf16_bits_to_f64(proj_t_bits)")
    assert mutant != src
    mod = {}
    exec(compile(mutant, "lowrank_mutant", "exec"), mod)

    class M:
        pass
    m = M()
    for k, v in mod.items():
        setattr(m, k, v)
    saved = lr.rel_from_lowrank
    failed = False
    try:
        lr.rel_from_lowrank = m.rel_from_lowrank
        test_one_hot_r_selects_a_projection_coefficient()
    except (AssertionError, ValueError):
        failed = True
    finally:
        lr.rel_from_lowrank = saved
    assert failed
