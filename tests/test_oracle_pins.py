"""The oracle against facts outside itself (runs on the CPU)."""
import math

import numpy as np
import pytest

import oracle
import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, orc):
    pin(orc)


def test_sketch_is_unbiased_on_average(orc):
    """With P ~ N(0, 1/r), E[(qP).(kP)] = q.k; the mean over many P must land near q.k.

    A statistical sanity check of the projection's shape and scale, not a parity check.
    """
    rng = np.random.default_rng(2024)
    hd, r, draws = 64, 32, 400
    q = rng.standard_normal(hd)
    k = q * 0.6 + rng.standard_normal(hd) * 0.8
    qb, kb = pins.to_bf16_bits(q), pins.to_bf16_bits(k)
    qf, kf = pins.from_bf16_bits(qb), pins.from_bf16_bits(kb)
    exact = float(qf @ kf)
    est = []
    for _ in range(draws):
        P = pins.bf16_normal_bits(rng, (hd, r), std=1 / math.sqrt(r))
        qp = pins.from_bf16_bits(oracle.project_q(qb.reshape(1, hd), P, L=orc))[0]
        A = np.zeros((1, 1, 1, 1, r), dtype=np.uint16)
        oracle.project_kv_blocks(P, kb.reshape(1, 1, 1, hd), 0, np.array([0]), A, L=orc)
        est.append(float(qp @ pins.from_bf16_bits(A[0, 0, 0, 0])))
    est = np.array(est)
    sigma = math.sqrt((float(qf @ qf) * float(kf @ kf) + exact ** 2) / r / draws)
    assert abs(est.mean() - exact) < 5 * sigma, (est.mean(), exact, sigma)


def test_threads_do_not_change_results(orc):
    rng = np.random.default_rng(4)
    nq, nkv, hd, r, bs, pool = 8, 4, 64, 32, 16, 37
    P = pins.bf16_normal_bits(rng, (hd, r), std=1 / math.sqrt(r))
    K = pins.bf16_normal_bits(rng, (pool, bs, nkv, hd))
    Q = pins.bf16_normal_bits(rng, (3, 2, nq, hd))
    A1 = np.zeros((2, pool, nkv, bs, r), dtype=np.uint16)
    A4 = np.zeros_like(A1)
    ids = rng.permutation(pool).astype(np.int32)
    oracle.project_kv_blocks(P, K, 1, ids, A1, nthreads=1, L=orc)
    oracle.project_kv_blocks(P, K, 1, ids, A4, nthreads=4, L=orc)
    assert np.array_equal(A1, A4)
    q1 = oracle.project_q(Q, P, nthreads=1, L=orc)
    assert np.array_equal(q1, oracle.project_q(Q, P, nthreads=3, L=orc))
    table = rng.permutation(pool).astype(np.int32)
    offs = np.array([0, 10, 11, 37])
    s1 = oracle.score_blocks(q1, A1, 1, table, offs, nthreads=1, L=orc)
    s4 = oracle.score_blocks(q1, A1, 1, table, offs, nthreads=4, L=orc)
    assert np.array_equal(s1[0], s4[0]) and np.array_equal(s1[1], s4[1])
    ent = np.array([36, 0, 10, 11, 5])
    se, te, _ = oracle.score_entries(q1, A1, 1, table, offs, ent, L=orc)
    assert np.array_equal(se, s1[0][ent]) and np.array_equal(te, s1[1][ent])
