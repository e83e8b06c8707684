"""Pins that tie the CPU oracle to facts outside itself.

Each pin takes the oracle library handle ``L`` so that the same checks can be
run against deliberately mutated copies of the oracle (see
test_oracle_mutants.py): a plausible slip anywhere in the oracle must make at
least one pin fail.

What the pins compare against (never the oracle's own formulas):
  * PyTorch's binary32 -> bf16 conversion (round to nearest even), a library
    routine, and hand-known bf16 bit patterns;
  * a brute-force full Q.K^T in numpy when P is the identity (r = head_dim),
    and when P selects coordinates (r < head_dim, P not symmetric);
  * a hand-worked three-block example (tests/golden/hand_three_block.json);
  * invariants: block-table permutation, exact power-of-two linearity;
  * hand-written victim orders with ties, signed zeros, NaN and k > n.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------- helpers
# Conversions done by numpy / torch, never by the oracle.

def to_bf16_bits(x) -> np.ndarray:
    """float values -> bf16 bit patterns via PyTorch (round to nearest even)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def from_bf16_bits(b) -> np.ndarray:
    """bf16 bit patterns -> float64 via numpy bit casting."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_normal_bits(rng: np.random.Generator, shape, std=1.0) -> np.ndarray:
    return to_bf16_bits(rng.standard_normal(shape) * std)


def brute_force_scores(Qv, Kv_by_id, table, seq_offsets, nkv):
    """max over rows, heads h and tokens t of q[row,h] . k[id][t, h // g] (numpy, fp64).

    Qv       [S, R, nq, e] float64 (e = the compared coordinates)
    Kv_by_id {id: [bs, nkv, e] float64}
    """
    S, R, nq, _ = Qv.shape
    g = nq // nkv
    out = []
    for s in range(S):
        for i in range(int(seq_offsets[s]), int(seq_offsets[s + 1])):
            kb = Kv_by_id[int(table[i])]
            best = -math.inf
            for h in range(nq):
                # Full products of every query row of head h with every token of its kv head.
                full = Qv[s, :, h, :] @ kb[:, h // g, :].T
                best = max(best, float(full.max()))
            out.append(best)
    return np.array(out)


# ----------------------------------------------------------------------------- bf16 rounding

def pin_bf16_hand_values(L):
    cases = [
        (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
        (1.0 + 2.0 ** -8, 0x3F80),                   # tie -> even (down)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),               # tie -> even (up)
        (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),      # just above a tie: must not double-round
        (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
        (2.0 ** -127, 0x0040),                       # bf16 subnormal
        (2.0 ** -134, 0x0000),                       # half the smallest subnormal: tie -> 0
        (3 * 2.0 ** -134, 0x0002),                   # 1.5 spacings -> even (2)
        (float.fromhex("0x1.FEp127"), 0x7F7F),       # largest finite
        (float.fromhex("0x1.FFp127"), 0x7F80),       # tie above the largest: even is +inf
        (math.inf, 0x7F80), (-math.inf, 0xFF80),
    ]
    got = oracle.bf16_from_double(np.array([c[0] for c in cases]), L=L)
    exp = np.array([c[1] for c in cases], dtype=np.uint16)
    assert np.array_equal(got, exp), (got, exp)
    assert (oracle.bf16_from_double([math.nan], L=L)[0] & 0x7FFF) > 0x7F80


def pin_bf16_matches_torch(L):
    """On every binary32 input the oracle's rounding equals PyTorch's f32 -> bf16."""
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([bits, np.arange(0, 70_000, dtype=np.uint32),       # subnormals
                           np.arange(0x7F7F0000, 0x7F800000, 7, dtype=np.uint32)])  # near max
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    exp = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_from_double(f.astype(np.float64), L=L)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at {f[bad[0]]!r}"
    back = oracle.bf16_to_double(exp, L=L)
    assert np.array_equal(back, from_bf16_bits(exp))


def pin_projection_single_rounding(L):
    """Every projection sums in more precision than binary32 and rounds once, to bf16.

    Hand case: a key/query row [1, 2^-8, 2^-30, 0, ...] against P columns of +-1 on the
    first three coordinates.  The exact sum 1 + 2^-8 + 2^-30 lies just above the midpoint
    between the bf16 neighbours 1 (0x3F80) and 1 + 2^-7 (0x3F81), so it rounds up to 0x3F81
    (and its negative to 0xBF81).  A binary32 running sum drops the 2^-30 term (it is below
    half a binary32 step at 1) and lands on the midpoint itself, which ties to even: 0x3F80.
    Rounding the exact sum to binary32 first does the same.  The row 1 + 2^-8 - 2^-30 lies
    just below the midpoint (0x3F80 either way), and 2^-30 alone is 0x3080.
    Checked through all three projections: queries, key blocks and key tokens.
    """
    hd, r, bs = 16, 4, 2
    row = np.zeros(hd)
    row[:3] = [1.0, 2.0 ** -8, 2.0 ** -30]
    Pf = np.zeros((hd, r))
    Pf[:3, 0] = 1.0
    Pf[:3, 1] = -1.0
    Pf[:3, 2] = [1.0, 1.0, -1.0]
    Pf[2, 3] = 1.0
    P = to_bf16_bits(Pf)
    # The row's entries are powers of two: exact in bf16.
    assert np.array_equal(from_bf16_bits(to_bf16_bits(row)), row)
    exp = np.array([0x3F81, 0xBF81, 0x3F80, 0x3080], dtype=np.uint16)
    rev = row.copy()
    rev[:3] = row[2::-1]                       # the same terms in reverse order
    Prev = to_bf16_bits(Pf[[2, 1, 0] + list(range(3, hd))])
    Q = to_bf16_bits(np.stack([row, row]))
    qp = oracle.project_q(Q, P, L=L)
    assert np.array_equal(qp[0], exp) and np.array_equal(qp[1], exp), qp
    qp_rev = oracle.project_q(to_bf16_bits(rev[None]), Prev, L=L)
    assert np.array_equal(qp_rev[0], exp), qp_rev
    # Key block: both tokens of the one kv head carry the row (second one negated).
    K = to_bf16_bits(np.stack([row, -row])[None, :, None, :])      # [1, bs, 1, hd]
    A = np.zeros((1, 1, 1, bs, r), dtype=np.uint16)
    assert oracle.project_kv_blocks(P, K, 0, np.array([0], dtype=np.int32), A, L=L) == 0
    assert np.array_equal(A[0, 0, 0, 0], exp), A[0, 0, 0, 0]
    assert np.array_equal(A[0, 0, 0, 1], exp ^ 0x8000), A[0, 0, 0, 1]
    # Key tokens: the same two rows written one token at a time, in reverse slot order.
    A_t = np.zeros_like(A)
    K_tok = to_bf16_bits(np.stack([-row, row])[:, None, :])        # [2, 1, hd]
    assert oracle.write_kv_tokens(P, K_tok, np.array([1, 0]), 0, A_t, L=L) == 0
    assert np.array_equal(A_t, A), A_t


# ----------------------------------------------------------------------------- method pins

def _grid_case(rng, *, nq, nkv, hd, bs, S, R, lengths, layers, layer, pool):
    total = sum(lengths)
    ids = rng.permutation(pool)[:pool].astype(np.int32)
    K = bf16_normal_bits(rng, (pool, bs, nkv, hd))
    Q = bf16_normal_bits(rng, (S, R, nq, hd))
    table = rng.permutation(pool)[:total].astype(np.int32)
    offs = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return Q, K, ids, table, offs


def pin_identity_projection_brute_force(L):
    """P = I (r = head_dim): Qp = Q and A_g = K exactly; scores = max of the full Q.K^T."""
    rng = np.random.default_rng(7)
    nq, nkv, hd, bs, S, R = 4, 2, 64, 16, 2, 3
    lengths, layers, layer, pool = [5, 9], 3, 2, 16
    Q, K, ids, table, offs = _grid_case(rng, nq=nq, nkv=nkv, hd=hd, bs=bs, S=S, R=R,
                                        lengths=lengths, layers=layers, layer=layer, pool=pool)
    P = to_bf16_bits(np.eye(hd))
    Qp = oracle.project_q(Q, P, L=L)
    assert np.array_equal(Qp, Q)
    A = np.zeros((layers, pool, nkv, bs, hd), dtype=np.uint16)
    assert oracle.project_kv_blocks(P, K, layer, ids, A, L=L) == 0
    for i, bid in enumerate(ids):
        assert np.array_equal(A[layer, bid], K[i].transpose(1, 0, 2)), "slot != K^T"
    assert not A[:layer].any() and not A[layer + 1:].any(), "wrote another layer"
    score, tsum, bad = oracle.score_blocks(Qp, A, layer, table, offs, L=L)
    assert bad == 0
    Kd = {int(bid): from_bf16_bits(K[i]) for i, bid in enumerate(ids)}
    exp = brute_force_scores(from_bf16_bits(Q), Kd, table, offs, nkv)
    assert np.array_equal(score, exp), np.max(np.abs(score - exp))
    assert np.all(tsum >= np.abs(score))


def pin_selection_projection_brute_force(L):
    """P selects r of head_dim coordinates (times 2): a non-symmetric, non-square P."""
    rng = np.random.default_rng(11)
    nq, nkv, hd, r, bs, S, R = 6, 3, 48, 16, 4, 3, 2
    lengths, layers, layer, pool = [4, 1, 6], 2, 1, 12
    Q, K, ids, table, offs = _grid_case(rng, nq=nq, nkv=nkv, hd=hd, bs=bs, S=S, R=R,
                                        lengths=lengths, layers=layers, layer=layer, pool=pool)
    sel = rng.permutation(hd)[:r]
    Pf = np.zeros((hd, r))
    Pf[sel, np.arange(r)] = 2.0
    P = to_bf16_bits(Pf)
    Qp = oracle.project_q(Q, P, L=L)
    assert np.array_equal(from_bf16_bits(Qp), 2.0 * from_bf16_bits(Q)[..., sel])
    A = np.zeros((layers, pool, nkv, bs, r), dtype=np.uint16)
    assert oracle.project_kv_blocks(P, K, layer, ids, A, L=L) == 0
    Kf = from_bf16_bits(K)
    for i, bid in enumerate(ids):
        assert np.array_equal(from_bf16_bits(A[layer, bid]),
                              2.0 * Kf[i][..., sel].transpose(1, 0, 2))
    score, _, bad = oracle.score_blocks(Qp, A, layer, table, offs, L=L)
    Kd = {int(bid): 2.0 * Kf[i][..., sel] for i, bid in enumerate(ids)}
    exp = brute_force_scores(2.0 * from_bf16_bits(Q)[..., sel], Kd, table, offs, nkv)
    assert bad == 0 and np.array_equal(score, exp)


def pin_gqa_contiguous_groups(L):
    """Query head h reads kv head h // g: a case where h % nkv would give another score."""
    nq, nkv, hd, bs = 4, 2, 16, 16
    P = to_bf16_bits(np.eye(hd))
    Q = np.zeros((1, 1, nq, hd))
    Q[0, 0, 2, 0] = Q[0, 0, 3, 0] = 1.0         # heads 2, 3 (group of kv head 1)
    K = np.zeros((1, bs, nkv, hd))
    K[0, :, 0, 0] = 4.0                         # kv head 0: large, read only by heads 0, 1
    K[0, 5, 1, 0] = 1.0                         # kv head 1: one token with a 1
    A = np.zeros((1, 1, nkv, bs, hd), dtype=np.uint16)
    oracle.project_kv_blocks(P, to_bf16_bits(K), 0, np.array([0]), A, L=L)
    score, _, _ = oracle.score_blocks(oracle.project_q(to_bf16_bits(Q), P, L=L), A, 0,
                                      np.array([0]), np.array([0, 1]), L=L)
    assert score[0] == 1.0, score


def pin_hand_example(L):
    g = json.load(open(os.path.join(GOLDEN, "hand_three_block.json")))
    d = g["dims"]
    P = to_bf16_bits(g["P"])
    Q = to_bf16_bits(np.array(g["Q"], dtype=np.float64).reshape(1, 1, d["num_q_heads"],
                                                                  d["head_dim"]))
    K = to_bf16_bits(g["K"])
    Qp = oracle.project_q(Q, P, L=L)
    assert np.array_equal(from_bf16_bits(Qp).reshape(d["num_q_heads"], d["r"]),
                          np.array(g["expected_Qp"], dtype=np.float64))
    A = np.zeros((1, d["max_blocks"], d["num_kv_heads"], d["block_size"], d["r"]),
                 dtype=np.uint16)
    assert oracle.project_kv_blocks(P, K, 0, np.arange(d["max_blocks"]), A, L=L) == 0
    assert np.array_equal(from_bf16_bits(A[0]), np.array(g["expected_A_g_slots"]))
    for c in g["cases"]:
        offs = np.array(c["seq_offsets"])
        S = len(offs) - 1
        QpS = np.repeat(Qp, S, axis=0)
        score, _, bad = oracle.score_blocks(QpS, A, 0, np.array(c["table"]), offs, L=L)
        assert bad == 0 and np.array_equal(score, np.array(c["expected_scores"], dtype=float))
        vic = oracle.rank_victims(score.astype(np.float32), offs, c["k"], L=L)
        assert np.array_equal(vic, np.array(c["expected_victims"])), (vic, c)


def pin_table_permutation(L):
    """Permuting a sequence's table permutes its scores the same way."""
    rng = np.random.default_rng(5)
    nq, nkv, hd, r, bs, pool = 8, 2, 32, 16, 16, 40
    P = bf16_normal_bits(rng, (hd, r), std=1 / math.sqrt(r))
    K = bf16_normal_bits(rng, (pool, bs, nkv, hd))
    Q = bf16_normal_bits(rng, (2, 2, nq, hd))
    A = np.zeros((1, pool, nkv, bs, r), dtype=np.uint16)
    oracle.project_kv_blocks(P, K, 0, np.arange(pool), A, L=L)
    Qp = oracle.project_q(Q, P, L=L)
    table = rng.permutation(pool)[:30].astype(np.int32)
    offs = np.array([0, 13, 30])
    base, _, _ = oracle.score_blocks(Qp, A, 0, table, offs, L=L)
    perm = np.concatenate([rng.permutation(13), 13 + rng.permutation(17)])
    moved, _, _ = oracle.score_blocks(Qp, A, 0, table[perm], offs, L=L)
    assert np.array_equal(moved, base[perm])
    k = 6
    v0 = oracle.rank_victims(base.astype(np.float32), offs, k, L=L)
    v1 = oracle.rank_victims(moved.astype(np.float32), offs, k, L=L)
    for s in range(2):
        a, b = offs[s], offs[s + 1]
        # The permuted table's victim j is entry perm[a + j] of the original table.
        mapped = perm[a + v1[s]] - a
        assert sorted(mapped.tolist()) == sorted(v0[s].tolist())


def pin_linearity(L):
    """Doubling K doubles A_g exactly; doubling Q doubles Qp; scores scale by 2 and 4."""
    rng = np.random.default_rng(9)
    nq, nkv, hd, r, bs, pool = 4, 2, 32, 16, 16, 8
    P = bf16_normal_bits(rng, (hd, r), std=1 / math.sqrt(r))
    K = bf16_normal_bits(rng, (pool, bs, nkv, hd))
    Q = bf16_normal_bits(rng, (1, 1, nq, hd))
    K2 = to_bf16_bits(2.0 * from_bf16_bits(K))
    Q2 = to_bf16_bits(2.0 * from_bf16_bits(Q))
    A1 = np.zeros((1, pool, nkv, bs, r), dtype=np.uint16)
    A2 = np.zeros_like(A1)
    oracle.project_kv_blocks(P, K, 0, np.arange(pool), A1, L=L)
    oracle.project_kv_blocks(P, K2, 0, np.arange(pool), A2, L=L)
    assert np.array_equal(from_bf16_bits(A2), 2.0 * from_bf16_bits(A1))
    q1 = oracle.project_q(Q, P, L=L)
    q2 = oracle.project_q(Q2, P, L=L)
    assert np.array_equal(from_bf16_bits(q2), 2.0 * from_bf16_bits(q1))
    t, offs = np.arange(pool), np.array([0, pool])
    s11, _, _ = oracle.score_blocks(q1, A1, 0, t, offs, L=L)
    s12, _, _ = oracle.score_blocks(q1, A2, 0, t, offs, L=L)
    s22, _, _ = oracle.score_blocks(q2, A2, 0, t, offs, L=L)
    assert np.array_equal(s12, 2.0 * s11) and np.array_equal(s22, 4.0 * s11)


def pin_out_of_range(L):
    """Bad layer: nothing written; bad block id: skipped, reported, scored +inf."""
    rng = np.random.default_rng(3)
    P = bf16_normal_bits(rng, (16, 16))
    K = bf16_normal_bits(rng, (3, 16, 1, 16))
    A = np.zeros((2, 4, 1, 16, 16), dtype=np.uint16)
    assert oracle.project_kv_blocks(P, K, 2, np.array([0, 1, 2]), A, L=L) == -1
    assert not A.any()
    assert oracle.project_kv_blocks(P, K, 1, np.array([0, 4, 2]), A, L=L) == 2
    assert A[1, 0].any() and A[1, 2].any() and not A[1, 1].any() and not A[0].any()
    Qp = bf16_normal_bits(rng, (1, 1, 1, 16))
    score, tsum, bad = oracle.score_blocks(Qp, A, 1, np.array([0, -1, 4, 2]),
                                           np.array([0, 4]), L=L)
    assert bad == 2 and math.isinf(score[1]) and math.isinf(score[2])
    assert np.isfinite(score[[0, 3]]).all() and tsum[1] == 0.0


def pin_victim_order(L):
    """Hand-written victim orders: ties, signed zeros, NaN, +-inf, k > n, empty sequences."""
    nan, inf = math.nan, math.inf
    scores = np.array([
        3.0, 1.0, 1.0, -2.0, 0.0, -0.0, 5.0,      # seq 0 (7 entries)
        nan, inf, -inf, 2.0,                       # seq 1 (4 entries)
                                                   # seq 2 (empty)
        0.5, 0.5, 0.5,                             # seq 3 (3 entries)
    ], dtype=np.float32)
    offs = np.array([0, 7, 11, 11, 14])
    k = 5
    exp = np.array([
        [3, 4, 5, 1, 2],           # -2, then 0 / -0 (equal: lower index first), then 1, 1
        [2, 3, 0, 1, -1],          # -inf, 2, NaN (as +inf, index 0) before +inf (index 1)
        [-1, -1, -1, -1, -1],
        [0, 1, 2, -1, -1],
    ])
    got = oracle.rank_victims(scores, offs, k, L=L)
    assert np.array_equal(got, exp), got


def pin_victims_brute_force(L):
    """Victims equal a plain Python sort of (score, index) on random data with ties."""
    rng = np.random.default_rng(21)
    lengths = [0, 1, 17, 64, 300]
    offs = np.concatenate([[0], np.cumsum(lengths)])
    s = np.round(rng.standard_normal(offs[-1]) * 4).astype(np.float32)  # many exact ties
    k = 20
    got = oracle.rank_victims(s, offs, k, L=L)
    for si in range(len(lengths)):
        seg = s[offs[si]:offs[si + 1]]
        order = sorted(range(len(seg)), key=lambda i: (float(seg[i]), i))[:k]
        exp = order + [-1] * (k - len(order))
        assert got[si].tolist() == exp


def _masked_case(rng, *, nq=4, nkv=2, hd=32, bs=4, S=3, R=3, lengths=(5, 0, 7), pool=16):
    Q, K, ids, table, offs = _grid_case(rng, nq=nq, nkv=nkv, hd=hd, bs=bs, S=S, R=R,
                                        lengths=list(lengths), layers=1, layer=0, pool=pool)
    P = to_bf16_bits(np.eye(hd))
    A = np.zeros((1, pool, nkv, bs, hd), dtype=np.uint16)
    return Q, K, ids, table, offs, P, A


def pin_masked_brute_force(L):
    """Length and causal masks against a numpy brute force over explicit token positions."""
    rng = np.random.default_rng(31)
    nq, nkv, hd, bs, S, R = 4, 2, 32, 4, 3, 3
    Q, K, ids, table, offs, P, A = _masked_case(rng, nq=nq, nkv=nkv, hd=hd, bs=bs, S=S, R=R)
    oracle.project_kv_blocks(P, K, 0, ids, A, L=L)
    Qp = oracle.project_q(Q, P, L=L)
    ctx = np.array([17, 3, 25])          # seq 0: 5 blocks = 20 tokens, 17 valid
    pos0 = np.array([9, 0, 12])
    Kd = {int(b): from_bf16_bits(K[i]) for i, b in enumerate(ids)}
    Qf = from_bf16_bits(Q)
    g = nq // nkv
    for use_len, use_causal in ((True, False), (False, True), (True, True)):
        got, _, _ = oracle.score_blocks_masked(Qp, A, 0, table, offs,
                                               ctx_len=ctx if use_len else None,
                                               row_pos0=pos0 if use_causal else None, L=L)
        exp = []
        for sq in range(S):
            for i in range(int(offs[sq]), int(offs[sq + 1])):
                j = i - int(offs[sq])
                kb = Kd[int(table[i])]
                best = -math.inf
                for row in range(R):
                    for h in range(nq):
                        for t in range(bs):
                            p = j * bs + t
                            if use_len and p >= ctx[sq]:
                                continue
                            if use_causal and p > pos0[sq] + row:
                                continue
                            best = max(best, float(Qf[sq, row, h] @ kb[t, h // g]))
                exp.append(best)
        assert np.array_equal(got, np.array(exp)), (use_len, use_causal)


def pin_masked_reduces_to_unmasked(L):
    """A length covering every token and row positions past the context change nothing;
    hiding everything gives -inf; a longer context never lowers a score."""
    rng = np.random.default_rng(32)
    Q, K, ids, table, offs, P, A = _masked_case(rng)
    oracle.project_kv_blocks(P, K, 0, ids, A, L=L)
    Qp = oracle.project_q(Q, P, L=L)
    base, tb, _ = oracle.score_blocks(Qp, A, 0, table, offs, L=L)
    lens = np.diff(offs) * 4
    full, tf, _ = oracle.score_blocks_masked(Qp, A, 0, table, offs, ctx_len=lens,
                                             row_pos0=np.full(3, 10 ** 6), L=L)
    assert np.array_equal(full, base) and np.array_equal(tf, tb)
    none, tn, _ = oracle.score_blocks_masked(Qp, A, 0, table, offs, ctx_len=np.zeros(3),
                                             L=L)
    assert np.all(np.isneginf(none)) and not tn.any()
    hidden, _, _ = oracle.score_blocks_masked(Qp, A, 0, table, offs, row_pos0=np.full(3, -3),
                                              L=L)
    assert np.all(np.isneginf(hidden))  # row r sees p <= -3 + r < 0 for r < 3
    prev = None
    for c in range(0, 30, 3):
        cur, _, _ = oracle.score_blocks_masked(Qp, A, 0, table, offs, ctx_len=np.full(3, c),
                                               L=L)
        if prev is not None:
            assert np.all(cur >= prev)
        prev = cur


def pin_masked_hand_case(L):
    """Hand case: block_size 2, two query rows at positions 1 and 2 (causal, row_pos0 = 1).
    Block 0 (positions 0, 1) is seen by both rows; of block 1 (positions 2, 3) only row 1
    sees position 2, and nobody sees position 3."""
    P = to_bf16_bits(np.eye(16))
    Q = np.zeros((1, 2, 1, 16))
    Q[0, :, 0, 0] = 1.0                          # both rows: the first coordinate
    K = np.zeros((2, 2, 1, 16))
    K[0, 0, 0, 0], K[0, 1, 0, 0] = 3.0, -1.0     # block 0 tokens: dots 3, -1
    K[1, 0, 0, 0], K[1, 1, 0, 0] = 0.5, 7.0      # block 1 tokens: dots 0.5 (row 1 only), 7
    A = np.zeros((1, 2, 1, 2, 16), dtype=np.uint16)
    oracle.project_kv_blocks(P, to_bf16_bits(K), 0, np.array([0, 1]), A, L=L)
    Qp = oracle.project_q(to_bf16_bits(Q), P, L=L)
    sc, _, _ = oracle.score_blocks_masked(Qp, A, 0, np.array([0, 1]), np.array([0, 2]),
                                          row_pos0=np.array([1]), L=L)
    assert sc.tolist() == [3.0, 0.5], sc
    sc, _, _ = oracle.score_blocks_masked(Qp, A, 0, np.array([0, 1]), np.array([0, 2]),
                                          ctx_len=np.array([1]), L=L)
    assert sc[0] == 3.0 and math.isinf(sc[1]) and sc[1] < 0
    sc, _, _ = oracle.score_blocks_masked(Qp, A, 0, np.array([1, 0]), np.array([0, 2]),
                                          ctx_len=np.array([3]), L=L)
    assert sc.tolist() == [7.0, 3.0], sc     # table order decides positions


# ----------------------------------------------------------------------------- token ingest

def _token_case(rng, *, nkv=3, hd=48, bs=4, pool=4, layers=2):
    """Fresh keys for every position of every block, in a shuffled token order with two
    padding tokens (slot -1) mixed in.  The token pins keep pool == block_size, so that an
    oracle that swapped block and position would still index inside its arrays (and fail an
    assertion instead of writing out of bounds)."""
    order = rng.permutation(pool * bs)
    slots = np.concatenate([order, [-1, -1]]).astype(np.int64)
    rng.shuffle(slots)
    K_tok = to_bf16_bits(rng.standard_normal((slots.size, nkv, hd)))
    return K_tok, slots


def pin_tokens_identity_brute_force(L):
    """P = I: every token's A_g row is its key row and its cache row a copy, at the position
    its slot names; padding writes nothing; other layers stay untouched."""
    rng = np.random.default_rng(41)
    nkv, hd, bs, pool, layers, layer = 3, 48, 4, 4, 3, 1
    K_tok, slots = _token_case(rng, nkv=nkv, hd=hd, bs=bs, pool=pool, layers=layers)
    P = to_bf16_bits(np.eye(hd))
    A = np.full((layers, pool, nkv, bs, hd), 0x7FC1, dtype=np.uint16)
    C = np.full((pool, bs, nkv, hd), 0x7FC1, dtype=np.uint16)
    assert oracle.write_kv_tokens(P, K_tok, slots, layer, A, K_cache=C, L=L) == 0
    for i, sl in enumerate(slots):
        if sl < 0:
            continue
        blk, t = divmod(int(sl), bs)
        assert np.array_equal(C[blk, t], K_tok[i]), "cache row is not the key row"
        assert np.array_equal(A[layer, blk, :, t], K_tok[i]), "A_g row is not K . I"
    assert (A[0] == 0x7FC1).all() and (A[2] == 0x7FC1).all(), "wrote another layer"


def pin_tokens_selection_projection(L):
    """P selects r coordinates, times 2: A_g rows are exact numpy slices of the keys."""
    rng = np.random.default_rng(43)
    nkv, hd, r, bs, pool = 2, 64, 16, 8, 8
    K_tok, slots = _token_case(rng, nkv=nkv, hd=hd, bs=bs, pool=pool)
    sel = rng.permutation(hd)[:r]
    Pf = np.zeros((hd, r))
    Pf[sel, np.arange(r)] = 2.0
    A = np.zeros((1, pool, nkv, bs, r), dtype=np.uint16)
    assert oracle.write_kv_tokens(to_bf16_bits(Pf), K_tok, slots, 0, A, L=L) == 0
    Kf = from_bf16_bits(K_tok)
    for i, sl in enumerate(slots):
        if sl >= 0:
            blk, t = divmod(int(sl), bs)
            assert np.array_equal(from_bf16_bits(A[0, blk, :, t]), 2.0 * Kf[i][:, sel])


def pin_tokens_equal_block_projection(L):
    """Writing a block's tokens one slot at a time (any order, general P) gives the slot the
    block projection gives; a block written only in part changes only those rows."""
    rng = np.random.default_rng(47)
    nkv, hd, r, bs, pool = 2, 64, 16, 4, 4
    P = to_bf16_bits(rng.standard_normal((hd, r)) / math.sqrt(r))
    Kb = to_bf16_bits(rng.standard_normal((pool, bs, nkv, hd)))
    ids = rng.permutation(pool).astype(np.int32)
    A_blk = np.zeros((1, pool, nkv, bs, r), dtype=np.uint16)
    assert oracle.project_kv_blocks(P, Kb[ids], 0, ids, A_blk, L=L) == 0
    A_tok = np.zeros_like(A_blk)
    order = rng.permutation(pool * bs)
    slots = order.astype(np.int64)
    K_tok = Kb.reshape(pool * bs, nkv, hd)[order]
    assert oracle.write_kv_tokens(P, K_tok, slots, 0, A_tok, L=L) == 0
    assert np.array_equal(A_tok, A_blk)
    part = np.full_like(A_blk, 0x7FC1)
    assert oracle.write_kv_tokens(P, K_tok[:3], slots[:3], 0, part, L=L) == 0
    written = np.zeros((pool, bs), dtype=bool)
    for sl in slots[:3]:
        written[divmod(int(sl), bs)] = True
    for blk in range(pool):
        for t in range(bs):
            row = part[0, blk, :, t]
            if written[blk, t]:
                assert np.array_equal(row, A_blk[0, blk, :, t])
            else:
                assert (row == 0x7FC1).all()


def pin_tokens_out_of_range(L):
    """A slot past the last block is skipped and reported (1-based position); a bad layer
    writes nothing."""
    rng = np.random.default_rng(53)
    nkv, hd, r, bs, pool = 2, 64, 16, 4, 4
    P = to_bf16_bits(rng.standard_normal((hd, r)))
    K_tok = to_bf16_bits(rng.standard_normal((3, nkv, hd)))
    A = np.zeros((1, pool, nkv, bs, r), dtype=np.uint16)
    st = oracle.write_kv_tokens(P, K_tok, np.array([5, pool * bs, -1]), 0, A, L=L)
    assert st == 2
    assert A[0, 1, :, 1].any() and np.count_nonzero(A.reshape(-1, r).any(axis=1)) == nkv
    B = np.zeros_like(A)
    assert oracle.write_kv_tokens(P, K_tok, np.array([0, 1, 2]), 1, B, L=L) == -1
    assert not B.any()


# ----------------------------------------------------------------------------- per-row selection

def pin_rows_identity_brute_force(L):
    """P = I: per-row scores are the per-row max of the full Q.K^T (numpy), exactly; their
    max over rows is the pinned block score; a bad id scores -inf."""
    rng = np.random.default_rng(61)
    nq, nkv, hd, bs, R, pool, n = 6, 2, 32, 4, 5, 9, 7
    P = to_bf16_bits(np.eye(hd))
    Q = bf16_normal_bits(rng, (R, nq, hd))
    K = bf16_normal_bits(rng, (pool, bs, nkv, hd))
    ids = np.arange(pool, dtype=np.int32)
    A = np.zeros((2, pool, nkv, bs, hd), dtype=np.uint16)
    assert oracle.project_kv_blocks(P, K, 1, ids, A, L=L) == 0
    table = rng.permutation(pool)[:n].astype(np.int32)
    score, tsum, bad = oracle.score_rows(Q, A, 1, table, L=L)
    assert bad == 0 and score.shape == (R, n)
    Qf, Kf = from_bf16_bits(Q), from_bf16_bits(K)
    g = nq // nkv
    for row in range(R):
        for j, bid in enumerate(table):
            exp = max(float((Kf[bid][:, h // g, :] @ Qf[row, h]).max()) for h in range(nq))
            assert score[row, j] == exp, (row, j)
    blk, btsum, _ = oracle.score_blocks(Q[None], A, 1, table, np.array([0, n]), L=L)
    assert np.array_equal(score.max(axis=0), blk)
    assert np.array_equal(tsum.max(axis=0), btsum)
    bad_table = table.copy()
    bad_table[2] = pool + 3
    sc2, _, bad2 = oracle.score_rows(Q, A, 1, bad_table, L=L)
    assert bad2 == 1 and np.all(np.isneginf(sc2[:, 2]))


def pin_rows_selection_brute_force(L):
    """Per-row top-k against a plain Python sort (larger first, lower index on ties), over
    the blocks each row has seen whole, with ties, signed zeros and NaN."""
    rng = np.random.default_rng(67)
    rows, n, stride, bs, topk = 9, 13, 16, 4, 5
    sc = rng.integers(-3, 4, size=(rows, stride)).astype(np.float32)  # many ties
    sc[1, 2] = -0.0
    sc[1, 3] = 0.0
    sc[2, 0] = np.nan
    sc[3, :] = np.nan
    for first_pos in (0, 3, 17, 40):
        got = oracle.select_rows(sc, n, first_pos, bs, topk, L=L)
        for r in range(rows):
            complete = min(n, (first_pos + r + 1) // bs)
            key = lambda j: (-math.inf if math.isnan(sc[r, j]) else float(sc[r, j]) + 0.0, -j)
            order = sorted(range(complete), key=key, reverse=True)
            exp = (order + [-1] * topk)[:topk]
            assert got[r].tolist() == exp, (first_pos, r, got[r].tolist(), exp)


def pin_rows_selection_hand_case(L):
    """Block size 4, three blocks with scores 2, 5, 5 (row 0) and 7, 1, 9 (row 1)."""
    sc = np.array([[2.0, 5.0, 5.0], [7.0, 1.0, 9.0]], dtype=np.float32)
    # first_pos 6: row 0 sits at 6 and has seen block 0 whole; row 1 (at 7) blocks 0, 1.
    assert oracle.select_rows(sc, 3, 6, 4, 2, L=L).tolist() == [[0, -1], [0, 1]]
    # first_pos 10: row 0 (at 10) sees blocks 0, 1; row 1 (at 11) all three.
    assert oracle.select_rows(sc, 3, 10, 4, 2, L=L).tolist() == [[1, 0], [2, 0]]
    # Equal scores: the lower index first.
    assert oracle.select_rows(sc, 3, 100, 4, 3, L=L).tolist() == [[1, 2, 0], [2, 0, 1]]


ALL_PINS = [
    pin_bf16_hand_values,
    pin_bf16_matches_torch,
    pin_projection_single_rounding,
    pin_identity_projection_brute_force,
    pin_selection_projection_brute_force,
    pin_gqa_contiguous_groups,
    pin_hand_example,
    pin_table_permutation,
    pin_linearity,
    pin_out_of_range,
    pin_victim_order,
    pin_victims_brute_force,
    pin_masked_brute_force,
    pin_masked_reduces_to_unmasked,
    pin_masked_hand_case,
    pin_tokens_identity_brute_force,
    pin_tokens_selection_projection,
    pin_tokens_equal_block_projection,
    pin_tokens_out_of_range,
    pin_rows_identity_brute_force,
    pin_rows_selection_brute_force,
    pin_rows_selection_hand_case,
]
