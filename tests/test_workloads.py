"""The seeded input generators: deterministic, correctly shaped, structurally valid."""
import torch

import workloads as W


def test_tiny_is_deterministic_and_shaped():
    a, b = W.tiny(seed=0), W.tiny(seed=0)
    for f in ("P", "Q", "K", "table", "seq_offsets", "block_ids"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    assert a.P.shape == (64, 16) and a.P.dtype == torch.bfloat16
    assert a.Q.shape == (1, 1, 1, 4, 64)
    assert a.K.shape == (1, 64, 16, 2, 64)
    assert a.table.tolist() == list(range(64)), "tiny uses the identity block table"
    assert a.seq_offsets.tolist() == [0, 64]
    c = W.tiny(seed=1)
    assert not torch.equal(a.K, c.K)


def test_projection_scale():
    g = torch.Generator().manual_seed(0)
    P = W.projection(g, 128, 32).float()
    assert abs(P.std().item() - (1 / 32) ** 0.5) < 0.01


def test_batched_lengths_fit_pool():
    g = torch.Generator().manual_seed(7)
    n = W.batched_lengths(g, 64, 1024, 16384, 16, 40000)
    assert len(n) == 64 and sum(n) <= 40000
    assert all(64 <= x <= 1024 for x in n)


def test_skewed_keys_have_outliers():
    g = torch.Generator().manual_seed(3)
    ch = torch.tensor([1, 5, 9, 30])
    K = W.skewed_keys(g, (64, 16, 2, 32), ch).float()
    per_ch = K.abs().mean(dim=(0, 1, 2))
    others = per_ch[[i for i in range(32) if i not in ch.tolist()]]
    assert per_ch[ch].min() > 8 * others.max()
    norms = K.norm(dim=-1).flatten()
    assert norms.max() / norms.min() > 20  # log-normal spread


def test_generic_permutation_and_offsets():
    d = W.Dims(2, 8, 2, 32, 16, 16, 50)
    c = W.generic("x", d, num_seqs=3, rows_per_seq=2, lengths=[5, 0, 7], k_victims=4, seed=3,
                  pool=20, score_layer=1)
    assert c.table.numel() == 12 and len(set(c.table.tolist())) == 12
    assert max(c.table.tolist()) < 20
    assert c.seq_offsets.tolist() == [0, 5, 5, 12]
    assert c.K.shape == (1, 20, 16, 2, 32) and c.ingest_layers == [1]


def test_random_scores_plants_ties_and_zeros():
    s, offs = W.random_scores(1, [100, 50], ties=0.3)
    assert offs.tolist() == [0, 100, 150]
    assert (s == 0).sum() >= 2 and torch.signbit(s[s == 0]).any()
    assert s.unique().numel() < 150
