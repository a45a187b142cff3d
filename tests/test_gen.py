"""Synthetic workload generators: shapes, dtypes, determinism (CPU)."""

import torch

import gen


def test_chain_tiny_shapes_and_seed():
    a = gen.chain_tiny(0)
    b = gen.chain_tiny(0)
    assert a.Lp.shape == (4, 5, 1000) and a.Lq.shape == (4, 4, 1000) and a.Lp.dtype == torch.float32
    assert a.x.dtype == torch.int32 and a.x.shape == (4, 4)
    assert torch.equal(a.Lp, b.Lp) and torch.equal(a.x, b.x) and torch.equal(a.ua, b.ua)
    assert not torch.equal(a.Lp, gen.chain_tiny(1).Lp)
    assert float(a.ua.min()) >= 0.0 and float(a.ua.max()) < 1.0


def test_zipf_small():
    c = gen.chain_zipf(3, 2, 512, torch.bfloat16, 0.7, 1.0, seed=5)
    assert c.Lp.dtype == torch.bfloat16 and c.Lp.shape == (3, 3, 512)
    assert int(c.x.min()) >= 0 and int(c.x.max()) < 512
    # 20 boosted ids per position stand well above the Gaussian tail
    assert int((c.Lp.float() > 5.5).sum(dim=-1).min()) >= 15
    g = gen.chain_zipf(2, 3, 300, torch.float32, 0.0, 0.5, seed=1)
    assert torch.equal(g.x, g.Lq.argmax(dim=-1).to(torch.int32))


def test_tree_batch_structure():
    tb = gen.tree_batch(3, n_per_tree=30, V=97, dtype=torch.float32, seed=2)
    assert tb.N == 61 and tb.R.shape[2] == 7 and tb.n1 == 30
    for b in range(tb.B):
        m = tb.mask[b]
        assert int(m.diagonal().sum()) == tb.N and bool((m[:, 0] == 1).all())
        assert int(tb.pos[b].max()) <= 6
        for row in tb.R[b].tolist():
            if row[0] == -1:
                continue
            path = [v for v in row if v != -1]
            for t in range(1, len(path)):
                assert m[path[t], path[t - 1]] == 1
