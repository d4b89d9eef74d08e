"""The seeded input generator: determinism, random access by row, roles and distributions."""
import numpy as np

import gen
from oracle import ce_oracle as O


def test_rows_equal_full_and_are_deterministic():
    p = gen.custom(300, 517, "bf16", seed=3, n_margin=30, n_ignore=7)
    full = p.full(threads=3)
    again = gen.custom(300, 517, "bf16", seed=3, n_margin=30, n_ignore=7).full(threads=1)
    assert np.array_equal(full, again)
    idx = [0, 5, 299, int(p.margin_rows[0]), int(p.ignore_rows[0])]
    assert np.array_equal(p.rows(idx), full[idx])


def test_roles_are_disjoint_and_counted():
    p = gen.pages()
    assert len(p.margin_rows) == 1638 and len(p.ignore_rows) == 164
    assert not set(p.margin_rows) & set(p.ignore_rows)
    assert np.all(p.labels[p.ignore_rows] == gen.IGNORE_INDEX)
    ok = np.ones(p.T, bool)
    ok[p.ignore_rows] = False
    assert np.all((p.labels[ok] >= 0) & (p.labels[ok] < p.V))
    m = p.margin[p.margin_rows]
    assert np.all((m >= 17) & (m <= 50))
    t = gen.tiny()
    assert len(t.margin_rows) == 8 and len(t.ignore_rows) == 4


def test_raised_target_rows():
    p = gen.tiny()
    rows = p.rows(p.margin_rows)
    z = O.widen(rows, "f32")
    for k, r in enumerate(p.margin_rows):
        t = p.labels[r]
        others = np.delete(z[k], t)
        gap = z[k, t] - others.max()
        assert 20 - 1e-4 <= gap <= 40 + 1e-4 or gap >= p.margin[r] - 1e-4


def test_distribution_moments():
    p = gen.custom(64, 20000, "bf16", seed=12, std=2.0)
    z = O.widen(p.full(), "bf16")
    assert abs(z.mean()) < 0.01 and abs(z.std() - 2.0) < 0.01
    lp = gen.linear_small()
    E = O.widen(lp.E(), "bf16")
    W = O.widen(lp.W(), "bf16")
    assert abs(E.std() - 1.0) < 0.01 and abs(W.std() - 0.02) < 0.001
    assert lp.T == 8191 and lp.D == 128 and lp.V == 32 and len(lp.ignore_rows) == 164


def test_copy_cols():
    p = gen.custom(20, 48, "bf16", seed=1)
    full = p.full()
    for c0, w in gen.chunk_bounds(48, 4):
        assert np.array_equal(gen.copy_cols(full, c0, w), full[:, c0: c0 + w])
