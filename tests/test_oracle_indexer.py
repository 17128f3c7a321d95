"""Pins for the oracle's indexer scores (oracle.indexer_scores), each against
a closed form rather than the same formula retyped: basis-vector keys pick
single query coordinates, a one-hot head weight isolates one head's ReLU, the
score is linear in the head weights and positively homogeneous in (scale,
bias), negative logits vanish, and the row windows place and clip scores."""
import numpy as np
import pytest

import oracle

H, D = oracle.INDEXER_HEADS, oracle.INDEXER_DIM


def _call(q, w, keys, L, bias=None, scale=0.5, ks=0, ss=0, n=None):
    n = ss + L if n is None else n
    return oracle.indexer_scores(q[None], w[None], None if bias is None else [bias], keys, [ks], [L],
                                 [ss], n, scale)


def test_basis_keys_pick_query_coordinates():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((H, D))
    w = rng.random(H)
    keys = np.eye(D)[:20]                                 # key t = e_t
    s, wr = _call(q, w, keys, 20, scale=0.25)
    assert wr.all()
    for t in range(20):
        want = sum(w[h] * max(0.0, 0.25 * q[h, t]) for h in range(H))
        assert s[t] == pytest.approx(want, rel=1e-12, abs=1e-15)


def test_one_hot_head_and_relu():
    q = np.zeros((H, D))
    q[5, :3] = [1.0, -2.0, 0.5]
    w = np.zeros(H)
    w[5] = 3.0
    keys = np.array([[1.0, 0, 0] + [0] * (D - 3), [0, 1.0, 0] + [0] * (D - 3), [2.0, 1.0, 4.0] + [0] * (D - 3)])
    s, _ = _call(q, w, keys, 3, scale=1.0)
    assert s.tolist() == [3.0, 0.0, 3.0 * (2.0 - 2.0 + 2.0)]     # 1; relu(-2) = 0; 2 - 2 + 2
    s, _ = _call(q, w, keys, 3, scale=1.0, bias=-1.5)
    assert s.tolist() == [0.0, 0.0, 3.0 * 0.5]


def test_linear_in_weights_and_homogeneous():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((H, D))
    keys = rng.standard_normal((50, D))
    w1, w2 = rng.random(H), rng.random(H)
    a, _ = _call(q, w1, keys, 50)
    b, _ = _call(q, w2, keys, 50)
    c, _ = _call(q, 2.0 * w1 + 3.0 * w2, keys, 50)
    np.testing.assert_allclose(c, 2.0 * a + 3.0 * b, rtol=1e-12, atol=1e-12)
    d, _ = _call(q, w1, keys, 50, scale=1.0, bias=0.25)
    e, _ = _call(q, w1, keys, 50, scale=4.0, bias=1.0)      # every logit times 4
    np.testing.assert_allclose(e, 4.0 * d, rtol=1e-12, atol=1e-12)
    f, _ = _call(-q, w1, keys, 50, scale=1.0)               # relu(x) - relu(-x) = x
    g, _ = _call(q, w1, keys, 50, scale=1.0)
    np.testing.assert_allclose(g - f, (keys @ q.T) @ w1, rtol=1e-10, atol=1e-10)


def test_windows_place_and_reject():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((2, H, D))
    w = rng.random((2, H))
    keys = rng.standard_normal((30, D))
    s, wr = oracle.indexer_scores(q, w, None, keys, [4, 25], [10, 10], [3, 20], 40, 1.0)
    assert wr.tolist() == [False] * 3 + [True] * 10 + [False] * 27      # row 1's keys leave the buffer
    alone, _ = _call(q[0], w[0], keys[4:14], 10, scale=1.0)
    np.testing.assert_array_equal(s[3:13], alone)
    s, wr = oracle.indexer_scores(q, w, [0.0, 0.0], keys, [0, 0], [5, 0], [0, 5], 5, 1.0)
    assert wr.tolist() == [True] * 5


PINS = (test_basis_keys_pick_query_coordinates, test_one_hot_head_and_relu,
        test_linear_in_weights_and_homogeneous, test_windows_place_and_reject)
MUTATIONS = {
    "no_relu": ("np.maximum(logits, 0.0) @ w[i]", "logits @ w[i]"),
    "bias_inside_scale": ("scale * (keys[ks:ks + L] @ q[i].T) + b[i]", "scale * (keys[ks:ks + L] @ q[i].T + b[i])"),
    "no_scale": ("scale * (keys[ks:ks + L] @ q[i].T) + b[i]", "(keys[ks:ks + L] @ q[i].T) + b[i]"),
    "window_off_by_one": ("ks + L > keys.shape[0]", "ks + L >= keys.shape[0]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_slip_is_caught(name, monkeypatch):
    import inspect
    import textwrap
    before, after = MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(oracle.indexer_scores))
    assert src.count(before) == 1, name
    ns = dict(vars(oracle))
    exec(compile(src.replace(before, after), f"<indexer_scores {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, "indexer_scores", ns["indexer_scores"])
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed, f"no pin caught {name}"
