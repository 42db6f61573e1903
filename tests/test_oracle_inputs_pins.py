"""Pins of the oracle's indexer-input projections and key-cache update.

The projections are pinned to a pure-Python triple loop on small inputs, to
identity and one-hot closed forms, and to the head/dim layout of the reshape;
the cache update to a worked example and to the rows it must leave alone.
"""
import numpy as np

import oracle.dsa_oracle as O


def _loop_linear(x, w):
    T, K = len(x), len(x[0])
    N = len(w)
    return [[sum(float(x[t][k]) * float(w[n][k]) for k in range(K)) for n in range(N)] for t in range(T)]


def test_linear_equals_a_triple_loop():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 7))
    w = rng.standard_normal((3, 7))
    assert np.allclose(O.linear(x, w), np.array(_loop_linear(x.tolist(), w.tolist())), rtol=0, atol=1e-12)


def test_linear_transposes_the_weight_not_the_input():
    # weight [N, K]: output column n is the dot product with weight row n
    x = np.array([[1.0, 2.0, 3.0]])
    w = np.array([[1.0, 0.0, 0.0], [0.0, 0.0, 1.0]])
    assert O.linear(x, w).tolist() == [[1.0, 3.0]]


def test_indexer_inputs_identity_and_one_hot():
    H, D, R, E = 2, 3, 6, 4     # heads, head dim, q_lora_rank, hidden
    T = 3
    rng = np.random.default_rng(1)
    q_lat = rng.standard_normal((T, R))
    x = rng.standard_normal((T, E))
    wq_b = np.eye(H * D, R)      # picks the first H * D latent components
    wk = np.zeros((D, E)); wk[0, 2] = 1.0; wk[2, 0] = -2.0
    wp = np.zeros((H, E)); wp[1, 3] = 0.5
    q_i, k_i, w = O.indexer_inputs(q_lat, x, wq_b, wk, wp, H, D)
    assert q_i.shape == (T, H, D) and k_i.shape == (T, D) and w.shape == (T, H)
    # head j, component d of q_I is latent component j * D + d (row-major reshape)
    assert np.array_equal(q_i, q_lat[:, : H * D].reshape(T, H, D))
    assert np.array_equal(k_i[:, 0], x[:, 2]) and np.array_equal(k_i[:, 2], -2.0 * x[:, 0])
    assert np.all(k_i[:, 1] == 0.0)
    assert np.all(w[:, 0] == 0.0) and np.array_equal(w[:, 1], 0.5 * x[:, 3])


def test_indexer_inputs_is_linear():
    rng = np.random.default_rng(2)
    H, D, R, E, T = 4, 8, 16, 12, 5
    q1, q2 = rng.standard_normal((2, T, R))
    x1, x2 = rng.standard_normal((2, T, E))
    ws = [rng.standard_normal(s) for s in [(H * D, R), (D, E), (H, E)]]
    a = O.indexer_inputs(q1, x1, *ws, H, D)
    b = O.indexer_inputs(q2, x2, *ws, H, D)
    c = O.indexer_inputs(2 * q1 - q2, 2 * x1 - x2, *ws, H, D)
    for u, v, s in zip(a, b, c):
        assert np.allclose(s, 2 * u - v, atol=1e-12)


def test_update_indexer_worked_example():
    idx = np.zeros((3, 4, 2))
    kv = np.zeros((3, 4, 3))
    lens = np.array([0, 2, 4])
    k_new = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]])
    kv_new = np.array([[7.0, 8.0, 9.0], [10.0, 11.0, 12.0], [13.0, 14.0, 15.0]])
    i2, kv2, l2, full = O.update_indexer(idx, kv, lens, k_new, kv_new)
    assert l2.tolist() == [1, 3, 4] and full.tolist() == [False, False, True]
    assert i2[0, 0].tolist() == [1.0, 2.0] and kv2[0, 0].tolist() == [7.0, 8.0, 9.0]
    assert i2[1, 2].tolist() == [3.0, 4.0] and kv2[1, 2].tolist() == [10.0, 11.0, 12.0]
    # nothing else changed, and the inputs are not modified
    m = np.ones(idx.shape[:2], dtype=bool); m[0, 0] = m[1, 2] = False
    assert np.all(i2[m] == 0.0) and np.all(kv2[m] == 0.0)
    assert np.all(idx == 0.0) and lens.tolist() == [0, 2, 4]


def test_update_indexer_then_decode_sees_the_new_token():
    # the appended key takes part in the next decode step's scores: a new key that matches
    # the query far better than the rest is selected first
    rng = np.random.default_rng(3)
    H, D, M = 2, 4, 6
    idx = rng.standard_normal((1, M, D)) * 0.01
    lens = np.array([3])
    q = np.ones((H, D))
    w = np.ones(H)
    k_new = np.full((1, D), 5.0)
    kv = np.zeros((1, M, 3))
    i2, _, l2, _ = O.update_indexer(idx, kv, lens, k_new, np.zeros((1, 3)))
    sc = O.index_scores_row(q, w, i2[0, : l2[0]])
    assert int(np.argmax(sc)) == 3 and l2[0] == 4


def test_paged_to_dense_worked_example():
    P = 2
    pool = np.arange(5 * P * 3).reshape(5 * P, 3)          # 5 pages of 2 positions, 3 values each
    table = np.array([[3, 0], [1, -1]])
    d = O.paged_to_dense(pool, table, P)
    assert d.shape == (2, 4, 3)
    assert d[0, 0].tolist() == pool[6].tolist() and d[0, 1].tolist() == pool[7].tolist()   # page 3
    assert d[0, 2].tolist() == pool[0].tolist() and d[0, 3].tolist() == pool[1].tolist()   # page 0
    assert d[1, 0].tolist() == pool[2].tolist() and d[1, 1].tolist() == pool[3].tolist()   # page 1
    assert np.all(d[1, 2:] == 0)                                                            # no page


def test_paged_to_dense_with_contiguous_pages_is_a_reshape():
    B, P, pages, D = 3, 4, 5, 2
    pool = np.random.default_rng(0).standard_normal((B * pages * P, D))
    table = np.arange(B * pages).reshape(B, pages)
    assert np.array_equal(O.paged_to_dense(pool, table, P), pool.reshape(B, pages * P, D))
