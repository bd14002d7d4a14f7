"""Pins for the fp64 oracle: checks against what mathematics fixes, not against the oracle itself.

The method (page "SGLang Lightning Attention 能力矩阵与 seg_la 线性注意力测试覆盖深度解析", section
"独立参考实现：逐 token 递推公式") is the recurrence
    S_t = S_{t-1} * exp(-s) + outer(k_t, v_t),    o_t = (q_t @ S_t) * D^-0.5.
Unrolled, it has the closed form
    o_t = D^-0.5 * [ e^{-s(t-t0+1)} q_t S_0 + sum_{u=t0..t} e^{-s(t-u)} (q_t . k_u) v_u ]
    S_end = e^{-s n} S_0 + sum_u e^{-s(t1-1-u)} outer(k_u, v_u),
which the tests below evaluate with independent O(T^2) loops.  Each pin is chosen so that a
plausible slip in the oracle (dropped decay, decay applied after the add, transposed outer
product, missing scale, wrong slot, wrong initial state) fails at least one of them; the mutation
tests in test_oracle_mutants.py show that they do.
"""
import math

import numpy as np
import pytest

import oracle


def rng_inputs(seed, T, H, D):
    r = np.random.default_rng(seed)
    q = r.standard_normal((T, H * D))
    k = r.standard_normal((T, H * D))
    v = r.standard_normal((T, H * D))
    return q, k, v


def closed_form(q, k, v, s, S0, D):
    """O(T^2) closed form of the recurrence for one request-head (rows are tokens)."""
    n = q.shape[0]
    scale = 1.0 / math.sqrt(D)
    out = np.zeros((n, D))
    for t in range(n):
        acc = math.exp(-s * (t + 1)) * (q[t] @ S0)
        for u in range(t + 1):
            acc = acc + math.exp(-s * (t - u)) * float(q[t] @ k[u]) * v[u]
        out[t] = scale * acc
    S = math.exp(-s * n) * S0
    for u in range(n):
        S = S + math.exp(-s * (n - 1 - u)) * np.outer(k[u], v[u])
    return out, S


def test_closed_form_varlen_with_prefix():
    H, D = 2, 16
    lens = [5, 0, 9, 1]
    B = len(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v = rng_inputs(1, T, H, D)
    slopes = np.array([0.3, 0.05])
    r = np.random.default_rng(7)
    num_slots = 6
    pool = r.standard_normal((num_slots, H, D, D)) * 0.05
    idx = np.array([4, 1, 0, 3], dtype=np.int32)
    pm = np.array([1, 1, 0, 1], dtype=np.uint8)
    out, pool_after = oracle.extend(q, k, v, slopes, pool, idx, cu, pm, H, D)
    for b in range(B):
        t0, t1 = cu[b], cu[b + 1]
        for h in range(H):
            sl = slice(h * D, (h + 1) * D)
            S0 = pool[idx[b], h] if pm[b] else np.zeros((D, D))
            o_ref, S_ref = closed_form(q[t0:t1, sl], k[t0:t1, sl], v[t0:t1, sl], slopes[h], S0, D)
            np.testing.assert_allclose(out[t0:t1, sl], o_ref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(pool_after[idx[b], h], S_ref, rtol=1e-12, atol=1e-13)
    # the slot no request names is untouched, bit for bit
    np.testing.assert_array_equal(pool_after[2], pool[2])
    np.testing.assert_array_equal(pool_after[5], pool[5])


def test_closed_form_head_dim_128():
    H, D, n = 1, 128, 12
    q, k, v = rng_inputs(3, n, H, D)
    s = 0.7071
    S0 = np.random.default_rng(4).standard_normal((D, D)) * 0.05
    pool = S0[None, None].copy()
    out, pool_after = oracle.extend(q, k, v, [s], pool, [0], [0, n], [1], H, D)
    o_ref, S_ref = closed_form(q, k, v, s, S0, D)
    np.testing.assert_allclose(out, o_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(pool_after[0, 0], S_ref, rtol=1e-11, atol=1e-12)


def test_geometric_series_scalar_head():
    """D = 1, q = k = v = 1, slope ln 2: S_t = c 2^-t + 2 - 2^(1-t) and o_t = S_t (scale 1)."""
    n, c = 10, 0.75
    ones = np.ones((n, 1))
    out, pool_after = oracle.extend(ones, ones, ones, [math.log(2.0)], np.full((1, 1, 1, 1), c),
                                    [0], [0, n], [1], 1, 1)
    t = np.arange(1, n + 1, dtype=np.float64)
    expect = c * 2.0 ** -t + 2.0 - 2.0 ** (1 - t)
    np.testing.assert_allclose(out[:, 0], expect, rtol=1e-14)
    assert abs(pool_after[0, 0, 0, 0] - expect[-1]) < 1e-14


def test_zero_slope_is_prefix_sum():
    """s = 0: o_t = D^-0.5 q_t (S_0 + sum_{u<=t} k_u v_u^T), a cumulative sum of outer products."""
    H, D, n = 1, 8, 20
    q, k, v = rng_inputs(5, n, H, D)
    S0 = np.random.default_rng(6).standard_normal((D, D))
    out, pool_after = oracle.extend(q, k, v, [0.0], S0[None, None], [0], [0, n], [1], H, D)
    outer = np.einsum("ti,tj->tij", k, v)
    S = S0[None] + np.cumsum(outer, axis=0)
    ref = np.einsum("ti,tij->tj", q, S) / math.sqrt(D)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(pool_after[0, 0], S[-1], rtol=1e-12, atol=1e-12)


def test_large_slope_limit():
    """s = 50: every older contribution is damped by e^-50, so o_t = D^-0.5 (q_t . k_t) v_t."""
    H, D, n = 1, 8, 6
    q, k, v = rng_inputs(8, n, H, D)
    S0 = np.ones((1, 1, D, D))
    out, _ = oracle.extend(q, k, v, [50.0], S0, [0], [0, n], [1], H, D)
    ref = np.einsum("ti,ti->t", q, k)[:, None] * v / math.sqrt(D)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-18)


@pytest.mark.parametrize("split", [0, 1, 7, 63, 64, 65, 127, 128, 129, 199, 200])
def test_split_invariance(split):
    """Extend of A then extend of B (prefix taken from the state A wrote) equals extend of A||B."""
    H, D, n = 2, 8, 200
    q, k, v = rng_inputs(9, n, H, D)
    slopes = np.array([0.2, 0.01])
    S0 = np.random.default_rng(10).standard_normal((3, H, D, D)) * 0.05
    full_out, full_pool = oracle.extend(q, k, v, slopes, S0, [2], [0, n], [1], H, D)
    o1, p1 = oracle.extend(q[:split], k[:split], v[:split], slopes, S0, [2], [0, split], [1], H, D)
    o2, p2 = oracle.extend(q[split:], k[split:], v[split:], slopes, p1, [2], [0, n - split], [1],
                           H, D)
    np.testing.assert_allclose(np.concatenate([o1, o2]), full_out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(p2, full_pool, rtol=1e-12, atol=1e-13)


def test_decode_equals_length_one_extend():
    H, D, B = 2, 16, 5
    q, k, v = rng_inputs(11, B, H, D)
    slopes = np.array([0.5, 0.001])
    pool = np.random.default_rng(12).standard_normal((8, H, D, D)) * 0.05
    idx = np.array([6, 0, 3, 2, 7], dtype=np.int32)
    d_out, d_pool = oracle.decode(q, k, v, slopes, pool, idx, H, D)
    e_out, e_pool = oracle.extend(q, k, v, slopes, pool, idx, np.arange(B + 1, dtype=np.int32),
                                  np.ones(B, np.uint8), H, D)
    np.testing.assert_array_equal(d_out, e_out)
    np.testing.assert_array_equal(d_pool, e_pool)
    # and against the one-step closed form: S' = e^-s S + k v^T, o = D^-0.5 q S'
    for b in range(B):
        for h in range(H):
            sl = slice(h * D, (h + 1) * D)
            S1 = math.exp(-slopes[h]) * pool[idx[b], h] + np.outer(k[b, sl], v[b, sl])
            np.testing.assert_allclose(d_pool[idx[b], h], S1, rtol=1e-14, atol=1e-16)
            np.testing.assert_allclose(d_out[b, sl], q[b, sl] @ S1 / math.sqrt(D), rtol=1e-12,
                                       atol=1e-14)


def test_verify_equals_extend_prefixes():
    H, D, B, N = 2, 8, 3, 4
    q, k, v = rng_inputs(13, B * N, H, D)
    slopes = np.array([0.9, 0.02])
    pool = np.random.default_rng(14).standard_normal((5, H, D, D)) * 0.05
    pool_before = pool.copy()
    idx = np.array([3, 0, 4], dtype=np.int32)
    out, inter = oracle.verify_chain(q, k, v, slopes, pool, idx, N, H, D)
    np.testing.assert_array_equal(pool, pool_before)  # the pool is only read
    for b in range(B):
        rows = slice(b * N, (b + 1) * N)
        e_out, _ = oracle.extend(q[rows], k[rows], v[rows], slopes, pool, [idx[b]], [0, N], [1],
                                 H, D)
        np.testing.assert_allclose(out[rows], e_out, rtol=1e-13, atol=1e-15)
        for t in range(N):
            _, p = oracle.extend(q[rows][: t + 1], k[rows][: t + 1], v[rows][: t + 1], slopes,
                                 pool, [idx[b]], [0, t + 1], [1], H, D)
            np.testing.assert_allclose(inter[b, t], p[idx[b]], rtol=1e-13, atol=1e-15)


def test_linearity():
    H, D, n = 1, 8, 15
    q, k, v = rng_inputs(15, n, H, D)
    _, _, v2 = rng_inputs(16, n, H, D)
    z = np.zeros((1, 1, D, D))
    s = [0.1]
    o1, _ = oracle.extend(q, k, v, s, z, [0], [0, n], [0], H, D)
    o2, _ = oracle.extend(q, k, v2, s, z, [0], [0, n], [0], H, D)
    o12, _ = oracle.extend(q, k, 2.0 * v + 3.0 * v2, s, z, [0], [0, n], [0], H, D)
    np.testing.assert_allclose(o12, 2.0 * o1 + 3.0 * o2, rtol=1e-12, atol=1e-12)
    oq, _ = oracle.extend(-0.5 * q, k, v, s, z, [0], [0, n], [0], H, D)
    np.testing.assert_allclose(oq, -0.5 * o1, rtol=1e-13, atol=1e-14)
    ok, pk = oracle.extend(q, 4.0 * k, v, s, z, [0], [0, n], [0], H, D)
    np.testing.assert_allclose(ok, 4.0 * o1, rtol=1e-13, atol=1e-14)


def test_prefix_flag_zero_never_reads_slot():
    H, D, n = 1, 8, 9
    q, k, v = rng_inputs(17, n, H, D)
    nan_pool = np.full((2, H, D, D), np.nan)
    out, pool_after = oracle.extend(q, k, v, [0.3], nan_pool, [1], [0, n], [0], H, D)
    assert np.isfinite(out).all() and np.isfinite(pool_after[1]).all()
    assert np.isnan(pool_after[0]).all()  # untouched slot keeps its contents
    z_out, z_pool = oracle.extend(q, k, v, [0.3], np.zeros((2, H, D, D)), [1], [0, n], [1], H, D)
    np.testing.assert_array_equal(out, z_out)
    np.testing.assert_array_equal(pool_after[1], z_pool[1])


def test_zero_length_request_writes_initial_state_back():
    H, D = 1, 4
    pool = np.random.default_rng(18).standard_normal((3, H, D, D))
    q = np.zeros((0, H * D))
    out, p = oracle.extend(q, q, q, [0.4], pool, [0, 2], [0, 0, 0], [1, 0], H, D)
    assert out.shape == (0, H * D)
    np.testing.assert_array_equal(p[0], pool[0])     # prefix kept as is
    np.testing.assert_array_equal(p[2], np.zeros((H, D, D)))  # no prefix: zero state written
    np.testing.assert_array_equal(p[1], pool[1])     # untouched


def test_slope_rule():
    """ALiBi base 2^(-8(i+1)/H) times (1 - l/(L-1) + 1e-5), or (1 + 1e-5) when L = 1."""
    s = oracle.slopes(8, 0, 1)
    base = np.array([2.0 ** -(i + 1) for i in range(8)])  # H = 8: 1/2, 1/4, ..., 1/256, exact
    np.testing.assert_allclose(s, base * (1 + 1e-5), rtol=1e-15)
    np.testing.assert_allclose(oracle.slopes(8, 0, 4), base * (1 + 1e-5), rtol=1e-15)
    np.testing.assert_allclose(oracle.slopes(8, 3, 4), base * 1e-5, rtol=1e-10)
    np.testing.assert_allclose(oracle.slopes(16, 3, 8), 2.0 ** (-0.5 * np.arange(1, 17))
                               * (1 - 3 / 7 + 1e-5), rtol=1e-15)
    # H = 2: 2^-4 and 2^-8
    np.testing.assert_allclose(oracle.slopes(2, 0, 1), np.array([1 / 16, 1 / 256]) * (1 + 1e-5),
                               rtol=1e-15)


def test_thread_count_does_not_change_results():
    H, D = 3, 8
    lens = [4, 7, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v = rng_inputs(19, int(cu[-1]), H, D)
    pool = np.random.default_rng(20).standard_normal((4, H, D, D))
    args = (q, k, v, [0.1, 0.2, 0.3], pool, [3, 1, 0, 2], cu, [1, 0, 1, 1], H, D)
    o1, p1 = oracle.extend(*args, nthreads=1)
    o8, p8 = oracle.extend(*args, nthreads=8)
    np.testing.assert_array_equal(o1, o8)
    np.testing.assert_array_equal(p1, p8)


def test_tree_verify_chain_shaped_tree_is_chain_verify():
    H, D, B, N = 2, 8, 3, 5
    q, k, v = rng_inputs(23, B * N, H, D)
    slopes = np.array([0.4, 0.03])
    pool = np.random.default_rng(24).standard_normal((4, H, D, D)) * 0.05
    idx = np.array([1, 3, 0], dtype=np.int32)
    chain = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    o_t, i_t = oracle.verify_tree(q, k, v, slopes, pool, idx, chain, N, H, D)
    o_c, i_c = oracle.verify_chain(q, k, v, slopes, pool, idx, N, H, D)
    np.testing.assert_array_equal(o_t, o_c)
    np.testing.assert_array_equal(i_t, i_c)


def test_tree_verify_star_is_independent_decodes():
    """Every parent the root: each draft token is one decode step from the pool state."""
    H, D, B, N = 2, 8, 2, 4
    q, k, v = rng_inputs(25, B * N, H, D)
    slopes = np.array([0.2, 0.7])
    pool = np.random.default_rng(26).standard_normal((3, H, D, D)) * 0.05
    idx = np.array([2, 0], dtype=np.int32)
    star = np.full((B, N), -1, dtype=np.int32)
    out, inter = oracle.verify_tree(q, k, v, slopes, pool, idx, star, N, H, D)
    for b in range(B):
        for t in range(N):
            row = b * N + t
            for h in range(H):
                sl = slice(h * D, (h + 1) * D)
                S1 = math.exp(-slopes[h]) * pool[idx[b], h] + np.outer(k[row, sl], v[row, sl])
                np.testing.assert_allclose(inter[b, t, h], S1, rtol=1e-14, atol=1e-16)
                np.testing.assert_allclose(out[row, sl], q[row, sl] @ S1 / math.sqrt(D),
                                           rtol=1e-12, atol=1e-14)


def test_tree_verify_equals_extend_along_root_paths():
    """Any tree: token t's state and output equal an extend over the tokens on its root path."""
    H, D, B, N = 2, 8, 2, 7
    q, k, v = rng_inputs(27, B * N, H, D)
    slopes = np.array([0.15, 0.05])
    pool = np.random.default_rng(28).standard_normal((3, H, D, D)) * 0.05
    idx = np.array([2, 1], dtype=np.int32)
    parents = np.array([[-1, 0, 0, 1, -1, 4, 2], [-1, -1, 1, 2, 2, 0, 5]], dtype=np.int32)
    out, inter = oracle.verify_tree(q, k, v, slopes, pool, idx, parents, N, H, D)
    for b in range(B):
        for t in range(N):
            path, x = [], t
            while x >= 0:
                path.append(b * N + x)
                x = parents[b, x]
            path = path[::-1]
            e_out, e_pool = oracle.extend(q[path], k[path], v[path], slopes, pool, [idx[b]],
                                          [0, len(path)], [1], H, D)
            np.testing.assert_allclose(inter[b, t], e_pool[idx[b]], rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(out[b * N + t], e_out[-1], rtol=1e-13, atol=1e-15)


def test_tree_verify_rejects_forward_parents():
    H, D = 1, 4
    q = np.zeros((3, H * D))
    with pytest.raises(ValueError):
        oracle.verify_tree(q, q, q, [0.1], np.zeros((1, H, D, D)), [0],
                           np.array([[-1, 2, 0]], dtype=np.int32), 3, H, D)
    with pytest.raises(ValueError):
        oracle.verify_tree(q, q, q, [0.1], np.zeros((1, H, D, D)), [0],
                           np.array([[-2, 0, 1]], dtype=np.int32), 3, H, D)


def test_commit_after_chain_verify_is_the_accepted_prefix_state():
    """Committing draft token a of a chain verify leaves in the slot the closed-form state after
    tokens 0..a; -1 leaves the slot as it was; slots no request names are untouched; and a decode
    from the committed slot continues the sequence."""
    H, D, B, N = 2, 6, 4, 4
    q, k, v = rng_inputs(31, B * N, H, D)
    slopes = np.array([0.4, 0.03])
    pool = np.random.default_rng(32).standard_normal((7, H, D, D)) * 0.05
    idx = np.array([5, 0, 3, 6], dtype=np.int32)
    accept = np.array([2, -1, 0, 3], dtype=np.int32)
    _, inter = oracle.verify_chain(q, k, v, slopes, pool, idx, N, H, D)
    new_pool = oracle.commit_accepted(inter, accept, pool, idx)
    for s in range(7):
        if s not in idx:
            np.testing.assert_array_equal(new_pool[s], pool[s])
    for b in range(B):
        a = int(accept[b])
        if a < 0:
            np.testing.assert_array_equal(new_pool[idx[b]], pool[idx[b]])
            continue
        rows = slice(b * N, b * N + a + 1)
        for h in range(H):
            sl = slice(h * D, (h + 1) * D)
            _, S = closed_form(q[rows, sl], k[rows, sl], v[rows, sl], slopes[h], pool[idx[b], h], D)
            np.testing.assert_allclose(new_pool[idx[b], h], S, rtol=1e-13, atol=1e-15)
    # one more token from the committed state equals the recurrence over a + 2 tokens
    qn, kn, vn = rng_inputs(33, B, H, D)
    d_out, d_pool = oracle.decode(qn, kn, vn, slopes, new_pool, idx, H, D)
    for b in (0, 2, 3):
        a = int(accept[b])
        rows = list(range(b * N, b * N + a + 1))
        for h in range(H):
            sl = slice(h * D, (h + 1) * D)
            qq = np.vstack([q[rows, sl], qn[b, sl]])
            kk = np.vstack([k[rows, sl], kn[b, sl]])
            vv = np.vstack([v[rows, sl], vn[b, sl]])
            o, S = closed_form(qq, kk, vv, slopes[h], pool[idx[b], h], D)
            np.testing.assert_allclose(d_out[b, sl], o[-1], rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(d_pool[idx[b], h], S, rtol=1e-13, atol=1e-15)


def test_commit_after_tree_verify_is_the_root_path_state():
    H, D, B, N = 1, 5, 3, 6
    q, k, v = rng_inputs(34, B * N, H, D)
    slopes = np.array([0.2])
    pool = np.random.default_rng(35).standard_normal((4, H, D, D)) * 0.05
    idx = np.array([1, 3, 0], dtype=np.int32)
    parents = np.array([[-1, 0, 0, 1, 2, 2]] * B, dtype=np.int32)
    accept = np.array([4, 3, 5], dtype=np.int32)
    _, inter = oracle.verify_tree(q, k, v, slopes, pool, idx, parents, N, H, D)
    new_pool = oracle.commit_accepted(inter, accept, pool, idx)
    np.testing.assert_array_equal(new_pool[2], pool[2])
    for b in range(B):
        path, x = [], int(accept[b])
        while x >= 0:
            path.append(b * N + x)
            x = parents[b, x]
        path = path[::-1]
        _, S = closed_form(q[path], k[path], v[path], slopes[0], pool[idx[b], 0], D)
        np.testing.assert_allclose(new_pool[idx[b], 0], S, rtol=1e-13, atol=1e-15)


def test_commit_rejects_out_of_range_index():
    inter = np.zeros((1, 3, 1, 4, 4))
    pool = np.ones((2, 1, 4, 4))
    for bad in (3, -2):
        with pytest.raises(ValueError):
            oracle.commit_accepted(inter, [bad], pool, [1])


def _tracked_case(seed=41):
    H, D = 2, 6
    lens = [9, 5, 0, 12, 7, 4]
    tls = [4, 0, 0, 12, -1, 0]
    pm = [1, 0, 0, 1, 1, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v = rng_inputs(seed, int(cu[-1]), H, D)
    slopes = np.array([0.3, 0.05])
    S = 16
    pool = np.full((S, H, D, D), 54321.0)
    r = np.random.default_rng(seed + 1)
    idx = np.array([3, 7, 1, 12, 0, 9], dtype=np.int32)
    tidx = np.array([5, 2, 15, 8, 6, 11], dtype=np.int32)
    for b in range(len(lens)):
        pool[idx[b]] = r.standard_normal((H, D, D)) * 0.05 if pm[b] else np.nan
    return H, D, lens, tls, pm, cu, q, k, v, slopes, pool, idx, tidx


def test_tracking_snapshot_is_the_state_after_track_len_tokens():
    """The track slot holds the closed-form state after the first track_len tokens (the initial
    state for 0, the final state for the full length); outputs and final states are those of a
    plain extend; slots that nothing names keep their bytes; -1 writes no snapshot."""
    H, D, lens, tls, pm, cu, q, k, v, slopes, pool, idx, tidx = _tracked_case()
    out, got = oracle.extend_tracked(q, k, v, slopes, pool, idx, cu, pm, tls, tidx, H, D)
    out_p, got_p = oracle.extend(q, k, v, slopes, pool, idx, cu, pm, H, D)
    np.testing.assert_array_equal(out, out_p)
    np.testing.assert_array_equal(got[idx], got_p[idx])
    snap = {int(tidx[b]) for b in range(len(lens)) if tls[b] >= 0}
    for s in range(pool.shape[0]):
        if s not in snap and s not in idx:
            np.testing.assert_array_equal(got[s], pool[s])
    np.testing.assert_array_equal(got[tidx[4]], pool[tidx[4]])  # track_len -1: untouched
    for b in range(len(lens)):
        if tls[b] < 0:
            continue
        rows = slice(int(cu[b]), int(cu[b]) + tls[b])
        for h in range(H):
            sl = slice(h * D, (h + 1) * D)
            S0 = pool[idx[b], h] if pm[b] else np.zeros((D, D))
            _, S = closed_form(q[rows, sl], k[rows, sl], v[rows, sl], slopes[h], S0, D)
            np.testing.assert_allclose(got[tidx[b], h], S, rtol=1e-13, atol=1e-15)


def test_tracking_snapshot_equals_verify_intermediate_state():
    """The check the page describes: the snapshot at track_len equals the per-token recurrence's
    state at that moment, here chain verify's state after draft token track_len - 1."""
    H, D, lens, tls, pm, cu, q, k, v, slopes, pool, idx, tidx = _tracked_case(43)
    _, got = oracle.extend_tracked(q, k, v, slopes, pool, idx, cu, pm, tls, tidx, H, D)
    for b in (0, 3):
        n = lens[b]
        rows = slice(int(cu[b]), int(cu[b]) + n)
        _, inter = oracle.verify_chain(q[rows], k[rows], v[rows], slopes, pool, [idx[b]], n, H, D)
        np.testing.assert_allclose(got[tidx[b]], inter[0, tls[b] - 1], rtol=1e-13, atol=1e-15)


def test_tracking_rejects_bad_track_lengths_and_own_slot():
    H, D, lens, tls, pm, cu, q, k, v, slopes, pool, idx, tidx = _tracked_case()
    for b, bad_tl in ((0, 10), (1, -2), (2, 1)):
        t = list(tls)
        t[b] = bad_tl
        with pytest.raises(ValueError):
            oracle.extend_tracked(q, k, v, slopes, pool, idx, cu, pm, t, tidx, H, D)
    ti = tidx.copy()
    ti[3] = idx[3]
    with pytest.raises(ValueError):
        oracle.extend_tracked(q, k, v, slopes, pool, idx, cu, pm, tls, ti, H, D)


# ------------------------------------------------------------------ grouped-query heads
# The page's seg_la takes one head count for q, k and v (section "输入与配置覆盖"); the grouped
# variant lets H query heads share Hkv key/value heads, with one state and one slope per kv head.

def _gqa_case(seed, H, Hkv, D, lens, num_slots=7):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    r = np.random.default_rng(seed)
    q = r.standard_normal((T, H * D))
    k = r.standard_normal((T, Hkv * D))
    v = r.standard_normal((T, Hkv * D))
    slopes = r.uniform(0.01, 0.9, size=Hkv)
    pool = r.standard_normal((num_slots, Hkv, D, D)) * 0.05
    idx = r.permutation(num_slots)[:len(lens)].astype(np.int32)
    pm = (np.arange(len(lens)) % 2 == 0).astype(np.uint8)
    return q, k, v, slopes, pool, idx, cu, pm


def test_gqa_closed_form_per_query_head():
    """Every query head h reads the closed-form state of kv head h // G, from the same k, v and
    slope; the kv head's final state is the closed-form end state."""
    H, Hkv, D = 6, 2, 8
    G = H // Hkv
    lens = [7, 0, 12]
    q, k, v, slopes, pool, idx, cu, pm = _gqa_case(21, H, Hkv, D, lens)
    out, pool_after = oracle.extend_gqa(q, k, v, slopes, pool, idx, cu, pm, H, Hkv, D)
    for b in range(len(lens)):
        t0, t1 = cu[b], cu[b + 1]
        for h in range(H):
            j = h // G
            sq, skv = slice(h * D, (h + 1) * D), slice(j * D, (j + 1) * D)
            S0 = pool[idx[b], j] if pm[b] else np.zeros((D, D))
            o_ref, S_ref = closed_form(q[t0:t1, sq], k[t0:t1, skv], v[t0:t1, skv], slopes[j], S0, D)
            np.testing.assert_allclose(out[t0:t1, sq], o_ref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(pool_after[idx[b], j], S_ref, rtol=1e-12, atol=1e-13)
    untouched = np.setdiff1d(np.arange(pool.shape[0]), idx)
    np.testing.assert_array_equal(pool_after[untouched], pool[untouched])


def test_gqa_with_one_query_head_per_kv_head_is_the_plain_extend():
    H = Hkv = 3
    D = 8
    q, k, v, slopes, pool, idx, cu, pm = _gqa_case(22, H, Hkv, D, [9, 4, 0, 17])
    g_out, g_pool = oracle.extend_gqa(q, k, v, slopes, pool, idx, cu, pm, H, Hkv, D)
    e_out, e_pool = oracle.extend(q, k, v, slopes, pool, idx, cu, pm, H, D)
    np.testing.assert_array_equal(g_out, e_out)
    np.testing.assert_array_equal(g_pool, e_pool)


def test_gqa_group_equals_the_recurrence_with_the_kv_head_repeated():
    """Repeating each kv head's k, v, slope and state G times turns the grouped call into the
    plain per-head recurrence: same outputs, and every copy of a group's state ends equal to the
    kv head's final state."""
    H, Hkv, D = 8, 2, 8
    G = H // Hkv
    q, k, v, slopes, pool, idx, cu, pm = _gqa_case(23, H, Hkv, D, [11, 3, 20])
    g_out, g_pool = oracle.extend_gqa(q, k, v, slopes, pool, idx, cu, pm, H, Hkv, D)
    rep = np.repeat(np.arange(Hkv), G)
    cols = np.concatenate([np.arange(j * D, (j + 1) * D) for j in rep])
    e_out, e_pool = oracle.extend(q, k[:, cols], v[:, cols], slopes[rep], pool[:, rep], idx, cu,
                                  pm, H, D)
    np.testing.assert_array_equal(g_out, e_out)
    for h in range(H):
        np.testing.assert_array_equal(e_pool[idx][:, h], g_pool[idx][:, h // G])


def test_gqa_decode_is_a_length_one_grouped_extend():
    H, Hkv, D, B = 4, 2, 8, 5
    q, k, v, slopes, pool, idx, _, _ = _gqa_case(24, H, Hkv, D, [1] * B, num_slots=9)
    d_out, d_pool = oracle.decode_gqa(q, k, v, slopes, pool, idx, H, Hkv, D)
    e_out, e_pool = oracle.extend_gqa(q, k, v, slopes, pool, idx,
                                      np.arange(B + 1, dtype=np.int32), np.ones(B, np.uint8),
                                      H, Hkv, D)
    np.testing.assert_array_equal(d_out, e_out)
    np.testing.assert_array_equal(d_pool, e_pool)
    # one step in closed form: S' = e^-s_j S + k_j v_j^T, o_h = D^-0.5 q_h S'
    G = H // Hkv
    for b in range(B):
        for h in range(H):
            j = h // G
            skv = slice(j * D, (j + 1) * D)
            S1 = math.exp(-slopes[j]) * pool[idx[b], j] + np.outer(k[b, skv], v[b, skv])
            np.testing.assert_allclose(d_out[b, h * D:(h + 1) * D], q[b, h * D:(h + 1) * D] @ S1
                                       / math.sqrt(D), rtol=1e-12, atol=1e-14)


def test_gqa_rejects_indivisible_heads():
    q, k, v, slopes, pool, idx, cu, pm = _gqa_case(25, 4, 2, 8, [3])
    with pytest.raises(ValueError):
        oracle.extend_gqa(q[:, :3 * 8], k, v, slopes, pool, idx, cu, pm, 3, 2, 8)
