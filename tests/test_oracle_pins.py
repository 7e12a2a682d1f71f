"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics.

None of these re-type the oracle's formula.  They check it against printed
values (tests/golden, each with its citation), closed forms, invariants and an
independent evaluation order, chosen so that a dropped term, a wrong sign or
index, a swapped read/write order or a transposed operand fails at least one.
"""
import numpy as np
import pytest

from conftest import golden


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_la(seed, B, H, N, dk, dv, scale=1.0):
    r = _rng(seed)
    q = r.normal(size=(B, H, N, dk)) * scale
    k = r.normal(size=(B, H, N, dk)) * scale
    v = r.normal(size=(B, H, N, dv)) * scale
    return q, k, v


def _relmax(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# --------------------------------------------------------------------------
# feature map

def test_phi_facts(orc):
    g = golden("phi_and_state_facts.json")
    u = np.array([p[0] for p in g["phi"]])
    want = np.array([p[1] for p in g["phi"]])
    got = orc.phi(u)
    assert got[0] == 1.0  # phi(0) = 1 exactly
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=0)
    # positive everywhere, continuous at 0 from both sides
    x = np.linspace(-30, 30, 10001)
    y = orc.phi(x)
    assert np.all(y > 0)
    eps = 1e-12
    assert abs(orc.phi(np.array([eps]))[0] - orc.phi(np.array([-eps]))[0]) < 1e-11


# --------------------------------------------------------------------------
# the printed seed-7 run of the first page

def _seed7_inputs():
    g = golden("p1_seed7_run.json")
    rng = np.random.default_rng(g["seed"])
    q = rng.normal(size=tuple(g["q_shape"]))
    k = rng.normal(size=tuple(g["k_shape"]))
    v = rng.normal(size=tuple(g["v_shape"]))
    return g, q, k, v


def _causal_softmax(q, k, v):
    # Test-only foil (a different operator): pins that the seeded draw matches
    # the page's, through the printed linear-vs-softmax difference.
    logits = q @ k.T / np.sqrt(q.shape[1])
    n = len(q)
    logits[np.triu_indices(n, k=1)] = -np.inf
    logits -= logits.max(axis=1, keepdims=True)
    w = np.exp(logits)
    w /= w.sum(axis=1, keepdims=True)
    return w @ v


def test_p1_seed7_printed_run(orc):
    g, q, k, v = _seed7_inputs()
    q4, k4, v4 = (x[None, None] for x in (q, k, v))
    o, S, z = orc.la_recurrent(q4, k4, v4, eps=g["eps"])
    o = o[0, 0]
    assert S.shape == (1, 1, 4, 3) and z.shape == (1, 1, 4)
    np.testing.assert_allclose(o[:2], np.array(g["first_two_outputs"]),
                               rtol=0, atol=0.5 * 10.0 ** -g["first_two_outputs_decimals"] + 1e-12)
    assert abs(o.min() - g["output_min"]) < 1e-12
    assert abs(o.max() - g["output_max"]) < 1e-12
    quad = orc.la_quadratic(q4, k4, v4, eps=g["eps"])[0, 0]
    assert np.max(np.abs(quad - o)) < g["explicit_recurrent_max_error_below"]
    soft = _causal_softmax(q, k, v)
    assert abs(np.max(np.abs(o - soft)) - g["linear_softmax_max_difference"]) < 1e-12


def test_p1_future_leak_is_exactly_zero(orc):
    g, q, k, v = _seed7_inputs()
    base = orc.la_recurrent(q[None, None], k[None, None], v[None, None])[0][0, 0]
    v2 = v.copy()
    v2[-1] += 100.0
    pert = orc.la_recurrent(q[None, None], k[None, None], v2[None, None])[0][0, 0]
    assert np.array_equal(base[:-1], pert[:-1])  # bit-identical
    assert not np.array_equal(base[-1], pert[-1])
    # the same through the quadratic and chunked forms, perturbing q, k and v
    qq, kk, vv = _rand_la(11, 1, 2, 37, 5, 3)
    t0 = 20
    q2, k2, v2 = qq.copy(), kk.copy(), vv.copy()
    q2[:, :, t0 + 1:] += 3.0
    k2[:, :, t0 + 1:] -= 2.0
    v2[:, :, t0 + 1:] *= -7.0
    for fn in (lambda a, b, c: orc.la_quadratic(a, b, c),
               lambda a, b, c: orc.la_chunked(a, b, c, C=8)[0],
               lambda a, b, c: orc.la_recurrent(a, b, c)[0]):
        a0 = fn(qq, kk, vv)
        a1 = fn(q2, k2, v2)
        assert np.array_equal(a0[:, :, :t0 + 1], a1[:, :, :t0 + 1])


# --------------------------------------------------------------------------
# closed forms

def test_first_step_closed_form(orc):
    q, k, v = _rand_la(3, 2, 3, 5, 7, 4)
    eps = 1e-3  # large enough to see
    o = orc.la_recurrent(q, k, v, eps=eps)[0]
    fq, fk = orc.phi(q[:, :, 0]), orc.phi(k[:, :, 0])
    s = np.sum(fq * fk, axis=-1, keepdims=True)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0] * s / (s + eps), rtol=1e-14)


def test_final_state_closed_form(orc):
    q, k, v = _rand_la(4, 2, 2, 33, 6, 5)
    r = _rng(5)
    S0 = r.normal(size=(2, 2, 6, 5))
    z0 = np.abs(r.normal(size=(2, 2, 6)))
    _, S, z = orc.la_recurrent(q, k, v, S0=S0, z0=z0)
    fk = orc.phi(k)
    S_ref = S0 + np.einsum("bhti,bhtj->bhij", fk, v)  # phi(K)^T V, no q
    z_ref = z0 + fk.sum(axis=2)
    np.testing.assert_allclose(S, S_ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(z, z_ref, rtol=1e-14)
    # the final state does not depend on q
    _, S2, z2 = orc.la_recurrent(q * -5.0 + 1.0, k, v, S0=S0, z0=z0)
    assert np.array_equal(S, S2) and np.array_equal(z, z2)


def test_convex_hull_bound_and_constant_values(orc):
    q, k, v = _rand_la(6, 1, 3, 64, 8, 4)
    o = orc.la_recurrent(q, k, v)[0]
    run_max = np.maximum.accumulate(np.abs(v), axis=2)
    assert np.all(np.abs(o) <= run_max * (1 + 1e-12))
    # constant value rows: o_t = c * w_t / (w_t + eps) with w_t = phi(q_t).z_t
    c = np.array([0.5, -2.0, 3.0, 1.25])
    vc = np.broadcast_to(c, v.shape).copy()
    eps = 1e-2
    o = orc.la_recurrent(q, k, vc, eps=eps)[0]
    zt = np.cumsum(orc.phi(k), axis=2)
    w = np.sum(orc.phi(q) * zt, axis=-1, keepdims=True)
    np.testing.assert_allclose(o, c * w / (w + eps), rtol=1e-13)


def test_eps_zero_single_key_returns_its_value(orc):
    # With one stored token and eps = 0 the normalized read returns that value
    # exactly (up to rounding), whatever the query.
    q, k, v = _rand_la(12, 1, 1, 1, 9, 6)
    o = orc.la_recurrent(q, k, v, eps=0.0)[0]
    np.testing.assert_allclose(o, v, rtol=1e-14)


def test_tiny_brute_force_by_hand(orc):
    # dk = dv = 1, N = 2: o_1 = a1 v1/(a1+eps), o_2 = (a1 v1 + a2 v2)/(a1+a2+eps)
    # with a_i = phi(q_t) phi(k_i); exp and +1 done here by hand.
    q = np.array([[[[-0.5], [1.5]]]])
    k = np.array([[[[2.0], [-1.0]]]])
    v = np.array([[[[3.0], [-4.0]]]])
    eps = 0.25
    pq = [np.exp(-0.5), 2.5]
    pk = [3.0, np.exp(-1.0)]
    o1 = pq[0] * pk[0] * 3.0 / (pq[0] * pk[0] + eps)
    o2 = (pq[1] * pk[0] * 3.0 + pq[1] * pk[1] * -4.0) / (pq[1] * pk[0] + pq[1] * pk[1] + eps)
    o, S, z = orc.la_recurrent(q, k, v, eps=eps)
    np.testing.assert_allclose(o.ravel(), [o1, o2], rtol=1e-15)
    np.testing.assert_allclose(S.ravel(), [3.0 * 3.0 + pk[1] * -4.0], rtol=1e-15)
    np.testing.assert_allclose(z.ravel(), [3.0 + pk[1]], rtol=1e-15)


# --------------------------------------------------------------------------
# independent evaluation orders agree

@pytest.mark.parametrize("dk,dv", [(1, 1), (3, 5), (8, 2)])
def test_quadratic_equals_recurrent_with_state(orc, dk, dv):
    q, k, v = _rand_la(7, 2, 2, 29, dk, dv)
    r = _rng(8)
    S0 = r.normal(size=(2, 2, dk, dv))
    z0 = np.abs(r.normal(size=(2, 2, dk))) + 0.5
    o_rec = orc.la_recurrent(q, k, v, S0=S0, z0=z0)[0]
    o_quad = orc.la_quadratic(q, k, v, S0=S0, z0=z0)
    assert _relmax(o_quad, o_rec) < 1e-12


@pytest.mark.parametrize("C", [1, 2, 3, 7, 16, 64, 100, 101])
def test_chunk_size_independence(orc, C):
    q, k, v = _rand_la(9, 1, 3, 100, 6, 4)
    r = _rng(10)
    S0 = r.normal(size=(1, 3, 6, 4))
    z0 = np.abs(r.normal(size=(1, 3, 6))) + 1.0
    o_rec, S_rec, z_rec = orc.la_recurrent(q, k, v, S0=S0, z0=z0)
    o_ch, S_ch, z_ch = orc.la_chunked(q, k, v, C, S0=S0, z0=z0)
    assert _relmax(o_ch, o_rec) < 1e-12
    assert _relmax(S_ch, S_rec) < 1e-12
    assert _relmax(z_ch, z_rec) < 1e-12


def test_split_stream_equals_whole(orc):
    # prefill(N1) then prefill(N2, S0 = S_N1, z0 = z_N1) == prefill(N1 + N2)
    q, k, v = _rand_la(13, 2, 1, 50, 4, 3)
    o, S, z = orc.la_recurrent(q, k, v)
    o1, S1, z1 = orc.la_recurrent(q[:, :, :17], k[:, :, :17], v[:, :, :17])
    o2, S2, z2 = orc.la_recurrent(q[:, :, 17:], k[:, :, 17:], v[:, :, 17:], S0=S1, z0=z1)
    assert _relmax(np.concatenate([o1, o2], axis=2), o) < 1e-13
    assert _relmax(S2, S) < 1e-13 and _relmax(z2, z) < 1e-13


def test_decode_steps_equal_recurrence(orc):
    q, k, v = _rand_la(14, 3, 2, 12, 5, 7)
    o_ref, S_ref, z_ref = orc.la_recurrent(q, k, v)
    S = np.zeros((3, 2, 5, 7))
    z = np.zeros((3, 2, 5))
    outs = []
    for t in range(12):
        o, S, z = orc.la_decode_step(q[:, :, t], k[:, :, t], v[:, :, t], S, z)
        outs.append(o)
    assert _relmax(np.stack(outs, axis=2), o_ref) < 1e-13
    assert _relmax(S, S_ref) < 1e-13 and _relmax(z, z_ref) < 1e-13


def test_zero_length_and_heads_independent(orc):
    q, k, v = _rand_la(15, 2, 3, 0, 4, 4)
    r = _rng(16)
    S0 = r.normal(size=(2, 3, 4, 4))
    z0 = np.abs(r.normal(size=(2, 3, 4)))
    o, S, z = orc.la_recurrent(q, k, v, S0=S0, z0=z0)
    assert o.shape == (2, 3, 0, 4)
    assert np.array_equal(S, S0) and np.array_equal(z, z0)
    # a head's output depends only on its own tokens
    q, k, v = _rand_la(17, 2, 2, 9, 3, 3)
    o = orc.la_recurrent(q, k, v)[0]
    k2 = k.copy()
    k2[1, 0] += 1.0
    o2 = orc.la_recurrent(q, k2, v)[0]
    assert np.array_equal(o[0], o2[0]) and np.array_equal(o[1, 1], o2[1, 1])
    assert not np.array_equal(o[1, 0], o2[1, 0])


# --------------------------------------------------------------------------
# associative-memory pages

def test_two_entry_outer_product_memory(orc):
    g = golden("two_entry_memory.json")
    keys, values = np.array(g["keys"]), np.array(g["values"])
    reads = orc.outer_read(keys, values, keys)
    np.testing.assert_allclose(reads[0], g["read_A"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(reads[1], g["read_B"], rtol=0, atol=1e-15)
    # the k v^T state is the transpose of the page's W = sum v k^T
    S = orc.outer_read(keys, values, np.eye(2))  # e_i^T S = row i of S
    np.testing.assert_allclose(S, np.array(g["W_vkT"]).T, rtol=0, atol=1e-15)
    # the same memory through delta_prefill's machinery: S0 = W^T, beta = 0
    k = keys[None, None]
    v = np.zeros((1, 1, 2, 2))
    rd, S_N = orc.delta(k, v, np.zeros((1, 1, 2)), S0=np.array(g["W_vkT"]).T[None, None])
    np.testing.assert_allclose(rd[0, 0], [g["read_A"], g["read_B"]], atol=1e-15)


def test_p3_memory_collision_additive(orc):
    g = golden("p3_memory_collision.json")
    keys, values = np.array(g["keys"]), np.array(g["values"])
    S4 = orc.outer_read(keys, values, np.eye(2))
    np.testing.assert_allclose(S4, np.array(g["additive_S4_page_vkT"]).T, atol=1e-15)
    read = orc.outer_read(keys, values, keys[:1])[0]
    np.testing.assert_allclose(read, g["additive_read_k1"], atol=1e-15)


def test_p3_memory_collision_delta(orc):
    g = golden("p3_memory_collision.json")
    keys, values = np.array(g["keys"]), np.array(g["values"])
    k = keys[None, None]
    v = values[None, None]
    beta = np.ones((1, 1, 4))
    reads, S_N = orc.delta(k, v, beta)
    np.testing.assert_allclose(reads[0, 0], g["delta_reads_before_write"], atol=1e-14)
    for t in range(4):
        _, S_t = orc.delta(k[:, :, :t + 1], v[:, :, :t + 1], beta[:, :, :t + 1])
        np.testing.assert_allclose(S_t[0, 0], np.array(g["delta_S_page_vkT"][t]).T, atol=1e-14)
    # a fifth token queried with k_1 reads the latest value written to k_1
    k5 = np.concatenate([k, keys[None, None, :1]], axis=2)
    v5 = np.concatenate([v, np.zeros((1, 1, 1, 2))], axis=2)
    r5, _ = orc.delta(k5, v5, np.ones((1, 1, 5)))
    np.testing.assert_allclose(r5[0, 0, 4], g["delta_read_k1_after"], atol=1e-14)


def test_p1_delta_memory_experiments(orc):
    g = golden("p1_delta_memory.json")
    key = np.array(g["key"])
    values = np.array(g["values"])
    # additive average over the two writes to the same key
    add = orc.outer_read(np.stack([key, key]), values, key[None])[0] / 2.0
    np.testing.assert_allclose(add, g["additive_average_read"], atol=1e-15)
    k = np.stack([key, key, key])[None, None]
    v = np.concatenate([values, np.zeros((1, 2))])[None, None]
    for beta, want in ((1.0, g["delta_beta1_read"]), (0.5, g["delta_beta_half_read"])):
        reads, _ = orc.delta(k, v, np.full((1, 1, 3), beta))
        np.testing.assert_allclose(reads[0, 0, 2], want, atol=1e-15)
    for item in g["crosstalk"]:
        rho = item["rho"]
        k2 = np.array([rho, np.sqrt(1.0 - rho ** 2)])
        kk = np.stack([key, k2, key])[None, None]
        reads, _ = orc.delta(kk, v, np.ones((1, 1, 3)))
        np.testing.assert_allclose(reads[0, 0, 2], item["old_key_read"], rtol=0, atol=1e-15)


def test_delta_exact_recall_orthonormal_keys(orc):
    d = 8
    r = _rng(20)
    Qm, _ = np.linalg.qr(r.normal(size=(d, d)))
    for keys in (np.eye(d), Qm.T):  # basis keys, random orthonormal keys
        vals = r.normal(size=(d, 5))
        S0 = r.normal(size=(d, 5))  # arbitrary old memory, overwritten
        k = np.concatenate([keys, keys])[None, None]
        v = np.concatenate([vals, np.zeros((d, 5))])[None, None]
        beta = np.concatenate([np.ones(d), np.zeros(d)])[None, None]
        reads, S_N = orc.delta(k, v, beta, S0=S0[None, None])
        np.testing.assert_allclose(reads[0, 0, d:], vals, atol=1e-12)
        np.testing.assert_allclose(S_N[0, 0], keys.T @ vals, atol=1e-12)


def test_delta_unit_key_identity_and_beta_zero(orc):
    r = _rng(21)
    d, dv, N = 6, 4, 40
    k = r.normal(size=(1, 2, N, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.normal(size=(1, 2, N, dv))
    beta = r.uniform(0, 1, size=(1, 2, N))
    S0 = r.normal(size=(1, 2, d, dv))
    reads, S_N = orc.delta(k, v, beta, S0=S0)
    # k_t^T S_t = (1 - beta_t) k_t^T S_{t-1} + beta_t v_t^T for unit keys
    for t in range(0, N - 1, 7):
        _, St = orc.delta(k[:, :, :t + 1], v[:, :, :t + 1], beta[:, :, :t + 1], S0=S0)
        lhs = np.einsum("bhi,bhij->bhj", k[:, :, t], St)
        rhs = (1 - beta[:, :, t, None]) * reads[:, :, t] + beta[:, :, t, None] * v[:, :, t]
        np.testing.assert_allclose(lhs, rhs, atol=1e-12)
    # beta = 0: reads are k_t^T S0 and the state is unchanged
    reads0, S0_N = orc.delta(k, v, np.zeros((1, 2, N)), S0=S0)
    assert np.array_equal(S0_N, S0)
    np.testing.assert_allclose(reads0, np.einsum("bhti,bhij->bhtj", k, S0), atol=1e-13)


def test_delta_first_read_is_initial_memory(orc):
    # reads come before the write: with S0 = 0 the first read is exactly 0
    r = _rng(22)
    k = r.normal(size=(2, 1, 3, 4))
    v = r.normal(size=(2, 1, 3, 5))
    reads, _ = orc.delta(k, v, np.full((2, 1, 3), 0.7))
    assert np.all(reads[:, :, 0] == 0.0)
    assert np.all(np.abs(reads[:, :, 1]) > 0)


def test_state_accounting(orc):
    g = golden("phi_and_state_facts.json")
    dk, dv, n = g["dk"], g["dv"], g["history_tokens"]
    history = n * (dk + dv) * 4
    state = (dk * dv + dk) * 4
    assert history == g["history_bytes"] == 32 * 2 ** 20
    assert state == g["state_bytes"]
    assert round(state / 2 ** 20, 6) == g["state_mib_rounded"]
    assert round(history / state, 2) == g["ratio_rounded"]


# --------------------------------------------------------------------------
# gated delta rule (forgetting alpha, then correction)

def test_p1_gated_delta_unrelated_key(orc):
    # the pages' experiment: identity state, write the first key with alpha
    # then read the orthogonal key (a second token with beta = 0 reads it)
    g = golden("p1_gated_delta.json")
    S0 = np.array(g["state"])[None, None]
    k = np.array([g["key"], g["orthogonal_key"]])[None, None]
    v = np.array([g["value"], [0.0, 0.0]])[None, None]
    beta = np.array([[[g["beta"], 0.0]]])
    for alpha_t, want in ((g["gated_alpha"], g["gated_unrelated_key_read"]),
                          (1.0, g["no_forgetting_unrelated_key_read"])):
        alpha = np.array([[[alpha_t, 1.0]]])
        reads, S = orc.gated_delta(k, v, beta, alpha, S0=S0)
        np.testing.assert_allclose(reads[0, 0, 1], want, rtol=0, atol=1e-15)
        # the written key reads the written value exactly (beta = 1, unit key)
        np.testing.assert_allclose(np.array(g["key"]) @ S[0, 0], g["value"], atol=1e-15)


def test_gated_delta_alpha_one_is_the_delta_rule(orc):
    r = _rng(60)
    k = r.normal(size=(2, 2, 30, 5))
    v = r.normal(size=(2, 2, 30, 3))
    beta = r.uniform(size=(2, 2, 30))
    S0 = r.normal(size=(2, 2, 5, 3))
    rg, Sg = orc.gated_delta(k, v, beta, np.ones((2, 2, 30)), S0=S0)
    rd, Sd = orc.delta(k, v, beta, S0=S0)
    np.testing.assert_allclose(rg, rd, rtol=0, atol=1e-13)
    np.testing.assert_allclose(Sg, Sd, rtol=0, atol=1e-13)


def test_gated_delta_pure_forgetting_closed_form(orc):
    # beta = 0: nothing is written; the state decays geometrically and every
    # read is the decayed prediction alpha^(t+1) k_t^T S0
    r = _rng(61)
    N, a = 12, 0.9
    k = r.normal(size=(1, 1, N, 4))
    v = r.normal(size=(1, 1, N, 2))
    S0 = r.normal(size=(1, 1, 4, 2))
    reads, S = orc.gated_delta(k, v, np.zeros((1, 1, N)), np.full((1, 1, N), a), S0=S0)
    for t in range(N):
        np.testing.assert_allclose(reads[0, 0, t], a ** (t + 1) * k[0, 0, t] @ S0[0, 0],
                                   rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S, a ** N * S0, rtol=1e-13)


def test_gated_delta_forgets_before_correcting(orc):
    # alpha = 0 erases the old memory before the correction: one token with a
    # unit key and beta = 1 leaves exactly k v^T, whatever S0 was
    r = _rng(62)
    k = np.array([0.6, 0.8, 0.0])[None, None, None]
    v = r.normal(size=(1, 1, 1, 2))
    S0 = r.normal(size=(1, 1, 3, 2))
    reads, S = orc.gated_delta(k, v, np.ones((1, 1, 1)), np.zeros((1, 1, 1)), S0=S0)
    np.testing.assert_allclose(reads[0, 0, 0], 0.0, atol=1e-15)
    np.testing.assert_allclose(S[0, 0], np.outer(k[0, 0, 0], v[0, 0, 0]), atol=1e-15)


# --------------------------------------------------------------------------
# variants: scalar decay, read before write, non-causal

def test_variant_causal_without_decay_is_the_recurrence(orc):
    q, k, v = _rand_la(63, 2, 2, 20, 4, 3)
    r = _rng(64)
    S0 = r.uniform(size=(2, 2, 4, 3))
    z0 = r.uniform(size=(2, 2, 4))
    o1, S1, z1 = orc.la_variant(q, k, v, None, orc.MODE_CAUSAL, S0=S0, z0=z0)
    o2, S2, z2 = orc.la_recurrent(q, k, v, S0=S0, z0=z0)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(S1, S2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(z1, z2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_variant_recurrence_equals_explicit_weights(orc, mode):
    # an independent evaluation order: the unrolled weights (decay products
    # and masks written out per pair of tokens) against the token loop
    q, k, v = _rand_la(65 + mode, 2, 3, 17, 5, 4)
    r = _rng(70 + mode)
    alpha = None if mode == 2 else r.uniform(0.3, 1.0, size=(2, 3, 17))
    S0 = r.uniform(size=(2, 3, 5, 4))
    z0 = r.uniform(size=(2, 3, 5))
    o_rec, _, _ = orc.la_variant(q, k, v, alpha, mode, S0=S0, z0=z0)
    o_quad = orc.la_variant_quadratic(q, k, v, alpha, mode, S0=S0, z0=z0)
    assert _relmax(o_rec, o_quad) < 1e-12


def test_read_before_write_first_read_is_zero_and_strictly_past(orc):
    # P1 section 09, first change: the first read is zero, later reads see
    # only strictly earlier tokens
    q, k, v = _rand_la(75, 1, 1, 9, 3, 2)
    o, _, _ = orc.la_variant(q, k, v, None, orc.MODE_READ_BEFORE_WRITE)
    np.testing.assert_array_equal(o[0, 0, 0], 0.0)
    # token t's value never reaches o_t: changing the last value changes nothing
    v2 = v.copy()
    v2[0, 0, -1] += 100.0
    o2, _, _ = orc.la_variant(q, k, v2, None, orc.MODE_READ_BEFORE_WRITE)
    np.testing.assert_array_equal(o, o2)
    # and o_t (read before write) is the write-then-read output one token late
    # when the query is held fixed: compare against the causal recurrence on
    # the shifted sequence
    oc, _, _ = orc.la_recurrent(q[:, :, 1:], k[:, :, :-1], v[:, :, :-1])
    np.testing.assert_allclose(o[:, :, 1:], oc, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("eps", [1e-6, 0.5])
def test_decayed_read_before_write_reads_the_state_one_token_late(orc, eps):
    # read before write with a decay: token t reads S_{t-1}, the state after
    # token t - 1's own decay and write, not yet decayed by alpha_t.  So with
    # the query held fixed it is the write-then-read output of the sequence
    # shifted by one token.  (A large eps exposes a stray alpha_t on the read:
    # such a factor scales numerator and denominator alike and cancels against
    # all but eps.)
    q, k, v = _rand_la(80, 2, 2, 13, 4, 3)
    r = _rng(81)
    alpha = r.uniform(0.2, 1.0, size=(2, 2, 13))
    S0 = r.uniform(size=(2, 2, 4, 3))
    z0 = r.uniform(size=(2, 2, 4)) + 0.5
    o, S, z = orc.la_variant(q, k, v, alpha, orc.MODE_READ_BEFORE_WRITE, eps=eps, S0=S0, z0=z0)
    oc, _, _ = orc.la_variant(q[:, :, 1:], k[:, :, :-1], v[:, :, :-1], alpha[:, :, :-1],
                              orc.MODE_CAUSAL, eps=eps, S0=S0, z0=z0)
    np.testing.assert_allclose(o[:, :, 1:], oc, rtol=1e-12, atol=1e-15)
    fq = orc.phi(q[:, :, 0])  # the first read is the initial state's
    want0 = np.einsum("bhi,bhij->bhj", fq, S0) / (np.einsum("bhi,bhi->bh", fq, z0)[..., None] + eps)
    np.testing.assert_allclose(o[:, :, 0], want0, rtol=1e-12)
    # the final state is the write-then-read one
    _, Sc, zc = orc.la_variant(q, k, v, alpha, orc.MODE_CAUSAL, eps=eps, S0=S0, z0=z0)
    np.testing.assert_allclose(S, Sc, rtol=1e-13)
    np.testing.assert_allclose(z, zc, rtol=1e-13)


def test_decay_zero_attends_to_the_current_token_only(orc):
    q, k, v = _rand_la(76, 1, 2, 7, 4, 3)
    eps = 1e-6
    o, S, z = orc.la_variant(q, k, v, np.zeros((1, 2, 7)), orc.MODE_CAUSAL, eps=eps)
    fq, fk = orc.phi(q), orc.phi(k)
    w = np.sum(fq * fk, axis=-1, keepdims=True)
    np.testing.assert_allclose(o, w * v / (w + eps), rtol=1e-13)
    np.testing.assert_allclose(S[0, 1], np.outer(fk[0, 1, -1], v[0, 1, -1]), rtol=1e-13)


def test_noncausal_reads_the_whole_sequence(orc):
    # P2 linear_attention: S = phi(K)^T V and z = sum phi(K) once, every query
    # reads the same state (with eps = 0, the page's form exactly)
    q, k, v = _rand_la(77, 1, 1, 11, 4, 3)
    o, S, z = orc.la_variant(q, k, v, None, orc.MODE_NONCAUSAL, eps=0.0)
    fq, fk = orc.phi(q[0, 0]), orc.phi(k[0, 0])
    Sx = fk.T @ v[0, 0]
    zx = fk.sum(axis=0)
    np.testing.assert_allclose(o[0, 0], (fq @ Sx) / (fq @ zx)[:, None], rtol=1e-13)
    np.testing.assert_allclose(S[0, 0], Sx, rtol=1e-13)
    # not causal: a change to the last value moves the first output
    v2 = v.copy()
    v2[0, 0, -1] += 1.0
    o2, _, _ = orc.la_variant(q, k, v2, None, orc.MODE_NONCAUSAL, eps=0.0)
    assert np.max(np.abs(o2[0, 0, 0] - o[0, 0, 0])) > 1e-6


def test_decayed_state_closed_form(orc):
    # constant decay a: S_N = a^N S0 + sum_t a^(N-1-t) phi(k_t) v_t^T
    q, k, v = _rand_la(78, 1, 1, 10, 3, 2)
    a = 0.7
    r = _rng(79)
    S0 = r.uniform(size=(1, 1, 3, 2))
    z0 = r.uniform(size=(1, 1, 3))
    _, S, z = orc.la_variant(q, k, v, np.full((1, 1, 10), a), orc.MODE_CAUSAL, S0=S0, z0=z0)
    fk = orc.phi(k[0, 0])
    Sx = a ** 10 * S0[0, 0] + sum(a ** (9 - t) * np.outer(fk[t], v[0, 0, t]) for t in range(10))
    zx = a ** 10 * z0[0, 0] + sum(a ** (9 - t) * fk[t] for t in range(10))
    np.testing.assert_allclose(S[0, 0], Sx, rtol=1e-13)
    np.testing.assert_allclose(z[0, 0], zx, rtol=1e-13)


# --------------------------------------------------------------------------
# gradient (the pages name recomputation; the derivative itself is fixed by
# the forward map): checked against central finite differences of la_recurrent

def _fd_loss(orc, q, k, v, S0, z0, w_o, w_S, w_z, eps):
    o, S, z = orc.la_recurrent(q, k, v, eps=eps, S0=S0, z0=z0)
    return float(np.sum(w_o * o) + np.sum(w_S * S) + np.sum(w_z * z))


@pytest.mark.parametrize("with_state", [False, True], ids=["zero", "state"])
def test_backward_matches_finite_differences(orc, with_state):
    r = _rng(140 + int(with_state))
    B, H, N, dk, dv, eps = 1, 2, 6, 3, 2, 1e-6
    q, k, v = _rand_la(141, B, H, N, dk, dv)
    S0 = r.uniform(size=(B, H, dk, dv)) if with_state else None
    z0 = r.uniform(size=(B, H, dk)) if with_state else None
    w_o = r.normal(size=(B, H, N, dv))        # dO
    w_S = r.normal(size=(B, H, dk, dv))       # dS_N
    w_z = r.normal(size=(B, H, dk))           # dz_N
    dq, dk_, dv_, dS0, dz0 = orc.la_backward(q, k, v, w_o, eps=eps, S0=S0, z0=z0,
                                             dS_N=w_S, dz_N=w_z)
    h = 1e-6
    args = {"q": q, "k": k, "v": v, "S0": S0, "z0": z0}
    grads = {"q": dq, "k": dk_, "v": dv_, "S0": dS0, "z0": dz0}
    for name in (["q", "k", "v"] + (["S0", "z0"] if with_state else [])):
        x = args[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            a_p = dict(args); a_p[name] = xp
            a_m = dict(args); a_m[name] = xm
            num[idx] = (_fd_loss(orc, a_p["q"], a_p["k"], a_p["v"], a_p["S0"], a_p["z0"], w_o, w_S, w_z, eps)
                        - _fd_loss(orc, a_m["q"], a_m["k"], a_m["v"], a_m["S0"], a_m["z0"], w_o, w_S, w_z, eps)) / (2 * h)
        np.testing.assert_allclose(grads[name], num, rtol=1e-6, atol=1e-7, err_msg=name)


def test_backward_state_only_passes_through(orc):
    # with dO = 0 only the final state's gradient flows: S_N = S0 + sum phi(k) v^T,
    # so dS0 = dS_N, dz0 = dz_N, dv_t = dS_N^T phi(k_t), dq = 0
    r = _rng(150)
    q, k, v = _rand_la(151, 1, 1, 5, 3, 2)
    dS = r.normal(size=(1, 1, 3, 2))
    dz = r.normal(size=(1, 1, 3))
    dq, dk_, dv_, dS0, dz0 = orc.la_backward(q, k, v, np.zeros((1, 1, 5, 2)), dS_N=dS, dz_N=dz)
    np.testing.assert_array_equal(dq, 0.0)
    np.testing.assert_allclose(dS0, dS, rtol=0, atol=0)
    np.testing.assert_allclose(dz0, dz, rtol=0, atol=0)
    fk = orc.phi(k)
    for t in range(5):
        np.testing.assert_allclose(dv_[0, 0, t], dS[0, 0].T @ fk[0, 0, t], rtol=1e-13, atol=1e-15)


def test_backward_single_token_closed_form(orc):
    # N = 1 from a zero state: o = v w / (w + eps) with w = phi(q).phi(k), so
    # do/dv = w / (w + eps) times dO exactly
    q, k, v = _rand_la(152, 1, 1, 1, 4, 3)
    dO = _rng(153).normal(size=(1, 1, 1, 3))
    eps = 0.25
    _, _, dv_, _, _ = orc.la_backward(q, k, v, dO, eps=eps)
    w = float(np.sum(orc.phi(q) * orc.phi(k)))
    np.testing.assert_allclose(dv_[0, 0, 0], dO[0, 0, 0] * w / (w + eps), rtol=1e-14)
