"""Pins of the fp64 oracle to facts other than itself (CPU only).

Each test checks the oracle against a closed form, an invariant, a brute-force
construction, or values worked by hand, chosen so that a plausible slip in the
oracle -- a dropped term, a wrong sign or index, a transposed state, a decay
applied at the wrong token -- fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rel(x, ref):
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-300))


def _rand_case(rng, lengths, H, dk, dv, unit_k=True, h0=True, gate_scale=0.1):
    T = sum(lengths)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    la = -np.log1p(np.exp(rng.standard_normal((T, H)))) * gate_scale
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    s0 = rng.standard_normal((len(lengths), H, dk, dv)) * 0.3 if h0 else None
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, la, b, s0, cu


# --- hand-worked values -----------------------------------------------------

def test_hand_cases():
    with open(os.path.join(GOLD, "hand_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        o, hT = oracle.gdn(np.array(c["q"]), np.array(c["k"]), np.array(c["v"]),
                           np.array(c["log_alpha"]), np.array(c["beta"]),
                           np.array(c["h0"]), np.array(c["cu_seqlens"]))
        np.testing.assert_allclose(o, np.array(c["o"]), rtol=0, atol=1e-14, err_msg=c["name"])
        np.testing.assert_allclose(hT, np.array(c["hT"]), rtol=0, atol=1e-14, err_msg=c["name"])
        # the chunked evaluation agrees on the same hand cases (chunk 1 and 64)
        for C in (1, 64):
            oc, hc = oracle.chunked(np.array(c["q"]), np.array(c["k"]), np.array(c["v"]),
                                    np.array(c["log_alpha"]), np.array(c["beta"]),
                                    np.array(c["h0"]), np.array(c["cu_seqlens"]), chunk=C)
            np.testing.assert_allclose(oc, np.array(c["o"]), rtol=0, atol=1e-14)
            np.testing.assert_allclose(hc, np.array(c["hT"]), rtol=0, atol=1e-14)


# --- P1: linear attention equals its quadratic masked form -------------------

@pytest.mark.parametrize("lengths,dk,dv", [([7], 3, 5), ([1, 9, 4], 4, 4), ([33, 0, 17], 8, 6)])
def test_linear_matches_quadratic_form(lengths, dk, dv):
    rng = np.random.default_rng(1)
    q, k, v, _, _, s0, cu = _rand_case(rng, lengths, 2, dk, dv, unit_k=False)
    o, hT = oracle.linear(q, k, v, s0, cu)
    oq, hq = oracle.linear_quadratic(q, k, v, s0, cu)
    assert _rel(o, oq) < 1e-13
    assert _rel(hT, hq) < 1e-13


def test_linear_quadratic_is_brute_force_sum():
    # (Q K^T ⊙ M) V written as the explicit double sum, tiny case
    rng = np.random.default_rng(2)
    T, dk, dv = 5, 2, 3
    q = rng.standard_normal((T, 1, dk)); k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    oq, _ = oracle.linear_quadratic(q, k, v)
    for t in range(T):
        ref = sum(float(q[t, 0] @ k[s, 0]) * v[s, 0] for s in range(t + 1))
        np.testing.assert_allclose(oq[t, 0], ref, rtol=1e-14, atol=1e-14)


# --- P2: with ||k||=1 and beta=1 the updated state stores v under key k ------

@pytest.mark.parametrize("dk,dv", [(3, 5), (16, 16), (64, 8)])
def test_delta_rule_overwrite_invariant(dk, dv):
    rng = np.random.default_rng(3)
    q, k, v, la, _, s0, cu = _rand_case(rng, [11, 6], 3, dk, dv, gate_scale=1.0)
    beta = np.ones(la.shape)
    # o_t = S_t q_t, so asking with q_t = k_t reads back S_t k_t, which must be v_t
    o, _ = oracle.gdn(k, k, v, la, beta, s0, cu)
    assert np.max(np.abs(o - v)) < 1e-13
    # and through the chunked form
    oc, _ = oracle.chunked(k, k, v, la, beta, s0, cu, chunk=4)
    assert np.max(np.abs(oc - v)) < 1e-12
    # with beta < 1 the invariant must NOT hold (the test has teeth)
    o2, _ = oracle.gdn(k, k, v, la, beta * 0.5, s0, cu)
    assert np.max(np.abs(o2 - v)) > 1e-3


# --- P3: chunk-wise evaluation equals the token recurrence -------------------

@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("delta", [True, False])
def test_chunked_equals_recurrent(C, delta):
    rng = np.random.default_rng(4)
    lengths = [1, 70, 0, 129, 64, 5]
    q, k, v, la, b, s0, cu = _rand_case(rng, lengths, 2, 8, 6)
    o, hT = oracle.recurrent(q, k, v, la, b, s0, cu, delta_rule=delta)
    oc, hc = oracle.chunked(q, k, v, la, b, s0, cu, chunk=C, delta_rule=delta)
    assert _rel(oc, o) < 1e-12
    assert _rel(hc, hT) < 1e-12


def test_chunked_strong_gates():
    # strongly negative log-gates: the chunked form must not form exp(g_i)*exp(-g_j)
    rng = np.random.default_rng(5)
    q, k, v, la, b, s0, cu = _rand_case(rng, [150], 1, 8, 8)
    la = la * 0 - 30.0  # alpha = e^-30 per token: g reaches -1920 in a 64-chunk
    o, hT = oracle.gdn(q, k, v, la, b, s0, cu)
    oc, hc = oracle.chunked(q, k, v, la, b, s0, cu, chunk=64)
    assert np.all(np.isfinite(oc))
    assert _rel(oc, o) < 1e-12 and _rel(hc, hT) < 1e-12


# --- P4: beta = 0 leaves only the decayed initial state ----------------------

def test_beta_zero_closed_form():
    rng = np.random.default_rng(6)
    q, k, v, la, _, s0, cu = _rand_case(rng, [9, 4], 2, 5, 3)
    beta = np.zeros(la.shape)
    o, hT = oracle.gdn(q, k, v, la, beta, s0, cu)
    for s in range(2):
        a, e = cu[s], cu[s + 1]
        for h in range(2):
            G = np.cumsum(la[a:e, h])
            ref = np.exp(G)[:, None] * (q[a:e, h] @ s0[s, h])
            np.testing.assert_allclose(o[a:e, h], ref, rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(hT[s, h], np.exp(G[-1]) * s0[s, h], rtol=1e-13)


# --- P5: decay without the delta term has a masked closed form ---------------

def test_decay_without_delta_closed_form():
    rng = np.random.default_rng(7)
    q, k, v, la, b, s0, cu = _rand_case(rng, [12], 1, 4, 3, unit_k=False, gate_scale=0.5)
    o, hT = oracle.recurrent(q, k, v, la, b, s0, cu, delta_rule=False)
    G = np.cumsum(la[:, 0])
    D = np.tril(np.exp(G[:, None] - G[None, :]))
    Q, K, V = q[:, 0], k[:, 0], v[:, 0] * b[:, 0:1]
    ref = (Q @ K.T * D) @ V + np.exp(G)[:, None] * (Q @ s0[0, 0])
    np.testing.assert_allclose(o[:, 0], ref, rtol=1e-12, atol=1e-13)
    refh = np.exp(G[-1]) * s0[0, 0] + (K * np.exp(G[-1] - G)[:, None]).T @ V
    np.testing.assert_allclose(hT[0, 0], refh, rtol=1e-12, atol=1e-13)


# --- P7: explicit solution of the linear recurrence on tiny inputs -----------

def test_transition_matrix_product():
    rng = np.random.default_rng(8)
    T, dk, dv = 6, 3, 2
    q, k, v, la, b, s0, cu = _rand_case(rng, [T], 1, dk, dv, unit_k=False, gate_scale=1.0)
    o, hT = oracle.gdn(q, k, v, la, b, s0, cu)
    # S_t = S_{t-1} M_t + b_t v_t k_t^T with M_t = a_t (I - b_t k_t k_t^T) (dk x dk)
    M = [math.exp(la[t, 0]) * (np.eye(dk) - b[t, 0] * np.outer(k[t, 0], k[t, 0])) for t in range(T)]
    S0 = s0[0, 0].T
    for t in range(T):
        # S_t = S0 M_1..M_t + sum_{r<=t} b_r v_r k_r^T M_{r+1}..M_t
        P = np.eye(dk)
        for r in range(t + 1):
            P = P @ M[r]
        St = S0 @ P
        for r in range(t + 1):
            Pr = np.eye(dk)
            for x in range(r + 1, t + 1):
                Pr = Pr @ M[x]
            St = St + b[r, 0] * np.outer(v[r, 0], k[r, 0]) @ Pr
        np.testing.assert_allclose(o[t, 0], St @ q[t, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hT[0, 0], St.T, rtol=1e-12, atol=1e-13)


# --- P8: sequences are independent; h_T chains into h0 ----------------------

def test_varlen_packing_and_state_chaining():
    rng = np.random.default_rng(9)
    lengths = [5, 0, 13, 2]
    q, k, v, la, b, s0, cu = _rand_case(rng, lengths, 2, 4, 4)
    o, hT = oracle.gdn(q, k, v, la, b, s0, cu)
    for s in range(len(lengths)):
        a, e = cu[s], cu[s + 1]
        os_, hs = oracle.gdn(q[a:e], k[a:e], v[a:e], la[a:e], b[a:e], s0[s:s + 1])
        np.testing.assert_array_equal(o[a:e], os_)
        np.testing.assert_array_equal(hT[s:s + 1], hs)
    # a zero-length sequence returns its initial state
    np.testing.assert_array_equal(hT[1], s0[1])
    # splitting sequence 2 in two calls, h_T of the first as h0 of the second
    a, e = cu[2], cu[3]
    m = a + 6
    o1, h1 = oracle.gdn(q[a:m], k[a:m], v[a:m], la[a:m], b[a:m], s0[2:3])
    o2, h2 = oracle.gdn(q[m:e], k[m:e], v[m:e], la[m:e], b[m:e], h1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o[a:e], rtol=0, atol=0)
    np.testing.assert_allclose(h2, hT[2:3], rtol=0, atol=0)


# --- P9: the per-chunk affine maps compose to the final state ----------------

def test_affine_chunk_maps_compose():
    """SparseGDN article, "Схема встраивания селектора…": each chunk acts on the
    state as an affine map S -> A_c S + B_c.  In h = S^T form, from the chunked
    oracle's w, u, g:  h -> (e^{g_C} I - K~^T W) h + K~^T U  with K~ = e^{g_C-g} K."""
    rng = np.random.default_rng(10)
    C = 8
    lengths = [29]
    q, k, v, la, b, s0, cu = _rand_case(rng, lengths, 1, 6, 5)
    _, hT = oracle.gdn(q, k, v, la, b, s0, cu)
    _, _, it = oracle.chunked(q, k, v, la, b, s0, cu, chunk=C, intermediates=True)
    h = s0[0, 0].copy()
    for c0 in range(0, lengths[0], C):
        c1 = min(c0 + C, lengths[0])
        g = it["g"][c0:c1, 0]
        Kt = k[c0:c1, 0] * np.exp(g[-1] - g)[:, None]
        Mc = np.exp(g[-1]) * np.eye(6) - Kt.T @ it["w"][c0:c1, 0]
        Bc = Kt.T @ it["u"][c0:c1, 0]
        h = Mc @ h + Bc
    assert _rel(h, hT[0, 0]) < 1e-12


def test_wy_intermediates_solve_the_delta_system():
    # Tm really is (I + A)^-1 and A is the beta-scaled, decay-masked K K^T
    rng = np.random.default_rng(11)
    q, k, v, la, b, s0, cu = _rand_case(rng, [40], 1, 8, 4)
    _, _, it = oracle.chunked(q, k, v, la, b, s0, cu, chunk=16, intermediates=True)
    for c in range(3):
        A, Tm = it["A"][c, 0], it["Tm"][c, 0]
        n = min(16, 40 - 16 * c)
        np.testing.assert_allclose(Tm @ (np.eye(16) + A), np.eye(16), atol=1e-12)
        t0 = 16 * c
        for i in range(n):
            for j in range(16):
                expect = 0.0
                if j < i:
                    gi = np.sum(la[t0:t0 + i + 1, 0]); gj = np.sum(la[t0:t0 + j + 1, 0])
                    expect = b[t0 + i, 0] * np.exp(gi - gj) * (k[t0 + i, 0] @ k[t0 + j, 0])
                assert abs(A[i, j] - expect) < 1e-13


# --- block-adjacent solver (SparseGDN article, first observation) -----------

@pytest.mark.parametrize("band", [32, 64, 128])
def test_block_adjacent_is_exact_when_two_blocks_cover_the_chunk(band):
    """With blocks of half a chunk or more no block is two blocks below
    another, so the banded solve is the exact one."""
    rng = np.random.default_rng(21)
    q, k, v, la, b, s0, cu = _rand_case(rng, [150, 64, 5], 2, 8, 6)
    oe, he = oracle.chunked(q, k, v, la, b, s0, cu, chunk=64)
    ob, hb = oracle.chunked(q, k, v, la, b, s0, cu, chunk=64, band=band)
    assert _rel(ob, oe) < 1e-13 and _rel(hb, he) < 1e-13


def test_block_adjacent_is_exact_for_keys_orthogonal_across_blocks():
    """Keys of different 16-token blocks on disjoint coordinates: A has no
    links between blocks, the inverse is block-diagonal, and dropping the
    far blocks changes nothing (while it does change a generic input)."""
    rng = np.random.default_rng(22)
    T, H, dk, dv = 128, 2, 8, 5
    q, k, v, la, b, s0, cu = _rand_case(rng, [T], H, dk, dv, unit_k=False)
    for t in range(T):
        blk = (t % 64) // 16
        mask = np.zeros(dk)
        mask[2 * blk:2 * blk + 2] = 1.0
        k[t] *= mask
    oe, he = oracle.chunked(q, k, v, la, b, s0, cu, chunk=64)
    ob, hb = oracle.chunked(q, k, v, la, b, s0, cu, chunk=64, band=16)
    assert _rel(ob, oe) < 1e-13 and _rel(hb, he) < 1e-13
    q, k, v, la, b, s0, cu = _rand_case(rng, [T], H, dk, dv, unit_k=False)
    oe, _ = oracle.chunked(q, k, v, la, b, s0, cu, chunk=64)
    ob, _ = oracle.chunked(q, k, v, la, b, s0, cu, chunk=64, band=16)
    assert _rel(ob, oe) > 1e-6


def test_block_adjacent_keeps_exactly_the_two_diagonals_of_blocks():
    """The banded Tm is the exact inverse with the blocks two or more below
    the diagonal set to zero, and w, u are that Tm applied to b e^g K and
    b V: blocks one below the diagonal are kept, farther ones dropped."""
    rng = np.random.default_rng(23)
    q, k, v, la, b, s0, cu = _rand_case(rng, [64, 40], 1, 6, 4, unit_k=False)
    _, _, ex = oracle.chunked(q, k, v, la, b, s0, cu, chunk=64, intermediates=True)
    _, _, bd = oracle.chunked(q, k, v, la, b, s0, cu, chunk=64, intermediates=True, band=16)
    blk = np.arange(64) // 16
    far = (blk[:, None] - blk[None, :]) >= 2
    for c in range(ex["Tm"].shape[0]):
        Te, Tb = ex["Tm"][c, 0], bd["Tm"][c, 0]
        np.testing.assert_array_equal(Tb[far], 0.0)
        np.testing.assert_array_equal(Tb[~far], Te[~far])
        assert np.any(Te[(blk[:, None] - blk[None, :]) == 1] != 0.0)
    for s in range(2):
        a, e = int(cu[s]), int(cu[s + 1])
        n = e - a
        Tb = bd["Tm"][s, 0][:n, :n]
        g = np.cumsum(la[a:e, 0])
        np.testing.assert_allclose(bd["w"][a:e, 0], Tb @ (b[a:e, 0, None] * np.exp(g)[:, None] * k[a:e, 0]),
                                   rtol=0, atol=1e-12)
        np.testing.assert_allclose(bd["u"][a:e, 0], Tb @ (b[a:e, 0, None] * v[a:e, 0]), rtol=0, atol=1e-12)


# --- linear-attention variants: causal or bidirectional, normalised or not ---

def _positive_case(rng, lengths, H, dk, dv):
    T = sum(lengths)
    elu1 = lambda x: np.where(x > 0, x + 1.0, np.exp(x))  # elu(x) + 1 > 0
    q = elu1(rng.standard_normal((T, H, dk)))
    k = elu1(rng.standard_normal((T, H, dk)))
    v = rng.standard_normal((T, H, dv))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, cu


def test_linear_variants_brute_force():
    """Element by element: o_t[j] = sum_s (q_t . k_s) v_s[j] / sum_s (q_t . k_s)
    over the causal or the whole range, with explicit loops."""
    rng = np.random.default_rng(31)
    q, k, v, cu = _positive_case(rng, [5, 0, 3], 2, 3, 2)
    for causal in (True, False):
        for norm in (True, False):
            o, kv, z = oracle.linear_variant(q, k, v, cu, causal=causal, normalize=norm)
            for sq in range(2):
                a, e = int(cu[sq]), int(cu[sq + 1])
                for h in range(2):
                    for t in range(a, e):
                        top = np.zeros(2)
                        bot = 0.0
                        for u in range(a, (t + 1) if causal else e):
                            w = sum(q[t, h, x] * k[u, h, x] for x in range(3))
                            top += w * v[u, h]
                            bot += w
                        ref = top / bot if norm else top
                        np.testing.assert_allclose(o[t, h], ref, rtol=1e-13, atol=1e-13)
                    np.testing.assert_allclose(z[sq, h], k[a:e, h].sum(axis=0), rtol=1e-13)
                    ref_kv = sum(np.outer(k[u, h], v[u, h]) for u in range(a, e)) if e > a else 0.0
                    np.testing.assert_allclose(kv[sq, h], ref_kv, rtol=1e-13, atol=1e-13)
            kv2, z2 = oracle.linear_sums(k, v, cu)
            np.testing.assert_allclose(kv2, kv, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(z2, z, rtol=1e-13, atol=1e-13)


def test_normalised_weights_sum_to_one():
    """With positive features the normalised weights of a token sum to one, so
    a value that is the same vector c for every token comes out as c."""
    rng = np.random.default_rng(32)
    q, k, v, cu = _positive_case(rng, [40, 7], 3, 8, 5)
    c = rng.standard_normal(5)
    v[:] = c
    for causal in (True, False):
        o, _, _ = oracle.linear_variant(q, k, v, cu, causal=causal, normalize=True)
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=1e-12, atol=1e-12)


def test_causal_variants_first_token_and_recurrence():
    """The causal normalised output of a sequence's first token is its own
    value; the causal unnormalised output is the plain recurrence."""
    rng = np.random.default_rng(33)
    q, k, v, cu = _positive_case(rng, [12, 1, 9], 2, 4, 3)
    o, _, _ = oracle.linear_variant(q, k, v, cu, causal=True, normalize=True)
    for sq in range(3):
        a = int(cu[sq])
        np.testing.assert_allclose(o[a], v[a], rtol=1e-13, atol=1e-13)
    o, kv, _ = oracle.linear_variant(q, k, v, cu, causal=True, normalize=False)
    ro, rh = oracle.linear(q, k, v, None, cu)
    assert _rel(o, ro) < 1e-13 and _rel(kv, rh) < 1e-13


def test_bidirectional_is_order_free_and_reassociates():
    """Bidirectional outputs do not depend on the order of the sequence's
    tokens (permuting k and v together leaves every o_t unchanged), and they
    equal the reassociated evaluation q_t (K^T V) / (q_t . K^T 1)."""
    rng = np.random.default_rng(34)
    q, k, v, cu = _positive_case(rng, [30], 2, 6, 4)
    for norm in (True, False):
        o, kv, z = oracle.linear_variant(q, k, v, cu, causal=False, normalize=norm)
        perm = rng.permutation(30)
        o2, _, _ = oracle.linear_variant(q, k[perm], v[perm], cu, causal=False, normalize=norm)
        np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-12)
        for h in range(2):
            num = q[:, h] @ kv[0, h]
            ref = num / (q[:, h] @ z[0, h])[:, None] if norm else num
            np.testing.assert_allclose(o[:, h], ref, rtol=1e-12, atol=1e-12)
    o, _, _ = oracle.linear_variant(q, k, v, cu, causal=True, normalize=True)
    o2, _, _ = oracle.linear_variant(q, k[perm], v[perm], cu, causal=True, normalize=True)
    assert _rel(o2, o) > 1e-3  # the causal form does depend on the order


def test_decode_step_equals_one_prefill_token():
    rng = np.random.default_rng(12)
    B, H, dk, dv = 3, 2, 5, 4
    q, k, v, la, b, s0, cu = _rand_case(rng, [1] * B, H, dk, dv)
    o, st = oracle.decode_step(q, k, v, la, b, s0)
    for i in range(B):
        o1, h1 = oracle.gdn(q[i:i + 1], k[i:i + 1], v[i:i + 1], la[i:i + 1], b[i:i + 1], s0[i:i + 1])
        np.testing.assert_array_equal(o[i:i + 1], o1)
        np.testing.assert_array_equal(st[i:i + 1], h1)


def test_oracle_rejects_bad_seqlens():
    rng = np.random.default_rng(13)
    q, k, v, la, b, s0, cu = _rand_case(rng, [4, 4], 1, 2, 2)
    with pytest.raises(ValueError):
        oracle.gdn(q, k, v, la, b, s0, np.array([0, 5, 3, 8]))


# --- the pins have teeth: planted mistakes in a private copy of the oracle ---
#
# Each entry is a plausible slip in the oracle's arithmetic (a dropped factor, a
# wrong sign, a wrong operand or index, a transposed read-back, a mask off by
# one, a decay taken the wrong way).  It is made in a copy of gdn_oracle.c
# compiled beside the test; the pins above, run against that copy, must reject
# every one of them.  The oracle itself is not changed.

MUTATIONS = {
    "delta term without the decay": ("x -= b * (a * Sk[j]) * kt[i];", "x -= b * Sk[j] * kt[i];"),
    "delta term with the wrong sign": ("x -= b * (a * Sk[j]) * kt[i];", "x += b * (a * Sk[j]) * kt[i];"),
    "write term without beta": ("x += b * vt[j] * kt[i];", "x += vt[j] * kt[i];"),
    "output read with k instead of q": ("acc += S[(size_t)j * dk + i] * qt[i];", "acc += S[(size_t)j * dk + i] * kt[i];"),
    "decay with the wrong sign": ("exp(log_alpha[row])", "exp(-log_alpha[row])"),
    "final state read back transposed": ("= S[(size_t)j * dk + i];", "= S[(size_t)(i % dv) * dk + (j % dk)];"),
    "chunk: decay factor reversed in A": ("bi * exp(g[i] - g[j]) * kk;", "bi * exp(g[j] - g[i]) * kk;"),
    "chunk: A including the diagonal": ("for (int j = 0; j < i; ++j) {\n                        double kk",
                                        "for (int j = 0; j <= i; ++j) {\n                        double kk"),
    "chunk: u without beta": ("acc += Tm[(size_t)i * C + j] * bj * v[ROW(j) * dv + y];",
                              "acc += Tm[(size_t)i * C + j] * v[ROW(j) * dv + y];"),
    "chunk: intra-chunk mask missing the diagonal": ("for (int j = 0; j <= i; ++j) {\n                        double qk",
                                                     "for (int j = 0; j < i; ++j) {\n                        double qk"),
    "chunk: state carried without the decay": ("double acc = exp(gl) * h[(size_t)x * dv + y];",
                                               "double acc = h[(size_t)x * dv + y];"),
    "band: the blocks right below the diagonal dropped too": ("if (i / band - col / band >= 2)",
                                                             "if (i / band - col / band >= 1)"),
    "band: no block dropped": ("if (i / band - col / band >= 2)", "if (i / band - col / band >= 4)"),
}

PINS = [
    ("hand cases", lambda: test_hand_cases()),
    ("overwrite invariant", lambda: test_delta_rule_overwrite_invariant(16, 16)),
    ("chunked = recurrent", lambda: test_chunked_equals_recurrent(16, True)),
    ("chunked = recurrent, no delta", lambda: test_chunked_equals_recurrent(4, False)),
    ("linear = quadratic form", lambda: test_linear_matches_quadratic_form([7, 0, 33], 5, 3)),
    ("beta = 0 closed form", lambda: test_beta_zero_closed_form()),
    ("decay without delta closed form", lambda: test_decay_without_delta_closed_form()),
    ("transition-matrix product", lambda: test_transition_matrix_product()),
    ("WY intermediates", lambda: test_wy_intermediates_solve_the_delta_system()),
    ("banded solve keeps two block diagonals", lambda: test_block_adjacent_keeps_exactly_the_two_diagonals_of_blocks()),
    ("banded solve exact for orthogonal blocks", lambda: test_block_adjacent_is_exact_for_keys_orthogonal_across_blocks()),
]


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    import subprocess

    old, new = MUTATIONS[name]
    src_path = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")
    with open(src_path) as f:
        src = f.read()
    assert src.count(old) == 1, "mutation site not unique: " + name
    mutant = tmp_path / "gdn_oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", str(lib), str(mutant), "-lm"],
                   check=True)
    caught = []
    with oracle.using_library(str(lib)):
        for pin, check in PINS:
            try:
                check()
            except Exception:  # an assertion, or a NaN the comparison trips over
                caught.append(pin)
    assert caught, "no pin rejects the planted mistake: " + name
