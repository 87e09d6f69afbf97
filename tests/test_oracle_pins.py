"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test checks the oracle against brute force on tiny inputs, a closed form, an
invariant of the recurrence, a hand-worked example (tests/golden/) or an independent
library routine, so that a dropped term, a wrong sign or index or a transposed operand
in the oracle fails at least one of them.

Recurrence (state [Dk, Dv]): S_t = exp(g_t)(I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
o_t = scale S_t^T q_t. Shapes and head mapping: "GDN CTE Kernel API Reference"
(parameters; Notes: value head h reads key head h // (Hv//Hk)). Decode step: "GDN TKG
Kernel API Reference" (Background: l2norm, sigmoid, softplus gate, RMSNormGated).
"""
import numpy as np
import pytest
from scipy.special import expit

from conftest import read_golden, rel_fro


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_prefill(rng, B, Hk, Hv, S, Dk, Dv, *, unit=True, g=(-0.5, -0.01),
                 beta=(0.05, 0.95), state=True):
    q = rng.standard_normal((B, Hk, S, Dk))
    k = rng.standard_normal((B, Hk, S, Dk))
    if unit:
        q, k = _unit(q), _unit(k)
    v = rng.standard_normal((B, Hv, S, Dv))
    gl = rng.uniform(g[0], g[1], (B, Hv, S))
    be = rng.uniform(beta[0], beta[1], (B, Hv, S))
    s0 = rng.standard_normal((B, Hv, Dk, Dv)) * 0.3 if state else None
    return q, k, v, gl, be, s0


def brute_force_head(q, k, v, g, beta, scale, s0):
    """One head, from explicit dense matrices M_t = exp(g_t)(I - beta_t k_t k_t^T):
    S_t = (M_t...M_1) S_0 + sum_s (M_t...M_{s+1}) beta_s k_s v_s^T, o_t = scale S_t^T q_t."""
    S, Dk = k.shape
    Dv = v.shape[1]
    M = [np.exp(g[t]) * (np.eye(Dk) - beta[t] * np.outer(k[t], k[t])) for t in range(S)]
    outs, St = [], None
    for t in range(S):
        prod = np.eye(Dk)
        St = np.zeros((Dk, Dv))
        for s in range(t, -1, -1):
            St = St + prod @ (beta[s] * np.outer(k[s], v[s]))
            prod = prod @ M[s]
        St = St + prod @ s0
        outs.append(scale * St.T @ q[t])
    return np.array(outs), St


# ----------------------------------------------------------------------------- prefill


@pytest.mark.parametrize("Hk,Hv,unit", [(1, 1, True), (1, 2, True), (2, 4, False)])
def test_prefill_matches_dense_brute_force(oracle_mod, Hk, Hv, unit):
    rng = np.random.default_rng(1)
    B, S, Dk, Dv, scale = 2, 9, 3, 5, 0.7
    q, k, v, g, be, s0 = rand_prefill(rng, B, Hk, Hv, S, Dk, Dv, unit=unit)
    out, st = oracle_mod.prefill(q, k, v, g, be, scale, s0)
    G = Hv // Hk
    for b in range(B):
        for h in range(Hv):
            kh = h // G
            o_ref, s_ref = brute_force_head(q[b, kh], k[b, kh], v[b, h], g[b, h], be[b, h],
                                            scale, s0[b, h])
            assert rel_fro(out[b, h], o_ref) < 1e-12
            assert rel_fro(st[b, h], s_ref) < 1e-12


def test_identity_when_beta_and_g_vanish(oracle_mod):
    rng = np.random.default_rng(2)
    q, k, v, g, be, s0 = rand_prefill(rng, 1, 2, 2, 7, 4, 6)
    g[:] = 0.0
    be[:] = 0.0
    out, st = oracle_mod.prefill(q, k, v, g, be, 0.5, s0)
    np.testing.assert_allclose(st, s0, rtol=0, atol=1e-15)
    expect = 0.5 * np.einsum("bhsk,bhkv->bhsv", q, s0)
    np.testing.assert_allclose(out, expect, rtol=1e-13, atol=1e-15)


def test_pure_decay_when_beta_vanishes(oracle_mod):
    rng = np.random.default_rng(3)
    q, k, v, g, be, s0 = rand_prefill(rng, 2, 1, 1, 11, 5, 3)
    be[:] = 0.0
    out, st = oracle_mod.prefill(q, k, v, g, be, 1.0, s0)
    decay = np.exp(np.cumsum(g, axis=-1))  # [B,H,S]
    np.testing.assert_allclose(st, decay[..., -1, None, None] * s0, rtol=1e-13)
    expect = decay[..., None] * np.einsum("bhsk,bhkv->bhsv", q, s0)
    np.testing.assert_allclose(out, expect, rtol=1e-12, atol=1e-15)


def test_exact_write_then_read(oracle_mod):
    """g = 0, beta = 1, |k| = 1: the update makes S_t^T k_t = v_t. Reading with q = k
    and scale 1 returns v_t at every step, whatever the history."""
    rng = np.random.default_rng(4)
    q, k, v, g, be, s0 = rand_prefill(rng, 1, 3, 3, 13, 6, 4)
    g[:] = 0.0
    be[:] = 1.0
    out, _ = oracle_mod.prefill(k, k, v, g, be, 1.0, s0)
    np.testing.assert_allclose(out, v, rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_form_an_associative_memory(oracle_mod):
    """With orthonormal keys, g = 0, beta = 1 and S_0 = 0, every write leaves the others
    intact: S_T = sum_i k_i v_i^T = K^T V, and S_T^T k_i = v_i for every i."""
    rng = np.random.default_rng(5)
    D, Dv = 8, 5
    K = np.linalg.qr(rng.standard_normal((D, D)))[0].T  # rows orthonormal
    V = rng.standard_normal((D, Dv))
    q = K[None, None]
    k = K[None, None]
    v = V[None, None]
    g = np.zeros((1, 1, D))
    be = np.ones((1, 1, D))
    _, st = oracle_mod.prefill(q, k, v, g, be, 1.0, None)
    np.testing.assert_allclose(st[0, 0], K.T @ V, atol=1e-13)
    np.testing.assert_allclose(st[0, 0].T @ K.T, V.T, atol=1e-13)


def test_first_token_from_zero_state(oracle_mod):
    rng = np.random.default_rng(6)
    q, k, v, g, be, _ = rand_prefill(rng, 2, 2, 4, 1, 5, 7, state=False)
    out, st = oracle_mod.prefill(q, k, v, g, be, 0.3, None)
    G = 2
    for b in range(2):
        for h in range(4):
            kk, qq = k[b, h // G, 0], q[b, h // G, 0]
            np.testing.assert_allclose(st[b, h], be[b, h, 0] * np.outer(kk, v[b, h, 0]),
                                       rtol=1e-13)
            np.testing.assert_allclose(out[b, h, 0],
                                       0.3 * be[b, h, 0] * (kk @ qq) * v[b, h, 0], rtol=1e-12)


def test_strong_decay_forgets_history(oracle_mod):
    """g = -1e4 makes exp(g) = 0 in fp64: each step restarts from beta_t k_t v_t^T."""
    rng = np.random.default_rng(7)
    q, k, v, g, be, s0 = rand_prefill(rng, 1, 1, 1, 6, 4, 4)
    g[:] = -1e4
    out, st = oracle_mod.prefill(q, k, v, g, be, 1.0, s0)
    kk, qq, vv, bb = k[0, 0], q[0, 0], v[0, 0], be[0, 0]
    np.testing.assert_allclose(st[0, 0], bb[-1] * np.outer(kk[-1], vv[-1]), rtol=1e-13)
    expect = (bb * np.einsum("sk,sk->s", kk, qq))[:, None] * vv
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-12)


def test_state_norm_bound(oracle_mod):
    """|k| = 1, beta in (0,1): ||I - beta k k^T||_2 = 1, so
    ||S_t||_2 <= exp(g_t) ||S_{t-1}||_2 + beta_t ||v_t||."""
    rng = np.random.default_rng(8)
    q, k, v, g, be, s0 = rand_prefill(rng, 1, 1, 1, 40, 6, 6, g=(-0.05, 0.0))
    st = s0
    for t in range(40):
        sl = slice(t, t + 1)
        _, nxt = oracle_mod.prefill(q[:, :, sl], k[:, :, sl], v[:, :, sl], g[:, :, sl],
                                    be[:, :, sl], 1.0, st)
        bound = (np.exp(g[0, 0, t]) * np.linalg.norm(st[0, 0], 2)
                 + be[0, 0, t] * np.linalg.norm(v[0, 0, t]))
        assert np.linalg.norm(nxt[0, 0], 2) <= bound * (1 + 1e-12)
        st = nxt


def test_gqa_head_map_is_repeat_interleave(oracle_mod):
    """Value head h reads key head h // (Hv // Hk). Expanding q,k by repeating each key
    head G times in place must give the same result; tiling them must not."""
    rng = np.random.default_rng(9)
    Hk, G = 2, 3
    q, k, v, g, be, s0 = rand_prefill(rng, 1, Hk, Hk * G, 10, 4, 5)
    out, st = oracle_mod.prefill(q, k, v, g, be, 0.9, s0)
    out_r, st_r = oracle_mod.prefill(np.repeat(q, G, axis=1), np.repeat(k, G, axis=1), v, g,
                                     be, 0.9, s0)
    np.testing.assert_allclose(out, out_r, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(st, st_r, rtol=1e-14, atol=1e-15)
    out_t, _ = oracle_mod.prefill(np.tile(q, (1, G, 1, 1)), np.tile(k, (1, G, 1, 1)), v, g,
                                  be, 0.9, s0)
    assert rel_fro(out_t, out) > 1e-2


def test_heads_and_batches_are_independent(oracle_mod):
    rng = np.random.default_rng(10)
    q, k, v, g, be, s0 = rand_prefill(rng, 3, 2, 4, 8, 4, 4)
    out, st = oracle_mod.prefill(q, k, v, g, be, 1.0, s0)
    perm = [2, 0, 1]
    out_p, st_p = oracle_mod.prefill(q[perm], k[perm], v[perm], g[perm], be[perm], 1.0,
                                     s0[perm])
    np.testing.assert_array_equal(out_p, out[perm])
    np.testing.assert_array_equal(st_p, st[perm])
    v2 = v.copy()
    v2[:, 1] += 1.0  # touch value head 1 only
    out2, _ = oracle_mod.prefill(q, k, v2, g, be, 1.0, s0)
    np.testing.assert_array_equal(out2[:, [0, 2, 3]], out[:, [0, 2, 3]])
    assert rel_fro(out2[:, 1], out[:, 1]) > 1e-3


def test_split_and_carry(oracle_mod):
    """Prefill of tokens [0,s) then of [s,S) from the carried state equals one prefill:
    the supplied state is the initial state ("GDN CTE Kernel API Reference",
    :param recurrent_state:)."""
    rng = np.random.default_rng(11)
    q, k, v, g, be, s0 = rand_prefill(rng, 2, 2, 4, 96, 8, 6)
    out, st = oracle_mod.prefill(q, k, v, g, be, 0.4, s0)
    for s in (1, 64, 95):
        a, b_ = slice(0, s), slice(s, 96)
        o1, s1 = oracle_mod.prefill(q[:, :, a], k[:, :, a], v[:, :, a], g[:, :, a],
                                    be[:, :, a], 0.4, s0)
        o2, s2 = oracle_mod.prefill(q[:, :, b_], k[:, :, b_], v[:, :, b_], g[:, :, b_],
                                    be[:, :, b_], 0.4, s1)
        np.testing.assert_allclose(np.concatenate([o1, o2], axis=2), out, rtol=1e-12,
                                   atol=1e-13)
        np.testing.assert_allclose(s2, st, rtol=1e-12, atol=1e-13)


def test_prefill_hand_worked_example(oracle_mod):
    gd = read_golden("prefill_hand_2x2.txt")
    q = gd["q"].reshape(1, 1, 2, 2)
    k = gd["k"].reshape(1, 1, 2, 2)
    v = gd["v"].reshape(1, 1, 2, 2)
    g = gd["g_log"].reshape(1, 1, 2)
    be = gd["beta"].reshape(1, 1, 2)
    s0 = gd["state0"].reshape(1, 1, 2, 2)
    out, st = oracle_mod.prefill(q, k, v, g, be, 1.0, s0)
    np.testing.assert_allclose(out.ravel(), gd["out"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(st.ravel(), gd["state"], rtol=1e-14, atol=1e-15)


# ----------------------------------------------------------------------- chunked form


@pytest.mark.parametrize("C", [1, 2, 16, 64, 128])
def test_chunked_form_equals_recurrence(oracle_mod, C):
    """The chunk-parallel (WY) algebra reproduces the token recurrence for every chunk
    size, including a ragged last chunk (S = 200 is no multiple of 16, 64 or 128)."""
    rng = np.random.default_rng(12)
    q, k, v, g, be, s0 = rand_prefill(rng, 1, 2, 4, 200, 16, 24, g=(-1.0, -0.001))
    out, st = oracle_mod.prefill(q, k, v, g, be, 0.25, s0)
    out_c, st_c = oracle_mod.prefill_chunked(q, k, v, g, be, 0.25, C, s0)
    assert rel_fro(out_c, out) < 1e-12
    assert rel_fro(st_c, st) < 1e-12


def test_chunked_form_zero_state(oracle_mod):
    rng = np.random.default_rng(13)
    q, k, v, g, be, _ = rand_prefill(rng, 2, 1, 1, 128, 8, 8, state=False)
    out, st = oracle_mod.prefill(q, k, v, g, be, 1.0, None)
    out_c, st_c = oracle_mod.prefill_chunked(q, k, v, g, be, 1.0, 64, None)
    assert rel_fro(out_c, out) < 1e-12 and rel_fro(st_c, st) < 1e-12


def test_unit_lower_inverse(oracle_mod):
    """T = (I + A)^-1 for strictly lower A: checked by T (I + A) = I and by the Neumann
    series sum_{n<N} (-A)^n, which is exact because A^N = 0."""
    rng = np.random.default_rng(14)
    N = 64
    kk = _unit(rng.standard_normal((N, 16)))
    gam = np.cumsum(rng.uniform(-0.5, -0.01, N))
    be = rng.uniform(0.05, 0.95, N)
    A = np.tril(be[:, None] * (kk @ kk.T) * np.exp(gam[:, None] - gam[None, :]), -1)
    T = oracle_mod.unit_lower_inverse(A)
    np.testing.assert_allclose(T @ (np.eye(N) + A), np.eye(N), atol=1e-12)
    neu = np.zeros((N, N))
    p = np.eye(N)
    for _ in range(N):
        neu += p
        p = p @ (-A)
    np.testing.assert_allclose(T, neu, rtol=1e-10, atol=1e-12)
    assert np.allclose(np.triu(T, 1), 0.0) and np.allclose(np.diag(T), 1.0)


# ------------------------------------------------------------------------ decode step


def rand_decode(rng, BH, H, K, V):
    return dict(q=rng.standard_normal((BH, K)), k=rng.standard_normal((BH, K)),
                v=rng.standard_normal((BH, V)), b=rng.standard_normal(BH),
                a=rng.standard_normal(BH), A_log=rng.uniform(-2, 1, H),
                dt_bias=rng.uniform(-1, 1, H), z=rng.standard_normal((BH, V)),
                norm_weight=rng.uniform(0.5, 1.5, V),
                state_in=rng.standard_normal((BH, K, V)) * 0.05, num_v_heads=H)


def _gates(d):
    """beta and g from an independent routine: scipy's expit and numpy's logaddexp."""
    h = np.arange(d["b"].shape[0]) % d["num_v_heads"]
    beta = expit(d["b"])
    g = -np.exp(d["A_log"][h]) * np.logaddexp(0.0, d["a"] + d["dt_bias"][h])
    return beta, g


def test_decode_core_equals_one_prefill_token(oracle_mod):
    """With eps_l2 = 0 the decode step's state is one prefill token on l2-normalised
    q,k, beta = sigmoid(b), g = -exp(A_log[h]) softplus(a + dt_bias[h]) with
    h = bh mod num_v_heads, scale 1/sqrt(K). Its output, divided by norm_weight and
    SiLU(z), is that token's o rescaled to unit RMS."""
    rng = np.random.default_rng(20)
    BH, H, K, V = 12, 4, 8, 6
    d = rand_decode(rng, BH, H, K, V)
    y, st = oracle_mod.decode_step(**d, eps_l2=0.0, eps_rms=0.0)
    beta, g = _gates(d)
    qn, kn = _unit(d["q"]), _unit(d["k"])
    out_p, st_p = oracle_mod.prefill(qn[:, None, None], kn[:, None, None],
                                     d["v"][:, None, None], g[:, None, None],
                                     beta[:, None, None], K ** -0.5,
                                     d["state_in"][:, None])
    np.testing.assert_allclose(st, st_p[:, 0], rtol=1e-12, atol=1e-14)
    o = out_p[:, 0, 0]
    r = y / (d["norm_weight"][None] * d["z"] * expit(d["z"]))
    np.testing.assert_allclose(r, o / np.sqrt(np.mean(o * o, axis=1, keepdims=True)),
                               rtol=1e-10)


def test_decode_steps_equal_one_prefill(oracle_mod):
    """T chained decode steps advance the state exactly like one T-token prefill."""
    rng = np.random.default_rng(21)
    BH, H, K, V, T = 6, 3, 8, 8, 5
    qs, ks, vs, bs, as_ = [], [], [], [], []
    d0 = rand_decode(rng, BH, H, K, V)
    st = d0["state_in"]
    gs, betas = [], []
    for _ in range(T):
        d = rand_decode(rng, BH, H, K, V)
        d.update(A_log=d0["A_log"], dt_bias=d0["dt_bias"], norm_weight=d0["norm_weight"],
                 state_in=st)
        _, st = oracle_mod.decode_step(**d, eps_l2=0.0)
        beta, g = _gates(d)
        qs.append(_unit(d["q"])), ks.append(_unit(d["k"])), vs.append(d["v"])
        gs.append(g), betas.append(beta)
    q = np.stack(qs, 1)[:, None]
    k = np.stack(ks, 1)[:, None]
    v = np.stack(vs, 1)[:, None]
    _, st_p = oracle_mod.prefill(q, k, v, np.stack(gs, 1)[:, None],
                                 np.stack(betas, 1)[:, None], K ** -0.5,
                                 d0["state_in"][:, None])
    np.testing.assert_allclose(st, st_p[:, 0], rtol=1e-12, atol=1e-14)


def test_decode_multi_equals_prefill(oracle_mod):
    """The multi-token decode (T tokens in one call) carries the state like one T-token
    prefill on the gated, l2-normalised inputs, and its first token is the single
    step."""
    rng = np.random.default_rng(23)
    BH, H, K, V, T = 6, 3, 8, 8, 4
    d0 = rand_decode(rng, BH, H, K, V)
    toks = [rand_decode(rng, BH, H, K, V) for _ in range(T)]
    seq = {n: np.stack([d[n] for d in toks]) for n in ("q", "k", "v", "b", "a", "z")}
    out, st = oracle_mod.decode_multi(seq["q"], seq["k"], seq["v"], seq["b"], seq["a"],
                                      d0["A_log"], d0["dt_bias"], seq["z"], d0["norm_weight"],
                                      d0["state_in"], H, eps_l2=0.0)
    gs, betas = [], []
    for d in toks:
        d.update(A_log=d0["A_log"], dt_bias=d0["dt_bias"], num_v_heads=H)
        beta, g = _gates(d)
        gs.append(g), betas.append(beta)
    q = np.stack([_unit(d["q"]) for d in toks], 1)[:, None]
    k = np.stack([_unit(d["k"]) for d in toks], 1)[:, None]
    v = np.stack([d["v"] for d in toks], 1)[:, None]
    _, st_p = oracle_mod.prefill(q, k, v, np.stack(gs, 1)[:, None],
                                 np.stack(betas, 1)[:, None], K ** -0.5,
                                 d0["state_in"][:, None])
    np.testing.assert_allclose(st, st_p[:, 0], rtol=1e-12, atol=1e-14)
    y1, _ = oracle_mod.decode_step(seq["q"][0], seq["k"][0], seq["v"][0], seq["b"][0],
                                   seq["a"][0], d0["A_log"], d0["dt_bias"], seq["z"][0],
                                   d0["norm_weight"], d0["state_in"], H, eps_l2=0.0)
    np.testing.assert_array_equal(out[0], y1)


def test_decode_gates_closed_forms(oracle_mod):
    """Read beta and alpha = exp(g) off the state and check closed forms:
    sigmoid(0) = 1/2; softplus(0) = ln 2 so A_log = ln 2 gives alpha = 2^-2;
    softplus(30) = 30 + 9.4e-14; softplus(-30) = 9.4e-14. Row bh uses head bh mod H."""
    K = V = 4
    H, BH = 2, 4
    e0 = np.eye(K)[0]
    base = dict(q=np.tile(e0, (BH, 1)), k=np.tile(e0, (BH, 1)), v=np.ones((BH, V)),
                z=np.ones((BH, V)), norm_weight=np.ones(V), num_v_heads=H)
    # beta from a zero state: S' = beta k^ v^T
    d = dict(base, b=np.array([0.0, 0.0, 2.0, -3.0]), a=np.zeros(BH), A_log=np.zeros(H),
             dt_bias=np.zeros(H), state_in=np.zeros((BH, K, V)))
    _, st = oracle_mod.decode_step(**d, eps_l2=0.0)
    np.testing.assert_allclose(st[:, 0, 0], 1 / (1 + np.exp(-d["b"])), rtol=1e-14)
    np.testing.assert_allclose(st[:, 0, 0], [0.5, 0.5, 0.8807970779778823, 0.04742587317756678],
                               rtol=1e-14)
    # alpha with beta ~ 0 (b = -80): S' = alpha S on rows orthogonal to k
    s0 = np.zeros((BH, K, V))
    s0[:, 1, :] = 1.0
    d = dict(base, b=np.full(BH, -80.0), a=np.array([0.0, 0.0, 30.0, -30.0]),
             A_log=np.array([0.0, np.log(2.0)]), dt_bias=np.zeros(H), state_in=s0)
    _, st = oracle_mod.decode_step(**d, eps_l2=0.0)
    alpha = st[:, 1, 0]
    sp30 = 30.0 + np.exp(-30.0)  # softplus(30) to fp64 precision
    expect = [0.5, 0.25, np.exp(-sp30), np.exp(-2.0 * np.exp(-30.0))]
    np.testing.assert_allclose(alpha, expect, rtol=1e-13)


def test_decode_l2norm_scale_invariance(oracle_mod):
    rng = np.random.default_rng(22)
    d = rand_decode(rng, 8, 2, 16, 8)
    y, st = oracle_mod.decode_step(**d, eps_l2=0.0)
    d2 = dict(d, q=d["q"] * 7.0, k=d["k"] * 0.3)
    y2, st2 = oracle_mod.decode_step(**d2, eps_l2=0.0)
    np.testing.assert_allclose(y2, y, rtol=1e-12)
    np.testing.assert_allclose(st2, st, rtol=1e-12, atol=1e-15)


def test_decode_epilogue_closed_forms(oracle_mod):
    """Zero state, q = k: o = scale beta v. A constant v gives a constant o, so the
    normalised output is sign(o) * norm_weight * SiLU(z) (eps_rms = 0). z varies per
    element, which tells norm-then-gate apart from gate-then-norm."""
    K, V, BH = 8, 6, 2
    rng = np.random.default_rng(23)
    qk = rng.standard_normal((BH, K))
    z = np.array([[-2.0, -0.5, 0.0, 0.5, 3.0, 20.0]] * BH)
    w = np.array([0.5, 0.7, 0.9, 1.1, 1.3, 1.5])
    d = dict(q=qk, k=qk, v=np.array([[2.5] * V, [-0.75] * V]), b=np.zeros(BH),
             a=np.zeros(BH), A_log=np.zeros(1), dt_bias=np.zeros(1), z=z, norm_weight=w,
             state_in=np.zeros((BH, K, V)), num_v_heads=1)
    y, _ = oracle_mod.decode_step(**d, eps_l2=0.0, eps_rms=0.0)
    silu = z / (1.0 + np.exp(-z))
    np.testing.assert_allclose(y[0], w * silu[0], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(y[1], -w * silu[1], rtol=1e-13, atol=1e-15)
    assert abs(y[0, 5] - 1.5 * 20.0) < 1e-6  # SiLU(20) = 20 (1 - 2e-9)


def test_decode_hand_worked_example(oracle_mod):
    gd = read_golden("decode_hand_2x2.txt")
    d = dict(q=gd["q"][None], k=gd["k"][None], v=gd["v"][None], b=gd["b"], a=gd["a"],
             A_log=gd["A_log"], dt_bias=gd["dt_bias"], z=gd["z"][None],
             norm_weight=gd["norm_weight"], state_in=gd["state_in"].reshape(1, 2, 2),
             num_v_heads=1)
    y, st = oracle_mod.decode_step(**d)  # default eps readings (1e-6)
    np.testing.assert_allclose(y.ravel(), gd["out"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(st.ravel(), gd["state_out"], rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------- conv1d decode token
def _silu(x):
    return x * expit(x)


def test_conv1d_impulse_response(oracle_mod):
    """A depthwise causal filter is fixed by its impulse response: an impulse of height a
    entered at step 0 into a zero window comes out at step t as silu(a w[c][K-1-t])."""
    rng = np.random.default_rng(30)
    B, C, K = 2, 5, 4
    w = rng.standard_normal((C, K))
    a = rng.standard_normal((B, C))
    st = np.zeros((B, C, K))
    for t in range(K + 1):
        x = a if t == 0 else np.zeros((B, C))
        y, st = oracle_mod.conv1d_decode(x, w, st)
        want = _silu(a * w[None, :, K - 1 - t]) if t < K else np.zeros((B, C))
        np.testing.assert_allclose(y, want, rtol=1e-14, atol=0)


def test_conv1d_window_is_a_shift_register(oracle_mod):
    """After K tokens the window holds exactly those tokens, oldest first; the next token
    drops the oldest."""
    rng = np.random.default_rng(31)
    B, C, K = 3, 4, 5
    w = rng.standard_normal((C, K))
    st = rng.standard_normal((B, C, K))
    xs = [rng.standard_normal((B, C)) for _ in range(K + 1)]
    for x in xs[:K]:
        _, st = oracle_mod.conv1d_decode(x, w, st)
    np.testing.assert_array_equal(st, np.stack(xs[:K], axis=2))
    _, st = oracle_mod.conv1d_decode(xs[K], w, st)
    np.testing.assert_array_equal(st, np.stack(xs[1:], axis=2))


def test_conv1d_pass_through_and_delay(oracle_mod):
    """A one-hot filter on the newest tap passes silu(x) through; on tap j it returns
    silu of the input j + 1 tokens older than the newest (state[j + 1])."""
    rng = np.random.default_rng(32)
    B, C, K = 2, 3, 4
    st = rng.standard_normal((B, C, K))
    x = rng.standard_normal((B, C))
    w = np.zeros((C, K))
    w[:, K - 1] = 1.0
    y, _ = oracle_mod.conv1d_decode(x, w, st)
    np.testing.assert_allclose(y, _silu(x), rtol=1e-15)
    for j in range(K - 1):
        w = np.zeros((C, K))
        w[:, j] = 1.0
        y, _ = oracle_mod.conv1d_decode(x, w, st)
        np.testing.assert_allclose(y, _silu(st[:, :, j + 1]), rtol=1e-15)


def test_conv1d_split_is_repeat_interleave(oracle_mod):
    """q | k | v split of the conv channels, q and k repeated over the value heads the
    way torch.repeat_interleave does it (value head h reads key head h // G)."""
    import torch
    rng = np.random.default_rng(33)
    B, Hk, Hv, Dk, Dv = 2, 2, 6, 3, 4
    y = rng.standard_normal((B, 2 * Hk * Dk + Hv * Dv))
    q, k, v = oracle_mod.conv1d_split(y, Hk, Hv, Dk, Dv)
    t = torch.from_numpy(y)
    qr = t[:, :Hk * Dk].reshape(B, Hk, Dk).repeat_interleave(Hv // Hk, dim=1)
    kr = t[:, Hk * Dk:2 * Hk * Dk].reshape(B, Hk, Dk).repeat_interleave(Hv // Hk, dim=1)
    np.testing.assert_array_equal(q, qr.reshape(B * Hv, Dk).numpy())
    np.testing.assert_array_equal(k, kr.reshape(B * Hv, Dk).numpy())
    np.testing.assert_array_equal(v, t[:, 2 * Hk * Dk:].reshape(B * Hv, Dv).numpy())


# ------------------------------------------------------------ variable-length batches
def test_varlen_equal_lengths_is_the_dense_batch(oracle_mod):
    """N sequences of one length L packed along the token axis give the dense batch
    (B = N, S = L) result, row for row."""
    rng = np.random.default_rng(40)
    N, Hk, Hv, L, D = 3, 2, 4, 7, 5
    q = _unit(rng.standard_normal((N, Hk, L, D)))
    k = _unit(rng.standard_normal((N, Hk, L, D)))
    v = rng.standard_normal((N, Hv, L, D))
    g = rng.uniform(-0.5, -0.01, (N, Hv, L))
    b = rng.uniform(0.05, 0.95, (N, Hv, L))
    s0 = rng.standard_normal((N, Hv, D, D)) * 0.1
    o_d, s_d = oracle_mod.prefill(q, k, v, g, b, 0.5, s0)
    pack = lambda x: np.concatenate(list(x), axis=1)  # [N, H, L, ...] -> [H, N*L, ...]
    cu = np.arange(N + 1) * L
    o_v, s_v = oracle_mod.prefill_varlen(pack(q), pack(k), pack(v), pack(g), pack(b), 0.5, cu,
                                         s0)
    np.testing.assert_allclose(o_v, pack(o_d), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(s_v, s_d, rtol=1e-13, atol=1e-15)


def test_varlen_empty_sequences_keep_their_state(oracle_mod):
    rng = np.random.default_rng(41)
    Hk, Hv, T, D = 1, 2, 6, 4
    q = _unit(rng.standard_normal((Hk, T, D)))
    k = _unit(rng.standard_normal((Hk, T, D)))
    v = rng.standard_normal((Hv, T, D))
    g = rng.uniform(-0.5, -0.01, (Hv, T))
    b = rng.uniform(0.05, 0.95, (Hv, T))
    s0 = rng.standard_normal((3, Hv, D, D))
    out, st = oracle_mod.prefill_varlen(q, k, v, g, b, 1.0, [0, 0, 6, 6], s0)
    np.testing.assert_array_equal(st[0], s0[0])
    np.testing.assert_array_equal(st[2], s0[2])
    o1, s1 = oracle_mod.prefill(q[None], k[None], v[None], g[None], b[None], 1.0, s0[1][None])
    np.testing.assert_array_equal(st[1], s1[0])
    np.testing.assert_array_equal(out, o1[0])
