"""Pins of the CPU oracle against what the mathematics fixes (CPU only, no GPU).

Build: brute force over every candidate tree, the k=1 -> flat-chain invariant, a
pruned exhaustive enumeration on mid sizes, log-sum-exp against an exactly rounded sum.
Attention: chain tree == plain causal attention; every row == per-path replay (the
check the research notes' proving ground used); closed forms for one key and for
equal keys.  GDN: per-path replay in projection form; beta=0 closed form; the delta
rule's read-back property; orthonormal keys; conv taps.  Walk: brute force over all
paths; planted paths.  Commit: indices, post-commit state, conv state, capacity.
"""
import math

import numpy as np
import pytest

import oracle
from tests import _np_ref as R

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rng(seed):
    return np.random.default_rng(seed)


# ============================================================================ build
def _check_canonical(out, b, D):
    tok, par, dep, rk = out["token"][b], out["parent"][b], out["depth"][b], out["rank"][b]
    n = int(out["n_nodes"][b])
    assert par[0] == -1 and dep[0] == 0
    keys = []
    for i in range(1, n):
        assert 0 <= par[i] < i
        assert dep[i] == dep[par[i]] + 1 and 1 <= dep[i] <= D
        keys.append((dep[i], par[i], rk[i]))
    assert keys == sorted(keys) and len(set(keys)) == len(keys)
    N = tok.shape[0]
    for i in range(n, N):
        assert tok[i] == -1 and par[i] == -1 and dep[i] == -1
    np.testing.assert_array_equal(out["anc"][b], R.anc_from_parent(par, n, N))
    np.testing.assert_array_equal(out["position"][b][:n], out["position"][b][0] + dep[:n])


@pytest.mark.parametrize("seed", range(40))
def test_build_matches_brute_force(seed):
    rng = _rng(seed)
    V = int(rng.integers(2, 9))
    D = int(rng.integers(1, 6))
    k = int(rng.integers(1, V + 1))
    lattice = sum(k ** d for d in range(1, D + 1))
    budget = int(rng.integers(0, min(lattice, 24) + 3))
    if seed % 3 == 0:   # integer logits: many exact ties, decided by token order
        logits = rng.integers(-2, 3, size=(1, D, V)).astype(np.float64)
    else:
        logits = rng.normal(0, 2, size=(1, D, V)).astype(np.float32).astype(np.float64)
    out = oracle.build_tree(logits, [3], [17], k, budget)
    _check_canonical(out, 0, D)
    sel, rest = R.brute_force_tree(logits[0], k, budget)
    got = R.tree_sequences(out["token"][0], out["parent"][0], out["n_nodes"][0])
    assert int(out["n_nodes"][0]) == len(sel) + 1
    assert set(got.values()) == {s for _, s in sel}
    # scores equal the exact log-probability of each path
    want = {s: sc for sc, s in sel}
    for i, s in got.items():
        assert abs(out["score"][0][i] - want[s]) < 1e-12
    if rest and sel:
        assert abs(out["margin"][0] - (sel[-1][0] - rest[0][0])) < 1e-12


@pytest.mark.parametrize("seed", range(6))
def test_build_k1_is_flat_chain(seed):
    """A one-per-depth tree is the flat DFlash chain of per-depth argmax tokens."""
    rng = _rng(100 + seed)
    D, V = int(rng.integers(1, 12)), int(rng.integers(2, 300))
    logits = rng.integers(-3, 4, size=(1, D, V)).astype(np.float64)  # ties on purpose
    budget = int(rng.integers(0, 20))
    out = oracle.build_tree(logits, [7], [0], 1, budget)
    n = min(budget, D)
    assert out["n_nodes"][0] == n + 1
    for i in range(1, n + 1):
        assert out["parent"][0][i] == i - 1
        row = logits[0, i - 1]
        assert out["token"][0][i] == int(np.flatnonzero(row == row.max())[0])


@pytest.mark.parametrize("seed", range(4))
def test_build_pruned_enumeration_mid_size(seed):
    """Mid sizes (lattice too big to sort): enumerate every path scoring at least the
    oracle's last selected score, pruning on the fact that scores fall along children and
    along ranks; that set must be the oracle's tree."""
    rng = _rng(200 + seed)
    D, V, k, budget = 8, 512, 8, 64
    logits = rng.normal(0, 3, size=(1, D, V)).astype(np.float32).astype(np.float64)
    logits[0, np.arange(D), rng.integers(0, V, D)] += 6.0
    out = oracle.build_tree(logits, [1], [5], k, budget)
    _check_canonical(out, 0, D)
    tops = [R.rank_order(logits[0, d])[:k] for d in range(D)]
    lses = [R.lse_exact(logits[0, d]) for d in range(D)]
    thr = min(out["score"][0][1:out["n_nodes"][0]]) - 1e-9
    found = []

    def dfs(prefix, logp):
        d = len(prefix)
        if d == D:
            return
        for t in tops[d]:
            s = logp + float(logits[0, d, t]) - lses[d]
            if s < thr:
                break        # later ranks only score lower
            found.append(prefix + (int(t),))
            dfs(prefix + (int(t),), s)

    dfs((), 0.0)
    got = R.tree_sequences(out["token"][0], out["parent"][0], out["n_nodes"][0])
    assert set(found) == set(got.values())
    assert out["margin"][0] > 1e-6


def test_build_lse_and_scores():
    rng = _rng(7)
    logits = rng.normal(0, 3, size=(2, 4, 5000)).astype(np.float32).astype(np.float64)
    out = oracle.build_tree(logits, [0, 1], [0, 0], 4, 10)
    for b in range(2):
        for d in range(4):
            assert abs(out["lse"][b, d] - R.lse_exact(logits[b, d])) < 1e-12
        top = R.rank_order(logits[b, 0])[0]
        i = int(np.flatnonzero((out["depth"][b] == 1) & (out["rank"][b] == 0))[0])
        assert out["token"][b, i] == top
        assert abs(out["score"][b, i] - (logits[b, 0, top] - R.lse_exact(logits[b, 0]))) < 1e-12


def test_build_empty_budget_and_multi_request():
    rng = _rng(8)
    logits = rng.normal(0, 2, size=(3, 3, 50))
    out = oracle.build_tree(logits, [4, 5, 6], [10, 0, 3], 3, 0)
    np.testing.assert_array_equal(out["n_nodes"], [1, 1, 1])
    np.testing.assert_array_equal(out["token"][:, 0], [4, 5, 6])
    np.testing.assert_array_equal(out["position"][:, 0], [10, 0, 3])


# ======================================================================== attention
def _attn_case(rng, P, N, d, parent, n_nodes):
    q = rng.normal(size=(N, d))
    kp, vp = rng.normal(size=(P, d)), rng.normal(size=(P, d))
    kt, vt = rng.normal(size=(N, d)), rng.normal(size=(N, d))
    anc = R.anc_from_parent(parent, n_nodes, N)
    return q, kp, vp, kt, vt, anc


@pytest.mark.parametrize("P", [0, 1, 7, 64])
def test_attn_chain_is_causal_attention(P):
    rng = _rng(P + 1)
    N, d = 9, 16
    parent = np.array([-1] + list(range(N - 1)))
    q, kp, vp, kt, vt, anc = _attn_case(rng, P, N, d, parent, N)
    scale = 1 / math.sqrt(d)
    qs = np.concatenate([np.zeros((P, d)), q])
    want = R.causal_attention(qs, np.concatenate([kp, kt]), np.concatenate([vp, vt]), scale)[P:]
    for i in range(N):
        got = oracle.attn_row(q[i], kp, vp, kt, vt, anc[i], N, scale)
        np.testing.assert_allclose(got, want[i], rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(5))
def test_attn_rows_equal_per_path_replay(seed):
    rng = _rng(300 + seed)
    logits = rng.normal(0, 2, size=(1, 6, 40))
    tree = oracle.build_tree(logits, [0], [0], 3, 20)
    parent, n = tree["parent"][0], int(tree["n_nodes"][0])
    N, d, P = parent.shape[0], 8, int(rng.integers(0, 30))
    q, kp, vp, kt, vt, anc = _attn_case(rng, P, N, d, parent, n)
    np.testing.assert_array_equal(anc, tree["anc"][0])
    for i in range(n):
        rows = R.path_rows(parent, i)
        seq_k = np.concatenate([kp, kt[rows]])
        seq_v = np.concatenate([vp, vt[rows]])
        seq_q = np.concatenate([np.zeros((P + len(rows) - 1, d)), q[i:i + 1]])
        want = R.causal_attention(seq_q, seq_k, seq_v, 0.5)[-1]
        got = oracle.attn_row(q[i], kp, vp, kt, vt, anc[i], n, 0.5)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_attn_closed_forms():
    rng = _rng(9)
    d = 8
    # one key: the output is that key's value
    q, kt, vt = rng.normal(size=d), rng.normal(size=(1, d)), rng.normal(size=(1, d))
    got = oracle.attn_row(q, np.zeros((0, d)), np.zeros((0, d)), kt, vt, [1], 1, 1.0)
    np.testing.assert_allclose(got, vt[0], atol=1e-15)
    # equal keys: the output is the mean of the visible values (siblings excluded)
    parent = np.array([-1, 0, 0, 1])
    anc = R.anc_from_parent(parent, 4, 4)
    kp = np.ones((5, d))
    vp = rng.normal(size=(5, d))
    kt = np.ones((4, d))
    vt = rng.normal(size=(4, d))
    got = oracle.attn_row(rng.normal(size=d), kp, vp, kt, vt, anc[3], 4, 0.3)
    np.testing.assert_allclose(got, np.concatenate([vp, vt[[0, 1, 3]]]).mean(0), atol=1e-13)


def test_tree_attn_batch_matches_rows():
    rng = _rng(10)
    L, B, Hq, Hkv, d, Pcap = 2, 2, 4, 2, 8, 12
    logits = rng.normal(0, 2, size=(B, 4, 30))
    tree = oracle.build_tree(logits, [0, 1], [5, 12], 3, 7)
    N = tree["token"].shape[1]
    q = rng.normal(size=(L, B, N, Hq, d))
    kt, vt = rng.normal(size=(L, B, N, Hkv, d)), rng.normal(size=(L, B, N, Hkv, d))
    kc, vc = rng.normal(size=(L, B, Hkv, Pcap, d)), rng.normal(size=(L, B, Hkv, Pcap, d))
    pl = np.array([5, 12])
    o = oracle.tree_attn(q, kt, vt, kc, vc, pl, tree["n_nodes"], tree["anc"], 0.4)["o"]
    for (l, b, i, h) in [(0, 0, 0, 0), (1, 1, 5, 3), (1, 0, 7, 2)]:
        g = h // (Hq // Hkv)
        want = oracle.attn_row(q[l, b, i, h], kc[l, b, g, :pl[b]], vc[l, b, g, :pl[b]], kt[l, b, :, g],
                               vt[l, b, :, g], tree["anc"][b, i], tree["n_nodes"][b], 0.4)
        np.testing.assert_allclose(o[l, b, i, h], want, atol=1e-14)


# ============================================================================== GDN
def _gdn_case(rng, N, Hk, Hv, dk, dv, K):
    C = 2 * Hk * dk + Hv * dv
    x = rng.normal(size=(N, C))
    w = 0.5 * rng.normal(size=(C, K))
    cs = rng.normal(size=(K - 1, C))
    beta = 1 / (1 + np.exp(-rng.normal(size=(N, Hv))))
    decay = np.exp(-np.log1p(np.exp(rng.normal(size=(N, Hv)))))
    S0 = rng.normal(size=(dk, dv))
    return x, w, cs, beta, decay, S0


@pytest.mark.parametrize("seed", range(4))
def test_gdn_per_path_replay(seed):
    rng = _rng(400 + seed)
    Hk, Hv, dk, dv, K = 2, 4, 6, 5, 4
    tree = oracle.build_tree(rng.normal(0, 2, size=(1, 7, 30)), [0], [0], 3, 18)
    parent, n = tree["parent"][0], int(tree["n_nodes"][0])
    N = parent.shape[0]
    x, w, cs, beta, decay, S0 = _gdn_case(rng, N, Hk, Hv, dk, dv, K)
    for h in (0, 3):
        got = oracle.gdn_unit(x, w, cs, beta, decay, S0, parent, n, Hk, Hv, h, want_states=True)
        for i in range(n):
            rows = R.path_rows(parent, i)
            o, S = R.gdn_sequence(x[rows], w, cs, beta[rows, h], decay[rows, h], S0, Hk, Hv, h)
            np.testing.assert_allclose(got["o"][i], o[-1], rtol=1e-10, atol=1e-10)
            np.testing.assert_allclose(got["S_node"][i], S[-1], rtol=1e-10, atol=1e-10)


def test_gdn_beta_zero_is_pure_decay():
    rng = _rng(11)
    Hk, Hv, dk, dv, K = 1, 2, 4, 3, 4
    parent = np.array([-1, 0, 1, 1, 0, 4])
    x, w, cs, beta, decay, S0 = _gdn_case(rng, 6, Hk, Hv, dk, dv, K)
    beta[:] = 0.0
    got = oracle.gdn_unit(x, w, cs, beta, decay, S0, parent, 6, Hk, Hv, 1, want_states=True)
    for i in range(6):
        g = np.prod([decay[r, 1] for r in R.path_rows(parent, i)])
        np.testing.assert_allclose(got["S_node"][i], g * S0, rtol=1e-13, atol=1e-14)


def _identity_tap(C, K):
    w = np.zeros((C, K))
    w[:, K - 1] = 1.0
    return w


def test_gdn_delta_rule_readback():
    """One delta step with key k^: S_n - a S_p is rank one along k^, and
    S_n^T k^ = a S_p^T k^ + b |k^|^2 (v - a S_p^T k^)."""
    rng = _rng(12)
    Hk, Hv, dk, dv, K = 1, 1, 5, 4, 4
    parent = np.array([-1, 0, 1, 0])
    x, _, cs, beta, decay, S0 = _gdn_case(rng, 4, Hk, Hv, dk, dv, K)
    w = _identity_tap(x.shape[1], K)
    got = oracle.gdn_unit(x, w, cs, beta, decay, S0, parent, 4, Hk, Hv, 0, want_states=True)
    for i in range(4):
        Sp = S0 if i == 0 else got["S_node"][parent[i]]
        y = R.silu(x[i])
        k = y[dk:2 * dk] / math.sqrt(float(y[dk:2 * dk] @ y[dk:2 * dk]) + 1e-6)
        v = y[2 * dk:]
        a, b = decay[i, 0], beta[i, 0]
        Sn = got["S_node"][i]
        delta = Sn - a * Sp
        sv = np.linalg.svd(delta, compute_uv=False)
        assert sv[1] < 1e-12 * max(1.0, sv[0])
        np.testing.assert_allclose(Sn.T @ k, a * Sp.T @ k + b * (k @ k) * (v - a * Sp.T @ k), atol=1e-12)


def test_gdn_orthonormal_keys_recall_values():
    """a = b = 1 with keys of disjoint support: every ancestor's value reads back exactly."""
    Hk, Hv, dk, dv, K = 1, 1, 8, 3, 4
    C = 2 * dk + dv
    parent = np.array([-1, 0, 1, 2, 0])
    x = np.zeros((5, C))
    for i in range(5):
        x[i, dk + i] = 20.0                    # k channel: one-hot, silu(0) = 0 elsewhere
        x[i, 2 * dk:] = np.arange(dv) + i + 1.0
    rng = _rng(13)
    S0 = rng.normal(size=(dk, dv))
    got = oracle.gdn_unit(x, _identity_tap(C, K), np.zeros((K - 1, C)), np.ones((5, 1)), np.ones((5, 1)),
                          S0, parent, 5, Hk, Hv, 0, want_states=True)
    for i in range(5):
        for j in R.path_rows(parent, i):
            kj = np.zeros(dk)
            kj[j] = 1.0
            np.testing.assert_allclose(got["S_node"][i].T @ kj, R.silu(x[j, 2 * dk:]), atol=1e-8)
        for j in set(range(5)) - set(R.path_rows(parent, i)):   # siblings stay invisible
            np.testing.assert_allclose(got["S_node"][i][j], S0[j], atol=1e-12)


@pytest.mark.parametrize("tap", [0, 1, 2, 3])
def test_gdn_conv_taps_follow_the_ancestor_path(tap):
    """decay 0, beta 1 and q == k channels: o_n = |k^|^2/sqrt(dk) * conv_v(n), exposing
    the conv output, which for a one-hot tap is SiLU of the input `3 - tap` steps up the
    node's own path (or the committed conv state past the root)."""
    rng = _rng(14 + tap)
    Hk, Hv, dk, dv, K = 1, 1, 4, 3, 4
    C = 2 * dk + dv
    parent = np.array([-1, 0, 1, 2, 0, 4, 2])
    N = 7
    x = rng.normal(size=(N, C))
    x[:, dk:2 * dk] = x[:, :dk]
    cs = rng.normal(size=(K - 1, C))
    w = np.zeros((C, K))
    w[:dk, K - 1] = 1.0
    w[dk:2 * dk, K - 1] = 1.0
    w[2 * dk:, tap] = 1.0
    got = oracle.gdn_unit(x, w, cs, np.ones((N, 1)), np.zeros((N, 1)), rng.normal(size=(dk, dv)),
                          parent, N, Hk, Hv, 0)
    for n in range(N):
        path = R.path_rows(parent, n)[::-1]          # n, parent, grandparent, ...
        back = K - 1 - tap
        src = x[path[back]] if back < len(path) else cs[K - 1 - (back - (len(path) - 1))]
        kq = R.silu(x[n, :dk])
        kk = (kq @ kq) / ((kq @ kq) + 1e-6)
        np.testing.assert_allclose(got["o"][n], kk / math.sqrt(dk) * R.silu(src[2 * dk:]), atol=1e-12)


def test_tree_gdn_batch_matches_units():
    rng = _rng(15)
    L, B, Hk, Hv, dk, dv, K = 2, 2, 1, 2, 4, 3, 4
    tree = oracle.build_tree(rng.normal(0, 2, size=(B, 4, 20)), [0, 1], [0, 0], 2, 6)
    N = tree["parent"].shape[1]
    C = 2 * Hk * dk + Hv * dv
    x = rng.normal(size=(L, B, N, C))
    w = rng.normal(size=(L, C, K))
    cs = rng.normal(size=(L, B, K - 1, C))
    beta, decay = rng.uniform(size=(L, B, N, Hv)), rng.uniform(size=(L, B, N, Hv))
    S = rng.normal(size=(L, B, Hv, dk, dv))
    out = oracle.tree_gdn(x, w, cs, beta, decay, S, tree["parent"], tree["n_nodes"], Hk, want_states=True)
    for (l, b, h) in [(0, 0, 0), (1, 1, 1), (1, 0, 1)]:
        u = oracle.gdn_unit(x[l, b], w[l], cs[l, b], beta[l, b], decay[l, b], S[l, b, h], tree["parent"][b],
                            tree["n_nodes"][b], Hk, Hv, h, want_states=True)
        np.testing.assert_allclose(out["o"][l, b, :, h], u["o"], atol=1e-14)
        n = tree["n_nodes"][b]
        np.testing.assert_allclose(out["S_node"][l, b, :n, h], u["S_node"][:n], atol=1e-14)


# ============================================================================= walk
@pytest.mark.parametrize("seed", range(10))
def test_walk_brute_force_planted(seed):
    rng = _rng(500 + seed)
    B, D, V = 2, 6, 12
    tree = oracle.build_tree(rng.normal(0, 2, size=(B, D, V)), [1, 2], [0, 0], 3, 20)
    N = tree["token"].shape[1]
    tl = rng.normal(size=(B, N, V))
    for b in range(B):   # plant a random root-to-node path
        cur = 0
        for _ in range(int(rng.integers(0, D + 1))):
            kids = [c for c in range(1, tree["n_nodes"][b]) if tree["parent"][b][c] == cur]
            if not kids:
                break
            nxt = kids[int(rng.integers(len(kids)))]
            tl[b, cur, tree["token"][b][nxt]] += 10.0
            cur = nxt
    if seed % 2:
        tl = np.round(tl)  # argmax ties -> lowest id
    out = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], D, target_logits=tl)
    for b in range(B):
        am = np.array([int(np.flatnonzero(tl[b, i] == tl[b, i].max())[0]) for i in range(N)])
        n = tree["n_nodes"][b]
        np.testing.assert_array_equal(out["target_argmax"][b][:n], am[:n])
        last, path = R.walk_bruteforce(tree["token"][b], tree["parent"][b], n, am)
        assert out["acc_len"][b] == len(path) - 1
        np.testing.assert_array_equal(out["acc_nodes"][b][:len(path)], path)
        assert (out["acc_nodes"][b][len(path):] == -1).all()
        assert out["bonus"][b] == am[last]
        em = [tree["token"][b][r] for r in path[1:]] + [am[last]]
        np.testing.assert_array_equal(out["emitted"][b][:len(em)], em)
        assert out["n_emitted"][b] == len(em)


def test_walk_chain_is_longest_prefix():
    """Flat chain: accepted = longest prefix where the draft equals the target's argmax."""
    D = 6
    token = np.array([[9, 3, 1, 4, 1, 5, 9]])
    parent = np.array([[-1, 0, 1, 2, 3, 4, 5]])
    am = np.array([[3, 1, 4, 2, 0, 0, 0]])
    out = oracle.walk(token, parent, [7], D, target_argmax=am)
    assert out["acc_len"][0] == 3 and out["bonus"][0] == 2
    np.testing.assert_array_equal(out["emitted"][0][:4], [3, 1, 4, 2])


# ==================================================== walk, rejection sampling
def _softmax(x, T):
    z = np.exp((x - x.max()) / T)
    return z / z.sum()


def _sample_case(lg, U, tok, par, D, C, T=1.0):
    N = len(tok)
    tl = np.asarray(lg, np.float64).reshape(1, N, -1)
    return oracle.walk_sample(np.array([tok]), np.array([par]), [N], D, tl, np.asarray(U)[None], T, C)


def test_walk_sample_worked_examples():
    """Hand-worked decisions of the rule (speculative sampling with point-mass drafts over
    a node's children): accept x with probability p(x) / (1 - R), R the rejected mass;
    otherwise the bonus comes from p with the rejected tokens removed."""
    p = np.array([0.5, 0.25, 0.125, 0.125])
    lg = np.log(np.tile(p, (3, 1)))
    tok, par = [7, 1, 2], [-1, 0, 0]   # root, children tokens 1 (p 1/4) then 2 (p 1/8)
    # 0.2 < 1/4: the first child is accepted; its node has no children, so the bonus
    # target is U = 0.6 and the running sum 0.5, 0.75 first passes it at id 1
    o = _sample_case(lg, [[0.2, 0.0, 0.0], [0.0, 0.0, 0.6]], tok, par, 1, 2)
    assert o["acc_len"][0] == 1 and o["acc_nodes"][0].tolist() == [0, 1]
    assert o["emitted"][0].tolist() == [1, 1] and o["bonus"][0] == 1
    assert o["margin"][0] == pytest.approx(0.05)            # min(|0.2-0.25|, 0.6-0.5, 0.75-0.6)
    # 0.3 >= 1/4 rejects token 1 (R = 1/4); 0.1 < (1/8)/(3/4) = 1/6 accepts token 2
    o = _sample_case(lg, [[0.3, 0.1, 0.0], [0.0, 0.0, 0.1]], tok, par, 1, 2)
    assert o["acc_nodes"][0].tolist() == [0, 2] and o["emitted"][0].tolist() == [2, 0]
    assert o["margin"][0] == pytest.approx(min(0.05, 1 / 6 - 0.1, 0.1))
    # both rejected (R = 3/8): target 0.9 * 5/8 = 0.5625 over ids 0, 3 (0.5, 0.625) -> 3
    o = _sample_case(lg, [[0.3, 0.9, 0.9], [0.0, 0.0, 0.0]], tok, par, 1, 2)
    assert o["acc_len"][0] == 0 and o["bonus"][0] == 3 and o["emitted"][0].tolist() == [3, -1]
    assert o["margin"][0] == pytest.approx(min(0.05, 0.9 - 1 / 6, 0.0625, 0.0625))
    # target 0.4 * 5/8 = 0.25 < 0.5 -> id 0 (the bonus never lands on a rejected token)
    o = _sample_case(lg, [[0.3, 0.9, 0.4], [0.0, 0.0, 0.0]], tok, par, 1, 2)
    assert o["bonus"][0] == 0
    # at max depth 0 no child is tried: the bonus comes from the whole p_root
    o = _sample_case(lg, [[0.0, 0.0, 0.55]], tok, par, 0, 2)
    assert o["acc_len"][0] == 0 and o["bonus"][0] == 1
    # temperature: the child token 1 is compared at softmax([2, 1, 0] / 2)[1], the tempered
    # probability, not at the untempered softmax([2, 1, 0])[1]
    lg2 = np.array([[2.0, 1.0, 0.0]] * 2)
    q = _softmax(lg2[0], 2.0)
    for u, acc in ((q[1] - 1e-3, 1), (q[1] + 1e-3, 0)):
        o = _sample_case(lg2, [[u, 0.0], [0.0, 0.0]], [5, 1], [-1, 0], 1, 1, T=2.0)
        assert o["acc_len"][0] == acc


def test_walk_sample_statuses():
    lg = np.zeros((4, 5))
    U = np.zeros((3, 3))
    # three children with C = 2
    o = _sample_case(lg, U, [0, 1, 2, 3], [-1, 0, 0, 0], 2, 2)
    assert o["status"][0] == 7 and o["n_emitted"][0] == 0 and o["bonus"][0] == -1
    # a repeated sibling token
    o = _sample_case(lg, U, [0, 1, 1, 3], [-1, 0, 0, 1], 2, 2)
    assert o["status"][0] == 7
    # a token outside the vocabulary
    o = _sample_case(lg, U, [0, 1, 5, 3], [-1, 0, 0, 1], 2, 2)
    assert o["status"][0] == 7
    # a parent after its child
    o = _sample_case(lg, U, [0, 1, 2, 3], [-1, 0, 3, 1], 2, 2)
    assert o["status"][0] == 7
    # a NaN logit in a row of the tree
    bad = lg.copy()
    bad[3, 4] = np.nan
    o = _sample_case(bad, U, [0, 1, 2, 3], [-1, 0, 0, 1], 2, 2)
    assert o["status"][0] == 6 and o["acc_len"][0] == 0 and (o["emitted"][0] == -1).all()
    o = _sample_case(lg, U, [0, 1, 2, 3], [-1, 0, 0, 1], 2, 2)
    assert o["status"][0] == 0


def _emission_law(tok, par, tl, T, D):
    """Closed form of the target's own sampling: each emitted token ~ p_u at the node the
    previous tokens lead to (the sequence stops at the first token that is not a child,
    or after D + 1 tokens).  Returns {tuple(emitted): probability}."""
    law = {}

    def rec(u, prefix, prob, depth):
        pu = _softmax(tl[u], T)
        kids = {tok[c]: c for c in range(1, len(tok)) if par[c] == u}
        for t, pt in enumerate(pu):
            if t in kids and depth < D:
                rec(kids[t], prefix + (t,), prob * pt, depth + 1)
            else:
                law[prefix + (t,)] = law.get(prefix + (t,), 0.0) + prob * pt
    rec(0, (), 1.0, 0)
    return law


@pytest.mark.parametrize("T,shape", [(1.0, "tree"), (0.6, "tree"), (1.5, "chain"), (1.0, "depth_cut")])
def test_walk_sample_is_lossless_monte_carlo(T, shape):
    """Lossless: the emitted sequence is distributed exactly as sampling the target token
    by token (each cell within 5 standard errors over 200k seeded walks).  A dropped
    renormalisation by 1 - R, a bonus that keeps rejected tokens, or a wrong step index
    into the uniforms moves some cell by far more."""
    rng = _rng(77)
    V = 6
    if shape == "chain":
        tok, par, D = [9, 2, 4, 1], [-1, 0, 1, 2], 3
    else:
        # root: children tokens 1, 3, 4; token 1's node: children 0, 2; token 0's node: child 5
        tok, par, D = [9, 1, 3, 4, 0, 2, 5], [-1, 0, 0, 0, 1, 1, 4], 3
        if shape == "depth_cut":
            D = 2
    N, C = len(tok), 3
    tl = rng.normal(0, 0.5, size=(N, V))
    # children tokens carry most of their parent's mass, so that rejections happen after
    # earlier rejections (R well above 0) and the deeper levels are visited often
    for u in range(N):
        for c in range(1, N):
            if par[c] == u:
                tl[u, tok[c]] += 1.5
    n = 200_000
    U = rng.random((n, D + 1, C + 1))
    o = oracle.walk_sample(np.tile(tok, (n, 1)), np.tile(par, (n, 1)), np.full(n, N), D,
                           np.broadcast_to(tl, (n, N, V)), U, T, C)
    assert (o["status"] == 0).all()
    law = _emission_law(tok, par, tl, T, D)
    counts = {}
    for b in range(n):
        key = tuple(o["emitted"][b][:o["n_emitted"][b]].tolist())
        counts[key] = counts.get(key, 0) + 1
    assert set(counts) <= set(law)
    for key, prob in law.items():
        f = counts.get(key, 0) / n
        assert abs(f - prob) <= 5 * math.sqrt(prob * (1 - prob) / n) + 1e-6, (key, f, prob)
    # accepted nodes are the emitted children: acc_len = n_emitted - 1 and the path's tokens
    for b in range(0, n, 997):
        a = o["acc_len"][b]
        assert o["n_emitted"][b] == a + 1
        assert [tok[r] for r in o["acc_nodes"][b][1:a + 1]] == o["emitted"][b][:a].tolist()


@pytest.mark.parametrize("seed", range(4))
def test_walk_sample_cold_limit_is_greedy(seed):
    """T -> 0: p_u becomes the point mass on the argmax (logit gaps of 0.1 at T = 1e-3 leave
    at most V e^-100 elsewhere), so for uniforms below 0.99 the sampler takes exactly the
    greedy walk: a child is accepted iff it is the argmax, and the bonus is the argmax."""
    rng = _rng(900 + seed)
    B, D, V, k = 3, 5, 40, 4
    tree = oracle.build_tree(rng.normal(0, 2, size=(B, D, V)), [1, 2, 3], [0, 0, 0], k, 24)
    N = tree["token"].shape[1]
    tl = np.stack([[rng.permutation(V) * 0.1 for _ in range(N)] for _ in range(B)]).astype(np.float64)
    for b in range(B):   # plant a path so the walk descends
        cur = 0
        for _ in range(int(rng.integers(1, D + 1))):
            kids = [c for c in range(1, tree["n_nodes"][b]) if tree["parent"][b][c] == cur]
            if not kids:
                break
            nxt = kids[int(rng.integers(len(kids)))]
            tl[b, cur, tree["token"][b][nxt]] = tl[b, cur].max() + 0.1
            cur = nxt
    U = rng.uniform(0, 0.99, size=(B, D + 1, k + 1))
    s = oracle.walk_sample(tree["token"], tree["parent"], tree["n_nodes"], D, tl, U, 1e-3, k)
    g = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], D, target_logits=tl)
    assert (s["status"] == 0).all() and (g["acc_len"] > 0).any()
    for key in ("acc_nodes", "acc_len", "bonus", "emitted", "n_emitted"):
        np.testing.assert_array_equal(s[key], g[key])


# =========================================================================== commit
def test_commit_kv_gdn_conv():
    rng = _rng(16)
    La, Lg, B, Hkv, d, Pcap = 2, 2, 2, 2, 4, 12
    Hk, Hv, dk, dv, K = 1, 2, 3, 2, 4
    tree = oracle.build_tree(rng.normal(0, 2, size=(B, 4, 9)), [0, 1], [3, 8], 2, 8)
    N = tree["token"].shape[1]
    C = 2 * Hk * dk + Hv * dv
    kt, vt = rng.normal(size=(La, B, N, Hkv, d)), rng.normal(size=(La, B, N, Hkv, d))
    kc, vc = rng.normal(size=(La, B, Hkv, Pcap, d)), rng.normal(size=(La, B, Hkv, Pcap, d))
    x = rng.normal(size=(Lg, B, N, C))
    w = rng.normal(size=(Lg, C, K))
    cs = rng.normal(size=(Lg, B, K - 1, C))
    beta, decay = rng.uniform(size=(Lg, B, N, Hv)), rng.uniform(size=(Lg, B, N, Hv))
    S = rng.normal(size=(Lg, B, Hv, dk, dv))
    tl = rng.normal(size=(B, N, 9))
    # accept the deepest first-child path of request 0, nothing of request 1
    cur = 0
    while True:
        kids = [c for c in range(1, tree["n_nodes"][0]) if tree["parent"][0][c] == cur]
        if not kids:
            break
        tl[0, cur, tree["token"][0][kids[0]]] += 50
        cur = kids[0]
    wk = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], 4, target_logits=tl)
    pl = np.array([3, 8])
    out = oracle.commit(wk["acc_nodes"], wk["acc_len"], pl, k_tree=kt, v_tree=vt, k_cache=kc, v_cache=vc,
                        x=x, conv_w=w, beta=beta, decay=decay, S=S, conv_state=cs, Hk=Hk)
    tg = oracle.tree_gdn(x, w, cs, beta, decay, S, tree["parent"], tree["n_nodes"], Hk, want_states=True)
    for b in range(B):
        a = int(wk["acc_len"][b])
        path = wk["acc_nodes"][b][:a + 1]
        assert out["status"][b] == 0 and out["prefix_len"][b] == pl[b] + a + 1
        np.testing.assert_array_equal(out["src_row"][b][:a + 1], path)
        np.testing.assert_array_equal(out["dst_pos"][b][:a + 1], pl[b] + np.arange(a + 1))
        for l in range(La):
            for g in range(Hkv):
                np.testing.assert_array_equal(out["k_cache"][l, b, g, pl[b]:pl[b] + a + 1], kt[l, b, path, g])
                np.testing.assert_array_equal(out["v_cache"][l, b, g, pl[b]:pl[b] + a + 1], vt[l, b, path, g])
                np.testing.assert_array_equal(out["k_cache"][l, b, g, :pl[b]], kc[l, b, g, :pl[b]])
                np.testing.assert_array_equal(out["k_cache"][l, b, g, pl[b] + a + 1:],
                                              kc[l, b, g, pl[b] + a + 1:])
        for l in range(Lg):
            for h in range(Hv):
                np.testing.assert_allclose(out["S"][l, b, h], tg["S_node"][l, b, path[-1], h], atol=1e-12)
                _, Sseq = R.gdn_sequence(x[l, b, path], w[l], cs[l, b], beta[l, b, path, h],
                                         decay[l, b, path, h], S[l, b, h], Hk, Hv, h)
                np.testing.assert_allclose(out["S"][l, b, h], Sseq[-1], rtol=1e-10, atol=1e-10)
            full = np.concatenate([cs[l, b], x[l, b, path]])
            np.testing.assert_array_equal(out["conv_state"][l, b], full[-(K - 1):])
    assert wk["acc_len"][0] >= 1


def test_commit_capacity_refused():
    rng = _rng(17)
    kt = rng.normal(size=(1, 1, 3, 1, 2))
    kc = rng.normal(size=(1, 1, 1, 5, 2))
    out = oracle.commit(np.array([[0, 1, 2]]), [2], [3], k_tree=kt, v_tree=kt, k_cache=kc, v_cache=kc)
    assert out["status"][0] == 3 and out["prefix_len"][0] == 3
    np.testing.assert_array_equal(out["k_cache"], kc)


# ------------------------------------------------------------------ paged KV layout
def _pages_from_cache(cache, page, perm=None):
    """Independent construction: cut each (layer, request, head) slab into pages of `page`
    rows with numpy reshapes; page index of (b, i) is b * max_pages + i, optionally
    relabelled by `perm`."""
    L, B, Hkv, Pcap, d = cache.shape
    mp = Pcap // page
    pages = cache.reshape(L, B, Hkv, mp, page, d).transpose(0, 1, 3, 2, 4, 5).reshape(L, B * mp, Hkv, page, d)
    table = np.arange(B * mp, dtype=np.int32).reshape(B, mp)
    if perm is not None:
        out = np.empty_like(pages)
        out[:, perm] = pages          # logical page j is stored at physical page perm[j]
        return out, perm[table].astype(np.int32)
    return pages, table


@pytest.mark.parametrize("page", [1, 4, 16])
def test_gather_pages_identity_and_permuted(page):
    rng = np.random.default_rng(11)
    L, B, Hkv, Pcap, d = 2, 3, 2, 32, 5
    cache = rng.standard_normal((L, B, Hkv, Pcap, d))
    P = np.array([0, 17, 32], np.int32)
    want = cache.copy()
    for b in range(B):
        want[:, b, :, P[b]:] = 0.0
    pages, table = _pages_from_cache(cache, page)
    assert np.array_equal(oracle.gather_pages(pages, table, P, Pcap), want)
    perm = rng.permutation(pages.shape[1])
    pages2, table2 = _pages_from_cache(cache, page, perm)
    assert np.array_equal(oracle.gather_pages(pages2, table2, P, Pcap), want)


def test_scatter_pages_inverts_gather_on_the_rows_written():
    rng = np.random.default_rng(12)
    L, B, Hkv, Pcap, d, page = 1, 2, 3, 24, 4, 8
    cache = rng.standard_normal((L, B, Hkv, Pcap, d))
    pages, table = _pages_from_cache(cache, page, rng.permutation(B * Pcap // page))
    blank = np.full_like(pages, np.nan)
    n = np.array([24, 9], np.int32)
    back = oracle.scatter_pages(cache, table, n, blank)
    got = oracle.gather_pages(np.nan_to_num(back, nan=0.0), table, n, Pcap)
    want = cache.copy()
    want[:, 1, :, 9:] = 0.0
    assert np.array_equal(got, want)
    # pages no row was written to stay untouched
    assert np.isnan(back[:, table[1, 2]]).all()


def test_gather_pages_rejects_bad_tables():
    pages = np.zeros((1, 4, 1, 8, 2))
    with pytest.raises(RuntimeError):
        oracle.gather_pages(pages, np.array([[0, 9]], np.int32), [12], 16)   # page 9 does not exist
    with pytest.raises(RuntimeError):
        oracle.gather_pages(pages, np.array([[0, 1]], np.int32), [17], 17)   # past max_pages * page


# ------------------------------------------------------------------ rotary by depth
def test_rope_closed_forms():
    """Position 0 is the identity; pair 0 (frequency 1) turns by exactly `position`
    radians; pair i turns by position * theta^(-2i/rot); channels past rot are kept."""
    d, rot = 8, 6
    x = np.zeros((1, 1, 3, 1, d))
    x[..., 0] = 1.0          # pair 0 -> (cos p, sin p) at channels (0, 3)
    x[..., 1] = 2.0          # pair 1: x1 = 2 at channel 1, 0 at channel 4
    x[..., 6:] = 5.0         # outside the rotated part
    pos = np.array([[0, 3, 7]], np.int32)
    y = oracle.rope_tree(x, pos, [3], rot, theta=100.0)
    assert np.allclose(y[0, 0, 0, 0], x[0, 0, 0, 0])
    for n, p in ((1, 3), (2, 7)):
        assert np.isclose(y[0, 0, n, 0, 0], np.cos(p)) and np.isclose(y[0, 0, n, 0, 3], np.sin(p))
        a1 = p * 100.0 ** (-2.0 / rot)
        assert np.isclose(y[0, 0, n, 0, 1], 2 * np.cos(a1)) and np.isclose(y[0, 0, n, 0, 4], 2 * np.sin(a1))
        assert (y[0, 0, n, 0, 6:] == 5.0).all()


def test_rope_dot_products_depend_on_position_difference_only():
    """<R(m) q, R(n) k> = <R(m - n) q, k>: the defining property of rotary embedding; also
    norms are kept and padding rows are untouched."""
    rng = np.random.default_rng(21)
    d = 16
    q = rng.standard_normal((1, 1, 4, 1, d))
    k = rng.standard_normal((1, 1, 4, 1, d))
    pos = np.array([[5, 12, 40, 40]], np.int32)
    qr = oracle.rope_tree(q, pos, [3], d, theta=500.0)
    kr = oracle.rope_tree(k, pos, [3], d, theta=500.0)
    for m in range(3):
        for n in range(3):
            rel = oracle.rope_tree(q[:, :, m:m + 1], np.array([[pos[0, m] - pos[0, n]]], np.int32), [1], d,
                                   theta=500.0)
            assert np.isclose(np.dot(qr[0, 0, m, 0], kr[0, 0, n, 0]), np.dot(rel[0, 0, 0, 0], k[0, 0, n, 0]))
        assert np.isclose(np.linalg.norm(qr[0, 0, m, 0]), np.linalg.norm(q[0, 0, m, 0]))
    assert np.array_equal(qr[0, 0, 3], q[0, 0, 3])   # row 3 is padding (n_nodes = 3)


# ------------------------------------------------------------------ flat-commit safe mode
def _paths(tree, b):
    """Token path (root excluded) of every row of request b."""
    out = []
    for i in range(int(tree["n_nodes"][b])):
        p = R.path_rows(tree["parent"][b], i)
        out.append(tuple(int(tree["token"][b][r]) for r in p[1:]))
    return out


@pytest.mark.parametrize("seed", range(6))
def test_flat_walk_is_the_dflash_chain_walk(seed):
    """The safe-mode walk on a k = 4 tree accepts exactly what the ordinary walk accepts on
    the k = 1 tree (the flat DFlash chain) of the same drafter logits, when the target's
    token is a function of the token path: the regression invariant against flat DFlash."""
    rng = np.random.default_rng(100 + seed)
    D, V = 5, 7
    logits = rng.integers(-3, 4, size=(1, D, V)).astype(np.float64) + rng.standard_normal((1, D, V)) * 0.1
    full = oracle.build_tree(logits, [1], [0], 4, 30)
    chain = oracle.build_tree(logits, [1], [0], 1, 30)
    spine = _paths(chain, 0)[-1]                  # c_1 .. c_D
    m = int(rng.integers(0, D + 1))
    table = {}

    def target(path):
        if path not in table:
            j = len(path)
            if j < m and path == spine[:j]:
                table[path] = spine[j]            # agree along the chain
            else:                                 # anything else (often a sibling's token)
                table[path] = int(rng.integers(0, V)) if j >= D or path != spine[:j] else (spine[j] + 1) % V
        return table[path]

    def argmax_rows(tree):
        return np.array([[target(p) for p in _paths(tree, 0)] + [0] * (tree["token"].shape[1] - tree["n_nodes"][0])],
                        np.int32)

    f = oracle.walk(full["token"], full["parent"], full["n_nodes"], D, target_argmax=argmax_rows(full), flat=True)
    c = oracle.walk(chain["token"], chain["parent"], chain["n_nodes"], D, target_argmax=argmax_rows(chain))
    assert int(f["acc_len"][0]) == int(c["acc_len"][0]) == min(m, D)
    assert f["emitted"].tolist() == c["emitted"].tolist() and int(f["bonus"][0]) == int(c["bonus"][0])


@pytest.mark.parametrize("seed", range(4))
def test_flat_walk_brute_force_on_the_first_child_spine(seed):
    """Brute force: follow first children while the edge matches the target argmax; also
    never longer than the ordinary walk, and equal to it on a chain tree."""
    rng = np.random.default_rng(200 + seed)
    tree, _ = C_tree(rng)
    tok, par, nn = tree["token"][0], tree["parent"][0], int(tree["n_nodes"][0])
    targ = np.zeros((1, tok.shape[0]), np.int32)
    for i in range(nn):                          # half the rows agree with some child
        kids = [c for c in range(1, nn) if par[c] == i]
        targ[0, i] = int(tok[kids[int(rng.integers(len(kids)))]]) if kids and rng.random() < 0.7 else 10 ** 6
    f = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], 8, target_argmax=targ, flat=True)
    g = oracle.walk(tree["token"], tree["parent"], tree["n_nodes"], 8, target_argmax=targ)
    cur, want = 0, [0]
    while True:
        kids = [c for c in range(1, nn) if par[c] == cur]
        if not kids or int(tok[kids[0]]) != int(targ[0, cur]) or len(want) > 8:
            break
        cur = kids[0]
        want.append(cur)
    assert f["acc_nodes"][0][:len(want)].tolist() == want and int(f["acc_len"][0]) == len(want) - 1
    assert int(f["acc_len"][0]) <= int(g["acc_len"][0])


def C_tree(rng):
    logits = rng.standard_normal((1, 8, 40)) * 2
    return oracle.build_tree(logits, [3], [0], 3, 40), logits
