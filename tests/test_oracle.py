"""Pins of the CPU oracle against things other than itself: hand-worked
golden cases, brute-force loops, closed forms, invariants, central finite
differences, autograd of a dense formulation, and planted mistakes that the
pins must catch.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from mixture_experts_atomic_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            out[k] = [float(t) if ("." in t or "e" in t) else int(t) for t in v]
    return out


def _rand_problem(L, d, h, E, K, act, seed, one_expert=None):
    ids, gates = I.random_routing(L, E, K, seed, one_expert=one_expert)
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((L, d))
    W1 = rng.standard_normal((E, d, h)) / math.sqrt(d)
    W2 = rng.standard_normal((E, d, h)) / math.sqrt(d) if act == "swiglu" else None
    W3 = rng.standard_normal((E, h, d)) / math.sqrt(h)
    dY = rng.standard_normal((L, d))
    if act == "identity":
        W1 = W2 = W3 = None
    return ids.numpy(), gates.numpy().astype(np.float64), x, W1, W2, W3, dY


# ---------------------------------------------------------------- dispatch

def _dispatch_bruteforce(ids, E):
    """Per-slot loops, no sort: walk experts, then tokens in ascending order."""
    L, K = ids.shape
    D1, D2 = [], [0]
    D4 = [[-1] * K for _ in range(L)]
    for e in range(E):
        for t in range(L):
            for k in range(K):
                if ids[t][k] == e:
                    D4[t][k] = len(D1)
                    D1.append(t)
        D2.append(len(D1))
    return np.array(D1, dtype=np.int64), np.array(D2), np.array(ids), np.array(D4)


def test_dispatch_golden_hand_worked():
    g = _read_golden("dispatch_L5_E4_K2.txt")
    L, E, K = g["L"][0], g["E"][0], g["K"][0]
    ids = np.array(g["topk_ids"]).reshape(L, K)
    D1, D2, D3, D4 = O.dispatch(ids, E)
    assert D1.tolist() == g["expert_token_indices"]
    assert D2.tolist() == g["expert_token_offsets"]
    assert D3.reshape(-1).tolist() == g["token_expert_indices"]
    assert D4.reshape(-1).tolist() == g["token_index_map"]


@pytest.mark.parametrize("L,E,K,seed", [(1, 1, 1, 0), (7, 3, 2, 1), (16, 4, 4, 2),
                                        (33, 8, 3, 3), (40, 5, 1, 4), (12, 6, 6, 5)])
def test_dispatch_matches_bruteforce(L, E, K, seed):
    ids, _ = I.random_routing(L, E, K, seed)
    ids = ids.numpy()
    got = O.dispatch(ids, E)
    ref = _dispatch_bruteforce(ids, E)
    for a, b in zip(got, ref):
        assert np.array_equal(a.reshape(-1), b.reshape(-1))


def test_dispatch_invariants_and_edge_cases():
    # empty input
    D1, D2, D3, D4 = O.dispatch(np.zeros((0, 2), dtype=np.int64), 4)
    assert D1.size == 0 and D2.tolist() == [0] * 5
    # every token on one expert with K = 1: D1 is 0..L-1
    L = 37
    D1, D2, _, D4 = O.dispatch(np.full((L, 1), 2), 5)
    assert D1.tolist() == list(range(L))
    assert D2.tolist() == [0, 0, 0, L, L, L]
    # randomised invariants with skewed loads and empty experts
    ids, _ = I.random_routing(500, 9, 3, 7, one_expert=4)
    ids = ids.numpy()
    E = 12  # experts 9..11 receive no token
    D1, D2, D3, D4 = O.dispatch(ids, E)
    L, K = ids.shape
    assert D2[-1] == L * K and D2[0] == 0 and np.all(np.diff(D2) >= 0)
    assert np.array_equal(D2[10:], [L * K] * 3)
    assert sorted(D4.reshape(-1).tolist()) == list(range(L * K))  # every slot once
    assert np.array_equal(D1[D4], np.repeat(np.arange(L)[:, None], K, 1))
    assert np.array_equal(D3, ids)
    for e in range(E):
        seg = D1[D2[e]:D2[e + 1]]
        assert np.all(np.diff(seg) > 0)  # ascending token ids
        assert np.all((ids[seg] == e).any(axis=1))
    with pytest.raises(ValueError):
        O.dispatch(np.array([[0, 5]]), 4)
    assert not O.check_distinct(np.array([[1, 1]]))
    assert O.check_distinct(np.array([[1, 2]]))


# ---------------------------------------------------------------- forward

def _bruteforce_token(xrow, e, W1, W2, W3, act):
    """One token through one expert with scalar Python loops and math.exp."""
    d = len(xrow)
    if act == "identity":
        return list(xrow)
    h = len(W1[e][0])
    H = []
    for j in range(h):
        a = sum(xrow[i] * W1[e][i][j] for i in range(d))
        s = a / (1.0 + math.exp(-a))
        if act == "swiglu":
            b = sum(xrow[i] * W2[e][i][j] for i in range(d))
            H.append(s * b)
        else:
            H.append(s)
    return [sum(H[j] * W3[e][j][c] for j in range(h)) for c in range(d)]


@pytest.mark.parametrize("act", ["swiglu", "silu", "identity"])
def test_forward_matches_per_token_bruteforce(act):
    L, d, h, E, K = 9, 5, 4, 4, 2
    ids, g, x, W1, W2, W3, _ = _rand_problem(L, d, h, E, K, act, 11)
    y = O.forward(ids, g, x, W1, W2, W3, act, E=E)
    for t in range(L):
        ref = [0.0] * d
        for k in range(K):
            out = _bruteforce_token(x[t].tolist(), int(ids[t, k]),
                                    None if W1 is None else W1.tolist(),
                                    None if W2 is None else W2.tolist(),
                                    None if W3 is None else W3.tolist(), act)
            ref = [r + g[t, k] * o for r, o in zip(ref, out)]
        np.testing.assert_allclose(y[t], ref, rtol=1e-12, atol=1e-12)


def test_forward_identity_closed_form():
    # identity experts: y = (sum_k g) x = x for Dirichlet gates (sum to 1)
    L, d, E, K = 64, 8, 16, 4
    ids, g = I.random_routing(L, E, K, 3)
    x = np.random.default_rng(0).standard_normal((L, d))
    y = O.forward(ids, g, x, act="identity", E=E)
    np.testing.assert_allclose(y, g.numpy().astype(np.float64).sum(1)[:, None] * x, rtol=1e-14)
    np.testing.assert_allclose(y, x, rtol=1e-6, atol=1e-6)  # gates are fp32-rounded


def test_forward_single_expert_silu_is_dense_mlp():
    # one expert, K = 1, gate 1: y = SiLU(x W1) W3 (torch.nn.functional.silu)
    L, d, h = 20, 6, 10
    rng = np.random.default_rng(5)
    x = rng.standard_normal((L, d)); W1 = rng.standard_normal((1, d, h)); W3 = rng.standard_normal((1, h, d))
    y = O.forward(np.zeros((L, 1), dtype=np.int64), np.ones((L, 1)), x, W1, None, W3, "silu", E=1)
    ref = torch.nn.functional.silu(torch.from_numpy(x) @ torch.from_numpy(W1[0])) @ torch.from_numpy(W3[0])
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_swiglu_scalar_golden():
    gd = _read_golden("swiglu_scalar_closed_form.txt")
    f = lambda k: np.array(gd[k], dtype=np.float64)
    x = f("x").reshape(1, 1)
    W1 = f("W1").reshape(1, 1, 1); W2 = f("W2").reshape(1, 1, 1); W3 = f("W3").reshape(1, 1, 1)
    ids = np.zeros((1, 1), dtype=np.int64); g = f("g").reshape(1, 1); dY = f("dY").reshape(1, 1)
    y = O.forward(ids, g, x, W1, W2, W3, "swiglu", E=1)
    dX, dW1, dW2, dW3, dg = O.backward(ids, g, x, dY, W1, W2, W3, "swiglu", E=1)
    for name, v in [("y", y), ("dX", dX), ("dW1", dW1), ("dW2", dW2), ("dW3", dW3), ("dgates", dg)]:
        assert float(v.reshape(-1)[0]) == pytest.approx(gd[name][0], rel=1e-14), name


# ---------------------------------------------------------------- backward

def _loss(ids, g, x, W1, W2, W3, dY, act, E):
    return float(np.sum(O.forward(ids, g, x, W1, W2, W3, act, E=E) * dY))


def _fd_errors(ids, g, x, W1, W2, W3, dY, act, E, eps=1e-5, n_samples=None, seed=0):
    """max relative error of the oracle's backward vs central differences."""
    dX, dW1, dW2, dW3, dg = O.backward(ids, g, x, dY, W1, W2, W3, act, E=E)
    rng = np.random.default_rng(seed)
    errs = {}
    for name, arr, grad in [("x", x, dX), ("W1", W1, dW1), ("W2", W2, dW2), ("W3", W3, dW3), ("gates", g, dg)]:
        if arr is None:
            continue
        flat = arr.reshape(-1)
        idxs = range(flat.size) if n_samples is None else rng.choice(flat.size, n_samples, replace=False)
        fd = []
        an = []
        for i in idxs:
            old = flat[i]
            flat[i] = old + eps
            lp = _loss(ids, g, x, W1, W2, W3, dY, act, E)
            flat[i] = old - eps
            lm = _loss(ids, g, x, W1, W2, W3, dY, act, E)
            flat[i] = old
            fd.append((lp - lm) / (2 * eps))
            an.append(grad.reshape(-1)[i])
        fd = np.array(fd); an = np.array(an)
        errs[name] = float(np.max(np.abs(fd - an)) / max(np.max(np.abs(fd)), 1e-30))
    return errs


@pytest.mark.parametrize("act", ["swiglu", "silu", "identity"])
def test_backward_central_finite_differences(act):
    L, d, h, E, K = 7, 4, 3, 3, 2
    ids, g, x, W1, W2, W3, dY = _rand_problem(L, d, h, E, K, act, 21)
    errs = _fd_errors(ids, g, x, W1, W2, W3, dY, act, E)
    assert max(errs.values()) < 1e-7, errs  # the benchmark spec's bound is 1e-3


def test_backward_fd_config0_shape_sampled():
    # the fp32 config's shape class with a smaller L; sampled entries
    cfg = I.CONFIGS[0].scaled(L=24)
    inp = I.make_inputs(cfg)
    args = [inp["ids"].numpy(), inp["gates"].numpy().astype(np.float64),
            O._f64(inp["x"]), O._f64(inp["W1"]), O._f64(inp["W2"]), O._f64(inp["W3"]), O._f64(inp["dY"])]
    errs = _fd_errors(*args, "swiglu", cfg.E, eps=1e-5, n_samples=12)
    assert max(errs.values()) < 1e-6, errs


@pytest.mark.parametrize("act", ["swiglu", "silu"])
def test_backward_matches_autograd_dense(act):
    """torch.autograd (fp64) of a dense formulation in which every token runs
    through every expert, masked by a dense gate matrix."""
    L, d, h, E, K = 11, 6, 5, 4, 2
    ids, g, x, W1, W2, W3, dY = _rand_problem(L, d, h, E, K, act, 31)
    T = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    xt, w1, w3, gt = T(x), T(W1), T(W3), T(g)
    w2 = T(W2) if act == "swiglu" else None
    onehot = torch.zeros(L, K, E, dtype=torch.float64)
    for t in range(L):
        for k in range(K):
            onehot[t, k, ids[t, k]] = 1.0
    Gd = torch.einsum("lk,lke->le", gt, onehot)
    a = torch.einsum("ld,edh->leh", xt, w1)
    H = torch.nn.functional.silu(a)
    if act == "swiglu":
        H = H * torch.einsum("ld,edh->leh", xt, w2)
    Y = torch.einsum("leh,ehd->led", H, w3)
    y = (Gd[:, :, None] * Y).sum(1)
    (y * torch.tensor(dY)).sum().backward()
    dX, dW1, dW2, dW3, dg = O.backward(ids, g, x, dY, W1, W2, W3, act, E=E)
    np.testing.assert_allclose(dX, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dW1, w1.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dW3, w3.grad.numpy(), rtol=1e-10, atol=1e-12)
    if act == "swiglu":
        np.testing.assert_allclose(dW2, w2.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(O.forward(ids, g, x, W1, W2, W3, act, E=E), y.detach().numpy(),
                               rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- sampled helpers

@pytest.mark.parametrize("act", ["swiglu", "silu", "identity"])
def test_sampled_helpers_agree_with_full_oracle(act):
    L, d, h, E, K = 30, 8, 6, 5, 3
    ids, g, x, W1, W2, W3, dY = _rand_problem(L, d, h, E, K, act, 41)
    y = O.forward(ids, g, x, W1, W2, W3, act, E=E)
    dX, dW1, dW2, dW3, dg = O.backward(ids, g, x, dY, W1, W2, W3, act, E=E)
    toks = [0, 3, 17, 29]
    np.testing.assert_allclose(O.forward_rows(toks, ids, g, x[toks], W1, W2, W3, act), y[toks], rtol=1e-12, atol=1e-13)
    rdx, rdg = O.backward_rows(toks, ids, g, x[toks], dY[toks], W1, W2, W3, act, with_dgates=True)
    np.testing.assert_allclose(rdx, dX[toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(rdg, dg[toks], rtol=1e-12, atol=1e-13)
    if act == "identity":
        return
    D1, D2, D3, D4 = O.dispatch(ids, E)
    gr = np.zeros(L * K)
    for k in range(K):
        gr[D4[:, k]] = g[:, k]
    for e in range(E):
        seg = D1[D2[e]:D2[e + 1]]
        c1, c2, r3 = O.weight_grad_slices(e, seg, gr[D2[e]:D2[e + 1]], x[seg], dY[seg], W1, W2, W3, act,
                                          h_cols=[0, h - 1], w3_rows=[1, 2])
        np.testing.assert_allclose(c1, dW1[e][:, [0, h - 1]], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(r3, dW3[e][[1, 2], :], rtol=1e-12, atol=1e-13)
        if act == "swiglu":
            np.testing.assert_allclose(c2, dW2[e][:, [0, h - 1]], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- planted mistakes

def test_pins_catch_planted_mistakes(monkeypatch):
    """A plausible mistake in the oracle makes at least one pin fail."""
    L, d, h, E, K = 6, 3, 4, 3, 2
    ids, g, x, W1, W2, W3, dY = _rand_problem(L, d, h, E, K, "swiglu", 51)

    # 1) dropped term in SiLU' -> finite differences disagree
    with monkeypatch.context() as m:
        m.setattr(O, "silu_grad", lambda a: O.sigmoid(a))
        assert max(_fd_errors(ids, g, x, W1, W2, W3, dY, "swiglu", E).values()) > 1e-3

    # 2) W1 and W2 swapped in the expert -> per-token brute force disagrees
    orig = O.expert_forward
    with monkeypatch.context() as m:
        m.setattr(O, "expert_forward", lambda X, a, b, c, act: orig(X, b, a, c, act))
        y = O.forward(ids, g, x, W1, W2, W3, "swiglu", E=E)
        out = _bruteforce_token(x[0].tolist(), int(ids[0, 0]), W1.tolist(), W2.tolist(), W3.tolist(), "swiglu")
        out2 = _bruteforce_token(x[0].tolist(), int(ids[0, 1]), W1.tolist(), W2.tolist(), W3.tolist(), "swiglu")
        ref0 = g[0, 0] * np.array(out) + g[0, 1] * np.array(out2)
        assert np.max(np.abs(y[0] - ref0)) > 1e-6

    # 3) descending tokens inside an expert -> brute-force dispatch disagrees
    D1, D2, D3, D4 = O.dispatch(ids, E)
    bad = D1.copy()
    for e in range(E):
        bad[D2[e]:D2[e + 1]] = bad[D2[e]:D2[e + 1]][::-1]
    assert not np.array_equal(bad, _dispatch_bruteforce(ids, E)[0])

    # 4) wrong sign of SiLU(a) in the gate-branch gradient dB = dH * SiLU(a)
    #    (the backward reads SiLU(a) as out["s"]) -> finite differences disagree
    with monkeypatch.context() as m:
        def bad_ef(X, a, b, c, act):
            out = orig(X, a, b, c, act)
            if "s" in out:
                out = dict(out); out["s"] = -out["s"]
            return out
        m.setattr(O, "expert_forward", bad_ef)
        errs = _fd_errors(ids, g, x, W1, W2, W3, dY, "swiglu", E)
        assert max(errs.values()) > 1e-3


# ---------------------------------------------------------------- router (the step before the dispatch)

def test_router_golden_hand_worked():
    gd = _read_golden("router_tiny.txt")
    Wr = np.array(gd["Wr"], dtype=np.float64).reshape(2, 4)
    for t in range(3):
        bias = np.array(gd[f"bias{t}"], dtype=np.float64) if f"bias{t}" in gd else None
        ids, g, _ = O.router(np.array([gd[f"x{t}"]], dtype=np.float64), Wr, bias, 2)
        assert ids[0].tolist() == gd[f"ids{t}"]
        np.testing.assert_allclose(g[0], gd[f"gates{t}"], rtol=0, atol=1e-15)


def test_router_k_equals_e_is_the_full_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(60)
    L, d, E = 40, 16, 7
    x, Wr, b = rng.standard_normal((L, d)), rng.standard_normal((d, E)), rng.standard_normal(E)
    ids, g, lg = O.router(x, Wr, b, E)
    p = softmax(np.einsum("td,de->te", x, Wr) + b, axis=1)
    for t in range(L):
        assert sorted(ids[t].tolist()) == list(range(E))
        assert np.all(np.diff(lg[t, ids[t]]) <= 0)
        np.testing.assert_allclose(g[t], p[t, ids[t]], rtol=1e-12)


def _router_bruteforce(logits, K):
    """Every K-subset: the one with the largest sum, among those the smallest
    sorted index tuple; slots ordered by value, then index; gates by a loop."""
    import itertools
    E = len(logits)
    best = None
    for sub in itertools.combinations(range(E), K):
        key = (sum(logits[e] for e in sub), [-e for e in sub])
        if best is None or key > best[0]:
            best = (key, sub)
    chosen = sorted(best[1], key=lambda e: (-logits[e], e))
    w = [math.exp(logits[e] - logits[chosen[0]]) for e in chosen]
    return chosen, [v / sum(w) for v in w]


def test_router_matches_bruteforce_over_subsets():
    rng = np.random.default_rng(61)
    for K in (1, 2, 3, 6):
        # small integer features and weights: many exact ties between logits
        x = rng.integers(-2, 3, size=(30, 3)).astype(np.float64)
        Wr = rng.integers(-1, 2, size=(3, 6)).astype(np.float64)
        ids, g, lg = O.router(x, Wr, None, K)
        for t in range(30):
            chosen, gates = _router_bruteforce(lg[t].tolist(), K)
            assert ids[t].tolist() == chosen
            np.testing.assert_allclose(g[t], gates, rtol=1e-13)


def test_router_shift_invariance():
    rng = np.random.default_rng(62)
    x, Wr = rng.standard_normal((25, 8)), rng.standard_normal((8, 9))
    ids0, g0, _ = O.router(x, Wr, None, 3)
    ids1, g1, _ = O.router(x, Wr, np.full(9, 4.5), 3)
    assert np.array_equal(ids0, ids1)
    np.testing.assert_allclose(g0, g1, rtol=1e-12)


def _router_loss(x, Wr, b, ids, dg):
    """sum_t,k dg * gates with the selection held at `ids` (fp64)."""
    lg = x @ Wr + b
    top = np.take_along_axis(lg, ids, axis=1)
    w = np.exp(top - top.max(axis=1, keepdims=True))
    return float(np.sum(dg * w / w.sum(axis=1, keepdims=True)))


def _router_fd_errors(rb=O.router_backward):
    rng = np.random.default_rng(63)
    L, d, E, K = 5, 4, 6, 3
    x, Wr, b = rng.standard_normal((L, d)), rng.standard_normal((d, E)), rng.standard_normal(E)
    ids, g, lg = O.router(x, Wr, b, K)
    srt = np.sort(lg, axis=1)[:, ::-1]
    assert np.min(srt[:, K - 1] - srt[:, K]) > 1e-3  # no near-tie at the selection boundary
    dg = rng.standard_normal((L, K))
    dWr, db, dx, _ = rb(x, Wr, ids, g, dg, E)
    eps, errs = 1e-6, {}
    for name, arr, grad in (("Wr", Wr, dWr), ("x", x, dx), ("bias", b, db)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a1 = arr.copy(); a1[idx] += eps
            a2 = arr.copy(); a2[idx] -= eps
            args1 = {"x": x, "Wr": Wr, "bias": b}; args1[name] = a1
            args2 = {"x": x, "Wr": Wr, "bias": b}; args2[name] = a2
            num[idx] = (_router_loss(args1["x"], args1["Wr"], args1["bias"], ids, dg)
                        - _router_loss(args2["x"], args2["Wr"], args2["bias"], ids, dg)) / (2 * eps)
        errs[name] = float(np.max(np.abs(num - grad)) / max(1e-12, np.max(np.abs(num))))
    return errs


def test_router_backward_finite_differences():
    errs = _router_fd_errors()
    assert max(errs.values()) < 1e-6, errs


def test_router_backward_matches_autograd():
    rng = np.random.default_rng(64)
    L, d, E, K = 50, 12, 10, 4
    x, Wr, b = rng.standard_normal((L, d)), rng.standard_normal((d, E)), rng.standard_normal(E)
    ids, g, _ = O.router(x, Wr, b, K)
    dg = rng.standard_normal((L, K))
    dWr, db, dx, _ = O.router_backward(x, Wr, ids, g, dg, E)
    tx, tW, tb = (torch.tensor(v, dtype=torch.float64, requires_grad=True) for v in (x, Wr, b))
    sel = torch.gather(tx @ tW + tb, 1, torch.from_numpy(ids))
    (torch.softmax(sel, dim=1) * torch.from_numpy(dg)).sum().backward()
    np.testing.assert_allclose(dWr, tW.grad.numpy(), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(db, tb.grad.numpy(), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dx, tx.grad.numpy(), rtol=1e-11, atol=1e-13)


def test_router_pins_catch_planted_mistakes():
    # 1) the centring term of the softmax gradient dropped -> finite differences disagree
    def bad_rb(x, Wr, topk_ids, gates, dgates, E):
        X = O._f64(x); ids = O._i64(topk_ids); g = O._f64(gates); dg = O._f64(dgates)
        dl = np.zeros((X.shape[0], E))
        np.put_along_axis(dl, ids, g * dg, axis=1)
        return X.T @ dl, dl.sum(axis=0), dl @ O._f64(Wr).T, dl
    assert max(_router_fd_errors(bad_rb).values()) > 1e-2
    # 2) ties broken towards the higher index -> the hand-worked golden case disagrees
    gd = _read_golden("router_tiny.txt")
    lg = np.array(gd["x0"], dtype=np.float64) @ np.array(gd["Wr"], dtype=np.float64).reshape(2, 4)
    wrong = sorted(range(4), key=lambda e: (-lg[e], -e))[:2]  # equal logits to the higher index
    assert wrong != gd["ids0"]
    # 3) gates over all E experts instead of the K selected -> the K = E softmax pin's
    #    renormalisation check fails for K < E
    ids, g, lg = O.router(np.array([gd["x0"]], dtype=np.float64), np.array(gd["Wr"], dtype=np.float64).reshape(2, 4), None, 2)
    full = np.exp(lg[0] - lg[0].max()); full /= full.sum()
    assert abs(full[ids[0]].sum() - 1.0) > 1e-3 and abs(g[0].sum() - 1.0) < 1e-15


# ---------------------------------------------------------------- the parity checker
# Every GPU parity test reduces to rel_err(got, ref) <= tol, the tolerance rule
# max|gpu - ref| / max|ref|.  Its cases are worked by hand here.

# (got, ref, expected value): a value None means "must not compare <= any tol"
_REL_ERR_CASES = [
    # |got - ref| = (0.25, 0.5, 0); max|ref| = 4 (the negative entry) -> 0.125
    ([1.25, 2.5, -4.0], [1.0, 2.0, -4.0], 0.125),
    # max|got| = 3 differs from max|ref| = 2: the denominator is the reference's
    ([-3.0, -1.0], [-2.0, -1.0], 0.5),
    # the largest deviation is a negative one: max of |.|, not of the signed difference
    ([0.0, 1.0], [2.0, 1.0], 1.0),
    # all-zero reference: the absolute deviation itself
    ([0.0, -0.25], [0.0, 0.0], 0.25),
    ([0.0, 0.0, 0.0], [0.0, 0.0, 0.0], 0.0),
    # one large deviation among many small ones: a max, not a mean (mean would give 0.0375)
    ([1.1, 1.0, 1.0, 1.0], [1.0, 1.0, 1.0, 1.0], 0.1),
    # a NaN in the GPU result never passes a tolerance
    ([1.0, float("nan")], [1.0, 1.0], None),
    # an infinite GPU result never passes either
    ([float("inf"), 1.0], [1.0, 1.0], None),
]


def _rel_err_cases_hold(fn):
    for got, ref, want in _REL_ERR_CASES:
        v = fn(np.array(got), np.array(ref))
        if want is None:
            if v <= 1e30:
                return False
        elif not abs(v - want) <= 1e-15:
            return False
    return True


def test_rel_err_hand_worked():
    assert _rel_err_cases_hold(O.rel_err)
    # 2-D inputs and bf16 torch tensors (widened exactly before subtracting)
    got = torch.tensor([[1.0, -2.0], [0.5, 3.0]]).to(torch.bfloat16)
    ref = np.array([[1.0, -2.0], [0.25, 4.0]])
    assert O.rel_err(got, ref) == 0.25  # max|.| = 1 (3 vs 4), max|ref| = 4


def test_rel_err_pins_catch_planted_variants():
    """Plausible slips in the checker each break at least one hand-worked case."""
    a = np.abs

    def den_from_got(g, r):      # denominator max|got|
        return float(np.max(a(g - r)) / np.max(a(g))) if np.max(a(g)) else float(np.max(a(g - r)))

    def no_abs(g, r):            # max(got - ref) / max(ref)
        return float(np.max(g - r) / np.max(r)) if np.max(r) else float(np.max(g - r))

    def mean_not_max(g, r):      # mean deviation
        return float(np.mean(a(g - r)) / np.max(a(r))) if np.max(a(r)) else float(np.mean(a(g - r)))

    def zero_for_zero_ref(g, r):  # 0 whenever the reference is all zero
        d = np.max(a(r))
        return float(np.max(a(g - r)) / d) if d else 0.0

    def nan_ignored(g, r):       # nanmax lets a NaN through
        d = np.nanmax(a(r))
        n = np.nanmax(a(g - r))
        return float(n / d) if d else float(n)

    def finite_only(g, r):       # drops non-finite entries before comparing
        m = np.isfinite(g)
        return O.rel_err(g[m], r[m])

    for bad in (den_from_got, no_abs, mean_not_max, zero_for_zero_ref, nan_ignored, finite_only):
        assert not _rel_err_cases_hold(bad), bad.__name__
