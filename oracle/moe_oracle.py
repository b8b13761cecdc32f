"""CPU oracle of the dropless top-K MoE layer: the conventional pipeline.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module; only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code with the CUDA path (it imports numpy and nothing else).

What it computes follows the "conventional" side of Figure 1 of MoEBlaze
(awesome-system-papers page, "核心方法 / 免物化 token dispatch" and the
Figure 1 caption on the sciencestack page): dispatch by sorting -> a
materialised per-expert buffer -> the expert MLP, unfused -> a weighted
reduce, followed by a hand-derived backward.  All arithmetic is fp64 on the
exact input values (bf16 or fp32 inputs are widened losslessly).

Index structures (page 1, data-structure table under "免物化 token dispatch"):

* ``expert_token_indices`` (L*K): token ids concatenated expert by expert;
  within one expert in ascending token id.
* ``expert_token_offsets`` (E+1): the interval of each expert in the above.
* ``token_expert_indices`` (L,K): the expert of each (token, slot), in the
  caller's slot order (the inverse map).
* ``token_index_map`` (L,K): the global position of each (token, slot) in
  ``expert_token_indices``, used by the combine.

Expert MLP (page 1, "SwiGLU kernel 融合 + activation checkpoint"):
a = x W1, b = x W2, SwiGLU output SiLU(a) * b, SiLU(a) = a * sigmoid(a);
the SiLU (non-gated) expert drops W2; the identity expert returns x.
The layer output is y[t] = sum_k g[t,k] * expert_{ids[t,k]}(x[t]).
The backward takes the loss as <y, dY> with ids and gates held constant.

Parity status of each function is pinned in tests/test_oracle.py; see the
module constants ``PINNED``.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence, Tuple

import numpy as np

PINNED = {
    "dispatch": "brute-force per-slot loops, hand-worked golden case, invariants",
    "forward": "per-token brute force, identity closed form, dense-MLP special case",
    "backward": "central finite differences (fp64), torch.autograd of a dense formulation",
    "backward dgates": "central finite differences in the gates, autograd, hand-worked golden case",
    "forward_rows / backward_rows / weight_grad_slices": "agree with forward/backward on every row and column at small sizes",
    "router": "hand-worked golden case (ties, bias), K = E equals the full softmax, brute force over all K-subsets, shift invariance",
    "router_backward": "central finite differences in Wr, x and the bias, torch.autograd of the softmax over the selected logits",
    "rel_err": "hand-worked cases (negative and all-zero references, NaN and inf in the result) and planted variants of the rule",
}


def _f64(a) -> np.ndarray:
    """Widen an array (numpy or torch, any float dtype incl. bf16) to fp64."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # a torch tensor: go through float32 for bf16
        import torch  # local: only when handed torch tensors
        t = a.detach().cpu()
        if t.dtype == torch.bfloat16:
            t = t.to(torch.float32)
        return t.numpy().astype(np.float64)
    return np.asarray(a, dtype=np.float64)


def _i64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        return a.detach().cpu().numpy().astype(np.int64)
    return np.asarray(a, dtype=np.int64)


# ---------------------------------------------------------------------------
# activation and its derivative (page 1, SwiGLU section)
# ---------------------------------------------------------------------------

def sigmoid(a: np.ndarray) -> np.ndarray:
    # split by sign so exp never overflows
    out = np.empty_like(a)
    pos = a >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-a[pos]))
    ea = np.exp(a[~pos])
    out[~pos] = ea / (1.0 + ea)
    return out


def silu(a: np.ndarray) -> np.ndarray:
    return a * sigmoid(a)


def silu_grad(a: np.ndarray) -> np.ndarray:
    """d/da [a sigmoid(a)] = sigmoid(a) (1 + a (1 - sigmoid(a)))."""
    s = sigmoid(a)
    return s * (1.0 + a * (1.0 - s))


# ---------------------------------------------------------------------------
# dispatch: the conventional sort-based build
# ---------------------------------------------------------------------------

def dispatch(topk_ids, E: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """Sort-based dispatch.

    The L*K (expert, token) pairs, enumerated token-major in (t, k) order, are
    sorted by expert with a stable sort; the token ids in sorted order are
    ``expert_token_indices``; a count per expert and its exclusive scan give
    ``expert_token_offsets``; the inverse of the sorting permutation gives
    ``token_index_map``; ``token_expert_indices`` is the ids array itself.

    Returns (expert_token_indices (LK,), expert_token_offsets (E+1,),
    token_expert_indices (L,K), token_index_map (L,K)), all int64.
    """
    ids = _i64(topk_ids)
    L, K = ids.shape
    flat_e = ids.reshape(-1)
    if flat_e.size and (flat_e.min() < 0 or flat_e.max() >= E):
        raise ValueError("expert id out of range")
    flat_t = np.repeat(np.arange(L, dtype=np.int64), K)
    perm = np.argsort(flat_e, kind="stable")          # sorted slot order
    expert_token_indices = flat_t[perm]
    counts = np.bincount(flat_e, minlength=E).astype(np.int64)
    expert_token_offsets = np.zeros(E + 1, dtype=np.int64)
    expert_token_offsets[1:] = np.cumsum(counts)
    inv = np.empty(L * K, dtype=np.int64)
    inv[perm] = np.arange(L * K, dtype=np.int64)
    token_index_map = inv.reshape(L, K)
    token_expert_indices = ids.copy()
    return expert_token_indices, expert_token_offsets, token_expert_indices, token_index_map


def check_distinct(topk_ids) -> bool:
    """True when every token's K ids are pairwise distinct (the pages'
    assumption that each (token, expert) cell is marked at most once)."""
    ids = _i64(topk_ids)
    s = np.sort(ids, axis=1)
    return bool(np.all(s[:, 1:] != s[:, :-1])) if ids.shape[1] > 1 else True


# ---------------------------------------------------------------------------
# expert MLP on a materialised buffer
# ---------------------------------------------------------------------------

def expert_forward(X: np.ndarray, W1: Optional[np.ndarray], W2: Optional[np.ndarray],
                   W3: Optional[np.ndarray], act: str) -> Dict[str, np.ndarray]:
    """Unfused expert MLP on rows X (n,d).  Returns a dict with the
    intermediates the conventional path materialises (a, b, sigma(a),
    SiLU(a), H) and the output Y."""
    if act == "identity":
        return {"Y": X.copy()}
    a = X @ W1
    sg = sigmoid(a)
    s = a * sg
    if act == "swiglu":
        b = X @ W2
        H = s * b
    elif act == "silu":
        b = None
        H = s
    else:
        raise ValueError(act)
    Y = H @ W3
    return {"a": a, "b": b, "sig": sg, "s": s, "H": H, "Y": Y}


def forward(topk_ids, gates, x, W1=None, W2=None, W3=None, act: str = "swiglu",
            E: Optional[int] = None, keep: bool = False):
    """Conventional forward: dispatch, per-expert materialise + MLP, weighted
    reduce over k in ascending slot order.

    Returns y (L,d) fp64, and when ``keep`` a dict with the dispatch result
    and per-expert 'a' and 'b' (the values the fused path checkpoints), keyed
    by expert.
    """
    ids = _i64(topk_ids)
    g = _f64(gates)
    X = _f64(x)
    w1, w2, w3 = _f64(W1), _f64(W2), _f64(W3)
    L, K = ids.shape
    if E is None:
        E = w1.shape[0] if w1 is not None else int(ids.max()) + 1
    D1, D2, D3, D4 = dispatch(ids, E)
    d = X.shape[1]
    # per-expert output buffers (the conventional routed layout, LK rows)
    Yrouted = np.zeros((L * K, d), dtype=np.float64)
    saved = {}
    for e in range(E):
        lo, hi = D2[e], D2[e + 1]
        if hi == lo:
            continue
        Xe = X[D1[lo:hi]]                       # materialise the routed rows
        out = expert_forward(Xe, None if w1 is None else w1[e],
                             None if w2 is None else w2[e],
                             None if w3 is None else w3[e], act)
        Yrouted[lo:hi] = out["Y"]
        if keep and act != "identity":
            saved[e] = {"a": out["a"], "b": out["b"]}
    y = np.zeros((L, d), dtype=np.float64)
    for k in range(K):                          # weighted reduce, ascending k
        y += g[:, k:k + 1] * Yrouted[D4[:, k]]
    if keep:
        return y, {"dispatch": (D1, D2, D3, D4), "saved": saved}
    return y


def backward(topk_ids, gates, x, dY, W1=None, W2=None, W3=None, act: str = "swiglu",
             E: Optional[int] = None):
    """Hand-derived backward of the loss <y, dY> with the ids held constant.
    Per expert e and its routed rows (token t, gate g):

        G      = g * dY[t]                       (the gradient scattered to the row)
        dW3_e += H^T G
        dH     = G W3_e^T
        dA     = dH * b * SiLU'(a)   (SiLU expert: dH * SiLU'(a))
        dB     = dH * SiLU(a)
        dW1_e += X_e^T dA ;  dW2_e += X_e^T dB
        dx[t] += dA W1_e^T + dB W2_e^T
    Identity expert: dx[t] = sum_k g[t,k] dY[t].
    Gate gradient (y is linear in the gates): dg[t,k] = <dY[t], Y_row>, the
    expert's output for that routed row before gating.

    Returns (dX (L,d), dW1, dW2, dW3, dgates (L,K)) in fp64 (None where the
    weight is absent).
    """
    ids = _i64(topk_ids)
    g = _f64(gates)
    X = _f64(x)
    gy = _f64(dY)
    w1, w2, w3 = _f64(W1), _f64(W2), _f64(W3)
    L, K = ids.shape
    if E is None:
        E = w1.shape[0] if w1 is not None else int(ids.max()) + 1
    D1, D2, D3, D4 = dispatch(ids, E)
    # gate of each routed row p: slot k of token D1[p] with D4[t,k] == p
    gate_routed = np.zeros(L * K, dtype=np.float64)
    for k in range(K):
        gate_routed[D4[:, k]] = g[:, k]
    dX = np.zeros_like(X)
    dg_routed = np.zeros(L * K, dtype=np.float64)     # <dY[t], Y_row> per routed row
    if act == "identity":
        np.add.at(dX, D1, gate_routed[:, None] * gy[D1])
        dg_routed[:] = np.sum(gy[D1] * X[D1], axis=1)
        return dX, None, None, None, dg_routed[D4]
    dW1 = np.zeros_like(w1)
    dW2 = np.zeros_like(w2) if act == "swiglu" else None
    dW3 = np.zeros_like(w3)
    for e in range(E):
        lo, hi = D2[e], D2[e + 1]
        if hi == lo:
            continue
        rows = D1[lo:hi]
        Xe = X[rows]
        out = expert_forward(Xe, w1[e], None if w2 is None else w2[e], w3[e], act)
        G = gate_routed[lo:hi, None] * gy[rows]  # expand dY to the routed rows
        dg_routed[lo:hi] = np.sum(gy[rows] * out["Y"], axis=1)
        dW3[e] = out["H"].T @ G
        dH = G @ w3[e].T
        if act == "swiglu":
            dA = dH * out["b"] * silu_grad(out["a"])
            dB = dH * out["s"]
            dW2[e] = Xe.T @ dB
            dXe = dA @ w1[e].T + dB @ w2[e].T
        else:
            dA = dH * silu_grad(out["a"])
            dXe = dA @ w1[e].T
        dW1[e] = Xe.T @ dA
        np.add.at(dX, rows, dXe)                 # reduce the routed rows
    return dX, dW1, dW2, dW3, dg_routed[D4]


# ---------------------------------------------------------------------------
# sampled outputs for full-size checks (same definitions, restricted)
# ---------------------------------------------------------------------------

def forward_rows(tokens: Sequence[int], topk_ids, gates, x_rows, W1=None, W2=None,
                 W3=None, act: str = "swiglu") -> np.ndarray:
    """y for a subset of tokens: y[t] = sum_k g[t,k] expert_{ids[t,k]}(x[t]).
    ``x_rows`` holds x for exactly these tokens (in this order); ids and
    gates are the full (L,K) arrays."""
    ids = _i64(topk_ids)
    g = _f64(gates)
    Xr = _f64(x_rows)
    tokens = np.asarray(tokens, dtype=np.int64)
    y = np.zeros_like(Xr)
    K = ids.shape[1]
    for k in range(K):
        ek = ids[tokens, k]
        for e in np.unique(ek):
            sel = np.nonzero(ek == e)[0]
            out = expert_forward(Xr[sel], None if W1 is None else _f64(W1[e]),
                                 None if W2 is None else _f64(W2[e]),
                                 None if W3 is None else _f64(W3[e]), act)
            y[sel] += g[tokens[sel], k:k + 1] * out["Y"]
    return y


def backward_rows(tokens: Sequence[int], topk_ids, gates, x_rows, dy_rows, W1=None,
                  W2=None, W3=None, act: str = "swiglu", with_dgates: bool = False):
    """dX for a subset of tokens (same formulas as ``backward``); with
    ``with_dgates`` also the (len(tokens), K) gate gradients."""
    ids = _i64(topk_ids)
    g = _f64(gates)
    Xr = _f64(x_rows)
    Gy = _f64(dy_rows)
    tokens = np.asarray(tokens, dtype=np.int64)
    K = ids.shape[1]
    dX = np.zeros_like(Xr)
    dg = np.zeros((len(tokens), K))
    for k in range(K):
        gk = g[tokens, k:k + 1]
        if act == "identity":
            dX += gk * Gy
            dg[:, k] = np.sum(Gy * Xr, axis=1)
            continue
        ek = ids[tokens, k]
        for e in np.unique(ek):
            sel = np.nonzero(ek == e)[0]
            w1 = _f64(W1[e]); w3 = _f64(W3[e])
            w2 = _f64(W2[e]) if act == "swiglu" else None
            out = expert_forward(Xr[sel], w1, w2, w3, act)
            dg[sel, k] = np.sum(Gy[sel] * out["Y"], axis=1)
            dH = (gk[sel] * Gy[sel]) @ w3.T
            if act == "swiglu":
                dA = dH * out["b"] * silu_grad(out["a"])
                dB = dH * out["s"]
                dX[sel] += dA @ w1.T + dB @ w2.T
            else:
                dA = dH * silu_grad(out["a"])
                dX[sel] += dA @ w1.T
    return (dX, dg) if with_dgates else dX


def weight_grad_slices(e: int, rows_tokens, row_gates, X_e, dY_e, W1, W2, W3,
                       act: str, h_cols: Sequence[int], w3_rows: Sequence[int]):
    """Selected slices of one expert's weight gradients.

    ``rows_tokens`` are expert e's routed tokens, ``row_gates`` their gates,
    ``X_e``/``dY_e`` the matching rows of x and dY.  Returns
    (dW1[e][:, h_cols], dW2[e][:, h_cols] or None, dW3[e][w3_rows, :]).
    Column j of dW1/dW2 needs only column j of W1, W2 and row j of W3;
    row i of dW3 needs only column i of W1, W2.
    """
    Xe = _f64(X_e)
    G = _f64(row_gates)[:, None] * _f64(dY_e)
    w1 = _f64(W1[e]); w3 = _f64(W3[e])
    w2 = _f64(W2[e]) if act == "swiglu" else None
    hc = np.asarray(h_cols, dtype=np.int64)
    a = Xe @ w1[:, hc]
    dH = G @ w3[hc, :].T
    if act == "swiglu":
        b = Xe @ w2[:, hc]
        dA = dH * b * silu_grad(a)
        dB = dH * silu(a)
        dW1c = Xe.T @ dA
        dW2c = Xe.T @ dB
    else:
        dA = dH * silu_grad(a)
        dW1c = Xe.T @ dA
        dW2c = None
    wr = np.asarray(w3_rows, dtype=np.int64)
    a_r = Xe @ w1[:, wr]
    H_r = silu(a_r) * (Xe @ w2[:, wr]) if act == "swiglu" else silu(a_r)
    dW3r = H_r.T @ G
    return dW1c, dW2c, dW3r


# ---------------------------------------------------------------------------
# router: the step before the dispatch (token-choice top-K routing, page 1,
# assumptions of the problem statement; the workloads' softmax router)
# ---------------------------------------------------------------------------

def router(x, Wr, bias, K: int):
    """Token-choice top-K softmax router.

    logits[t, e] = x[t] . Wr[:, e] (+ bias[e]); the K experts of token t are
    its K largest logits, equal logits ordered by the lower expert index, slot
    0 the largest; the gates are the softmax over those K logits (the top-K
    probabilities renormalised to sum 1).  fp64.  Returns ids (L,K) int64,
    gates (L,K) and the logits (L,E)."""
    lg = _f64(x) @ _f64(Wr)
    if bias is not None:
        lg = lg + _f64(bias)[None, :]
    ids = np.argsort(-lg, axis=1, kind="stable")[:, :K]
    top = np.take_along_axis(lg, ids, axis=1)
    w = np.exp(top - top[:, :1])
    return ids.astype(np.int64), w / w.sum(axis=1, keepdims=True), lg


def router_backward(x, Wr, topk_ids, gates, dgates, E: int):
    """Gradients through the router, given dgates = dLoss/dgates.

    The selection is piecewise constant in the logits, so only the K selected
    logits of a token receive a gradient: with g the softmax over them,
    dlogit[t, ids[t,k]] = g_k (dg_k - sum_j g_j dg_j).  Then dWr = x^T dlogit,
    dbias = sum_t dlogit[t], dx = dlogit Wr^T.  Returns dWr (d,E), dbias (E),
    dx (L,d) and the dense dlogit (L,E)."""
    X = _f64(x); W = _f64(Wr); ids = _i64(topk_ids); g = _f64(gates); dg = _f64(dgates)
    L = X.shape[0]
    dl_k = g * (dg - np.sum(g * dg, axis=1, keepdims=True))
    dl = np.zeros((L, E))
    np.put_along_axis(dl, ids, dl_k, axis=1)
    return X.T @ dl, dl.sum(axis=0), dl @ W.T, dl


def rel_err(got, ref) -> float:
    """max|got - ref| / max|ref| (0 when both are all zero)."""
    got = _f64(got); ref = _f64(ref)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(got - ref)) if ref.size else 0.0
    if den == 0.0:
        return float(num)
    return float(num / den)
