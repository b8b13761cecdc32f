"""Shared helpers of the GPU parity tests (imported by test_gpu_*.py)."""
from __future__ import annotations

import numpy as np
import torch

import oracle.moe_oracle as O
from mixture_experts_atomic_gb300 import binding as B
from mixture_experts_atomic_gb300 import inputs as I
from mixture_experts_atomic_gb300.layer import MoELayer

TOL = {"f32": 1e-4, "bf16": 2e-2}


def ensure_built():
    try:
        B.lib()
    except RuntimeError:
        import __graft_entry__
        __graft_entry__.build()


def check_dispatch(layer: MoELayer, ids_cpu: torch.Tensor, E: int):
    """Bit-exact comparison of the four index structures with the oracle, and
    consistency of the tile metadata."""
    D1, D2, D3, D4 = O.dispatch(ids_cpu, E)
    g1, g2, g3, g4 = (t.cpu().numpy().astype(np.int64) for t in B.index_views(layer.shape, layer.disp))
    assert np.array_equal(g2, D2), "expert_token_offsets"
    assert np.array_equal(g1, D1), "expert_token_indices"
    assert np.array_equal(g3, D3), "token_expert_indices"
    assert np.array_equal(g4, D4), "token_index_map"
    num_mt, n_e, pad, order = layer.meta()
    n_e = n_e.numpy(); pad = pad.numpy(); order = order.numpy()
    assert np.array_equal(n_e, np.diff(D2))
    padded = (n_e + 127) // 128 * 128
    assert np.array_equal(pad, np.concatenate([[0], np.cumsum(padded)]))
    assert num_mt == pad[-1] // 128
    # experts by descending load, equal loads by index
    assert order.tolist() == sorted(range(E), key=lambda e: (-int(n_e[e]), e))
    return D1, D2, D3, D4


def run_layer(cfg, inp_dev) -> MoELayer:
    layer = MoELayer.for_config(cfg, "cuda")
    layer.step(inp_dev)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    return layer


def full_compare(cfg, inp_cpu, tol=None, check_saved=True):
    """Whole-tensor comparison of every output with the oracle."""
    tol = TOL[cfg.dtype] if tol is None else tol
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp_cpu.items()}
    layer = run_layer(cfg, dev)
    D1, D2, D3, D4 = check_dispatch(layer, inp_cpu["ids"], cfg.E)
    a = inp_cpu
    y, keep = O.forward(a["ids"], a["gates"], a["x"], a["W1"], a["W2"], a["W3"], cfg.act, E=cfg.E, keep=True)
    dX, dW1, dW2, dW3, dg = O.backward(a["ids"], a["gates"], a["x"], a["dY"], a["W1"], a["W2"], a["W3"], cfg.act,
                                       E=cfg.E)
    errs = {"y": O.rel_err(layer.y, y), "dX": O.rel_err(layer.dX, dX), "dgates": O.rel_err(layer.dgates, dg)}
    if cfg.act != "identity":
        errs["dW1"] = O.rel_err(layer.dW1, dW1)
        errs["dW3"] = O.rel_err(layer.dW3, dW3)
        if cfg.act == "swiglu":
            errs["dW2"] = O.rel_err(layer.dW2, dW2)
        if check_saved:
            A, Bv = layer.saved()
            _, _, pad, _ = layer.meta()
            A = O._f64(A); Bv = O._f64(Bv) if Bv is not None else None
            ra, rb = [], []
            ga, gb = [], []
            for e, s in keep["saved"].items():
                p0 = int(pad[e]); n = s["a"].shape[0]
                ra.append(s["a"]); ga.append(A[p0:p0 + n])
                if Bv is not None:
                    rb.append(s["b"]); gb.append(Bv[p0:p0 + n])
            errs["A"] = O.rel_err(np.concatenate(ga), np.concatenate(ra))
            if Bv is not None:
                errs["B"] = O.rel_err(np.concatenate(gb), np.concatenate(rb))
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{cfg.name}: {bad} (tol {tol}); all {errs}"
    return errs, layer


def sampled_compare(cfg, n_tok=48, n_cols=3, seed=0, tol=None):
    """Full-size run on the device; the oracle computes sampled token rows of
    y and dX and sampled columns/rows of the weight gradients one by one."""
    tol = TOL[cfg.dtype] if tol is None else tol
    inp = I.make_inputs(cfg, "cuda")
    layer = run_layer(cfg, inp)
    ids = inp["ids"].cpu()
    gates = inp["gates"].cpu()
    D1, D2, D3, D4 = check_dispatch(layer, ids, cfg.E)
    rng = np.random.default_rng(seed)
    toks = np.unique(np.concatenate([[0, cfg.L - 1], rng.choice(cfg.L, n_tok, replace=False)]))
    tt = torch.from_numpy(toks).cuda()
    W = {k: (inp[k].cpu() if inp.get(k) is not None else None) for k in ("W1", "W2", "W3")}
    xr = inp["x"][tt].cpu()
    dyr = inp["dY"][tt].cpu()
    y_ref = O.forward_rows(toks, ids, gates, xr, W["W1"], W["W2"], W["W3"], cfg.act)
    dx_ref, dg_ref = O.backward_rows(toks, ids, gates, xr, dyr, W["W1"], W["W2"], W["W3"], cfg.act, with_dgates=True)
    errs = {"y": O.rel_err(layer.y[tt], y_ref), "dX": O.rel_err(layer.dX[tt], dx_ref),
            "dgates": O.rel_err(layer.dgates[tt], dg_ref)}
    if cfg.act != "identity":
        n_e = np.diff(D2)
        nz = np.nonzero(n_e)[0]
        experts = sorted({int(nz[np.argmax(n_e[nz])]), int(nz[np.argmin(n_e[nz])])})
        gr = np.zeros(cfg.L * cfg.K)
        g_np = gates.numpy().astype(np.float64)
        for k in range(cfg.K):
            gr[D4[:, k]] = g_np[:, k]
        hc = sorted(set(rng.choice(cfg.h, n_cols, replace=False).tolist() + [0, cfg.h - 1]))
        wr = sorted(set(rng.choice(cfg.h, n_cols, replace=False).tolist() + [cfg.h - 1]))
        e1, e2, e3 = [], [], []
        for e in experts:
            seg = D1[D2[e]:D2[e + 1]]
            st = torch.from_numpy(seg).cuda()
            c1, c2, r3 = O.weight_grad_slices(e, seg, gr[D2[e]:D2[e + 1]], inp["x"][st].cpu(), inp["dY"][st].cpu(),
                                              W["W1"], W["W2"], W["W3"], cfg.act, hc, wr)
            e1.append(O.rel_err(layer.dW1[e][:, hc], c1))
            e3.append(O.rel_err(layer.dW3[e][wr, :], r3))
            if c2 is not None:
                e2.append(O.rel_err(layer.dW2[e][:, hc], c2))
        errs["dW1"] = max(e1)
        errs["dW3"] = max(e3)
        if e2:
            errs["dW2"] = max(e2)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{cfg.name}: {bad} (tol {tol}); all {errs}"
    return errs
