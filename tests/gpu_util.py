"""Shared helpers of the GPU parity tests (imported by test_gpu_*.py)."""
from __future__ import annotations

import ctypes

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
    # the header records the (L, E, K) the build was made for; the forward and
    # backward kernels compare it with their own shape (the same comparison
    # as this host-side call)
    hdr = ctypes.create_string_buffer(layer.disp.meta[:32].cpu().numpy().tobytes(), 32)
    assert B.moeblaze_dispatch_meta_check(layer.shape, hdr) == B.OK
    num_mt, n_e, pad, order = layer.meta()
    n_e = n_e.numpy(); pad = pad.numpy(); order = order.numpy()
    assert np.array_equal(n_e, np.diff(D2))
    padded = (n_e + 255) // 256 * 256   # expert segments padded to a pair of 128-row tiles
    assert np.array_equal(pad, np.concatenate([[0], np.cumsum(padded)]))
    assert num_mt == pad[-1] // 128
    # experts by descending load, equal loads by index
    assert order.tolist() == sorted(range(E), key=lambda e: (-int(n_e[e]), e))
    return D1, D2, D3, D4


def run_layer(cfg, inp_dev, recompute_h=False, keep_saved=False):
    """One step; with keep_saved also a copy of the saved A (B) taken after
    the forward (the bf16 backward overwrites them with dA, dB)."""
    layer = MoELayer.for_config(cfg, "cuda", recompute_h=recompute_h)
    W = (inp_dev.get("W1"), inp_dev.get("W2"), inp_dev.get("W3"))
    layer.dispatch(inp_dev["ids"])
    layer.forward(inp_dev["x"], inp_dev["gates"], *W)
    saved = None
    if keep_saved:
        saved = tuple(None if v is None else v.clone() for v in layer.saved())
    layer.backward(inp_dev["dY"], inp_dev["x"], inp_dev["gates"], *W)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    return (layer, saved) if keep_saved else layer


def full_compare(cfg, inp_cpu, tol=None, check_saved=True, recompute_h=False):
    """Whole-tensor comparison of every output with the oracle."""
    tol = TOL[cfg.dtype] if tol is None else tol
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp_cpu.items()}
    layer, saved = run_layer(cfg, dev, recompute_h, keep_saved=True)
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
            A, Bv = saved
            _, _, pad, _ = layer.meta()
            ra, rb = [], []
            ga, gb = [], []
            # only the rows the forward wrote are widened: the padding rows
            # of a segment and the tail past the last segment hold no data
            for e, s in keep["saved"].items():
                p0 = int(pad[e]); n = s["a"].shape[0]
                ra.append(s["a"]); ga.append(O._f64(A[p0:p0 + n]))
                if Bv is not None:
                    rb.append(s["b"]); gb.append(O._f64(Bv[p0:p0 + n]))
            errs["A"] = O.rel_err(np.concatenate(ga), np.concatenate(ra))
            if Bv is not None:
                errs["B"] = O.rel_err(np.concatenate(gb), np.concatenate(rb))
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{cfg.name}: {bad} (tol {tol}); all {errs}"
    return errs, layer


def spread_indices(n, tile, per_tile, rng, extra=0):
    """Indices into [0, n) that cover the first, a middle and the last tile
    of width `tile`: each tile's first and last index plus `per_tile` random
    ones inside it, and `extra` uniform picks anywhere."""
    nt = (n + tile - 1) // tile
    picks = set()
    for t in sorted({0, nt // 2, nt - 1}):
        lo, hi = t * tile, min(n, (t + 1) * tile)
        picks.update([lo, hi - 1])
        picks.update(rng.choice(np.arange(lo, hi), min(per_tile, hi - lo), replace=False).tolist())
    if extra:
        picks.update(rng.choice(n, min(extra, n), replace=False).tolist())
    return sorted(int(i) for i in picks)


def sampled_compare(cfg, n_tok=62, per_tile=10, seed=0, tol=None, recompute_h=False):
    """Full-size run on the device; the oracle computes sampled outputs one
    by one:
      - y, dX and dgates on n_tok random token rows plus the first and last;
      - for EVERY expert with tokens, columns of dW1 (and dW2) and rows of
        dW3 spread over the first, a middle and the last output tile of the
        GEMM that writes them (128-column tiles of dW1|dW2 for SwiGLU,
        256 for SiLU; 128-row tiles of dW3), at least 32 of each plus 4
        uniform picks.
    Returns the errors and the sampled fractions."""
    tol = TOL[cfg.dtype] if tol is None else tol
    inp = I.make_inputs(cfg, "cuda")
    layer = run_layer(cfg, inp, recompute_h)
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
    frac = {"token_rows": len(toks) / cfg.L}
    if cfg.act != "identity":
        n_e = np.diff(D2)
        experts = [int(e) for e in np.nonzero(n_e)[0]]
        gr = np.zeros(cfg.L * cfg.K)
        g_np = gates.numpy().astype(np.float64)
        for k in range(cfg.K):
            gr[D4[:, k]] = g_np[:, k]
        ntile = 128 if cfg.act == "swiglu" else 256
        hc = spread_indices(cfg.h, ntile, per_tile, rng, extra=4)
        wr = spread_indices(cfg.h, 128, per_tile, rng, extra=4)
        assert len(hc) >= 32 and len(wr) >= 32
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
        frac.update({"experts_checked": len(experts), "experts_with_tokens": len(experts),
                     "dW12_columns": len(hc) / cfg.h, "dW3_rows": len(wr) / cfg.h})
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{cfg.name}: {bad} (tol {tol}); all {errs}"
    return errs, frac
