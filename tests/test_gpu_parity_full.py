"""GPU parity at the full workload sizes (the launch configuration bench.py
times), on outputs the oracle can compute piece by piece:

* routing: every integer output is checked in full (validity against the
  kernel's own logits, bit-exact agreement with the oracle's fp64 routing
  except at reported near-ties), logits in full;
* y and dx on sampled tokens (each depends only on its token's own row);
* dW_gate / dW_up columns and dW_down rows of sampled experts;
* the dW_r column of the expert with the fewest (non-zero) tokens.
bf16 tolerance: relative Frobenius error <= 1e-2 on each stacked sample; the
MXFP8 workloads (all six expert GEMMs, or only the backward's) are held to 3e-2
against the oracle run with the same quantisation points."""

import numpy as np
import pytest
import torch

import synth_inputs as si
from oracle import moe_oracle as mo
from gpu_support import (BF16_TOL, LOGIT_TOL, check_route_properties, f64, rel_fro,
                         routing_mismatches)

pytestmark = pytest.mark.gpu

N_TOKENS = 48
N_COLS = 4


MX_TOL = 3e-2   # MXFP8 tolerance
N_TOKENS_MX = 12


def _tokens_sharing_experts(ref_idx, cand, n, rng):
    """Greedy sample of n tokens whose selected experts overlap as much as
    possible (fewer distinct experts = fewer fp64 weight quantisations)."""
    chosen = [int(rng.choice(cand))]
    union = set(ref_idx[chosen[0]].tolist())
    while len(chosen) < n:
        pool = rng.choice(cand, size=min(4096, len(cand)), replace=False)
        new = [len(set(ref_idx[t].tolist()) - union) if t not in chosen else 99 for t in pool]
        t = int(pool[int(np.argmin(new))])
        chosen.append(t)
        union |= set(ref_idx[t].tolist())
    return np.sort(np.array(chosen))


def _report_and_check(name, errs, prec, bad):
    print(name, {k: f"{v:.2e}" for k, v in errs.items()}, "near-ties:", len(bad))
    for k, v in errs.items():
        tol = BF16_TOL if prec is None or (prec == "fp8_bwd" and k == "y") else MX_TOL
        assert v <= tol, (k, v)


@pytest.mark.parametrize("name", ["qwen3_30b", "qwen3_30b_skew", "qwen3_235b",
                                  "qwen3_235b_mxfp8", "qwen3_235b_fp8_bwd",
                                  "qwen3_235b_mxfp8_skew"])
def test_full_size_sampled(name):
    from mixture_experts_layer_17_gb300 import MoeLayer
    sh = si.shape(name)
    prec = None if sh.precision == "bf16" else sh.precision
    inp = si.make_inputs(sh, "cuda")
    layer = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, sh.precision)
    route = layer.route(inp["x"], inp["W_r"], inp["logit_bias"])
    y = layer.forward(inp["x"], inp["W_r"], inp["W_gate"], inp["W_up"], inp["W_down"],
                      inp["logit_bias"])
    g = layer.backward(inp["x"], inp["W_r"], inp["W_gate"], inp["W_up"], inp["W_down"],
                       inp["dY"])
    torch.cuda.synchronize()
    assert layer.device_status("fwd") == 0 and layer.device_status("bwd") == 0

    r = {k: v.cpu().numpy() for k, v in route.items()}
    check_route_properties(r, sh.T, sh.E, sh.top_k)

    # host copies for the oracle (exact widening of the bf16 inputs)
    x = inp["x"].float().cpu().numpy()
    dY = inp["dY"].float().cpu().numpy()
    W_r = inp["W_r"].float().cpu().numpy()
    Wg = inp["W_gate"].float().cpu().numpy()
    Wu = inp["W_up"].float().cpu().numpy()
    Wd = inp["W_down"].float().cpu().numpy()
    bias = f64(inp["logit_bias"])

    ref_logits = mo.router_logits(x, W_r, bias)
    assert rel_fro(r["logits"], ref_logits) < LOGIT_TOL
    bad = set(routing_mismatches(r["topk_idx"], ref_logits, sh.top_k).tolist())
    assert len(bad) <= 2, f"{len(bad)} routing near-ties"
    ref_idx = mo.select_topk(ref_logits, sh.top_k)
    ref_w = mo.topk_weights(ref_logits, ref_idx)
    ok = np.array([t not in bad for t in range(sh.T)])
    assert np.array_equal(r["topk_idx"][ok], ref_idx[ok])
    assert rel_fro(r["topk_w"][ok], ref_w[ok]) < LOGIT_TOL
    if sh.skew:
        assert (r["counts"] == 0).sum() >= 4

    # --- y and dx on sampled tokens
    rng = np.random.default_rng(sh.seed + 100)
    cand = np.nonzero(ok)[0]
    if prec is None:
        S = np.sort(rng.choice(cand, size=N_TOKENS, replace=False))
    else:
        # MX oracle cost grows with the experts the sample touches (each one's
        # weights are quantised in fp64): pick tokens that share experts
        S = _tokens_sharing_experts(ref_idx, cand, N_TOKENS_MX, rng)
    sub = mo.backward(x[S], W_r, Wg, Wu, Wd, sh.top_k, dY[S], logit_bias=bias,
                      keep_weight_grads=False, precision=prec)
    e_y = rel_fro(f64(y[torch.from_numpy(S).cuda()]), sub["fwd"]["y"])
    e_dx = rel_fro(f64(g["dx"][torch.from_numpy(S).cuda()]), sub["dx"])

    # --- expert weight gradients: sampled columns of three experts
    counts = np.bincount(ref_idx.reshape(-1), minlength=sh.E)
    nz = np.nonzero(counts)[0]
    experts = sorted({int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])]),
                      int(nz[len(nz) // 2])})
    got_g, got_u, got_d, want_g, want_u, want_d = [], [], [], [], [], []
    for e in experts:
        t_e, j_e = np.nonzero(ref_idx == e)               # ascending tokens
        rows_w = ref_w[t_e, j_e]
        cols = np.sort(rng.choice(sh.F, size=N_COLS, replace=False))
        if prec is None:
            c = mo.expert_weight_grad_columns(e, cols, x, dY, Wg, Wu, Wd, t_e, rows_w)
        else:
            c = mo.expert_weight_grad_columns_mx(e, cols, x, dY, Wg, Wu, Wd, t_e, rows_w, prec)
        want_g.append(c["dW_gate_col"])
        want_u.append(c["dW_up_col"])
        want_d.append(c["dW_down_row"])
        got_g.append(f64(g["dW_gate"][e][:, torch.from_numpy(cols).cuda()]).T)
        got_u.append(f64(g["dW_up"][e][:, torch.from_numpy(cols).cuda()]).T)
        got_d.append(f64(g["dW_down"][e][torch.from_numpy(cols).cuda(), :]))
    e_g = rel_fro(np.concatenate(got_g), np.concatenate(want_g))
    e_u = rel_fro(np.concatenate(got_u), np.concatenate(want_u))
    e_d = rel_fro(np.concatenate(got_d), np.concatenate(want_d))

    errs = {"y": e_y, "dx": e_dx, "dW_gate": e_g, "dW_up": e_u, "dW_down": e_d}
    if prec is not None:
        # the dW_r column needs every expert's weights quantised (all 128
        # experts of the tokens of one expert); MXFP8 dW_r is covered in full on
        # the small shapes of test_gpu_mxfp8.py
        _report_and_check(name, errs, prec, bad)
        return
    # --- router weight gradient: the column of the least-loaded expert
    e_min = int(nz[np.argmin(counts[nz])])
    S_e = np.nonzero(np.any(ref_idx == e_min, axis=1))[0]
    sub_e = mo.backward(x[S_e], W_r, Wg, Wu, Wd, sh.top_k, dY[S_e], logit_bias=bias,
                        keep_weight_grads=False, precision=prec)
    want_r = x[S_e].astype(np.float64).T @ sub_e["dl"][:, e_min]
    e_r = rel_fro(f64(g["dW_r"][:, e_min]), want_r)

    errs["dW_r"] = e_r
    _report_and_check(name, errs, prec, bad)
    # experts with no tokens: exact zeros
    for e in np.nonzero(r["counts"] == 0)[0]:
        for nm in ("dW_gate", "dW_up", "dW_down"):
            assert int(torch.count_nonzero(g[nm][e]).item()) == 0, (nm, e)
