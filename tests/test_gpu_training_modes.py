"""Training modes of the layer on the GPU:

* MOE_FLAG_RECOMPUTE (activation checkpointing): ctx keeps only the routing;
  the backward dispatches x again and recomputes h.  The kernels and their
  schedules are deterministic, so every output must equal, bit for bit, the
  run that kept x_perm and h in ctx, even after the forward workspace (where
  the recompute-mode forward put them) has been overwritten.
* moe_backward_accumulate: the weight gradients are added into fp32 buffers.
  Two calls on top of random fp32 contents must add 2·g exactly as fp32 sums
  of the same fp32 increments; the increment itself is the bf16 backward's
  gradient before rounding (checked against the bf16 outputs and against the
  oracle), and experts without tokens leave their slices untouched.
* moe_config_t.max_sms: the persistent grids shrink to the budget; each
  output tile is still computed by one CTA in a fixed K order, so everything
  but dW_r (whose split-K depth follows the budget) is bit-identical.
"""

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_support import BF16_TOL, f64, rel_fro
from oracle import moe_oracle as mo

pytestmark = pytest.mark.gpu

MX_TOL = 3e-2
GRAD_KEYS = ("dx", "dW_r", "dW_gate", "dW_up", "dW_down")


def _inputs(shape, precision="bf16", zero_experts=()):
    T, H, F, E, k, seed = shape
    sh = si.custom_shape(T, H, F, E, k, seed=seed, precision=precision)
    inp = si.make_inputs(sh, "cuda")
    if zero_experts:
        bias = torch.zeros(E)
        bias[list(zero_experts)] = -30.0
        inp["logit_bias"] = bias.cuda()
    return sh, inp


def _weights(inp):
    return inp["x"], inp["W_r"], inp["W_gate"], inp["W_up"], inp["W_down"]


def _run(layer, inp):
    args = _weights(inp)
    y = layer.forward(*args, inp["logit_bias"])
    g = layer.backward(*args, inp["dY"])
    torch.cuda.synchronize()
    assert layer.device_status("fwd") == 0 and layer.device_status("bwd") == 0
    return y, g


@pytest.mark.parametrize("precision", ["bf16", "mxfp8", "fp8_bwd"])
@pytest.mark.parametrize("shape", [(517, 512, 384, 16, 4, 61), (1024, 512, 256, 8, 4, 62),
                                   # 367 rows per expert, F = 2 x 192: the MXFP8 down dgrad
                                   # runs on 256 x 192 CTA pairs
                                   (1100, 256, 384, 6, 2, 67)])
def test_recompute_is_bit_identical(precision, shape):
    from mixture_experts_layer_17_gb300 import MoeLayer, libmoe
    sh, inp = _inputs(shape, precision)
    keep = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, precision)
    rec = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, precision, flags=libmoe.MOE_FLAG_RECOMPUTE)
    # ctx loses h [Pa, 2F] (Pa = P + 64 E rows, bf16) and x: x_perm [Pa, H] bf16,
    # or in mxfp8 x along the tokens [128 mt, H] E4M3 with its scale atoms
    Pa = sh.P + 64 * sh.E
    mt = (sh.P + 127) // 128 + sh.E
    x_bytes = 128 * mt * sh.H + mt * (sh.H // 128) * 512 if precision == "mxfp8" else 2 * Pa * sh.H
    saved = keep.ctx.numel() - rec.ctx.numel()
    assert x_bytes + 4 * Pa * sh.F <= saved <= x_bytes + 4 * Pa * sh.F + 768
    y0, g0 = _run(keep, inp)
    args = _weights(inp)
    y1 = rec.forward(*args, inp["logit_bias"])
    rec.fwd_ws.fill_(0xFF)          # the recompute-mode forward's x_perm and h are gone
    g1 = rec.backward(*args, inp["dY"])
    torch.cuda.synchronize()
    assert rec.device_status("bwd") == 0
    assert torch.equal(y0, y1)
    for key in GRAD_KEYS:
        assert torch.equal(g0[key], g1[key]), key
    if precision == "bf16":
        ref = mo.backward(*(f64(a) for a in args), sh.top_k, f64(inp["dY"]))
        for key in GRAD_KEYS:
            assert rel_fro(f64(g1[key]), ref[key]) <= BF16_TOL, key


@pytest.mark.parametrize("precision,flags,F", [("bf16", 0, 256), ("bf16", "pairs", 256),
                                               ("mxfp8", 0, 256), ("mxfp8", "pairs", 384)])
def test_accumulate_into_fp32(precision, flags, F):
    from mixture_experts_layer_17_gb300 import MoeLayer, libmoe
    fl = libmoe.MOE_FLAG_CTA_PAIRS_ON if flags == "pairs" else 0
    sh, inp = _inputs((1024, 512, F, 12, 4, 63), precision, zero_experts=(3, 7))
    layer = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, precision, flags=fl)
    args = _weights(inp)
    y, g = _run(layer, inp)
    gen = torch.Generator(device="cuda").manual_seed(5)
    acc0 = {k: torch.randn(inp[k.replace("dW", "W")].shape, device="cuda", generator=gen)
            for k in ("dW_r", "dW_gate", "dW_up", "dW_down")}
    acc = {k: v.clone() for k, v in acc0.items()}
    dx1 = layer.backward_accumulate(*args, inp["dY"], acc)
    torch.cuda.synchronize()
    assert layer.device_status("bwd") == 0
    acc1 = {k: v.clone() for k, v in acc.items()}
    dx2 = layer.backward_accumulate(*args, inp["dY"], acc)
    torch.cuda.synchronize()
    assert torch.equal(dx1, g["dx"]) and torch.equal(dx2, g["dx"])
    ref = mo.backward(*(f64(a) for a in args), sh.top_k, f64(inp["dY"]),
                      logit_bias=f64(inp["logit_bias"]),
                      precision=None if precision == "bf16" else precision)
    assert ref["fwd"]["counts"][3] == 0 and ref["fwd"]["counts"][7] == 0
    tol = BF16_TOL if precision == "bf16" else MX_TOL
    for k in acc:
        inc = (f64(acc[k]) - f64(acc0[k])) / 2.0
        # the increment is the bf16 output before rounding
        assert rel_fro(f64(g[k]), inc) <= 4e-3, k
        assert rel_fro(inc, ref[k]) <= tol, k
        # both calls added the same fp32 increment: acc1 = fl(acc0 + g), acc = fl(acc1 + g)
        a0, a1, a2 = f64(acc0[k]), f64(acc1[k]), f64(acc[k])
        slack = 2.0 ** -23 * (np.abs(a1) + np.abs(a2)) + 1e-30
        assert np.all(np.abs((a2 - a1) - (a1 - a0)) <= slack), k
    for e in (3, 7):
        for k in ("dW_gate", "dW_up", "dW_down"):
            assert torch.equal(acc[k][e], acc0[k][e]), (k, e)


@pytest.mark.parametrize("max_sms", [1, 7, 16, 1000])
def test_sm_budget_gives_the_same_results(max_sms):
    from mixture_experts_layer_17_gb300 import MoeLayer
    sh, inp = _inputs((1024, 512, 256, 8, 4, 64))     # 512 rows per expert: CTA pairs by default
    full = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k)
    part = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, max_sms=max_sms)
    y0, g0 = _run(full, inp)
    y1, g1 = _run(part, inp)
    assert torch.equal(y0, y1)
    for key in ("dx", "dW_gate", "dW_up", "dW_down"):
        assert torch.equal(g0[key], g1[key]), key
    # the budgeted run against the oracle (dW_r's split-K depth follows the budget)
    ref = mo.backward(*(f64(a) for a in _weights(inp)), sh.top_k, f64(inp["dY"]))
    assert rel_fro(f64(y1), ref["fwd"]["y"]) <= BF16_TOL
    for key in GRAD_KEYS:
        assert rel_fro(f64(g1[key]), ref[key]) <= BF16_TOL, key


def test_sm_budget_mxfp8_and_recompute_together():
    from mixture_experts_layer_17_gb300 import MoeLayer, libmoe
    sh, inp = _inputs((517, 512, 384, 16, 4, 65), "mxfp8")
    full = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, "mxfp8")
    part = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, "mxfp8",
                    flags=libmoe.MOE_FLAG_RECOMPUTE, max_sms=20)
    y0, g0 = _run(full, inp)
    y1, g1 = _run(part, inp)
    assert torch.equal(y0, y1)
    for key in ("dx", "dW_gate", "dW_up", "dW_down"):
        assert torch.equal(g0[key], g1[key]), key
    # the budgeted recompute run against the oracle with the MXFP8 quantisation points
    ref = mo.backward(*(f64(a) for a in _weights(inp)), sh.top_k, f64(inp["dY"]),
                      precision="mxfp8")
    assert rel_fro(f64(y1), ref["fwd"]["y"]) <= MX_TOL
    for key in GRAD_KEYS:
        assert rel_fro(f64(g1[key]), ref[key]) <= MX_TOL, key


@pytest.mark.parametrize("precision,extra", [("mxfp8", 0), ("fp8_bwd", 0), ("mxfp8", "recompute"),
                                             ("mxfp8", "pairs"), ("fp8_bwd", "pairs")])
def test_prepared_weights_are_bit_identical(precision, extra):
    """moe_prepare_weights writes the bytes the calls would quantise
    themselves, and the calls read them instead of the bf16 weights.  With
    CTA pairs (F = 384: the down dgrad's 256 x 192 tiles, which read W_down's
    scales in 192-row blocks) the weights are prepared under
    MOE_FLAG_CTA_PAIRS_OFF and used under MOE_FLAG_CTA_PAIRS_ON: the buffer
    holds both scale layouts."""
    from mixture_experts_layer_17_gb300 import MoeLayer, libmoe
    fl = {"recompute": libmoe.MOE_FLAG_RECOMPUTE, "pairs": libmoe.MOE_FLAG_CTA_PAIRS_ON}.get(extra, 0)
    sh, inp = _inputs((517, 512, 384, 16, 4, 66), precision)
    plain = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, precision, flags=fl)
    prep = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, precision, flags=fl)
    if extra == "pairs":
        prep.cfg.flags = libmoe.MOE_FLAG_CTA_PAIRS_OFF
    prep.prepare_weights(inp["W_gate"], inp["W_up"], inp["W_down"])
    prep.cfg.flags = fl
    y0, g0 = _run(plain, inp)
    y1, g1 = _run(prep, inp)
    assert torch.equal(y0, y1)
    for key in GRAD_KEYS:
        assert torch.equal(g0[key], g1[key]), key
    if precision == "mxfp8":
        # weights prepared from 2 * W_down: doubling moves only the MX scale
        # exponents, so the layer output doubles exactly
        prep.prepare_weights(inp["W_gate"], inp["W_up"], 2 * inp["W_down"])
        y2 = prep.forward(*_weights(inp), inp["logit_bias"])
        torch.cuda.synchronize()
        assert torch.equal(y2, 2 * y0)
