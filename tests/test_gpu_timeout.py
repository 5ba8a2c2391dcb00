"""Failure detection without a GPU fault: with MOE_FLAG_TEST_TIMEOUT the first
grouped GEMM of a call waits on a barrier that nothing signals, with a 20 ms
limit.  The kernel must give up, record MOE_ERR_TIMEOUT in the workspace
status word, free its tensor memory and return, leaving the context usable.
Run on the single-CTA bf16 kernels, on CTA pairs (where each CTA of a pair
gives up on its own and both still meet at the closing cluster barrier) and on
the MXFP8 kernels, single-CTA and paired (F = 384 adds the down dgrad's 256 x
192 pair tiles with two accumulators)."""

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_support import BF16_TOL, f64, rel_fro
from oracle import moe_oracle as mo

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("precision,extra,F", [("bf16", 0, 256), ("bf16", "pairs", 256),
                                               ("mxfp8", 0, 256), ("mxfp8", "pairs", 256),
                                               ("mxfp8", "pairs", 384)])
def test_bounded_wait_times_out_and_context_survives(precision, extra, F):
    from mixture_experts_layer_17_gb300 import MoeLayer, libmoe
    sh = si.custom_shape(384, 256, F, 8, 2, seed=31)
    inp = si.make_inputs(sh, "cuda")
    args = (inp["x"], inp["W_r"], inp["W_gate"], inp["W_up"], inp["W_down"])
    flags = libmoe.MOE_FLAG_TEST_TIMEOUT
    if extra == "pairs":
        flags |= libmoe.MOE_FLAG_CTA_PAIRS_ON
    bad = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, precision, flags=flags)
    bad.forward(*args)
    torch.cuda.synchronize()
    assert bad.device_status("fwd") == 5          # MOE_ERR_TIMEOUT
    assert libmoe.moe_status_string(5) == "MOE_ERR_TIMEOUT"
    bad.backward(*args, inp["dY"])
    torch.cuda.synchronize()
    assert bad.device_status("bwd") == 5
    # the context is still usable: a normal call afterwards is correct
    good = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k)
    y = good.forward(*args)
    torch.cuda.synchronize()
    assert good.device_status("fwd") == 0
    ref = mo.forward(*(f64(a) for a in args), sh.top_k)
    assert rel_fro(f64(y), ref["y"]) <= BF16_TOL
