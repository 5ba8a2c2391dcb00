"""The index-checking debug build of the library (-DMOE_DEVICE_CHECKS).

In that build every kernel that reads an index from memory (the router's
expert ids in the permutation, the un-permute and the router backward; the
destination rows of the dispatch gathers; the (token, slot) rows of the
scatter epilogues; the permuted rows the router backward reads) checks it
against its array and, if it is out of range,
records MOE_ERR_INVALID_ARG with the value in the status word and skips the
access instead of trapping.  This test builds that variant, loads it in a
child process (LIBMOE_PATH), and runs the tiny workload, a ragged shape on
single-CTA and CTA-pair tiles and an MXFP8 layer: every call must finish with
a clean status and match the oracle as the normal build does.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, ROOT)
sys.path.insert(0, ROOT + "/tests")
import numpy as np
import synth_inputs as si
from gpu_support import BF16_TOL, f64, rel_fro, run_layer
from oracle import moe_oracle as mo
from mixture_experts_layer_17_gb300 import libmoe
cases = [("tiny", None, 0, None), ("ragged", (300, 256, 256, 16, 4, 11), 0x4, None),
         ("ragged pairs", (300, 256, 256, 16, 4, 11), 0x8, None),
         ("mxfp8", (517, 512, 384, 16, 4, 65), 0, "mxfp8")]
for name, shape, flags, prec in cases:
    if shape is None:
        sh = si.shape("tiny")
    else:
        sh = si.custom_shape(*shape[:5], seed=shape[5], precision=prec or "bf16")
    inp = si.make_inputs(sh, "cuda")
    out = run_layer(sh, inp, flags=flags)      # asserts a clean device status
    args = [f64(inp[k]) for k in ("x", "W_r", "W_gate", "W_up", "W_down")]
    ref = mo.backward(*args, sh.top_k, f64(inp["dY"]), logit_bias=f64(inp["logit_bias"]),
                      precision=prec)
    tol = BF16_TOL if prec is None else 3e-2
    assert rel_fro(out["y"], ref["fwd"]["y"]) <= tol, name
    for key in ("dx", "dW_gate", "dW_up", "dW_down"):
        assert rel_fro(out[key], ref[key]) <= tol, (name, key)
    print("checked build clean:", name)
print("LOADED", libmoe.load()._name)
"""


def test_checked_build_runs_clean():
    from mixture_experts_layer_17_gb300 import build
    path = build.build(checked=True)
    env = dict(os.environ, LIBMOE_PATH=path)
    res = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + CHILD], env=env,
                         capture_output=True, text=True, timeout=600)
    print(res.stdout)
    assert res.returncode == 0, res.stderr[-4000:]
    assert f"LOADED {path}" in res.stdout
