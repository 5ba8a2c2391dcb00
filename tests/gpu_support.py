"""Shared pieces of the GPU parity tests: run the CUDA path through the C ABI
(via the ctypes binding) and compare it with the CPU oracle.  The oracle is
only ever fed the seeded inputs, never a result of the CUDA path."""

from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as mo

# relative Frobenius tolerance for bf16 results (fp32 accumulation)
BF16_TOL = 1e-2
# router logits: fp32 accumulation of bf16 products against fp64
LOGIT_TOL = 1e-3
# a routing decision may differ from the fp64 oracle only at a near-tie
NEAR_TIE = 1e-4


def f64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def rel_fro(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def run_layer(sh, inp, flags: int = 0):
    """Route, forward and backward on the GPU; returns numpy copies."""
    from mixture_experts_layer_17_gb300 import MoeLayer
    layer = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, sh.precision, flags)
    route = layer.route(inp["x"], inp["W_r"], inp["logit_bias"])
    y = layer.forward(inp["x"], inp["W_r"], inp["W_gate"], inp["W_up"], inp["W_down"],
                      inp["logit_bias"])
    grads = layer.backward(inp["x"], inp["W_r"], inp["W_gate"], inp["W_up"], inp["W_down"],
                           inp["dY"])
    torch.cuda.synchronize()
    assert layer.device_status("fwd") == 0
    assert layer.device_status("bwd") == 0
    out = {k: (v.cpu().numpy() if v is not None else None) for k, v in route.items()}
    out["y"] = f64(y)
    for k, v in grads.items():
        out[k] = f64(v)
    return out


def check_route_properties(r, T: int, E: int, k: int) -> None:
    """The integer outputs are a valid top-k of the kernel's own fp32 logits and
    a valid expert-major permutation of them (bit-exact, no tolerance)."""
    logits = r["logits"].astype(np.float32)
    idx = r["topk_idx"].astype(np.int64)
    # top-k by (-logit, id) of the exported logits
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    assert np.array_equal(idx, order), "topk_idx is not the top-k of the kernel's logits"
    # weights: softmax of the selected logits (fp32 kernel arithmetic vs fp64)
    sel = np.take_along_axis(logits.astype(np.float64), idx, axis=1)
    w_ref = np.exp(sel - sel[:, :1])
    w_ref /= w_ref.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(r["topk_w"], w_ref, rtol=2e-5, atol=1e-7)
    counts = np.bincount(idx.reshape(-1), minlength=E)
    assert np.array_equal(r["counts"], counts)
    assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(counts)]))
    perm = r["perm_token"].astype(np.int64)
    slot = r["slot_row"].astype(np.int64)
    P = T * k
    assert np.array_equal(np.sort(slot.reshape(-1)), np.arange(P))
    assert np.array_equal(perm[slot], np.repeat(np.arange(T)[:, None], k, axis=1))
    row_expert = np.repeat(np.arange(E), counts)
    assert np.array_equal(row_expert[slot], idx)
    for e in range(E):
        seg = perm[r["offsets"][e]:r["offsets"][e + 1]]
        assert np.all(np.diff(seg) > 0)


def routing_mismatches(gpu_idx, ref_logits, k: int) -> np.ndarray:
    """Tokens whose GPU selection differs from the oracle's (fp64 logits);
    each must be a near-tie between the k-th and (k+1)-th oracle logit."""
    ref_idx = mo.select_topk(ref_logits, k)
    bad = np.nonzero(np.any(ref_idx != gpu_idx.astype(np.int64), axis=1))[0]
    E = ref_logits.shape[1]
    for t in bad:
        srt = np.sort(ref_logits[t])[::-1]
        # same set in a different order, or a swap across the cut: both need a tie
        gaps = np.abs(np.diff(srt[: min(k + 1, E)]))
        assert np.min(gaps) < NEAR_TIE * max(1.0, abs(srt[0])), f"token {t} is not a near-tie"
    return bad
