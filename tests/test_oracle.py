"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a brute-force loop, a finite difference, a
closed form, a special case that reduces to a textbook or library routine, or
the hand-derived golden example; a plausible slip in the oracle (a dropped
term, a wrong sign, a transposed operand, a wrong tie rule) fails one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe_oracle as mo
import synth_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    return None if t is None else t.double().cpu().numpy()


def _rand_layer(rng, T, H, F, E, k, std=0.3):
    x = rng.standard_normal((T, H))
    W_r = rng.standard_normal((H, E)) * std
    Wg = rng.standard_normal((E, H, F)) * std
    Wu = rng.standard_normal((E, H, F)) * std
    Wd = rng.standard_normal((E, F, H)) * std
    dY = rng.standard_normal((T, H))
    return x, W_r, Wg, Wu, Wd, dY


# ----------------------------------------------------------------- routing


def test_select_topk_matches_python_sort_with_ties():
    rng = np.random.default_rng(1)
    T, E = 300, 16
    logits = rng.integers(-3, 4, size=(T, E)).astype(np.float32)   # many exact ties
    for k in (1, 2, 5, 16):
        idx = mo.select_topk(logits, k)
        for t in range(T):
            ref = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
            assert idx[t].tolist() == ref


def test_weights_are_softmax_of_selected_logits():
    # softmax over E then renormalising over S equals softmax over S alone
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((64, 12)) * 3
    idx, w = mo.route(logits, 4)
    ref = scipy.special.softmax(np.take_along_axis(logits, idx, axis=1), axis=1)
    np.testing.assert_allclose(w, ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
    # k = E: the renormalisation is the identity and w is the full softmax
    idx, w = mo.route(logits, 12)
    full = scipy.special.softmax(logits, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, idx, axis=1), rtol=1e-13)


def test_permutation_matches_loop_and_invariants():
    rng = np.random.default_rng(3)
    T, E, k = 97, 11, 3
    logits = rng.standard_normal((T, E))
    idx = mo.select_topk(logits, k)
    p = mo.permutation(idx, E)
    rows = []
    for e in range(E):                       # expert-major, ascending token
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    rows.append((t, j))
    assert [t for t, _ in rows] == p["perm_token"].tolist()
    for r, (t, j) in enumerate(rows):
        assert p["slot_row"][t, j] == r
    assert p["counts"].sum() == T * k
    assert np.array_equal(p["offsets"], np.concatenate([[0], np.cumsum(p["counts"])]))
    assert np.array_equal(np.bincount(p["perm_token"], minlength=T), np.full(T, k))
    for e in range(E):
        seg = p["perm_token"][p["offsets"][e]:p["offsets"][e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_zero_router_picks_first_experts_uniformly():
    rng = np.random.default_rng(4)
    x, W_r, Wg, Wu, Wd, dY = _rand_layer(rng, 8, 16, 8, 6, 3)
    W_r[:] = 0.0
    f = mo.forward(x, W_r, Wg, Wu, Wd, 3)
    assert np.array_equal(f["idx"], np.tile([0, 1, 2], (8, 1)))
    np.testing.assert_allclose(f["w"], 1.0 / 3.0, rtol=1e-15)


def test_skewed_workload_loads():
    """The Zipf-biased 30B workload: the largest expert carries 5-7x the mean
    load and at least four experts receive no tokens."""
    sh = si.shape("qwen3_30b_skew")
    inp = si.make_inputs(sh, "cpu", with_grad=False, with_weights=False)
    logits = mo.router_logits(_np(inp["x"]), _np(inp["W_r"]), _np(inp["logit_bias"]))
    idx = mo.select_topk(logits, sh.top_k)
    counts = np.bincount(idx.reshape(-1), minlength=sh.E)
    mean = sh.T * sh.top_k / sh.E
    assert 5.0 <= counts.max() / mean <= 7.0
    assert (counts == 0).sum() >= 4


# ----------------------------------------------------------------- forward


def test_grouped_forward_matches_per_token_loop():
    rng = np.random.default_rng(5)
    x, W_r, Wg, Wu, Wd, _ = _rand_layer(rng, 40, 24, 10, 7, 3)
    bias = rng.standard_normal(7)
    y_loop = mo.forward_per_token(x, W_r, Wg, Wu, Wd, 3, logit_bias=bias)
    y_grp = mo.forward(x, W_r, Wg, Wu, Wd, 3, logit_bias=bias)["y"]
    np.testing.assert_allclose(y_grp, y_loop, rtol=1e-12, atol=1e-12)


def test_single_expert_is_plain_swiglu_ffn():
    rng = np.random.default_rng(6)
    x, W_r, Wg, Wu, Wd, _ = _rand_layer(rng, 20, 16, 12, 1, 1)
    y = mo.forward(x, W_r, Wg, Wu, Wd, 1)["y"]
    xt = torch.from_numpy(x)
    ref = (torch.nn.functional.silu(xt @ torch.from_numpy(Wg[0]))
           * (xt @ torch.from_numpy(Wu[0]))) @ torch.from_numpy(Wd[0])
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_k_equals_E_is_dense_softmax_mixture():
    rng = np.random.default_rng(7)
    E = 5
    x, W_r, Wg, Wu, Wd, _ = _rand_layer(rng, 12, 16, 8, E, E)
    y = mo.forward(x, W_r, Wg, Wu, Wd, E)["y"]
    p = scipy.special.softmax(x @ W_r, axis=1)
    xt = torch.from_numpy(x)
    ref = np.zeros_like(y)
    for e in range(E):
        ffn = (torch.nn.functional.silu(xt @ torch.from_numpy(Wg[e]))
               * (xt @ torch.from_numpy(Wu[e]))) @ torch.from_numpy(Wd[e])
        ref += p[:, e:e + 1] * ffn.numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_output_scales_with_down_projection():
    rng = np.random.default_rng(8)
    x, W_r, Wg, Wu, Wd, _ = _rand_layer(rng, 16, 16, 8, 4, 2)
    y1 = mo.forward(x, W_r, Wg, Wu, Wd, 2)["y"]
    y3 = mo.forward(x, W_r, Wg, Wu, 3.0 * Wd, 2)["y"]
    np.testing.assert_allclose(y3, 3.0 * y1, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------- backward


def _loss(x, W_r, Wg, Wu, Wd, k, dY, bias=None, idx=None):
    return float(np.sum(dY * mo.forward(x, W_r, Wg, Wu, Wd, k, bias, idx=idx)["y"]))


def _fd_check(x, W_r, Wg, Wu, Wd, k, dY, n_coords, bias=None, seed=0):
    rng = np.random.default_rng(seed)
    g = mo.backward(x, W_r, Wg, Wu, Wd, k, dY, logit_bias=bias)
    idx0 = g["fwd"]["idx"]
    eps = 1e-6
    params = {"x": x, "W_r": W_r, "W_gate": Wg, "W_up": Wu, "W_down": Wd}
    grads = {"x": g["dx"], "W_r": g["dW_r"], "W_gate": g["dW_gate"], "W_up": g["dW_up"],
             "W_down": g["dW_down"]}
    checked = 0
    for name, arr in params.items():
        scale = np.max(np.abs(grads[name]))
        for flat in rng.choice(arr.size, size=min(n_coords, arr.size), replace=False):
            i = np.unravel_index(flat, arr.shape)
            old = arr[i]
            vals = []
            for s in (+1, -1):
                arr[i] = old + s * eps
                ps = dict(params)
                if name in ("x", "W_r"):          # skip if the selection would change
                    sel = mo.select_topk(mo.router_logits(ps["x"], ps["W_r"], bias), k)
                    if not np.array_equal(sel, idx0):
                        vals = None
                        break
                vals.append(_loss(ps["x"], ps["W_r"], ps["W_gate"], ps["W_up"], ps["W_down"],
                                  k, dY, bias))
            arr[i] = old
            if vals is None:
                continue
            fd = (vals[0] - vals[1]) / (2 * eps)
            an = grads[name][i]
            assert abs(fd - an) <= 1e-6 * max(abs(an), 1e-2 * scale), (name, i, fd, an)
            checked += 1
    return checked


def test_gradients_match_finite_differences_micro():
    rng = np.random.default_rng(9)
    x, W_r, Wg, Wu, Wd, dY = _rand_layer(rng, 16, 256, 128, 4, 2, std=0.05)
    assert _fd_check(x, W_r, Wg, Wu, Wd, 2, dY, n_coords=200, seed=1) > 900


@pytest.mark.slow
def test_gradients_match_finite_differences_tiny_fp32_draws():
    sh = si.shape("tiny")
    inp = si.make_inputs(sh, "cpu")
    args = [_np(inp[k + "_f32"]).copy() for k in ("x", "W_r", "W_gate", "W_up", "W_down")]
    dY = _np(inp["dY_f32"])
    assert _fd_check(*args, sh.top_k, dY, n_coords=60, seed=2) > 250


def test_gradients_match_autograd_with_bias():
    rng = np.random.default_rng(10)
    T, H, F, E, k = 24, 32, 16, 6, 3
    x, W_r, Wg, Wu, Wd, dY = _rand_layer(rng, T, H, F, E, k)
    bias = rng.standard_normal(E)
    g = mo.backward(x, W_r, Wg, Wu, Wd, k, dY, logit_bias=bias)
    idx = torch.from_numpy(g["fwd"]["idx"])
    tx, tr, tg, tu, td = (torch.tensor(a, requires_grad=True) for a in (x, W_r, Wg, Wu, Wd))
    logits = tx @ tr + torch.from_numpy(bias)
    w = torch.softmax(torch.gather(logits, 1, idx), dim=1)
    y = torch.zeros(T, H, dtype=torch.float64)
    for j in range(k):
        e = idx[:, j]
        h_g = torch.einsum("th,thf->tf", tx, tg[e])
        h_u = torch.einsum("th,thf->tf", tx, tu[e])
        o = torch.einsum("tf,tfh->th", torch.nn.functional.silu(h_g) * h_u, td[e])
        y = y + w[:, j:j + 1] * o
    (y * torch.from_numpy(dY)).sum().backward()
    for name, t in (("dx", tx), ("dW_r", tr), ("dW_gate", tg), ("dW_up", tu), ("dW_down", td)):
        np.testing.assert_allclose(g[name], t.grad.numpy(), rtol=1e-10, atol=1e-11)


def test_top1_router_gets_no_gradient():
    rng = np.random.default_rng(11)
    x, W_r, Wg, Wu, Wd, dY = _rand_layer(rng, 20, 16, 8, 5, 1)
    g = mo.backward(x, W_r, Wg, Wu, Wd, 1, dY)
    assert np.all(g["dl"] == 0.0)
    assert np.all(g["dW_r"] == 0.0)


def test_expert_without_tokens_gets_exact_zero_weight_grads():
    rng = np.random.default_rng(12)
    E = 6
    x, W_r, Wg, Wu, Wd, dY = _rand_layer(rng, 30, 16, 8, E, 2)
    bias = np.zeros(E)
    bias[4] = -1e3
    g = mo.backward(x, W_r, Wg, Wu, Wd, 2, dY, logit_bias=bias)
    assert g["fwd"]["counts"][4] == 0
    for name in ("dW_gate", "dW_up", "dW_down"):
        assert np.all(g[name][4] == 0.0)
        assert np.any(g[name][0] != 0.0)


def test_per_token_pieces_match_full_backward():
    rng = np.random.default_rng(13)
    x, W_r, Wg, Wu, Wd, dY = _rand_layer(rng, 18, 16, 8, 5, 2)
    bias = rng.standard_normal(5)
    g = mo.backward(x, W_r, Wg, Wu, Wd, 2, dY, logit_bias=bias)
    for t in (0, 7, 17):
        p = mo.token_forward_backward(t, x, W_r, Wg, Wu, Wd, 2, dY, logit_bias=bias)
        np.testing.assert_allclose(p["y"], g["fwd"]["y"][t], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(p["dx"], g["dx"][t], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(p["dw"], g["dw"][t], rtol=1e-12, atol=1e-13)
    fwd = g["fwd"]
    e = 2
    r0, r1 = fwd["offsets"][e], fwd["offsets"][e + 1]
    cols = mo.expert_weight_grad_columns(e, [0, 5], x, dY, Wg, Wu, Wd,
                                         fwd["perm_token"][r0:r1], fwd["w_row"][r0:r1])
    np.testing.assert_allclose(cols["dW_gate_col"], g["dW_gate"][e][:, [0, 5]].T, rtol=1e-12)
    np.testing.assert_allclose(cols["dW_up_col"], g["dW_up"][e][:, [0, 5]].T, rtol=1e-12)
    np.testing.assert_allclose(cols["dW_down_row"], g["dW_down"][e][[0, 5], :], rtol=1e-12)


def test_hand_worked_golden_example():
    with open(os.path.join(GOLDEN, "hand_worked_two_experts.json")) as fh:
        gold = json.load(fh)

    def ev(v):
        if isinstance(v, list):
            return np.array([ev(u) for u in v], dtype=np.float64)
        return float(eval(v, {"log": math.log}))  # closed forms written in the fixture

    i = gold["inputs"]
    x, W_r, Wg, Wu, Wd, dY = (ev(i[n]) for n in ("x", "W_r", "W_gate", "W_up", "W_down", "dY"))
    g = mo.backward(x, W_r, Wg, Wu, Wd, i["top_k"], dY)
    ex = gold["expected"]
    assert g["fwd"]["idx"].tolist() == ex["idx"]
    np.testing.assert_allclose(g["fwd"]["w"], ev(ex["w"]), rtol=1e-14)
    np.testing.assert_allclose(g["fwd"]["y"], ev(ex["y"]), rtol=1e-14, atol=1e-15)
    for name in ("dw", "dl", "dx", "dW_r", "dW_gate", "dW_up", "dW_down"):
        np.testing.assert_allclose(g[name], ev(ex[name]), rtol=1e-13, atol=1e-15, err_msg=name)


# ----------------------------------------------------------------- MXFP8


def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = mo.e4m3_decode(codes)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))
    assert np.nanmax(got) == 448.0 and np.sum(np.isnan(got)) == 2


def test_e4m3_round_trip_and_rne_against_torch_cast():
    codes = np.arange(256)
    vals = mo.e4m3_decode(codes)
    fin = np.isfinite(vals)
    assert np.array_equal(mo.e4m3_round(vals[fin]), vals[fin])
    rng = np.random.default_rng(14)
    v = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(20000) * 0.01,
                        (vals[fin][:-1] + vals[fin][1:]) / 2])     # midpoints: ties
    v = np.clip(v, -448, 448)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64)
    got = mo.e4m3_round(v.astype(np.float32).astype(np.float64))
    assert np.array_equal(got, ref.numpy())


def test_mx_scale_exponent_edges():
    for n in (-20, -3, 0, 1, 7, 30):
        assert mo.mx_scale_exponent(np.array(2.0 ** n)) == n - 8
        assert mo.mx_scale_exponent(np.array(np.nextafter(2.0 ** n, 0))) == n - 9
    assert mo.mx_scale_exponent(np.array(0.0)) == -127
    blk = np.zeros((1, 32))
    q, X = mo.mx_quantize(blk, 1)
    assert np.all(q == 0) and X[0, 0] == -127


def test_mx_quantize_properties():
    rng = np.random.default_rng(15)
    v = rng.standard_normal((8, 128)) * np.exp2(rng.integers(-10, 10, size=(8, 1)))
    q, X = mo.mx_quantize(v, 1)
    assert X.shape == (8, 4)
    assert np.all(np.abs(q) <= 448)
    blocks = np.abs(q).reshape(8, 4, 32).max(axis=2)
    assert np.all(blocks >= 256)                 # the largest element lands in [2^8, 448]
    deq = mo.mx_dequantize(q, X, 1)
    scale = np.repeat(np.exp2(X), 32, axis=1)
    err = np.abs(deq - v)
    inside = np.abs(v) <= 448 * scale
    # below the saturation point: at most half an E4M3 step (2^-4 relative for
    # normal numbers, half of 2^-9 in scaled units for subnormals)
    assert np.all(err[inside] <= np.maximum(np.abs(v[inside]) * 2.0 ** -4,
                                            2.0 ** -10 * scale[inside]) * (1 + 1e-12))
    # above it the element saturates to 448 * 2^X
    np.testing.assert_array_equal(np.abs(deq[~inside]), 448 * scale[~inside])
    # quantising along axis 0 of the transpose is the same thing
    q2, X2 = mo.mx_quantize(v.T, 0)
    assert np.array_equal(q2, q.T) and np.array_equal(X2, X.T)


def test_mx_segments_restart_blocks_per_expert():
    rng = np.random.default_rng(16)
    v = rng.standard_normal((75, 4))
    v[40:] *= 1000.0                            # second segment much larger
    offs = np.array([0, 40, 40, 75])
    out = mo.mx_round_trip_segments(v, offs)
    for a, b in ((0, 40), (40, 75)):
        seg = np.concatenate([v[a:b], np.zeros(((-(b - a)) % 32, 4))])
        np.testing.assert_array_equal(out[a:b], mo.mx_round_trip(seg, 0)[: b - a])
    # blocks of the first segment never see the large second segment
    assert np.max(np.abs(out[:40] - v[:40])) < 0.2


def test_mxfp8_forward_is_close_to_exact_and_fp8_bwd_forward_is_exact():
    rng = np.random.default_rng(17)
    x, W_r, Wg, Wu, Wd, dY = _rand_layer(rng, 32, 64, 32, 3, 2, std=0.1)
    exact = mo.forward(x, W_r, Wg, Wu, Wd, 2)
    q = mo.forward(x, W_r, Wg, Wu, Wd, 2, precision="mxfp8")
    rel = np.linalg.norm(q["y"] - exact["y"]) / np.linalg.norm(exact["y"])
    assert 1e-4 < rel < 0.1
    # fp8_bwd leaves the forward exact
    fb = mo.forward(x, W_r, Wg, Wu, Wd, 2, precision="fp8_bwd")
    np.testing.assert_array_equal(fb["y"], exact["y"])
    gb = mo.backward(x, W_r, Wg, Wu, Wd, 2, dY, precision="fp8_bwd")
    ge = mo.backward(x, W_r, Wg, Wu, Wd, 2, dY)
    for name in ("dx", "dW_gate", "dW_up", "dW_down"):
        rel = np.linalg.norm(gb[name] - ge[name]) / np.linalg.norm(ge[name])
        assert 1e-4 < rel < 0.1, name


# ----------------------------------------------------------------- MXFP8 block axes
#
# Which axis each GEMM operand is blocked along is a reading (E8M0 scales per
# 32 elements along the GEMM's reduction dimension K).  The mathematics fixes
# a pin for it: with blocks along K, multiplying one M-row of the A operand
# (or one N-column of B) by 2^j moves only that row's (column's) scale
# exponents by j and leaves its E4M3 codes unchanged, so exactly that row
# (column) of the product scales by 2^j and every other element stays
# bit-identical.  Blocks along any other axis mix the scaled row with its
# neighbours and break both halves of the statement.  Every quantisation
# point of the oracle is covered by one of the pins below.

MX_SHAPE = (96, 64, 64, 3, 2)    # T, H, F, E, k: 50-80 rows per expert, 2 blocks along H and F


def _mx_layer(seed):
    return _rand_layer(np.random.default_rng(seed), *MX_SHAPE, std=0.1)


def _token_rows(fwd, t):
    """Mask of the permuted rows that hold token t."""
    return fwd["perm_token"] == t


@pytest.mark.parametrize("j", [4, -3])
def test_mx_forward_activation_blocks_run_along_k(j):
    """x along H (gate/up GEMM) and a along F (down GEMM): scaling token t's
    input scales its rows of h exactly and leaves every other token's rows of
    h and o, and every other token's output, bit-identical."""
    x, W_r, Wg, Wu, Wd, _ = _mx_layer(40)
    t = 7
    base = mo.forward(x, W_r, Wg, Wu, Wd, 2, precision="mxfp8")
    x2 = x.copy()
    x2[t] *= 2.0 ** j
    got = mo.forward(x2, W_r, Wg, Wu, Wd, 2, precision="mxfp8")
    assert np.array_equal(got["idx"], base["idx"])    # logits scale exactly: same routing
    rows = _token_rows(base, t)
    for name in ("h_gate", "h_up"):
        np.testing.assert_array_equal(got[name][rows], base[name][rows] * 2.0 ** j)
        np.testing.assert_array_equal(got[name][~rows], base[name][~rows])
    np.testing.assert_array_equal(got["o"][~rows], base["o"][~rows])
    assert not np.array_equal(got["o"][rows], base["o"][rows])
    keep = np.arange(x.shape[0]) != t
    np.testing.assert_array_equal(got["y"][keep], base["y"][keep])


@pytest.mark.parametrize("which", ["gate", "up"])
def test_mx_forward_gate_up_weight_blocks_run_along_h(which):
    """W_gate / W_up along H: scaling column f of one expert's weight scales
    exactly that column of its rows of h and nothing else."""
    x, W_r, Wg, Wu, Wd, _ = _mx_layer(41)
    e, f, j = 1, 37, 3
    base = mo.forward(x, W_r, Wg, Wu, Wd, 2, precision="mxfp8")
    W2 = (Wg if which == "gate" else Wu).copy()
    W2[e][:, f] *= 2.0 ** j
    args = (W2, Wu) if which == "gate" else (Wg, W2)
    got = mo.forward(x, W_r, *args, Wd, 2, precision="mxfp8")
    r0, r1 = base["offsets"][e], base["offsets"][e + 1]
    name, other = ("h_gate", "h_up") if which == "gate" else ("h_up", "h_gate")
    want = base[name].copy()
    want[r0:r1, f] *= 2.0 ** j
    np.testing.assert_array_equal(got[name], want)
    np.testing.assert_array_equal(got[other], base[other])


def test_mx_forward_down_weight_blocks_run_along_f():
    """W_down along F: scaling column c of one expert's W_down scales exactly
    that column of its rows of o and nothing else."""
    x, W_r, Wg, Wu, Wd, _ = _mx_layer(42)
    e, c, j = 2, 21, 3
    base = mo.forward(x, W_r, Wg, Wu, Wd, 2, precision="mxfp8")
    Wd2 = Wd.copy()
    Wd2[e][:, c] *= 2.0 ** j
    got = mo.forward(x, W_r, Wg, Wu, Wd2, 2, precision="mxfp8")
    r0, r1 = base["offsets"][e], base["offsets"][e + 1]
    want = base["o"].copy()
    want[r0:r1, c] *= 2.0 ** j
    np.testing.assert_array_equal(got["o"], want)


@pytest.mark.parametrize("precision", ["mxfp8", "fp8_bwd"])
@pytest.mark.parametrize("j", [3, -4])
def test_mx_backward_dgrad_activation_blocks_run_along_k(precision, j):
    """dY along H (down dgrad) and dh along F (gate/up dgrad): scaling token
    t's upstream gradient scales its dx exactly and leaves every other token's
    dx bit-identical."""
    x, W_r, Wg, Wu, Wd, dY = _mx_layer(43)
    t = 11
    g0 = mo.backward(x, W_r, Wg, Wu, Wd, 2, dY, precision=precision)
    dY2 = dY.copy()
    dY2[t] *= 2.0 ** j
    g1 = mo.backward(x, W_r, Wg, Wu, Wd, 2, dY2, precision=precision)
    np.testing.assert_array_equal(g1["dx"][t], g0["dx"][t] * 2.0 ** j)
    keep = np.arange(x.shape[0]) != t
    np.testing.assert_array_equal(g1["dx"][keep], g0["dx"][keep])
    np.testing.assert_array_equal(g1["dw"][t], g0["dw"][t] * 2.0 ** j)


@pytest.mark.parametrize("precision", ["mxfp8", "fp8_bwd"])
def test_mx_backward_down_weight_and_dh_token_blocks(precision):
    """W_down along H (down dgrad) and dh along the expert's tokens (gate/up
    wgrad): scaling row f of one expert's W_down scales exactly column f of
    its dW_gate and dW_up; every other element of both stays bit-identical."""
    x, W_r, Wg, Wu, Wd, dY = _mx_layer(44)
    e, f, j = 0, 45, 2
    g0 = mo.backward(x, W_r, Wg, Wu, Wd, 2, dY, precision=precision)
    Wd2 = Wd.copy()
    Wd2[e][f, :] *= 2.0 ** j
    g1 = mo.backward(x, W_r, Wg, Wu, Wd2, 2, dY, precision=precision)
    for name in ("dW_gate", "dW_up"):
        want = g0[name].copy()
        want[e][:, f] *= 2.0 ** j
        np.testing.assert_array_equal(g1[name], want)


@pytest.mark.parametrize("precision", ["mxfp8", "fp8_bwd"])
def test_mx_backward_down_wgrad_a_operand_token_blocks(precision):
    """w*a along the expert's tokens (down wgrad): scaling column f of one
    expert's W_up scales column f of its a exactly, hence exactly row f of its
    dW_down, and leaves every other row of dW_down bit-identical."""
    x, W_r, Wg, Wu, Wd, dY = _mx_layer(45)
    e, f, j = 1, 9, 3
    g0 = mo.backward(x, W_r, Wg, Wu, Wd, 2, dY, precision=precision)
    Wu2 = Wu.copy()
    Wu2[e][:, f] *= 2.0 ** j
    g1 = mo.backward(x, W_r, Wg, Wu2, Wd, 2, dY, precision=precision)
    want = g0["dW_down"].copy()
    want[e][f, :] *= 2.0 ** j
    np.testing.assert_array_equal(g1["dW_down"], want)


@pytest.mark.parametrize("precision", ["mxfp8", "fp8_bwd"])
def test_mx_backward_down_wgrad_dy_token_blocks(precision):
    """dY along the expert's tokens (down wgrad): scaling column c of dY for
    every token scales exactly column c of every expert's dW_down."""
    x, W_r, Wg, Wu, Wd, dY = _mx_layer(46)
    c, j = 50, -3
    g0 = mo.backward(x, W_r, Wg, Wu, Wd, 2, dY, precision=precision)
    dY2 = dY.copy()
    dY2[:, c] *= 2.0 ** j
    g1 = mo.backward(x, W_r, Wg, Wu, Wd, 2, dY2, precision=precision)
    want = g0["dW_down"].copy()
    want[:, :, c] *= 2.0 ** j
    np.testing.assert_array_equal(g1["dW_down"], want)


@pytest.mark.parametrize("precision", ["mxfp8", "fp8_bwd"])
def test_mx_backward_gate_up_dgrad_weight_blocks_run_along_f(precision):
    """W_gate and W_up along F (gate/up dgrad), with the forward held fixed:
    scaling row h of one expert's W_gate and W_up scales exactly column h of
    its rows of dx and nothing else."""
    x, W_r, Wg, Wu, Wd, dY = _mx_layer(47)
    e, h, j = 2, 33, 2
    fwd = mo.forward(x, W_r, Wg, Wu, Wd, 2, precision=precision)
    b0 = mo.expert_backward(e, fwd, x, dY, Wg, Wu, Wd, precision)
    Wg2, Wu2 = Wg.copy(), Wu.copy()
    Wg2[e][h, :] *= 2.0 ** j
    Wu2[e][h, :] *= 2.0 ** j
    b1 = mo.expert_backward(e, fwd, x, dY, Wg2, Wu2, Wd, precision)
    want = b0["dx_row"].copy()
    want[:, h] *= 2.0 ** j
    np.testing.assert_array_equal(b1["dx_row"], want)


@pytest.mark.parametrize("precision", ["mxfp8", "fp8_bwd"])
def test_mx_backward_gate_up_wgrad_x_token_blocks(precision):
    """x along the expert's tokens (gate/up wgrad), with the forward held
    fixed: scaling column h of x scales exactly row h of the expert's dW_gate
    and dW_up and nothing else."""
    x, W_r, Wg, Wu, Wd, dY = _mx_layer(48)
    e, h, j = 0, 14, 3
    fwd = mo.forward(x, W_r, Wg, Wu, Wd, 2, precision=precision)
    b0 = mo.expert_backward(e, fwd, x, dY, Wg, Wu, Wd, precision)
    x2 = x.copy()
    x2[:, h] *= 2.0 ** j
    b1 = mo.expert_backward(e, fwd, x2, dY, Wg, Wu, Wd, precision)
    for name in ("dW_gate", "dW_up"):
        want = b0[name].copy()
        want[h, :] *= 2.0 ** j
        np.testing.assert_array_equal(b1[name], want)


@pytest.mark.parametrize("precision", ["mxfp8", "fp8_bwd"])
def test_mx_weight_grad_columns_match_full_backward(precision):
    rng = np.random.default_rng(18)
    x, W_r, Wg, Wu, Wd, dY = _rand_layer(rng, 70, 64, 64, 3, 2, std=0.1)
    g = mo.backward(x, W_r, Wg, Wu, Wd, 2, dY, precision=precision)
    fwd = g["fwd"]
    for e in range(3):
        r0, r1 = fwd["offsets"][e], fwd["offsets"][e + 1]
        cols = [0, 17, 63]
        c = mo.expert_weight_grad_columns_mx(e, cols, x, dY, Wg, Wu, Wd, fwd["perm_token"][r0:r1],
                                             fwd["w_row"][r0:r1], precision)
        np.testing.assert_allclose(c["dW_gate_col"], g["dW_gate"][e][:, cols].T, rtol=1e-10,
                                   atol=1e-12)
        np.testing.assert_allclose(c["dW_up_col"], g["dW_up"][e][:, cols].T, rtol=1e-10,
                                   atol=1e-12)
        np.testing.assert_allclose(c["dW_down_row"], g["dW_down"][e][cols, :], rtol=1e-10,
                                   atol=1e-12)
