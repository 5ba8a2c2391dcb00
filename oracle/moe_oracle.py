"""Plain CPU oracle of the fused Mixture-of-Experts layer, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path imports, calls
or links this module; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` use it.  It shares no code with the CUDA path.

What it computes (numpy, float64 throughout, slow and direct):

* The layer of "Prime Mega MoE" (Prime Intellect's fused MoE training kernel,
  which adds a fused backward pass to DeepSeek's forward-only Mega MoE): each
  token goes to a few experts, each expert is a gated SwiGLU feed-forward block
  with no bias, and the expert outputs are combined with the router weights
  (bitsgeniais.com.br/?p=10788, "A Magia da Fusão" and "Detalhes Técnicos
  Rápidos"; ai-daily-news.org, "Qué se ha publicado").
* Routing: a linear router, softmax over all E experts, top-k selection and
  renormalisation of the k selected probabilities.  The pages name top-8 of
  128 experts ("Os Números..." on bitsgeniais.com.br; "Analisi dei kernel
  layer" on roccomilluzzo.it) but print no formula; the softmax/top-k/
  renormalise form is the textbook one.
* The backward pass is the exact vector-Jacobian product of the forward at an
  upstream gradient dY (the routing indices are piecewise constant and get no
  gradient).
* MXFP8 (OCP Microscaling v1.0): E4M3 elements with one E8M0 power-of-two
  scale per 32 consecutive elements along a GEMM's reduction dimension.  The
  pages name the format only ("Supporto di precisione" on roccomilluzzo.it).

Readings where the pages are silent (each one is listed with its reason in the
design notes of the repository):

* selection is made on the router logits, which orders experts exactly as the
  softmax probabilities do; equal logits go to the lower expert id;
* silu(z) = z * sigmoid(z) applies to x·W_gate and multiplies x·W_up;
* the optional per-expert ``logit_bias`` is added to the logits before
  selection and weighting and receives no gradient;
* the permuted layout is expert-major with ascending token id inside an expert.

Pins: every function here is checked by ``tests/test_oracle.py`` against
something other than itself (brute-force loops, finite differences, closed
forms, special cases, library casts and hand-derived golden values).
"""

from __future__ import annotations

from typing import Dict, Iterator, Optional, Tuple

import numpy as np

# --------------------------------------------------------------------------
# element-wise pieces
# --------------------------------------------------------------------------


def sigmoid(z: np.ndarray) -> np.ndarray:
    """Logistic function 1 / (1 + exp(-z)), evaluated without overflow."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = ez / (1.0 + ez)
    return out


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU (swish-1): z * sigmoid(z)."""
    return z * sigmoid(z)


def silu_grad(z: np.ndarray) -> np.ndarray:
    """d silu / dz = sigmoid(z) * (1 + z * (1 - sigmoid(z)))."""
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def swiglu(h_gate: np.ndarray, h_up: np.ndarray) -> np.ndarray:
    """Gated SwiGLU activation: silu(x W_gate) * (x W_up)."""
    return silu(h_gate) * h_up


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------


def router_logits(x: np.ndarray, W_r: np.ndarray,
                  logit_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] W_r[h, e] (+ logit_bias[e])."""
    logits = np.asarray(x, np.float64) @ np.asarray(W_r, np.float64)
    if logit_bias is not None:
        logits = logits + np.asarray(logit_bias, np.float64)[None, :]
    return logits


def softmax(logits: np.ndarray) -> np.ndarray:
    """Softmax over the last axis."""
    m = np.max(logits, axis=-1, keepdims=True)
    ex = np.exp(logits - m)
    return ex / np.sum(ex, axis=-1, keepdims=True)


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """The k experts with the largest logit per token, ordered by (-logit, id).

    A stable sort of -logits keeps, among equal values, the lower expert id
    first; this is the tie rule.  Works on fp32 or fp64 logits: the decision is
    made on exactly the values given.
    """
    order = np.argsort(-np.asarray(logits), axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def topk_weights(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Renormalised top-k probabilities: w_j = p[S_j] / sum_{i in S} p[S_i],
    with p the softmax over all E experts."""
    p = softmax(np.asarray(logits, np.float64))
    pS = np.take_along_axis(p, idx, axis=1)
    return pS / np.sum(pS, axis=1, keepdims=True)


def route(logits: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Top-k indices and renormalised weights from router logits."""
    idx = select_topk(logits, k)
    return idx, topk_weights(logits, idx)


def permutation(idx: np.ndarray, E: int) -> Dict[str, np.ndarray]:
    """Counting-sort permutation of the (token, slot) pairs by expert.

    Rows of the permuted layout are expert-major and, inside an expert, in
    ascending token order.  Returns counts[E], offsets[E+1] (unpadded),
    perm_token[P] (row -> token) and slot_row[T, k] ((t, j) -> row).
    """
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    order = np.argsort(flat, kind="stable")          # row -> flat (t*k + j)
    perm_token = order // k
    slot_row = np.empty(T * k, np.int64)
    slot_row[order] = np.arange(T * k)
    return {"counts": counts, "offsets": offsets, "perm_token": perm_token,
            "slot_row": slot_row.reshape(T, k), "row_flat": order}


# --------------------------------------------------------------------------
# MXFP8 (OCP MX v1.0): E4M3 elements, E8M0 scale per 32 elements
# --------------------------------------------------------------------------

E4M3_MAX = 448.0
E4M3_EMAX = 8            # exponent of the largest power of two in E4M3 (2^8 = 256)
MX_BLOCK = 32


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    """Value of each 8-bit E4M3 code (1 sign, 4 exponent bits biased by 7,
    3 mantissa bits, no infinities, S.1111.111 is NaN)."""
    code = np.asarray(code, np.int64) & 0xFF
    s = np.where(code & 0x80, -1.0, 1.0)
    e = (code >> 3) & 0xF
    m = code & 0x7
    normal = s * (1.0 + m / 8.0) * np.exp2(e - 7.0)
    sub = s * (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, val)


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to even mantissa, saturating at
    +-448.  E4M3 has 3 mantissa bits, so inside the binade [2^e, 2^(e+1)) the
    representable values are multiples of 2^(e-3); subnormals share the step
    2^-9 of the lowest binade (e = -6).  Rounding |v| / step half-to-even is
    mantissa-parity rounding because every binade starts at the even multiple 8."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    _, ex = np.frexp(a)                     # a = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex.astype(np.int64) - 1, -6)
    step = np.exp2((e - 3).astype(np.float64))
    r = np.minimum(np.rint(a / step) * step, E4M3_MAX)
    return np.sign(v) * r


def mx_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Shared exponent X = floor(log2(amax)) - 8, clamped to E8M0's [-127, 127];
    an all-zero block takes -127."""
    amax = np.asarray(amax, np.float64)
    _, ex = np.frexp(amax)                  # amax = m * 2^ex, m in [0.5, 1)
    fl = ex.astype(np.int64) - 1            # floor(log2(amax)) for amax > 0
    X = fl - E4M3_EMAX
    X = np.where(amax > 0, X, -127)
    return np.clip(X, -127, 127)


def mx_quantize(v: np.ndarray, axis: int) -> Tuple[np.ndarray, np.ndarray]:
    """Quantise ``v`` in blocks of 32 consecutive elements along ``axis``.

    Returns (q, X): q the E4M3 values (as float64) with the same shape as v and
    X the integer scale exponents, one per block (the block axis shrinks by 32).
    The dequantised tensor is q * 2^X broadcast over each block.  The length
    along ``axis`` must be a multiple of 32 (callers zero-pad ragged tails).
    """
    v = np.moveaxis(np.asarray(v, np.float64), axis, -1)
    n = v.shape[-1]
    assert n % MX_BLOCK == 0, "MX blocks need a length that is a multiple of 32"
    blocks = v.reshape(*v.shape[:-1], n // MX_BLOCK, MX_BLOCK)
    amax = np.max(np.abs(blocks), axis=-1)
    X = mx_scale_exponent(amax)
    q = e4m3_round(blocks / np.exp2(X)[..., None])
    q = np.moveaxis(q.reshape(v.shape), -1, axis)
    return q, np.moveaxis(X, -1, axis)


def mx_dequantize(q: np.ndarray, X: np.ndarray, axis: int) -> np.ndarray:
    q = np.moveaxis(q, axis, -1)
    X = np.moveaxis(X, axis, -1)
    out = q * np.repeat(np.exp2(X), MX_BLOCK, axis=-1)
    return np.moveaxis(out, -1, axis)


def mx_round_trip(v: np.ndarray, axis: int) -> np.ndarray:
    """Quantise and dequantise along ``axis``."""
    q, X = mx_quantize(v, axis)
    return mx_dequantize(q, X, axis)


def mx_round_trip_segments(v: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """MX round trip along axis 0 where the blocks restart at every segment
    start ``offsets[e]`` (the tokens of one expert); a segment's ragged tail is
    padded with zeros to 32 rows for the scale computation."""
    out = np.zeros_like(np.asarray(v, np.float64))
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b == a:
            continue
        seg = np.asarray(v[a:b], np.float64)
        pad = (-seg.shape[0]) % MX_BLOCK
        if pad:
            seg = np.concatenate([seg, np.zeros((pad,) + seg.shape[1:])], axis=0)
        out[a:b] = mx_round_trip(seg, 0)[: b - a]
    return out


# --------------------------------------------------------------------------
# forward
# --------------------------------------------------------------------------


def _q(mode: Optional[str], which: str) -> bool:
    """Whether an expert GEMM runs on MXFP8 operands in precision ``mode``.
    'fwd' GEMMs: gate/up and down; 'bwd' GEMMs: both dgrads and both wgrads."""
    if mode == "mxfp8":
        return True
    if mode == "fp8_bwd":
        return which == "bwd"
    return False


def forward_per_token(x, W_r, W_gate, W_up, W_down, top_k: int,
                      logit_bias=None, idx=None) -> np.ndarray:
    """Brute-force forward: a Python loop over tokens and their k experts.

    y_t = sum_j w_tj * (silu(x_t W_gate[e]) * (x_t W_up[e])) W_down[e], e = S_tj.
    """
    x = np.asarray(x, np.float64)
    logits = router_logits(x, W_r, logit_bias)
    if idx is None:
        idx = select_topk(logits, top_k)
    w = topk_weights(logits, idx)
    T, H = x.shape
    y = np.zeros((T, H))
    for t in range(T):
        for j in range(top_k):
            e = int(idx[t, j])
            hg = x[t] @ W_gate[e]
            hu = x[t] @ W_up[e]
            y[t] += w[t, j] * (swiglu(hg, hu) @ W_down[e])
    return y


def forward(x, W_r, W_gate, W_up, W_down, top_k: int, logit_bias=None,
            precision: Optional[str] = None, idx=None) -> Dict[str, np.ndarray]:
    """Grouped forward: route, permute rows expert-major, one GEMM pair per
    expert, then the weighted combine back to token order.

    Returns y plus the intermediates (logits, idx, w, the permutation, h_gate,
    h_up and a in permuted row order).
    """
    x = np.asarray(x, np.float64)
    T, H = x.shape
    E = W_gate.shape[0]
    logits = router_logits(x, W_r, logit_bias)
    if idx is None:
        idx = select_topk(logits, top_k)
    w = topk_weights(logits, idx)
    perm = permutation(idx, E)
    offs, ptok = perm["offsets"], perm["perm_token"]
    w_row = w.reshape(-1)[perm["row_flat"]]
    xp = x[ptok]
    F = W_gate.shape[2]
    P = T * top_k
    hg = np.zeros((P, F))
    hu = np.zeros((P, F))
    a = np.zeros((P, F))
    o = np.zeros((P, H))
    qf = _q(precision, "fwd")
    for e in range(E):
        r0, r1 = int(offs[e]), int(offs[e + 1])
        if r1 == r0:
            continue
        xe = xp[r0:r1]
        Wg, Wu, Wd = (np.asarray(W, np.float64) for W in (W_gate[e], W_up[e], W_down[e]))
        if qf:   # K = H for gate/up: x rows along H, weights along their H axis
            xe = mx_round_trip(xe, 1)
            Wg, Wu = mx_round_trip(Wg, 0), mx_round_trip(Wu, 0)
        hg[r0:r1] = xe @ Wg
        hu[r0:r1] = xe @ Wu
        a[r0:r1] = swiglu(hg[r0:r1], hu[r0:r1])
        ae = a[r0:r1]
        if qf:   # K = F for down: a along F, W_down along its F axis
            ae = mx_round_trip(ae, 1)
            Wd = mx_round_trip(Wd, 0)
        o[r0:r1] = ae @ Wd
    y = np.zeros((T, H))
    np.add.at(y, ptok, w_row[:, None] * o)
    return {"y": y, "logits": logits, "idx": idx, "w": w, "w_row": w_row,
            "h_gate": hg, "h_up": hu, "a": a, "o": o, **perm}


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------


def router_logit_grad(w: np.ndarray, dw: np.ndarray) -> np.ndarray:
    """d loss / d logit at the selected experts: w_j (dw_j - sum_i w_i dw_i).

    w_j = exp(l_j) / sum_{i in S} exp(l_i) gives dw_j/dl_m = w_j (delta_jm - w_m);
    unselected logits get zero."""
    return w * (dw - np.sum(w * dw, axis=1, keepdims=True))


def expert_backward(e: int, fwd: Dict[str, np.ndarray], x, dY, W_gate, W_up, W_down,
                    precision: Optional[str] = None) -> Dict[str, np.ndarray]:
    """Backward pass restricted to the rows of expert e.

    Returns dW_gate[e], dW_up[e], dW_down[e] ([H,F], [H,F], [F,H]), the per-row
    router-weight gradients dw_row and the per-row input gradients dx_row.
    """
    offs, ptok = fwd["offsets"], fwd["perm_token"]
    r0, r1 = int(offs[e]), int(offs[e + 1])
    H = x.shape[1]
    F = W_gate.shape[2]
    if r1 == r0:
        return {"dW_gate": np.zeros((H, F)), "dW_up": np.zeros((H, F)),
                "dW_down": np.zeros((F, H)), "dw_row": np.zeros(0),
                "dx_row": np.zeros((0, H)), "rows": (r0, r1)}
    qb = _q(precision, "bwd")
    xe = np.asarray(x, np.float64)[ptok[r0:r1]]
    dYe = np.asarray(dY, np.float64)[ptok[r0:r1]]
    we = fwd["w_row"][r0:r1]
    hg, hu, a = fwd["h_gate"][r0:r1], fwd["h_up"][r0:r1], fwd["a"][r0:r1]
    Wg, Wu, Wd = (np.asarray(W, np.float64) for W in (W_gate[e], W_up[e], W_down[e]))
    seg = np.array([0, r1 - r0])
    # down dgrad: g = dY_perm W_down^T (K = H)
    if qb:
        g = mx_round_trip(dYe, 1) @ mx_round_trip(Wd, 1).T
    else:
        g = dYe @ Wd.T
    dw_row = np.sum(g * a, axis=1)                       # = <dY_t, o_r>
    da = we[:, None] * g
    dhg = da * hu * silu_grad(hg)
    dhu = da * silu(hg)
    aw = we[:, None] * a
    # down wgrad: (w a)^T dY_perm (K = tokens of the expert)
    if qb:
        dW_down = mx_round_trip_segments(aw, seg).T @ mx_round_trip_segments(dYe, seg)
    else:
        dW_down = aw.T @ dYe
    # gate/up dgrad (K = F for each half) and wgrad (K = tokens)
    if qb:
        dx_row = (mx_round_trip(dhg, 1) @ mx_round_trip(Wg, 1).T
                  + mx_round_trip(dhu, 1) @ mx_round_trip(Wu, 1).T)
        xq = mx_round_trip_segments(xe, seg)
        dW_gate = xq.T @ mx_round_trip_segments(dhg, seg)
        dW_up = xq.T @ mx_round_trip_segments(dhu, seg)
    else:
        dx_row = dhg @ Wg.T + dhu @ Wu.T
        dW_gate = xe.T @ dhg
        dW_up = xe.T @ dhu
    return {"dW_gate": dW_gate, "dW_up": dW_up, "dW_down": dW_down, "dw_row": dw_row,
            "dx_row": dx_row, "rows": (r0, r1)}


def iter_expert_backward(fwd, x, dY, W_gate, W_up, W_down,
                         precision: Optional[str] = None) -> Iterator[Tuple[int, Dict]]:
    """Expert-by-expert backward, so that large layers fit in host memory."""
    for e in range(W_gate.shape[0]):
        yield e, expert_backward(e, fwd, x, dY, W_gate, W_up, W_down, precision)


def backward(x, W_r, W_gate, W_up, W_down, top_k: int, dY, logit_bias=None,
             precision: Optional[str] = None, fwd=None, idx=None,
             keep_weight_grads: bool = True) -> Dict[str, np.ndarray]:
    """Full VJP of the layer at dY: dx, dW_r, dW_gate, dW_up, dW_down, and the
    router intermediates dw [T,k] and dl [T,E].  With keep_weight_grads=False
    the expert weight gradients are computed expert by expert and dropped, so
    the token-local results (dx, dw, dl) of a token subset of a large layer
    fit in host memory."""
    x = np.asarray(x, np.float64)
    if fwd is None:
        fwd = forward(x, W_r, W_gate, W_up, W_down, top_k, logit_bias, precision, idx=idx)
    T, H = x.shape
    E, _, F = W_gate.shape
    P = T * top_k
    if keep_weight_grads:
        dW_gate = np.zeros((E, H, F))
        dW_up = np.zeros((E, H, F))
        dW_down = np.zeros((E, F, H))
    else:
        dW_gate = dW_up = dW_down = None
    dw_rows = np.zeros(P)
    dx_rows = np.zeros((P, H))
    for e, g in iter_expert_backward(fwd, x, dY, W_gate, W_up, W_down, precision):
        r0, r1 = g["rows"]
        if keep_weight_grads:
            dW_gate[e], dW_up[e], dW_down[e] = g["dW_gate"], g["dW_up"], g["dW_down"]
        dw_rows[r0:r1] = g["dw_row"]
        dx_rows[r0:r1] = g["dx_row"]
    dw = dw_rows[fwd["slot_row"]]                        # [T, k]
    dl_sel = router_logit_grad(fwd["w"], dw)
    dl = np.zeros((T, E))
    np.put_along_axis(dl, fwd["idx"], dl_sel, axis=1)
    dx = np.zeros((T, H))
    np.add.at(dx, fwd["perm_token"], dx_rows)
    dx += dl @ np.asarray(W_r, np.float64).T
    dW_r = x.T @ dl
    return {"dx": dx, "dW_r": dW_r, "dW_gate": dW_gate, "dW_up": dW_up,
            "dW_down": dW_down, "dw": dw, "dl": dl, "fwd": fwd}


# --------------------------------------------------------------------------
# per-token and per-expert pieces for sampled checks of large layers
# --------------------------------------------------------------------------


def token_forward_backward(t: int, x, W_r, W_gate, W_up, W_down, top_k: int, dY,
                           logit_bias=None) -> Dict[str, np.ndarray]:
    """y_t, dw_t, dl_t (at the selected experts) and dx_t for one token.

    Every one of these depends only on token t's own row, so large layers can
    be checked on sampled tokens."""
    xt = np.asarray(x[t], np.float64)
    dYt = np.asarray(dY[t], np.float64)
    l = router_logits(xt[None, :], W_r, logit_bias)
    idx = select_topk(l, top_k)
    w = topk_weights(l, idx)[0]
    idx = idx[0]
    H = xt.shape[0]
    y = np.zeros(H)
    dw = np.zeros(top_k)
    dx = np.zeros(H)
    for j, e in enumerate(idx):
        Wg, Wu, Wd = (np.asarray(W[e], np.float64) for W in (W_gate, W_up, W_down))
        hg, hu = xt @ Wg, xt @ Wu
        a = swiglu(hg, hu)
        o = a @ Wd
        y += w[j] * o
        dw[j] = dYt @ o
        g = Wd @ dYt
        da = w[j] * g
        dx += (da * hu * silu_grad(hg)) @ Wg.T + (da * silu(hg)) @ Wu.T
    dl_sel = router_logit_grad(w[None, :], dw[None, :])[0]
    dx += np.asarray(W_r, np.float64)[:, idx] @ dl_sel
    return {"y": y, "idx": idx, "w": w, "dw": dw, "dl_sel": dl_sel, "dx": dx,
            "logits": l[0]}


def expert_weight_grad_columns(e: int, cols, x, dY, W_gate, W_up, W_down, rows_tokens,
                               rows_w) -> Dict[str, np.ndarray]:
    """Columns f of dW_gate[e] and dW_up[e] ([H] each) and rows f of dW_down[e]
    ([H]) from the tokens routed to expert e (``rows_tokens``, ascending) and
    their router weights ``rows_w``."""
    xe = np.asarray(x[rows_tokens], np.float64)
    dYe = np.asarray(dY[rows_tokens], np.float64)
    out = {"dW_gate_col": [], "dW_up_col": [], "dW_down_row": []}
    for f in cols:
        hg = xe @ np.asarray(W_gate[e][:, f], np.float64)
        hu = xe @ np.asarray(W_up[e][:, f], np.float64)
        a = swiglu(hg, hu)
        g = dYe @ np.asarray(W_down[e][f, :], np.float64)
        da = rows_w * g
        out["dW_gate_col"].append(xe.T @ (da * hu * silu_grad(hg)))
        out["dW_up_col"].append(xe.T @ (da * silu(hg)))
        out["dW_down_row"].append((rows_w * a) @ dYe)
    return {k: np.array(v) for k, v in out.items()}


def expert_weight_grad_columns_mx(e: int, cols, x, dY, W_gate, W_up, W_down, rows_tokens,
                                  rows_w, precision: str) -> Dict[str, np.ndarray]:
    """expert_weight_grad_columns with the MXFP8 quantisation points of
    ``precision`` ('mxfp8' or 'fp8_bwd'): columns f of dW_gate[e] / dW_up[e]
    and rows f of dW_down[e].

    Forward (mxfp8 only): x rows and W_gate / W_up columns along H, a along F
    (the whole row of a is needed for that block, so full rows of h are formed).
    Backward: dY rows and W_down rows along H for g; the weight gradients take
    x, dh, w*a and dY quantised along the expert's tokens (blocks of 32 from the
    segment start, zero-padded), which only needs whole token columns."""
    qf = _q(precision, "fwd")
    xe = np.asarray(x[rows_tokens], np.float64)
    dYe = np.asarray(dY[rows_tokens], np.float64)
    Wg = np.asarray(W_gate[e], np.float64)
    Wu = np.asarray(W_up[e], np.float64)
    Wd = np.asarray(W_down[e], np.float64)
    seg = np.array([0, xe.shape[0]])
    xf = mx_round_trip(xe, 1) if qf else xe
    Wgf = mx_round_trip(Wg, 0) if qf else Wg
    Wuf = mx_round_trip(Wu, 0) if qf else Wu
    hg = xf @ Wgf
    hu = xf @ Wuf
    a = swiglu(hg, hu)
    g = mx_round_trip(dYe, 1) @ mx_round_trip(Wd, 1).T
    xq = mx_round_trip_segments(xe, seg)
    dYq = mx_round_trip_segments(dYe, seg)
    out = {"dW_gate_col": [], "dW_up_col": [], "dW_down_row": []}
    for f in cols:
        da = rows_w * g[:, f]
        dhg = (da * hu[:, f] * silu_grad(hg[:, f]))[:, None]
        dhu = (da * silu(hg[:, f]))[:, None]
        aw = (rows_w * a[:, f])[:, None]
        out["dW_gate_col"].append(xq.T @ mx_round_trip_segments(dhg, seg)[:, 0])
        out["dW_up_col"].append(xq.T @ mx_round_trip_segments(dhu, seg)[:, 0])
        out["dW_down_row"].append(mx_round_trip_segments(aw, seg)[:, 0] @ dYq)
    return {k: np.array(v) for k, v in out.items()}
