"""Oracle: top-K routed SwiGLU MoE layer, forward and backward in float64 (test infrastructure only).

Forward being differentiated (the plainest reading shared by the three pages): for each token t and
each of its K routing slots k, with e = ids[t, k] and score s[t, k],

    h   = x_t @ W1_e + b1_e                 W1_e [H, 2I]: columns 0..I-1 gate, I..2I-1 up
    a   = SiLU(gate) * up                   SiLU(z) = z * sigmoid(z)
    y   = a @ W2_e + b2_e                   W2_e [I, H]
    out_t = sum_k s[t, k] * y

Backward (sonic-moe backward.py `_down_projection_backward_act` with `gemm_dgated(...,
colvec_scale=s, colvec_reduce=True)`, `db2_and_ds_kernel`, `_down_projection_backward_weight`,
`_up_projection_backward_act`, `db1_kernel`, `_up_projection_backward_weight`,
`_token_broadcast_backward`; blockwise MoE backward page, returned gradients):

    dA_raw = dout_t @ W2_e^T                ds[t,k] = <dA_raw, a> + <dout_t, b2_e>
    dA     = s * dA_raw                     a'      = s * a
    dgate  = dA * up * SiLU'(gate)          dup     = dA * SiLU(gate)        dh = [dgate | dup]
    dW2_e  = sum_rows a'^T dout_t           db2_e   = sum_rows s * dout_t
    dW1_e  = sum_rows x_t^T dh              db1_e   = sum_rows dh
    dx_t   = sum_k dh @ W1_e^T

The gate/up pre-activation h of each (t, k) is an input (the forward's checkpoint), always as
[gate | up].  Variants: `activation` "geglu" replaces SiLU by GELU (exact normal CDF); `gate_up`
"interleaved" puts gate_i and up_i in columns 2i, 2i+1 of W1_e (and of dh, dW1_e, db1_e).
"""
from __future__ import annotations

import numpy as np

from . import mxfp8 as mx


def _f64(a):
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a, dtype=np.float64)


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


def dsilu(z):
    sg = sigmoid(z)
    return sg * (1.0 + z * (1.0 - sg))


def gelu(z):
    """GELU(z) = z * Phi(z) with the exact normal CDF (the GeGLU activation of sonic-moe's
    `activation_type` "geglu"; the page names the activation but prints no formula)."""
    from scipy.special import erf
    return 0.5 * z * (1.0 + erf(z / np.sqrt(2.0)))


def dgelu(z):
    from scipy.special import erf
    return 0.5 * (1.0 + erf(z / np.sqrt(2.0))) + z * np.exp(-0.5 * z * z) / np.sqrt(2.0 * np.pi)


ACTIVATIONS = {"swiglu": (silu, dsilu), "geglu": (gelu, dgelu)}


def gate_up_columns(I, layout="concat"):
    """Columns of W1_e (and of dh, dW1_e, db1_e) holding gate_i and up_i: concat (gate block then up
    block) or interleaved (gate_i at 2i, up_i at 2i+1; sonic-moe's interleaved gate/up layout that
    its db1 kernel remaps to concat)."""
    i = np.arange(I)
    if layout == "concat":
        return i, I + i
    if layout == "interleaved":
        return 2 * i, 2 * i + 1
    raise ValueError(layout)


def rows_of_expert(ids: np.ndarray, e: int):
    """(t, k) of every row routed to expert e, in ascending flat order t*K + k."""
    flat = np.nonzero(np.asarray(ids).reshape(-1) == e)[0]
    K = ids.shape[1]
    return flat // K, flat % K


def moe_forward(x, W1, b1, W2, b2, s, ids, activation="swiglu", gate_up="concat"):
    """out [T,H] and the pre-activations h [T,K,2I] as [gate | up] whatever W1's layout (used by the
    pins, never by the GPU path)."""
    x, W1, W2, s = _f64(x), _f64(W1), _f64(W2), _f64(s)
    b1, b2 = _f64(b1), _f64(b2)
    ids = np.asarray(ids)
    T, H = x.shape
    E, _, I2 = W1.shape
    I = I2 // 2
    K = ids.shape[1]
    out = np.zeros((T, H))
    h = np.zeros((T, K, I2))
    for e in range(E):
        t, k = rows_of_expert(ids, e)
        if t.size == 0:
            continue
        gc, uc = gate_up_columns(I, gate_up)
        he = x[t] @ W1[e] + (b1[e] if b1 is not None else 0.0)
        he = np.concatenate([he[:, gc], he[:, uc]], axis=1)
        a = ACTIVATIONS[activation][0](he[:, :I]) * he[:, I:]
        y = a @ W2[e] + (b2[e] if b2 is not None else 0.0)
        np.add.at(out, t, s[t, k][:, None] * y)
        h[t, k] = he
    return out, h


def recompute_h(x, W1, ids, b1=None, mxfp8=False, fp8_act=mx.E5M2, fp8_w=mx.E4M3):
    """Gate/up pre-activations recomputed from the layer input, h[t,k] = x_t @ W1_e + b1_e, stored in
    bfloat16 (the checkpoint's dtype).  With mxfp8 both operands are quantised along H (the
    contraction of this GEMM) first: x rows with fp8_act, W1_e columns with fp8_w."""
    x, b1 = _f64(x), _f64(b1)
    ids = np.asarray(ids)
    T, H = x.shape
    E, _, I2 = W1.shape
    K = ids.shape[1]
    h = np.zeros((T, K, I2))
    for e in range(E):
        t, k = rows_of_expert(ids, e)
        if t.size == 0:
            continue
        W1e = _f64(W1[e])
        xe = x[t]
        if mxfp8:
            xe = mx.mx_roundtrip(xe, fp8_act, 1)
            W1e = mx.mx_roundtrip(W1e, fp8_w, 0)
        h[t, k] = _to_bf16(xe @ W1e + (b1[e] if b1 is not None else 0.0))
    return h


def ds_masked(ds, ids, E):
    """[BW] `expert_affinities_masked_grad` [T*E]: the score gradient laid out over all E experts of
    each token, entry t*E + e = sum of ds[t,k] over the slots k with ids[t,k] = e (the derivative of
    the loss by the token's affinity for e when those slots share it), zero for experts the token
    did not select.  Ids outside [0, E) contribute nothing."""
    ds = _f64(ds)
    ids = np.asarray(ids)
    T, K = ids.shape
    out = np.zeros((T, E))
    for t in range(T):
        for k in range(K):
            if 0 <= ids[t, k] < E:
                out[t, ids[t, k]] += ds[t, k]
    return out.reshape(T * E)


def valid_token_ids(ids, num_valid):
    """Routing of a problem whose leading num_valid tokens hold real rows ([BW] `num_valid_tokens`):
    the slots of later tokens become unused (-1); num_valid <= 0 routes no token, above T all."""
    ids = np.array(ids, copy=True)
    n = max(0, min(int(num_valid), ids.shape[0]))
    ids[n:] = -1
    return ids


def moe_backward(x, dout, W1, W2, s, ids, h, b2=None, with_bias=False, activation="swiglu", gate_up="concat",
                 affinity=1, inter=None, sdout=None, gate_act=None):
    """All gradients of the MoE layer in float64 (the BF16 path's reference).

    x, dout [T,H]; W1 [E,H,2I]; W2 [E,I,H]; s [T,K]; ids [T,K]; h [T,K,2I] ([gate | up]); b2 [E,H]
    or None.  Returns dict(dx [T,H], dW1 [E,H,2I], dW2 [E,I,H], ds [T,K], db1 [E,2I], db2 [E,H]);
    db1/db2 are None unless with_bias.  dW1 and db1 follow W1's gate/up layout.

    Forward values saved by the caller ([BW] optional checkpoints) replace recomputed ones in the
    dW_down product dW2_e = sum a'^T (s dout) with the affinity on I (affinity=1) or H (0):
      inter [T,K,I]  the factor that carries the activation: s*a on I, a on H
                     (`scaled_intermediate_checkpoint_T` / `intermediate_checkpoint_T`)
      sdout [T,K,H]  s*dout on H (`down_proj_act_checkpoint`), also summed into db2
    and `gate_act` [T,K,I] (`gate_act_checkpoint_T`, a saved act(gate)) replaces the recomputed
    act(gate) wherever the activation's value enters: a = act(gate)*up (ds, the dW_down factor) and
    dup = dA*act(gate); act'(gate) in dgate still comes from the pre-activation.
    """
    x, dout, s, h = map(_f64, (x, dout, s, h))
    b2 = _f64(b2)
    ids = np.asarray(ids)
    T, H = x.shape
    E, _, I2 = W1.shape
    I = I2 // 2
    K = ids.shape[1]
    dx = np.zeros((T, H))
    ds = np.zeros((T, K))
    dW1 = np.zeros((E, H, I2))
    dW2 = np.zeros((E, I, H))
    db1 = np.zeros((E, I2)) if with_bias else None
    db2 = np.zeros((E, H)) if with_bias else None
    act, dact = ACTIVATIONS[activation]
    gc, uc = gate_up_columns(I, gate_up)
    for e in range(E):
        t, k = rows_of_expert(ids, e)
        if t.size == 0:
            continue
        W1e, W2e = _f64(W1[e]), _f64(W2[e])
        g = dout[t]                                   # gathered upstream gradient rows
        gate, up = h[t, k, :I], h[t, k, I:]
        ag = act(gate) if gate_act is None else _f64(gate_act)[t, k]
        a = ag * up
        sr = s[t, k][:, None]
        dA_raw = g @ W2e.T
        ds[t, k] = np.sum(dA_raw * a, axis=1)
        if b2 is not None:
            ds[t, k] += g @ b2[e]
        dA = sr * dA_raw
        dh = np.zeros((t.size, I2))
        dh[:, gc] = dA * up * dact(gate)
        dh[:, uc] = dA * ag
        av = (sr * a if affinity == 1 else a) if inter is None else _f64(inter)[t, k]
        gv = (g if affinity == 1 else sr * g) if sdout is None or affinity == 1 else _f64(sdout)[t, k]
        dW2[e] = av.T @ gv
        dW1[e] = x[t].T @ dh
        if with_bias:
            db2[e] = np.sum(sr * g if sdout is None or affinity == 1 else gv, axis=0)
            db1[e] = np.sum(dh, axis=0)
        np.add.at(dx, t, dh @ W1e.T)
    return dict(dx=dx, dW1=dW1, dW2=dW2, ds=ds, db1=db1, db2=db2)


# ----------------------------------------------------------------------------------------------
# MXFP8 path
# ----------------------------------------------------------------------------------------------

def _to_f32(a):
    """Round float64 to the nearest float32 (where the kernel takes a quantisation decision)."""
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _to_bf16(a):
    """Round float64 to the nearest bfloat16 (round-to-nearest-even on the float32 value)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).to(torch.bfloat16).to(
        torch.float64).numpy()


def _col_roundtrip(v, fmt, quant):
    """Quantise along rows (axis 0) in groups of 32 consecutive rows; zero-pad the last group."""
    n = v.shape[0]
    npad = -(-n // 32) * 32
    if npad != n:
        v = np.concatenate([v, np.zeros((npad - n,) + v.shape[1:])], axis=0)
    return quant(v, fmt, 0)[:n]


def moe_backward_mxfp8(x, dout, W1, W2, s, ids, h, affinity=1, fp8_act=mx.E5M2, fp8_w=mx.E4M3,
                       b2=None, with_bias=False, experts=None, tokens=None, quant=None, activation="swiglu",
                       gate_up="concat", inter=None, sdout=None, gate_act=None):
    """MoE backward with every GEMM operand MXFP8-quantised along its contraction dimension.

    Quantisation points (reading of the MXFP8 blockwise backward page; weights pre-quantised,
    activations quantised after the per-expert gather):
      G1  dA_raw  = Q_H(dout_g) @ Q_H(W2_e)^T                 groups along H
      G2  dx_exp  = Q_2I(dh) @ Q_2I(W1_e)^T, stored BF16      groups along 2I
      G3  dW2_e   = Q_tok(a')^T @ Q_tok(dout_g)    (affinity on I, a' = s*a)
                  = Q_tok(a)^T  @ Q_tok(s*dout_g)  (affinity on H)
      G4  dW1_e   = Q_tok(x_g)^T @ Q_tok(dh)                  groups of 32 grouped rows
    Activation-side operands use fp8_act, weights fp8_w.  dh, a' and s*dout are rounded to float32
    before their quantisation, as the kernel quantises float32 values.  ds, db1 and db2 use the
    unquantised epilogue values.  `experts` limits dW1/dW2/db1/db2 to those experts, `tokens`
    limits dx/ds to those tokens (both default to all).  `quant(v, fmt, axis)` defaults to the
    MX round trip; tests substitute the identity to check the wiring.  dh, W1_e, dW1 and db1 are in
    W1's gate/up layout, so the 32-column groups of Q_2I follow that layout.  `inter` and `sdout`
    replace the dW_down factors and `gate_act` the activation's value, as in moe_backward (saved
    forward values; quantised the same way).
    """
    quant = quant or mx.mx_roundtrip
    x, dout, s, h = map(_f64, (x, dout, s, h))
    b2 = _f64(b2)
    ids = np.asarray(ids)
    T, H = x.shape
    E, _, I2 = W1.shape
    I = I2 // 2
    K = ids.shape[1]
    expert_set = range(E) if experts is None else experts
    token_mask = np.ones(T, bool)
    if tokens is not None:
        token_mask[:] = False
        token_mask[np.asarray(tokens, dtype=np.int64)] = True
    dx = np.zeros((T, H))
    ds = np.zeros((T, K))
    dW1 = np.zeros((E, H, I2))
    dW2 = np.zeros((E, I, H))
    db1 = np.zeros((E, I2)) if with_bias else None
    db2 = np.zeros((E, H)) if with_bias else None
    want_w = set(expert_set)
    act, dact = ACTIVATIONS[activation]
    gc, uc = gate_up_columns(I, gate_up)
    for e in range(E):
        t, k = rows_of_expert(ids, e)
        if t.size == 0:
            continue
        need_w = e in want_w
        sel = np.ones(t.size, bool) if need_w else token_mask[t]
        if not sel.any():
            continue
        t, k = t[sel], k[sel]            # need_w keeps every row, so column groups stay intact
        W2q = quant(_f64(W2[e]), fp8_w, 1)     # [I,H] groups along H
        W1q = quant(_f64(W1[e]), fp8_w, 1)     # [H,2I] groups along 2I
        g = dout[t]
        gq = quant(g, fp8_act, 1)
        gate, up = h[t, k, :I], h[t, k, I:]
        ag = act(gate) if gate_act is None else _f64(gate_act)[t, k]
        a = ag * up
        sr = s[t, k][:, None]
        dA_raw = gq @ W2q.T
        dsv = np.sum(dA_raw * a, axis=1)
        if b2 is not None:
            dsv = dsv + g @ b2[e]
        dA = sr * dA_raw
        dh = np.zeros((t.size, I2))
        dh[:, gc] = dA * up * dact(gate)
        dh[:, uc] = dA * ag
        dh = _to_f32(dh)
        tm = token_mask[t]
        ds[t[tm], k[tm]] = dsv[tm]
        if tm.any():   # dx_expanded only for rows whose token is wanted
            dx_exp = _to_bf16(quant(dh[tm], fp8_act, 1) @ W1q.T)
            np.add.at(dx, t[tm], dx_exp)
        if need_w:
            av = _to_f32(sr * a if affinity == 1 else a) if inter is None else _f64(inter)[t, k]
            if affinity == 1:
                dW2[e] = _col_roundtrip(av, fp8_act, quant).T @ _col_roundtrip(g, fp8_act, quant)
            else:
                gv = _to_f32(sr * g) if sdout is None else _f64(sdout)[t, k]
                dW2[e] = _col_roundtrip(av, fp8_act, quant).T @ _col_roundtrip(gv, fp8_act, quant)
            dW1[e] = _col_roundtrip(x[t], fp8_act, quant).T @ _col_roundtrip(dh, fp8_act, quant)
            if with_bias:
                db2[e] = np.sum(sr * g, axis=0)
                db1[e] = np.sum(dh, axis=0)
    return dict(dx=dx, dW1=dW1, dW2=dW2, ds=ds, db1=db1, db2=db2)


def moe_backward_sampled(x, dout, W1, W2, s, ids, h, experts, tokens, b2=None, with_bias=False):
    """BF16-path backward restricted to dW/db of `experts` and dx/ds of `tokens` (same formulas;
    SwiGLU, concatenated gate/up)."""
    x, dout, W1, W2, s, h = map(_f64, (x, dout, W1, W2, s, h))
    b2 = _f64(b2)
    ids = np.asarray(ids)
    T, H = x.shape
    E, _, I2 = W1.shape
    I = I2 // 2
    K = ids.shape[1]
    out = dict(dx={}, ds={}, dW1={}, dW2={}, db1={}, db2={})
    for e in experts:
        t, k = rows_of_expert(ids, e)
        g = dout[t]
        gate, up = h[t, k, :I], h[t, k, I:]
        a = silu(gate) * up
        sr = s[t, k][:, None]
        dA = sr * (g @ W2[e].T)
        dh = np.concatenate([dA * up * dsilu(gate), dA * silu(gate)], axis=1)
        out["dW2"][e] = (sr * a).T @ g
        out["dW1"][e] = x[t].T @ dh
        if with_bias:
            out["db2"][e] = np.sum(sr * g, axis=0)
            out["db1"][e] = np.sum(dh, axis=0)
    for tt in tokens:
        dxt = np.zeros(H)
        dst = np.zeros(K)
        for kk in range(K):
            e = int(ids[tt, kk])
            gate, up = h[tt, kk, :I], h[tt, kk, I:]
            a = silu(gate) * up
            dA_raw = dout[tt] @ W2[e].T
            dst[kk] = dA_raw @ a + (dout[tt] @ b2[e] if b2 is not None else 0.0)
            dA = s[tt, kk] * dA_raw
            dh = np.concatenate([dA * up * dsilu(gate), dA * silu(gate)])
            dxt += dh @ W1[e].T
        out["dx"][tt] = dxt
        out["ds"][tt] = dst
    return out
