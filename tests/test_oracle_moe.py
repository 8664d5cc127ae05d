"""Pins for oracle.moe: finite differences, float64 torch autograd, the dense-MLP reduction,
token-permutation invariance, closed-form identities and the MXFP8 quantisation points."""
import numpy as np
import pytest
import torch

from oracle import moe as om
from oracle import mxfp8 as mx


def _problem(T=6, H=8, I=4, E=3, K=2, seed=0, bias=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    dout = rng.standard_normal((T, H))
    W1 = rng.standard_normal((E, H, 2 * I)) * 0.3
    W2 = rng.standard_normal((E, I, H)) * 0.3
    b1 = rng.standard_normal((E, 2 * I)) * 0.1 if bias else None
    b2 = rng.standard_normal((E, H)) * 0.1 if bias else None
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)])
    s = rng.random((T, K)) + 0.1
    s = s / s.sum(1, keepdims=True)
    return x, dout, W1, b1, W2, b2, s, ids


def _grads(x, dout, W1, b1, W2, b2, s, ids, activation="swiglu", gate_up="concat"):
    _, h = om.moe_forward(x, W1, b1, W2, b2, s, ids, activation, gate_up)
    return om.moe_backward(x, dout, W1, W2, s, ids, h, b2=b2, with_bias=b1 is not None, activation=activation,
                           gate_up=gate_up)


@pytest.mark.parametrize("activation,gate_up", [("swiglu", "concat"), ("geglu", "concat"),
                                                ("swiglu", "interleaved"), ("geglu", "interleaved")])
def test_finite_differences(activation, gate_up):
    x, dout, W1, b1, W2, b2, s, ids = _problem()
    g = _grads(x, dout, W1, b1, W2, b2, s, ids, activation, gate_up)

    def loss(x, W1, b1, W2, b2, s):
        out, _ = om.moe_forward(x, W1, b1, W2, b2, s, ids, activation, gate_up)
        return float(np.sum(out * dout))

    args = dict(x=x, W1=W1, b1=b1, W2=W2, b2=b2, s=s)
    names = dict(x="dx", W1="dW1", b1="db1", W2="dW2", b2="db2", s="ds")
    eps = 1e-6
    for name, arr in args.items():
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus = {k: v.copy() for k, v in args.items()}
            minus = {k: v.copy() for k, v in args.items()}
            plus[name][idx] += eps
            minus[name][idx] -= eps
            num[idx] = (loss(**plus) - loss(**minus)) / (2 * eps)
        ana = g[names[name]]
        rel = np.max(np.abs(num - ana)) / max(np.max(np.abs(ana)), 1e-30)
        assert rel < 1e-7, (name, rel)


def _torch_forward(x, W1, b1, W2, b2, s, ids, activation="swiglu", gate_up="concat"):
    """Loop-over-experts forward in torch float64 (differentiated by torch autograd).  Interleaved
    gate/up: gate_i in column 2i, up_i in 2i+1."""
    T, H = x.shape
    I = W1.shape[2] // 2
    act = torch.nn.functional.silu if activation == "swiglu" else torch.nn.functional.gelu
    out = torch.zeros(T, H, dtype=torch.float64)
    for e in range(W1.shape[0]):
        t, k = torch.nonzero(ids == e, as_tuple=True)
        if t.numel() == 0:
            continue
        h = x[t] @ W1[e] + (b1[e] if b1 is not None else 0)
        gate, up = (h[:, :I], h[:, I:]) if gate_up == "concat" else (h[:, 0::2], h[:, 1::2])
        a = act(gate) * up
        y = a @ W2[e] + (b2[e] if b2 is not None else 0)
        out = out.index_add(0, t, s[t, k][:, None] * y)
    return out


@pytest.mark.parametrize("bias", [False, True])
def test_torch_autograd_tiny_config_shapes(bias):
    T, H, I, E, K = 256, 128, 256, 4, 2
    x, dout, W1, b1, W2, b2, s, ids = _problem(T, H, I, E, K, seed=11, bias=bias)
    g = _grads(x, dout, W1, b1, W2, b2, s, ids)
    tt = {n: torch.tensor(v, requires_grad=True) for n, v in
          dict(x=x, W1=W1, W2=W2, s=s).items()}
    tb1 = torch.tensor(b1, requires_grad=True) if bias else None
    tb2 = torch.tensor(b2, requires_grad=True) if bias else None
    out = _torch_forward(tt["x"], tt["W1"], tb1, tt["W2"], tb2, tt["s"], torch.tensor(ids))
    (out * torch.tensor(dout)).sum().backward()
    pairs = [("dx", tt["x"]), ("dW1", tt["W1"]), ("dW2", tt["W2"]), ("ds", tt["s"])]
    if bias:
        pairs += [("db1", tb1), ("db2", tb2)]
    for name, t in pairs:
        ref = t.grad.numpy()
        err = np.linalg.norm(g[name] - ref) / np.linalg.norm(ref)
        assert err < 1e-12, (name, err)


@pytest.mark.parametrize("activation,gate_up", [("geglu", "concat"), ("swiglu", "interleaved"),
                                                ("geglu", "interleaved")])
def test_torch_autograd_variants(activation, gate_up):
    """GeGLU (torch's exact-erf GELU) and the interleaved gate/up layout against torch autograd."""
    T, H, I, E, K = 64, 32, 16, 3, 2
    x, dout, W1, b1, W2, b2, s, ids = _problem(T, H, I, E, K, seed=13, bias=True)
    g = _grads(x, dout, W1, b1, W2, b2, s, ids, activation, gate_up)
    tt = {n: torch.tensor(v, requires_grad=True) for n, v in dict(x=x, W1=W1, b1=b1, W2=W2, b2=b2, s=s).items()}
    out = _torch_forward(tt["x"], tt["W1"], tt["b1"], tt["W2"], tt["b2"], tt["s"], torch.tensor(ids), activation,
                         gate_up)
    (out * torch.tensor(dout)).sum().backward()
    for name, key in (("dx", "x"), ("dW1", "W1"), ("dW2", "W2"), ("ds", "s"), ("db1", "b1"), ("db2", "b2")):
        ref = tt[key].grad.numpy()
        err = np.linalg.norm(g[name] - ref) / np.linalg.norm(ref)
        assert err < 1e-12, (name, err)


def test_interleaved_layout_is_a_column_permutation():
    """The interleaved layout is the concat layout with W1's columns (and so dW1's, db1's) permuted."""
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=8, H=6, I=3, E=2, K=1, seed=14)
    perm = np.empty(6, dtype=int)
    perm[0::2], perm[1::2] = np.arange(3), 3 + np.arange(3)   # interleaved column j <- concat column perm[j]
    gi = _grads(x, dout, W1[:, :, perm], b1[:, perm], W2, b2, s, ids, "swiglu", "interleaved")
    gc = _grads(x, dout, W1, b1, W2, b2, s, ids, "swiglu", "concat")
    assert np.allclose(gi["dW1"], gc["dW1"][:, :, perm], rtol=0, atol=1e-13)
    assert np.allclose(gi["db1"], gc["db1"][:, perm], rtol=0, atol=1e-13)
    for name in ("dx", "dW2", "ds", "db2"):
        assert np.allclose(gi[name], gc[name], rtol=0, atol=1e-13), name


def test_dense_mlp_reduction():
    """E=1, K=1, s=1: the layer is a dense SwiGLU MLP; compare with autograd of that MLP."""
    rng = np.random.default_rng(2)
    T, H, I = 16, 12, 10
    x, dout = rng.standard_normal((T, H)), rng.standard_normal((T, H))
    W1 = rng.standard_normal((1, H, 2 * I)) * 0.3
    W2 = rng.standard_normal((1, I, H)) * 0.3
    ids = np.zeros((T, 1), dtype=np.int64)
    s = np.ones((T, 1))
    g = _grads(x, dout, W1, None, W2, None, s, ids)
    tx = torch.tensor(x, requires_grad=True)
    tg = torch.tensor(W1[0][:, :I], requires_grad=True)
    tu = torch.tensor(W1[0][:, I:], requires_grad=True)
    td = torch.tensor(W2[0], requires_grad=True)
    y = (torch.nn.functional.silu(tx @ tg) * (tx @ tu)) @ td
    (y * torch.tensor(dout)).sum().backward()
    assert np.allclose(g["dx"], tx.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(g["dW1"][0], np.concatenate([tg.grad.numpy(), tu.grad.numpy()], 1), rtol=1e-12, atol=1e-12)
    assert np.allclose(g["dW2"][0], td.grad.numpy(), rtol=1e-12, atol=1e-12)
    y_np = y.detach().numpy()
    assert np.allclose(g["ds"][:, 0], np.sum(dout * y_np, 1), rtol=1e-12, atol=1e-12)


def test_token_permutation_invariance():
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=20, H=8, I=6, E=4, K=2, seed=4)
    g = _grads(x, dout, W1, b1, W2, b2, s, ids)
    p = np.random.default_rng(9).permutation(20)
    gp = _grads(x[p], dout[p], W1, b1, W2, b2, s[p], ids[p])
    for n in ("dx", "ds"):
        assert np.allclose(gp[n], g[n][p], rtol=1e-12, atol=1e-12)
    for n in ("dW1", "dW2", "db1", "db2"):
        assert np.allclose(gp[n], g[n], rtol=1e-12, atol=1e-12)


def test_closed_form_identities():
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=30, H=10, I=6, E=5, K=3, seed=6)
    out, h = om.moe_forward(x, W1, b1, W2, b2, s, ids)
    g = om.moe_backward(x, dout, W1, W2, s, ids, h, b2=b2, with_bias=True)
    lhs = np.sum(dout * out)
    assert np.isclose(np.sum(s * g["ds"]), lhs, rtol=1e-12)
    assert np.isclose(np.sum(g["dW2"] * W2) + np.sum(g["db2"] * b2), lhs, rtol=1e-12)
    # <dx, x> = sum_r <dh_r, x_r W1_e> = sum_e <dW1_e, W1_e>
    assert np.isclose(np.sum(g["dx"] * x), np.sum(g["dW1"] * W1), rtol=1e-12)
    # renormalised scores: sum_e db2_e = sum_t dout_t
    assert np.allclose(g["db2"].sum(0), dout.sum(0), rtol=1e-12, atol=1e-12)


def test_linearity_in_scores():
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=12, seed=8)
    _, h = om.moe_forward(x, W1, b1, W2, b2, s, ids)
    g1 = om.moe_backward(x, dout, W1, W2, s, ids, h, b2=b2, with_bias=True)
    g3 = om.moe_backward(x, dout, W1, W2, 3 * s, ids, h, b2=b2, with_bias=True)
    for n in ("dx", "dW1", "dW2", "db1", "db2"):
        assert np.allclose(g3[n], 3 * g1[n], rtol=1e-12, atol=1e-12)
    assert np.allclose(g3["ds"], g1["ds"], rtol=1e-12, atol=1e-12)


def test_sampled_matches_full():
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=24, H=8, I=6, E=4, K=2, seed=12)
    _, h = om.moe_forward(x, W1, b1, W2, b2, s, ids)
    g = om.moe_backward(x, dout, W1, W2, s, ids, h, b2=b2, with_bias=True)
    sm = om.moe_backward_sampled(x, dout, W1, W2, s, ids, h, experts=[1, 3], tokens=[0, 5, 23],
                                 b2=b2, with_bias=True)
    for e in (1, 3):
        for n in ("dW1", "dW2", "db1", "db2"):
            assert np.allclose(sm[n][e], g[n][e], rtol=1e-12, atol=1e-12)
    for t in (0, 5, 23):
        assert np.allclose(sm["dx"][t], g["dx"][t], rtol=1e-12, atol=1e-12)
        assert np.allclose(sm["ds"][t], g["ds"][t], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# MXFP8 path
# ---------------------------------------------------------------------------------------------

def _identity(v, fmt, axis):
    return v


@pytest.mark.parametrize("affinity", [0, 1])
def test_mxfp8_wiring_without_quantisation(affinity):
    """With the quantiser replaced by the identity, the MXFP8 path is the plain backward up to
    the float32 / bfloat16 roundings of its stored intermediates."""
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=40, H=32, I=32, E=3, K=2, seed=13)
    _, h = om.moe_forward(x, W1, b1, W2, b2, s, ids)
    ref = om.moe_backward(x, dout, W1, W2, s, ids, h, b2=b2, with_bias=True)
    got = om.moe_backward_mxfp8(x, dout, W1, W2, s, ids, h, affinity=affinity, b2=b2,
                                with_bias=True, quant=_identity)
    for n, tol in (("dW1", 1e-6), ("dW2", 1e-6), ("ds", 1e-12), ("db1", 1e-6), ("db2", 1e-12),
                   ("dx", 4e-3)):
        err = np.linalg.norm(got[n] - ref[n]) / np.linalg.norm(ref[n])
        assert err < tol, (n, err)


def test_mxfp8_error_within_quantisation_bound():
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=64, H=64, I=64, E=2, K=2, seed=14, bias=False)
    _, h = om.moe_forward(x, W1, None, W2, None, s, ids)
    ref = om.moe_backward(x, dout, W1, W2, s, ids, h)
    got = om.moe_backward_mxfp8(x, dout, W1, W2, s, ids, h)
    for n in ("dx", "dW1", "dW2", "ds"):
        err = np.linalg.norm(got[n] - ref[n]) / np.linalg.norm(ref[n])
        assert 1e-3 < err < 0.15, (n, err)   # quantisation applied, and only quantisation error


def test_mxfp8_groups_follow_contraction_axes():
    """Scaling one token's dout row by 2^j must scale exactly that token's ds and dx by 2^j (G1
    and G2 group along H and 2I, per row); scaling one feature column of x by 2^j must scale
    exactly that row of every dW1_e by 2^j (G4 groups along tokens, per feature).  Grouping along
    the other axis would mix rows of different scale into one group and break the equalities."""
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=64, H=64, I=32, E=2, K=2, seed=15, bias=False)
    _, h = om.moe_forward(x, W1, None, W2, None, s, ids)
    base = om.moe_backward_mxfp8(x, dout, W1, W2, s, ids, h)
    j = np.where(np.arange(64) % 3 == 0, 7, np.where(np.arange(64) % 3 == 1, -6, 0))
    row = np.ldexp(1.0, j)[:, None]
    g = om.moe_backward_mxfp8(x, dout * row, W1, W2, s, ids, h)
    assert np.array_equal(g["ds"], base["ds"] * row)
    assert np.array_equal(g["dx"], base["dx"] * row)
    g = om.moe_backward_mxfp8(x * row.T, dout, W1, W2, s, ids, h)   # h kept: only G4 sees x
    assert np.array_equal(g["dW1"], base["dW1"] * row[None, :, :])
    assert np.array_equal(g["dW2"], base["dW2"]) and np.array_equal(g["ds"], base["ds"])


def test_mxfp8_restrictions_match_full():
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=64, H=32, I=32, E=3, K=2, seed=16, bias=False)
    _, h = om.moe_forward(x, W1, None, W2, None, s, ids)
    full = om.moe_backward_mxfp8(x, dout, W1, W2, s, ids, h)
    part = om.moe_backward_mxfp8(x, dout, W1, W2, s, ids, h, experts=[2], tokens=[3, 40])
    assert np.array_equal(part["dW1"][2], full["dW1"][2])
    assert np.array_equal(part["dW2"][2], full["dW2"][2])
    for t in (3, 40):
        assert np.allclose(part["dx"][t], full["dx"][t], rtol=0, atol=1e-12)
        assert np.array_equal(part["ds"][t], full["ds"][t])


@pytest.mark.parametrize("mxfp8", [False, True])
def test_subproblems_reproduce_full_problem(mxfp8):
    """oracle.sample: expert samples keep those experts' weight gradients, token samples keep those
    tokens' dx and ds, exactly."""
    from oracle import route_meta as orm
    from oracle import sample as osm
    rng = np.random.default_rng(17)
    T, H, I, E, K, B = 90, 64, 32, 5, 2, 128
    x = torch.from_numpy(rng.standard_normal((T, H))).to(torch.bfloat16)
    dout = torch.from_numpy(rng.standard_normal((T, H))).to(torch.bfloat16)
    W1 = torch.from_numpy(rng.standard_normal((E, H, 2 * I)) * 0.1).to(torch.bfloat16)
    W2 = torch.from_numpy(rng.standard_normal((E, I, H)) * 0.1).to(torch.bfloat16)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    s = rng.random((T, K))
    N = orm.num_blocks_bound(T, K, E, B)
    ckpt = torch.from_numpy(rng.standard_normal((N, 2, I, B))).to(torch.bfloat16)
    meta = orm.route_meta(ids, E, B)
    h = orm.checkpoint_rows(ckpt.double().numpy(), meta, T, K)
    run = (lambda xx, dd, w1, w2, ss, ii, hh: om.moe_backward_mxfp8(xx, dd, w1, w2, ss, ii, hh)) if mxfp8 else \
          (lambda xx, dd, w1, w2, ss, ii, hh: om.moe_backward(xx, dd, w1, w2, ss, ii, hh))
    full = run(x, dout, W1, W2, s, ids, h)
    sub = osm.subproblem(x, dout, W1, W2, s, ids, ckpt, B, experts=[1, 3])
    g = run(sub["x"], sub["dout"], sub["W1"], sub["W2"], sub["s"], sub["ids"], sub["h"])
    for j, e in enumerate(sub["experts"]):
        assert np.array_equal(g["dW1"][j], full["dW1"][e]) and np.array_equal(g["dW2"][j], full["dW2"][e])
    sub = osm.subproblem(x, dout, W1, W2, s, ids, ckpt, B, tokens=[0, 7, 44, 89])
    g = run(sub["x"], sub["dout"], sub["W1"], sub["W2"], sub["s"], sub["ids"], sub["h"])
    assert np.allclose(g["dx"], full["dx"][sub["tokens"]], rtol=0, atol=1e-12)
    assert np.array_equal(g["ds"], full["ds"][sub["tokens"]])


def test_recompute_h_is_the_forward_preactivation():
    """recompute_h equals the forward's h up to its bfloat16 storage, and with MXFP8 it quantises
    x along H (row groups) and W1 along H (column groups): power-of-two scaling of one token row
    scales exactly that row of h."""
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=20, H=64, I=32, E=3, K=2, seed=21)
    _, h = om.moe_forward(x, W1, b1, W2, b2, s, ids)
    r = om.recompute_h(x, W1, ids, b1=b1)
    assert np.max(np.abs(r - h)) <= np.max(np.abs(h)) * 2.0 ** -8
    rq = om.recompute_h(x, W1, ids, mxfp8=True)
    x2 = x.copy()
    x2[3] *= 2.0 ** 5
    rq2 = om.recompute_h(x2, W1, ids, mxfp8=True)
    assert np.array_equal(rq2[3], rq[3] * 2.0 ** 5) and np.array_equal(np.delete(rq2, 3, 0), np.delete(rq, 3, 0))
    r0 = om.recompute_h(x, W1, ids)
    err = np.linalg.norm(rq - r0) / np.linalg.norm(r0)
    assert 1e-3 < err < 0.15


def test_ds_masked_is_the_gradient_of_the_masked_affinities():
    """[T*E] affinity gradient: finite differences of <dout, out> by the affinity A[t,e] that every
    slot of token t routed to e carries (two slots of one token share an expert here); zero where
    no slot selects e."""
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=5, H=6, I=3, E=4, K=3, seed=31)
    ids[2] = [1, 1, 3]  # a repeated selection
    g = _grads(x, dout, W1, b1, W2, b2, s, ids)
    m = om.ds_masked(g["ds"], ids, 4).reshape(5, 4)
    eps = 1e-6
    for t in range(5):
        for e in range(4):
            sel = ids[t] == e
            sp, sm = s.copy(), s.copy()
            sp[t, sel] += eps
            sm[t, sel] -= eps
            fp = np.sum(dout * om.moe_forward(x, W1, b1, W2, b2, sp, ids)[0])
            fm = np.sum(dout * om.moe_forward(x, W1, b1, W2, b2, sm, ids)[0])
            assert abs((fp - fm) / (2 * eps) - m[t, e]) < 1e-7, (t, e)
            if not sel.any():
                assert m[t, e] == 0.0


def test_num_valid_tokens_equals_the_truncated_problem():
    """Routing only the leading n tokens gives the gradients of the n-token problem, with zero dx
    rows and ds entries for the others."""
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=9, H=8, I=4, E=3, K=2, seed=32)
    n = 5
    v = om.valid_token_ids(ids, n)
    full = _grads(x, dout, W1, b1, W2, b2, s, v)
    part = _grads(x[:n], dout[:n], W1, b1, W2, b2, s[:n], ids[:n])
    for name in ("dW1", "dW2", "db1", "db2"):
        assert np.allclose(full[name], part[name], rtol=0, atol=1e-12), name
    assert np.allclose(full["dx"][:n], part["dx"]) and np.all(full["dx"][n:] == 0)
    assert np.allclose(full["ds"][:n], part["ds"]) and np.all(full["ds"][n:] == 0)
    assert np.array_equal(om.valid_token_ids(ids, 0), np.full_like(ids, -1))
    assert np.array_equal(om.valid_token_ids(ids, 100), ids)


@pytest.mark.parametrize("affinity", [0, 1])
def test_saved_dw_down_factors_reproduce_the_recomputed_ones(affinity):
    """Passing the forward's own a (or s*a) and s*dout as saved factors changes nothing; a saved
    factor that differs only in its affinity placement still gives the same dW2 (a' dout = a (s dout))."""
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=7, H=6, I=3, E=3, K=2, seed=33)
    _, h = om.moe_forward(x, W1, b1, W2, b2, s, ids)
    ref = om.moe_backward(x, dout, W1, W2, s, ids, h, b2=b2, with_bias=True, affinity=affinity)
    a = om.silu(h[..., :3]) * h[..., 3:]
    inter = s[..., None] * a if affinity == 1 else a
    sdout = s[..., None] * dout[:, None, :]
    got = om.moe_backward(x, dout, W1, W2, s, ids, h, b2=b2, with_bias=True, affinity=affinity, inter=inter,
                          sdout=sdout)
    for name in ("dx", "dW1", "dW2", "ds", "db1", "db2"):
        assert np.allclose(got[name], ref[name], rtol=1e-13, atol=1e-13), name
    other = om.moe_backward(x, dout, W1, W2, s, ids, h, b2=b2, with_bias=True, affinity=1 - affinity)
    assert np.allclose(other["dW2"], ref["dW2"], rtol=1e-13, atol=1e-13)
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=40, H=64, I=32, E=3, K=2, seed=34)
    _, h = om.moe_forward(x, W1, b1, W2, b2, s, ids)
    a = om.silu(h[..., :32]) * h[..., 32:]
    inter = s[..., None] * a if affinity == 1 else a
    sdout = s[..., None] * dout[:, None, :]
    mq = om.moe_backward_mxfp8(x, dout, W1, W2, s, ids, h, affinity=affinity)
    mg = om.moe_backward_mxfp8(x, dout, W1, W2, s, ids, h, affinity=affinity, inter=om._to_f32(inter),
                               sdout=om._to_f32(sdout) if affinity == 0 else None)
    assert np.array_equal(mq["dW2"], mg["dW2"])


@pytest.mark.parametrize("activation,gate_up", [("swiglu", "concat"), ("geglu", "interleaved")])
def test_saved_gate_act_enters_only_through_the_activation_value(activation, gate_up):
    """A saved act(gate) equal to the recomputed one changes nothing (both precisions); scaled by c it
    moves exactly the terms that carry the activation's value: ds, dW2, the up columns of dW1 and
    db1 scale by c, the gate columns (act'(gate) from the pre-activation) do not move, and dx is
    affine in c with its c = 0 part the gate columns' contribution alone."""
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=9, H=6, I=4, E=3, K=2, seed=35)
    _, h = om.moe_forward(x, W1, b1, W2, None, s, ids, activation, gate_up)
    act = om.ACTIVATIONS[activation][0](h[..., :4])
    gc, uc = om.gate_up_columns(4, gate_up)
    kw = dict(with_bias=True, activation=activation, gate_up=gate_up)
    ref = om.moe_backward(x, dout, W1, W2, s, ids, h, **kw)
    same = om.moe_backward(x, dout, W1, W2, s, ids, h, gate_act=act, **kw)
    for name in ("dx", "dW1", "dW2", "ds", "db1"):
        assert np.array_equal(same[name], ref[name]), name
    by = {c: om.moe_backward(x, dout, W1, W2, s, ids, h, gate_act=c * act, **kw) for c in (0.0, 2.0, 3.0)}
    assert np.all(by[0.0]["ds"] == 0) and np.all(by[0.0]["dW2"] == 0)
    assert np.all(by[0.0]["dW1"][:, :, uc] == 0) and np.all(by[0.0]["db1"][:, uc] == 0)
    for c in (0.0, 2.0, 3.0):
        g = by[c]
        assert np.allclose(g["ds"], c * ref["ds"], rtol=1e-12, atol=1e-14)
        assert np.allclose(g["dW2"], c * ref["dW2"], rtol=1e-12, atol=1e-14)
        assert np.allclose(g["dW1"][:, :, uc], c * ref["dW1"][:, :, uc], rtol=1e-12, atol=1e-14)
        assert np.allclose(g["db1"][:, uc], c * ref["db1"][:, uc], rtol=1e-12, atol=1e-14)
        assert np.array_equal(g["dW1"][:, :, gc], ref["dW1"][:, :, gc])
        assert np.allclose(g["dx"], by[0.0]["dx"] + c * (ref["dx"] - by[0.0]["dx"]), rtol=1e-12, atol=1e-13)
    # the gate columns' dx part, written out: (dA up act'(gate)) W1_gate^T summed over the slots
    dact = om.ACTIVATIONS[activation][1]
    dxg = np.zeros_like(x)
    for t in range(x.shape[0]):
        for k in range(ids.shape[1]):
            e = ids[t, k]
            dA = s[t, k] * (dout[t] @ W2[e].T)
            dxg[t] += (dA * h[t, k, 4:] * dact(h[t, k, :4])) @ W1[e][:, gc].T
    assert np.allclose(by[0.0]["dx"], dxg, rtol=1e-12, atol=1e-13)
    # MXFP8: the recomputed act in float64 as the saved value reproduces the quantised path exactly
    x, dout, W1, b1, W2, b2, s, ids = _problem(T=40, H=64, I=32, E=3, K=2, seed=36)
    _, h = om.moe_forward(x, W1, b1, W2, None, s, ids, activation, gate_up)
    act = om.ACTIVATIONS[activation][0](h[..., :32])
    mq = om.moe_backward_mxfp8(x, dout, W1, W2, s, ids, h, activation=activation, gate_up=gate_up)
    mg = om.moe_backward_mxfp8(x, dout, W1, W2, s, ids, h, activation=activation, gate_up=gate_up, gate_act=act)
    for name in ("dx", "dW1", "dW2", "ds"):
        assert np.array_equal(mq[name], mg[name]), name


@pytest.mark.parametrize("mxfp8", [False, True])
def test_feature_slice_reproduces_full_weight_gradients(mxfp8):
    """oracle.sample features mode: one expert with all its rows and a range of 32 intermediate
    features gives that expert's dW1 columns (gate and up) and dW2 rows of those features, and its
    db1 columns and db2, as the full problem does; the MXFP8 problem is run with the torch-cast round
    trip the full-size tests use, which must give the same values as the default one."""
    from oracle import mxfp8 as mxq
    from oracle import route_meta as orm
    from oracle import sample as osm
    rng = np.random.default_rng(23)
    T, H, I, E, K, B = 200, 64, 96, 4, 2, 128
    x = torch.from_numpy(rng.standard_normal((T, H))).to(torch.bfloat16)
    dout = torch.from_numpy(rng.standard_normal((T, H))).to(torch.bfloat16)
    W1 = torch.from_numpy(rng.standard_normal((E, H, 2 * I)) * 0.1).to(torch.bfloat16)
    W2 = torch.from_numpy(rng.standard_normal((E, I, H)) * 0.1).to(torch.bfloat16)
    b2 = torch.from_numpy(rng.standard_normal((E, H)) * 0.01).to(torch.bfloat16)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    ids[:150, 0] = 2                                   # expert 2 hot: several 32-row token groups
    ids[:150, 1] = np.where(ids[:150, 1] == 2, 0, ids[:150, 1])
    s = rng.random((T, K))
    N = orm.num_blocks_bound(T, K, E, B)
    ckpt = torch.from_numpy(rng.standard_normal((N, 2, I, B))).to(torch.bfloat16)
    meta = orm.route_meta(ids, E, B)
    h = orm.checkpoint_rows(ckpt.double().numpy(), meta, T, K)
    if mxfp8:
        full = om.moe_backward_mxfp8(x, dout, W1, W2, s, ids, h)
    else:
        full = om.moe_backward(x, dout, W1, W2, s, ids, h, b2=b2, with_bias=True)
    for e in (2, 1):
        sub = osm.subproblem(x, dout, W1, W2, s, ids, ckpt, B, experts=[e], features=(32, 32), b2=b2)
        cols = sub["columns"]
        assert list(cols[:32]) == list(range(32, 64)) and list(cols[32:]) == list(range(I + 32, I + 64))
        if mxfp8:
            g = om.moe_backward_mxfp8(sub["x"], sub["dout"], sub["W1"], sub["W2"], sub["s"], sub["ids"], sub["h"],
                                      tokens=[], quant=mxq.mx_roundtrip_torch)
        else:
            g = om.moe_backward(sub["x"], sub["dout"], sub["W1"], sub["W2"], sub["s"], sub["ids"], sub["h"],
                                b2=sub["b2"], with_bias=True)
            assert np.allclose(g["db1"][0], full["db1"][e][cols], rtol=1e-12, atol=1e-12)
            assert np.allclose(g["db2"][0], full["db2"][e], rtol=1e-12, atol=1e-12)
        assert np.allclose(g["dW1"][0], full["dW1"][e][:, cols], rtol=1e-12, atol=1e-12)
        assert np.allclose(g["dW2"][0], full["dW2"][e][32:64], rtol=1e-12, atol=1e-12)
        assert not np.allclose(g["dW1"][0], full["dW1"][e][:, :64])   # the slice is not the leading one
