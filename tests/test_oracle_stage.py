"""Pins for the numerics oracle (CPU only).

Each pin ties ``oracle.stage`` to something other than itself:
* central finite differences of the scalar loss sum(y * G), so dY = G;
* torch.autograd in float64 on a forward written here independently;
* "Zero-Bubble Pipeline Parallelism Guide for LLMs", section "2. Convergence
  and Numerical Stability": split B + W is the same arithmetic as the fused
  backward (checked against a separately written fused backward);
* every op except the weight contractions works per token, so the weight
  gradient summed over microbatches equals the weight gradient of the
  concatenated batch;
* closed-form special cases of the forward.
The last test plants mistakes in the oracle (on the CPU) and checks that one
of these pins catches each of them.
"""
import numpy as np
import pytest
import torch

from oracle import stage as S

SHAPES = {
    "transformer": dict(kind="transformer", n_layers=2, hidden=8, ffn=16, n_heads=2,
                        n_kv_heads=1, head_dim=4, eps=1e-5),
    "gqa4": dict(kind="transformer", n_layers=1, hidden=16, ffn=8, n_heads=4,
                 n_kv_heads=1, head_dim=4, eps=1e-5),
    "mlp": dict(kind="mlp", n_layers=2, hidden=8, ffn=16, n_heads=0, n_kv_heads=0,
                head_dim=0, eps=1e-5),
    "linear": dict(kind="linear", n_layers=1, hidden=8, ffn=12, n_heads=0, n_kv_heads=0,
                   head_dim=0, eps=1e-5),
    # causal softmax attention: sequences of 3 tokens (the 4- to 6-token cases hold a
    # whole sequence and a shorter last one), 4 query heads on 2 kv heads
    "causal": dict(kind="transformer", n_layers=2, hidden=16, ffn=8, n_heads=4, n_kv_heads=2,
                   head_dim=4, eps=1e-5, attention="causal", seq_len=3),
    "causal_one_seq": dict(kind="transformer", n_layers=1, hidden=8, ffn=8, n_heads=2, n_kv_heads=1,
                           head_dim=4, eps=1e-5, attention="causal", seq_len=0),
}


def make_case(shp, tokens=4, seed=1, wstd=0.3):
    rng = np.random.default_rng(seed)
    params = []
    for _ in range(shp["n_layers"]):
        sh = S.weight_shapes(shp["kind"], shp["hidden"], shp["ffn"], shp["n_heads"],
                             shp["n_kv_heads"], shp["head_dim"])
        prm = {}
        for k, s in sh.items():
            if k.startswith("gamma"):
                prm[k] = 1.0 + 0.1 * rng.standard_normal(s)
            else:
                prm[k] = wstd * rng.standard_normal(s)
        params.append(prm)
    x = rng.standard_normal((tokens, shp["hidden"]))
    out = shp["ffn"] if shp["kind"] == "linear" else shp["hidden"]
    G = rng.standard_normal((tokens, out))
    return params, x, G


def split_grads(params, x, G, shp):
    _, saved = S.stage_forward(x, params, shp)
    dx, kept = S.stage_backward_input(G, params, saved, shp)
    acc = S.zero_grads(params)
    S.stage_backward_weight(acc, saved, kept, shp)
    return dx, acc


def loss(params, x, G, shp):
    y, _ = S.stage_forward(x, params, shp)
    return float(np.sum(y * G))


def fd_max_rel_err(params, x, G, shp, step=1e-6):
    """Largest relative error (per gradient array) of the oracle's split grads vs central differences."""
    dx, acc = split_grads(params, x, G, shp)
    worst = 0.0

    def check(arr, analytic):
        nonlocal worst
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + step
            lp = loss(params, x, G, shp)
            arr[idx] = old - step
            lm = loss(params, x, G, shp)
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * step)
        err = np.max(np.abs(num - analytic)) / max(1e-12, np.max(np.abs(num)))
        worst = max(worst, err)

    check(x, dx)
    for li, prm in enumerate(params):
        for k in prm:
            check(prm[k], acc[li][k])
    return worst


# ----------------------------------------------------------------------------
# torch.autograd in float64, forward written independently
# ----------------------------------------------------------------------------


def torch_forward(x, params, shp):
    def norm(v, g):
        return g * v * torch.rsqrt((v * v).mean(dim=1, keepdim=True) + shp["eps"])

    for prm in params:
        if shp["kind"] == "linear":
            x = x @ prm["w"].t()
            continue
        if shp["kind"] == "transformer":
            nh, nkv, d = shp["n_heads"], shp["n_kv_heads"], shp["head_dim"]
            qkv = norm(x, prm["gamma1"]) @ prm["w_qkv"].t()
            q, k, v = torch.split(qkv, [nh * d, nkv * d, nkv * d], dim=1)
            t = x.shape[0]
            rep = nh // nkv
            kk = k.reshape(t, nkv, 1, d).expand(t, nkv, rep, d).reshape(t, nh * d)
            vv = v.reshape(t, nkv, 1, d).expand(t, nkv, rep, d).reshape(t, nh * d)
            if shp.get("attention") == "causal":
                a = torch_causal_attention(q, kk, vv, nh, d, shp["seq_len"])
            else:
                a = q + kk + vv
            h = x + a @ prm["w_o"].t()
        else:
            h = x
        gate, up = torch.chunk(norm(h, prm["gamma2"]) @ prm["w_gu"].t(), 2, dim=1)
        x = h + (torch.nn.functional.silu(gate) * up) @ prm["w_down"].t()
    return x


def torch_causal_attention(q, k, v, nh, d, seq_len):
    """Per head and per sequence: masked scores, softmax, weighted values (k, v already
    repeated to one per query head)."""
    t = q.shape[0]
    step = seq_len or t
    outs = []
    for s0 in range(0, t, step):
        s1 = min(t, s0 + step)
        n = s1 - s0
        qh = q[s0:s1].reshape(n, nh, d).transpose(0, 1)
        kh = k[s0:s1].reshape(n, nh, d).transpose(0, 1)
        vh = v[s0:s1].reshape(n, nh, d).transpose(0, 1)
        scores = qh @ kh.transpose(1, 2) / d ** 0.5
        future = torch.triu(torch.ones(n, n, dtype=torch.bool), diagonal=1)
        w = torch.softmax(scores.masked_fill(future, float("-inf")), dim=-1)
        outs.append((w @ vh).transpose(0, 1).reshape(n, nh * d))
    return torch.cat(outs)


def autograd_grads(params, x, G, shp):
    tp = [{k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in prm.items()}
          for prm in params]
    tx = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    y = torch_forward(tx, tp, shp)
    (y * torch.tensor(G)).sum().backward()
    return y.detach().numpy(), tx.grad.numpy(), [{k: v.grad.numpy() for k, v in prm.items()} for prm in tp]


def autograd_max_rel_err(params, x, G, shp):
    y_t, dx_t, g_t = autograd_grads(params, x, G, shp)
    y, _ = S.stage_forward(x, params, shp)
    dx, acc = split_grads(params, x, G, shp)
    errs = [np.max(np.abs(y - y_t)) / np.max(np.abs(y_t)),
            np.max(np.abs(dx - dx_t)) / np.max(np.abs(dx_t))]
    for li in range(len(params)):
        for k in params[li]:
            errs.append(np.max(np.abs(acc[li][k] - g_t[li][k])) / np.max(np.abs(g_t[li][k])))
    return max(errs)


def split_vs_fused_err(params, x, G, shp):
    _, saved = S.stage_forward(x, params, shp)
    dx_f, g_f = S.stage_backward_fused(G, params, saved, shp)
    dx, acc = split_grads(params, x, G, shp)
    errs = [np.max(np.abs(dx - dx_f)) / np.max(np.abs(dx_f))]
    for li in range(len(params)):
        for k in params[li]:
            errs.append(np.max(np.abs(acc[li][k] - g_f[li][k])) / np.max(np.abs(g_f[li][k])))
    return max(errs)


@pytest.mark.parametrize("name", list(SHAPES))
def test_finite_differences(name):
    shp = SHAPES[name]
    params, x, G = make_case(shp)
    assert fd_max_rel_err(params, x, G, shp) < 1e-6


@pytest.mark.parametrize("name", list(SHAPES))
def test_autograd_fp64(name):
    shp = SHAPES[name]
    params, x, G = make_case(shp, tokens=6, seed=2)
    assert autograd_max_rel_err(params, x, G, shp) < 1e-12


@pytest.mark.parametrize("name", list(SHAPES))
def test_split_equals_fused(name):
    shp = SHAPES[name]
    params, x, G = make_case(shp, tokens=5, seed=3)
    assert split_vs_fused_err(params, x, G, shp) < 1e-12


@pytest.mark.parametrize("name", ["transformer", "mlp", "linear", "causal"])
def test_concat_identity(name):
    """sum over microbatches of dW(mb) == dW(concatenation of the microbatches); with
    causal attention the microbatches hold whole sequences."""
    shp = SHAPES[name]
    params, _, _ = make_case(shp)
    rng = np.random.default_rng(7)
    out = shp["ffn"] if shp["kind"] == "linear" else shp["hidden"]
    sizes = (3, 6, 3) if shp.get("attention") == "causal" else (3, 5, 2)
    mbs = [(rng.standard_normal((t, shp["hidden"])), rng.standard_normal((t, out))) for t in sizes]
    st = S.StageOracle(params, shp)
    dxs = []
    for i, (x, g) in enumerate(mbs):
        st.forward(i, x)
    for i, (x, g) in enumerate(mbs):
        dxs.append(st.backward_input(i, g))
    for i in range(len(mbs)):
        st.backward_weight(i)
    xc = np.concatenate([m[0] for m in mbs])
    gc = np.concatenate([m[1] for m in mbs])
    dxc, accc = split_grads(params, xc, gc, shp)
    assert np.allclose(np.concatenate(dxs), dxc, rtol=1e-12, atol=1e-12)
    for li in range(len(params)):
        for k in params[li]:
            ref = accc[li][k]
            assert np.max(np.abs(st.grads[li][k] - ref)) <= 1e-12 * np.max(np.abs(ref))
    assert not st.saved and not st.kept  # W released every microbatch


def test_forward_closed_forms():
    # RMSNorm of a constant row c: r = 1 / sqrt(c^2 + eps), n = gamma * c * r
    eps = 1e-5
    x = np.full((2, 4), 3.0)
    g = np.array([1.0, 2.0, -1.0, 0.5])
    n, r = S.rmsnorm(x, g, eps)
    assert np.allclose(r, 1.0 / np.sqrt(9.0 + eps), rtol=1e-15)
    assert np.allclose(n, g * 3.0 / np.sqrt(9.0 + eps), rtol=1e-15)
    # silu(0) = 0, silu(z) -> z for large z, silu(-z) = silu(z) - z
    assert S.silu(np.array([0.0]))[0] == 0.0
    z = np.linspace(-4, 4, 9)
    assert np.allclose(S.silu(-z), S.silu(z) - z, rtol=1e-14, atol=1e-15)
    # stand-in with one head per kv head: a = q + k + v
    qkv = np.arange(24.0).reshape(2, 12)
    a = S.attention_standin(qkv, 2, 2, 2)
    assert np.array_equal(a, qkv[:, 0:4] + qkv[:, 4:8] + qkv[:, 8:12])
    # single linear with the guide's layout: y = x W^T
    w = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]])
    y, _ = S.layer_forward(np.array([[1.0, -1.0]]), {"w": w}, {"kind": "linear"})
    assert np.array_equal(y, [[-1.0, -1.0, -1.0]])


def test_causal_attention_special_cases():
    """Closed forms of the causal attention core, and the library's own attention routine."""
    rng = np.random.default_rng(3)
    t, nh, nkv, d = 7, 4, 2, 8
    qkv = rng.standard_normal((t, (nh + 2 * nkv) * d))
    q, k, v = S._heads(qkv, nh, nkv, d)
    # sequences of one token: each query sees only its own key, so a_h = v_j
    a = S.attention_causal(qkv, nh, nkv, d, 1).reshape(t, nh, d)
    for h in range(nh):
        assert np.allclose(a[:, h], v[:, h // 2], rtol=0, atol=1e-15)
    # q = 0: equal weights over the keys so far, so a is the running mean of v
    q0 = qkv.copy()
    q0[:, : nh * d] = 0.0
    a = S.attention_causal(q0, nh, nkv, d, 0).reshape(t, nh, d)
    run_mean = np.cumsum(v, axis=0) / np.arange(1, t + 1)[:, None, None]
    for h in range(nh):
        assert np.allclose(a[:, h], run_mean[:, h // 2], rtol=1e-14, atol=1e-14)
    # sequences of 3: the second sequence does not see the first
    a3 = S.attention_causal(qkv, nh, nkv, d, 3)
    assert np.allclose(a3[3:6], S.attention_causal(qkv[3:6], nh, nkv, d, 0), rtol=0, atol=1e-15)
    # torch's scaled_dot_product_attention (float64, causal) on the same heads
    tq = torch.tensor(q).transpose(0, 1)
    tk = torch.tensor(k).repeat_interleave(nh // nkv, dim=1).transpose(0, 1)
    tv = torch.tensor(v).repeat_interleave(nh // nkv, dim=1).transpose(0, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    got = S.attention_causal(qkv, nh, nkv, d, 0).reshape(t, nh, d)
    assert np.allclose(got, ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_linear_textbook_case():
    """Section "Core Innovation 1": dX = dY W (weights [out, in]) and dW = dY^T X.

    A 1x1x1 case worked by hand: y = w x, loss = g y, so dx = g w and dw = g x.
    """
    shp = {"kind": "linear"}
    params = [{"w": np.array([[3.0]])}]
    x = np.array([[2.0]])
    g = np.array([[5.0]])
    dx, acc = split_grads(params, x, g, shp)
    assert dx[0, 0] == 15.0 and acc[0]["w"][0, 0] == 10.0


# ----------------------------------------------------------------------------
# planted mistakes: every one must be caught by some pin above
# ----------------------------------------------------------------------------


def _bad_rms_sign(dn, x, r, gamma):
    xh = x * r[:, None]
    gdn = gamma[None, :] * dn
    return r[:, None] * (gdn + xh * np.mean(gdn * xh, axis=1)[:, None])


def _bad_swiglu(ds, g, u):
    sg = S.sigmoid(g)
    return ds * u * sg, ds * S.silu(g)


def _bad_standin_grad(da, nh, nkv, d):
    t = da.shape[0]
    dkv = da.reshape(t, nh, d)[:, :nkv, :].reshape(t, nkv * d)  # no group sum
    return np.concatenate([da, dkv, dkv], axis=1)


def _bad_causal_grad(da, qkv, nh, nkv, d, seq_len):
    """Drops the rowsum(dP * P) term of the softmax backward."""
    t = qkv.shape[0]
    q, k, v = S._heads(qkv, nh, nkv, d)
    da3 = da.reshape(t, nh, d)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s0, s1 in S.sequences(t, seq_len):
        for h in range(nh):
            j = h // (nh // nkv)
            p = S.causal_probs(q[s0:s1, h], k[s0:s1, j], 1 / np.sqrt(d))
            dv[s0:s1, j] += p.T @ da3[s0:s1, h]
            ds = p * (da3[s0:s1, h] @ v[s0:s1, j].T)
            dq[s0:s1, h] = ds @ k[s0:s1, j] / np.sqrt(d)
            dk[s0:s1, j] += ds.T @ q[s0:s1, h] / np.sqrt(d)
    return np.concatenate([dq.reshape(t, -1), dk.reshape(t, -1), dv.reshape(t, -1)], axis=1)


def _bad_causal_mask(q, k, scale):
    """Lets each query see the next key too."""
    n = q.shape[0]
    scores = scale * (q @ k.T)
    scores = np.where(np.tril(np.ones((n, n), dtype=bool), k=1), scores, -np.inf)
    e = np.exp(scores - scores.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def _bad_gamma_grad(dn, x, r):
    return np.sum(dn * x, axis=0)  # dropped r


def _bad_rmsnorm_fwd(x, gamma, eps):
    r = 1.0 / (np.sqrt(np.mean(x * x, axis=1)) + eps)
    return gamma[None, :] * x * r[:, None], r


MUTANTS = {
    "rms_sign": ("rmsnorm_input_grad", _bad_rms_sign),
    "swiglu_dropped_term": ("swiglu_grads", _bad_swiglu),
    "standin_no_group_sum": ("attention_standin_grad", _bad_standin_grad),
    "gamma_dropped_r": ("rmsnorm_gamma_grad", _bad_gamma_grad),
    "rmsnorm_eps_outside": ("rmsnorm", _bad_rmsnorm_fwd),
    "causal_no_rowsum": ("attention_causal_grad", _bad_causal_grad),
    "causal_mask_off_by_one": ("causal_probs", _bad_causal_mask),
}


@pytest.mark.parametrize("mutant", list(MUTANTS))
def test_planted_mistakes_are_caught(mutant, monkeypatch):
    name, fn = MUTANTS[mutant]
    monkeypatch.setattr(S, name, fn)
    shp = SHAPES["causal" if mutant.startswith("causal") else "gqa4"]
    params, x, G = make_case(shp, tokens=3, seed=5)
    caught = (autograd_max_rel_err(params, x, G, shp) > 1e-6
              or fd_max_rel_err(params, x, G, shp) > 1e-6)
    assert caught, mutant
