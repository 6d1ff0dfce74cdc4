"""Oracle: one pipeline stage's forward pass and its split backward, numpy float64.

TEST INFRASTRUCTURE (see the package docstring): plain, slow, no blocking,
no fusion, no rounding.  Inputs are the exact bf16 values the GPU side gets,
already widened to float64 by the caller.

The method ("Zero-Bubble Pipeline Parallelism Guide for LLMs", section
"Core Innovation 1: Mathematical Decomposition of the Backward Pass") splits
the backward of every linear Y = X W into
  B  (input gradient, on the critical path):  dX = dY W^T
  W  (weight gradient, deferrable):           dW = X^T dY
With the weight stored [out, in] and y = x W^T (section "Step-by-Step
Implementation") these read dX = dY W and dW = dY^T X.  Section
"2. Convergence and Numerical Stability" states that B + W is the same
arithmetic as the usual fused backward, so the oracle is the plain gradient of
the stage's forward, split into the part that feeds dX and the part that feeds
dW.

Readings where the pages are silent (the pages show a single linear only):
* Layer kinds.  "linear": y = x W^T (the guide's listing itself).
  "mlp": h = x; n2 = RMSNorm(h; g2); [g|u] = n2 W_gu^T; s = silu(g) * u;
  y = h + s W_down^T.  "transformer": n1 = RMSNorm(x; g1);
  qkv = n1 W_qkv^T; a = A(qkv); h = x + a W_o^T; then the mlp part.
* RMSNorm(x; g) = g * x * r with r = (mean_j x_j^2 + eps)^(-1/2) per token.
* W_gu = [W_gate; W_up]: gate rows first.
* A is the attention core, in one of two forms (``shp["attention"]``):
  - "standin" (the default): a weight-free stand-in; head h of the output is
    q_h + k_j + v_j with j = floor(h / (n_heads / n_kv_heads)) (a
    grouped-query broadcast sum).  It is linear and per token, so every
    identity the tests use still holds.
  - "causal": softmax attention with a causal mask and grouped K/V heads,
    a_h = softmax(q_h k_j^T / sqrt(head_dim), keys <= query) v_j, over
    independent sequences of ``shp["seq_len"]`` consecutive tokens of the
    microbatch (0: the whole microbatch is one sequence; a last, shorter
    sequence takes the remaining tokens).  No position encoding is applied.
    Tokens mix only inside a sequence, so the concatenated-batch identity
    holds for microbatches made of whole sequences.
* Weight gradients accumulate: the caller's float64 accumulators start at zero
  and every W adds into them (section "Memory Management & Activation
  Rollback": gradients are accumulated in place in fixed buffers).
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# shapes
# ----------------------------------------------------------------------------

KINDS = ("linear", "mlp", "transformer")


def weight_shapes(kind, hidden, ffn, n_heads=0, n_kv_heads=0, head_dim=0):
    """Per-layer parameter shapes, weights [out, in].

    For kind "linear", ``hidden`` is in_features and ``ffn`` out_features.
    """
    if kind == "linear":
        return {"w": (ffn, hidden)}
    shapes = {"w_gu": (2 * ffn, hidden), "w_down": (hidden, ffn), "gamma2": (hidden,)}
    if kind == "transformer":
        qkv_out = (n_heads + 2 * n_kv_heads) * head_dim
        assert n_heads * head_dim == hidden, "attention width must equal hidden"
        shapes.update({"w_qkv": (qkv_out, hidden), "w_o": (hidden, hidden), "gamma1": (hidden,)})
    return shapes


# ----------------------------------------------------------------------------
# pieces of the forward pass and their exact derivatives
# ----------------------------------------------------------------------------


def rmsnorm(x, gamma, eps):
    """n = gamma * x * r, r = 1 / sqrt(mean(x^2) + eps) per row.  Returns (n, r)."""
    r = 1.0 / np.sqrt(np.mean(x * x, axis=1) + eps)
    return gamma[None, :] * x * r[:, None], r


def rmsnorm_input_grad(dn, x, r, gamma):
    """d(loss)/dx for n = RMSNorm(x; gamma), given dn = d(loss)/dn.

    With xh = x r:  dx = r * (gamma * dn - xh * mean_j(gamma_j dn_j xh_j)).
    Derivation: d r / d x_j = -r^3 x_j / H, so
    dx_j = r gamma_j dn_j - (r^3 x_j / H) sum_i gamma_i dn_i x_i.
    """
    xh = x * r[:, None]
    gdn = gamma[None, :] * dn
    c = np.mean(gdn * xh, axis=1)
    return r[:, None] * (gdn - xh * c[:, None])


def rmsnorm_gamma_grad(dn, x, r):
    """d(loss)/dgamma for n = RMSNorm(x; gamma): sum over tokens of dn * x r."""
    return np.sum(dn * (x * r[:, None]), axis=0)


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


def swiglu_grads(ds, g, u):
    """For s = silu(g) * u: returns (dg, du).

    d silu(g)/dg = sigma(g) (1 + g (1 - sigma(g))).
    """
    sg = sigmoid(g)
    dg = ds * u * sg * (1.0 + g * (1.0 - sg))
    du = ds * silu(g)
    return dg, du


def attention_standin(qkv, n_heads, n_kv_heads, head_dim):
    """a[:, head h] = q_h + k_j + v_j, j = h // (n_heads // n_kv_heads)."""
    t = qkv.shape[0]
    d = head_dim
    q = qkv[:, : n_heads * d].reshape(t, n_heads, d)
    k = qkv[:, n_heads * d : (n_heads + n_kv_heads) * d].reshape(t, n_kv_heads, d)
    v = qkv[:, (n_heads + n_kv_heads) * d :].reshape(t, n_kv_heads, d)
    a = np.empty_like(q)
    group = n_heads // n_kv_heads
    for h in range(n_heads):
        j = h // group
        a[:, h, :] = q[:, h, :] + k[:, j, :] + v[:, j, :]
    return a.reshape(t, n_heads * d)


def attention_standin_grad(da, n_heads, n_kv_heads, head_dim):
    """Transpose of the stand-in: dq_h = da_h, dk_j = dv_j = sum of da_h over group j."""
    t = da.shape[0]
    d = head_dim
    group = n_heads // n_kv_heads
    da3 = da.reshape(t, n_heads, d)
    dkv = np.zeros((t, n_kv_heads, d))
    for h in range(n_heads):
        dkv[:, h // group, :] += da3[:, h, :]
    dkv = dkv.reshape(t, n_kv_heads * d)
    return np.concatenate([da, dkv, dkv], axis=1)


def _heads(qkv, n_heads, n_kv_heads, head_dim):
    t, d = qkv.shape[0], head_dim
    q = qkv[:, : n_heads * d].reshape(t, n_heads, d)
    k = qkv[:, n_heads * d : (n_heads + n_kv_heads) * d].reshape(t, n_kv_heads, d)
    v = qkv[:, (n_heads + n_kv_heads) * d :].reshape(t, n_kv_heads, d)
    return q, k, v


def sequences(t, seq_len):
    """(start, end) of the consecutive sequences of a microbatch of t tokens."""
    step = seq_len if seq_len else max(t, 1)
    return [(s0, min(t, s0 + step)) for s0 in range(0, t, step)]


def causal_probs(q, k, scale):
    """Softmax over keys of scale * q k^T with keys after the query masked out."""
    n = q.shape[0]
    scores = scale * (q @ k.T)
    scores = np.where(np.tril(np.ones((n, n), dtype=bool)), scores, -np.inf)
    e = np.exp(scores - scores.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def attention_causal(qkv, n_heads, n_kv_heads, head_dim, seq_len):
    """a[:, head h] = softmax(q_h k_j^T / sqrt(d), causal) v_j per sequence, j = h // group."""
    t = qkv.shape[0]
    q, k, v = _heads(qkv, n_heads, n_kv_heads, head_dim)
    group = n_heads // n_kv_heads
    scale = 1.0 / np.sqrt(head_dim)
    a = np.zeros((t, n_heads, head_dim))
    for s0, s1 in sequences(t, seq_len):
        for h in range(n_heads):
            j = h // group
            p = causal_probs(q[s0:s1, h], k[s0:s1, j], scale)
            a[s0:s1, h] = p @ v[s0:s1, j]
    return a.reshape(t, n_heads * head_dim)


def attention_causal_grad(da, qkv, n_heads, n_kv_heads, head_dim, seq_len):
    """Gradient of attention_causal with respect to qkv, given da.

    With P = softmax(S), S = scale q k^T and a = P v:
      dv += P^T da,  dP = da v^T,  dS = P * (dP - rowsum(dP * P)),
      dq = scale dS k,  dk += scale dS^T q,
    the sums over the heads of a group going to the shared k and v.
    """
    t = qkv.shape[0]
    q, k, v = _heads(qkv, n_heads, n_kv_heads, head_dim)
    group = n_heads // n_kv_heads
    scale = 1.0 / np.sqrt(head_dim)
    da3 = da.reshape(t, n_heads, head_dim)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for s0, s1 in sequences(t, seq_len):
        for h in range(n_heads):
            j = h // group
            p = causal_probs(q[s0:s1, h], k[s0:s1, j], scale)
            dv[s0:s1, j] += p.T @ da3[s0:s1, h]
            dp = da3[s0:s1, h] @ v[s0:s1, j].T
            ds = p * (dp - np.sum(dp * p, axis=1, keepdims=True))
            dq[s0:s1, h] = scale * (ds @ k[s0:s1, j])
            dk[s0:s1, j] += scale * (ds.T @ q[s0:s1, h])
    return np.concatenate([dq.reshape(t, -1), dk.reshape(t, -1), dv.reshape(t, -1)], axis=1)


def attention_forward(qkv, shp):
    if shp.get("attention", "standin") == "causal":
        return attention_causal(qkv, shp["n_heads"], shp["n_kv_heads"], shp["head_dim"], shp.get("seq_len", 0))
    return attention_standin(qkv, shp["n_heads"], shp["n_kv_heads"], shp["head_dim"])


def attention_backward(da, qkv, shp):
    if shp.get("attention", "standin") == "causal":
        return attention_causal_grad(da, qkv, shp["n_heads"], shp["n_kv_heads"], shp["head_dim"],
                                     shp.get("seq_len", 0))
    return attention_standin_grad(da, shp["n_heads"], shp["n_kv_heads"], shp["head_dim"])


# ----------------------------------------------------------------------------
# F: forward of one layer and of the stage
# ----------------------------------------------------------------------------


def layer_forward(x, prm, shp):
    """Forward of one layer.  Returns (y, saved) where ``saved`` holds what B and W read."""
    kind = shp["kind"]
    if kind == "linear":
        return x @ prm["w"].T, {"x": x}
    saved = {"x": x}
    if kind == "transformer":
        n1, r1 = rmsnorm(x, prm["gamma1"], shp["eps"])
        qkv = n1 @ prm["w_qkv"].T
        a = attention_forward(qkv, shp)
        h = x + a @ prm["w_o"].T
        saved.update({"n1": n1, "r1": r1, "a": a, "qkv": qkv})
    else:
        h = x
    n2, r2 = rmsnorm(h, prm["gamma2"], shp["eps"])
    gu = n2 @ prm["w_gu"].T
    f = shp["ffn"]
    g, u = gu[:, :f], gu[:, f:]
    s = silu(g) * u
    y = h + s @ prm["w_down"].T
    saved.update({"h": h, "n2": n2, "r2": r2, "g": g, "u": u, "s": s})
    return y, saved


def stage_forward(x, params, shp):
    """F of one microbatch through all layers.  Returns (y, [saved per layer])."""
    saved = []
    for prm in params:
        x, sv = layer_forward(x, prm, shp)
        saved.append(sv)
    return x, saved


# ----------------------------------------------------------------------------
# B: input gradient (critical path)
# ----------------------------------------------------------------------------


def layer_backward_input(dy, prm, saved, shp):
    """B of one layer: returns (dx, kept) where ``kept`` holds the dY of every linear.

    Only products with weights (dY W) appear here; no weight gradient is formed.
    """
    kind = shp["kind"]
    if kind == "linear":
        return dy @ prm["w"], {"dy": dy}
    kept = {"dy_down": dy}
    ds = dy @ prm["w_down"]  # B of the down projection
    dg, du = swiglu_grads(ds, saved["g"], saved["u"])
    dgu = np.concatenate([dg, du], axis=1)
    dn2 = dgu @ prm["w_gu"]  # B of gate|up
    dh = dy + rmsnorm_input_grad(dn2, saved["h"], saved["r2"], prm["gamma2"])
    kept.update({"dgu": dgu, "dn2": dn2})
    if kind == "mlp":
        return dh, kept
    da = dh @ prm["w_o"]  # B of the output projection
    dqkv = attention_backward(da, saved["qkv"], shp)
    dn1 = dqkv @ prm["w_qkv"]  # B of qkv
    dx = dh + rmsnorm_input_grad(dn1, saved["x"], saved["r1"], prm["gamma1"])
    kept.update({"dh": dh, "dqkv": dqkv, "dn1": dn1})
    return dx, kept


def stage_backward_input(dy, params, saved, shp):
    """B of one microbatch, top layer first.  Returns (dx, [kept per layer])."""
    kept = [None] * len(params)
    for li in range(len(params) - 1, -1, -1):
        dy, kept[li] = layer_backward_input(dy, params[li], saved[li], shp)
    return dy, kept


# ----------------------------------------------------------------------------
# W: weight gradient (deferred), accumulated
# ----------------------------------------------------------------------------


def zero_grads(params):
    """float64 accumulators, one per parameter, zero-initialised."""
    return [{k: np.zeros_like(v) for k, v in prm.items()} for prm in params]


def layer_backward_weight(acc, saved, kept, shp):
    """W of one layer: dW += dY^T X for every linear, dgamma += sum_t dn * xhat."""
    kind = shp["kind"]
    if kind == "linear":
        acc["w"] += kept["dy"].T @ saved["x"]
        return
    acc["w_down"] += kept["dy_down"].T @ saved["s"]
    acc["w_gu"] += kept["dgu"].T @ saved["n2"]
    acc["gamma2"] += rmsnorm_gamma_grad(kept["dn2"], saved["h"], saved["r2"])
    if kind == "transformer":
        acc["w_o"] += kept["dh"].T @ saved["a"]
        acc["w_qkv"] += kept["dqkv"].T @ saved["n1"]
        acc["gamma1"] += rmsnorm_gamma_grad(kept["dn1"], saved["x"], saved["r1"])


def stage_backward_weight(acc, saved, kept, shp):
    """W of one microbatch for every layer, into the accumulators ``acc``."""
    for li in range(len(acc)):
        layer_backward_weight(acc[li], saved[li], kept[li], shp)


# ----------------------------------------------------------------------------
# the usual fused backward, written on its own (for the split == fused identity)
# ----------------------------------------------------------------------------


def stage_backward_fused(dy, params, saved, shp):
    """Textbook backward: each layer forms its weight gradients and its input
    gradient together, top layer first.  Returns (dx, grads) with fresh grads.

    Written without calling the split functions above, so that comparing the
    two checks the split itself.  Each op is differentiated in reverse order of
    the forward, weight gradient first.
    """
    f = shp["ffn"]
    grads = []
    for li in range(len(params) - 1, -1, -1):
        prm, sv = params[li], saved[li]
        gr = {}
        if shp["kind"] == "linear":
            gr["w"] = dy.T @ sv["x"]
            dy = dy @ prm["w"]
            grads.append(gr)
            continue
        # y = h + s W_down^T
        gr["w_down"] = dy.T @ sv["s"]
        ds = dy @ prm["w_down"]
        # s = silu(g) * u, written with the product rule on g * sigma(g) * u
        sig = 1.0 / (1.0 + np.exp(-sv["g"]))
        dsig = sig * (1.0 - sig)
        dg = ds * sv["u"] * (sig + sv["g"] * dsig)
        du = ds * sv["g"] * sig
        dgu = np.hstack([dg, du])
        gr["w_gu"] = dgu.T @ sv["n2"]
        dn2 = dgu @ prm["w_gu"]
        # n2 = gamma2 * h * r2
        xh = sv["h"] * sv["r2"][:, None]
        gr["gamma2"] = (dn2 * xh).sum(axis=0)
        hidden = xh.shape[1]
        dxh = dn2 * prm["gamma2"][None, :]
        dh_norm = (dxh - xh * (dxh * xh).sum(axis=1, keepdims=True) / hidden) * sv["r2"][:, None]
        dh = dy + dh_norm
        if shp["kind"] == "mlp":
            dy = dh
            grads.append(gr)
            continue
        # h = x + a W_o^T
        gr["w_o"] = dh.T @ sv["a"]
        da = dh @ prm["w_o"]
        nh, nkv, d = shp["n_heads"], shp["n_kv_heads"], shp["head_dim"]
        t = da.shape[0]
        if shp.get("attention", "standin") == "causal":
            dqkv = _causal_grad_by_rows(da, sv["qkv"], nh, nkv, d, shp.get("seq_len", 0))
        else:
            da_heads = da.reshape(t, nkv, nh // nkv, d)
            dk = da_heads.sum(axis=2).reshape(t, nkv * d)
            dqkv = np.hstack([da, dk, dk])
        gr["w_qkv"] = dqkv.T @ sv["n1"]
        dn1 = dqkv @ prm["w_qkv"]
        xh1 = sv["x"] * sv["r1"][:, None]
        gr["gamma1"] = (dn1 * xh1).sum(axis=0)
        dxh1 = dn1 * prm["gamma1"][None, :]
        dx_norm = (dxh1 - xh1 * (dxh1 * xh1).sum(axis=1, keepdims=True) / hidden) * sv["r1"][:, None]
        dy = dh + dx_norm
        grads.append(gr)
    grads.reverse()
    return dy, grads


def _causal_grad_by_rows(da, qkv, nh, nkv, d, seq_len):
    """The causal attention gradient written query row by query row, with the
    softmax Jacobian diag(p) - p p^T formed explicitly (for the fused backward)."""
    t = qkv.shape[0]
    q = qkv[:, : nh * d]
    k = qkv[:, nh * d : (nh + nkv) * d]
    v = qkv[:, (nh + nkv) * d :]
    out = np.zeros_like(qkv)
    rep = nh // nkv
    step = seq_len if seq_len else max(t, 1)
    for h in range(nh):
        qc = slice(h * d, (h + 1) * d)
        kc = slice((h // rep) * d, (h // rep + 1) * d)
        for i in range(t):
            s0 = (i // step) * step
            keys = np.arange(s0, i + 1)
            z = (k[keys][:, kc] @ q[i, qc]) / np.sqrt(d)
            p = np.exp(z - z.max())
            p = p / p.sum()
            jac = np.diag(p) - np.outer(p, p)
            dz = jac @ (v[keys][:, kc] @ da[i, qc])
            out[i, qc] += (dz @ k[keys][:, kc]) / np.sqrt(d)
            out[keys, nh * d + kc.start : nh * d + kc.stop] += np.outer(dz, q[i, qc]) / np.sqrt(d)
            out[keys, (nh + nkv) * d + kc.start : (nh + nkv) * d + kc.stop] += np.outer(p, da[i, qc])
    return out


# ----------------------------------------------------------------------------
# the guide's single-linear stage object, for a whole sequence of F / B / W calls
# ----------------------------------------------------------------------------


class StageOracle:
    """Mirror of the guide's ``ZeroBubbleLinearStage`` (section "Step-by-Step
    Implementation") for any layer kind: F keeps its activations per
    microbatch id, B keeps dY and returns dX, W pops both and accumulates."""

    def __init__(self, params, shp):
        self.params = params
        self.shp = shp
        self.grads = zero_grads(params)
        self.saved = {}
        self.kept = {}

    def forward(self, mb, x):
        y, self.saved[mb] = stage_forward(x, self.params, self.shp)
        return y

    def backward_input(self, mb, dy):
        dx, self.kept[mb] = stage_backward_input(dy, self.params, self.saved[mb], self.shp)
        return dx

    def backward_weight(self, mb):
        saved = self.saved.pop(mb)
        kept = self.kept.pop(mb)
        stage_backward_weight(self.grads, saved, kept, self.shp)
