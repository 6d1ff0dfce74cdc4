"""A float64 replay of the stage's GPU arithmetic with every tensor the GPU stores or feeds to
the tensor cores rounded to bf16 (RNE), compared with the exact oracle.

TEST INFRASTRUCTURE: the source of the whole-stage tolerances in tests/parity.py, run by
tests/test_bf16_replay.py (collected, CPU only).  It can also be run by hand on the workloads'
own widths:

    python tests/bf16_replay.py causal     # the causal 8B-shaped two-layer stage
    python tests/bf16_replay.py standin    # the same stage with the weight-free stand-in

It follows the order of the GPU path (F: n1, qkv, a, h, n2, [g|u], s, y rounded; B: dgu,
dn2, dh, da, dqkv, dn1, dx rounded; attention: P rounded for the P V and dV products, dS
rounded, D from the rounded output) and keeps sums exact, so what it reports is the error
that bf16 storage alone implies.  It uses the oracle's functions as building blocks and
shares nothing with the CUDA path.
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from backward_split_linear_gb300 import synth  # noqa: E402
from oracle import stage as S  # noqa: E402
from parity import errors  # noqa: E402


def bf(x):
    """Round to bf16 (RNE) and widen back to float64."""
    return synth.bf16_to_f64(synth.bf16_bits(np.asarray(x, dtype=np.float32)))


def attn_fwd(qkv, nh, nkv, d, seq_len):
    t = qkv.shape[0]
    q, k, v = S._heads(qkv, nh, nkv, d)
    a = np.zeros((t, nh, d))
    for s0, s1 in S.sequences(t, seq_len):
        for h in range(nh):
            j = h // (nh // nkv)
            p = S.causal_probs(q[s0:s1, h], k[s0:s1, j], 1 / np.sqrt(d))
            a[s0:s1, h] = bf(p) @ v[s0:s1, j]  # P rounded for the P V product
    return a.reshape(t, -1)


def attn_bwd(da, qkv, a, nh, nkv, d, seq_len):
    t = qkv.shape[0]
    q, k, v = S._heads(qkv, nh, nkv, d)
    da3, a3 = da.reshape(t, nh, d), a.reshape(t, nh, d)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s0, s1 in S.sequences(t, seq_len):
        for h in range(nh):
            j = h // (nh // nkv)
            p = S.causal_probs(q[s0:s1, h], k[s0:s1, j], 1 / np.sqrt(d))
            dp = da3[s0:s1, h] @ v[s0:s1, j].T
            rowsum = np.sum(da3[s0:s1, h] * a3[s0:s1, h], axis=1)  # from the rounded output
            ds = bf(p * (dp - rowsum[:, None]))
            dv[s0:s1, j] += bf(p).T @ da3[s0:s1, h]
            dq[s0:s1, h] = ds @ k[s0:s1, j] / np.sqrt(d)
            dk[s0:s1, j] += ds.T @ q[s0:s1, h] / np.sqrt(d)
    return np.concatenate([dq.reshape(t, -1), dk.reshape(t, -1), dv.reshape(t, -1)], axis=1)


def run(c, params, xs, dys):
    """F, B and W of every microbatch with the GPU's bf16 roundings.  Returns (dx per
    microbatch, float64 accumulators per layer)."""
    nh, nkv, d, ffn = c["n_heads"], c["n_kv_heads"], c["head_dim"], c["ffn"]
    seq_len = c.get("seq_len", 0)
    causal = c.get("attention") == "causal"
    grads = [{k: np.zeros_like(v) for k, v in p.items()} for p in params]
    dxs = []
    for x, dy in zip(xs, dys):
        saved = []
        for prm in params:
            n1, r1 = S.rmsnorm(x, prm["gamma1"], c["eps"])
            n1 = bf(n1)
            qkv = bf(n1 @ prm["w_qkv"].T)
            a = bf(attn_fwd(qkv, nh, nkv, d, seq_len) if causal else S.attention_standin(qkv, nh, nkv, d))
            h = bf(x + a @ prm["w_o"].T)
            n2, r2 = S.rmsnorm(h, prm["gamma2"], c["eps"])
            n2 = bf(n2)
            gu = bf(n2 @ prm["w_gu"].T)
            g, u = gu[:, :ffn], gu[:, ffn:]
            s = bf(S.silu(g) * u)
            y = bf(h + s @ prm["w_down"].T)
            saved.append(dict(x=x, n1=n1, r1=r1, qkv=qkv, a=a, h=h, n2=n2, r2=r2, g=g, u=u, s=s))
            x = y
        dyl = dy
        for li in range(len(params) - 1, -1, -1):
            prm, v = params[li], saved[li]
            dg, du = S.swiglu_grads(dyl @ prm["w_down"], v["g"], v["u"])
            dgu = bf(np.concatenate([dg, du], axis=1))
            dn2 = bf(dgu @ prm["w_gu"])
            dh = bf(dyl + S.rmsnorm_input_grad(dn2, v["h"], v["r2"], prm["gamma2"]))
            da = bf(dh @ prm["w_o"])
            if causal:
                dqkv = bf(attn_bwd(da, v["qkv"], v["a"], nh, nkv, d, seq_len))
            else:
                dqkv = bf(S.attention_standin_grad(da, nh, nkv, d))
            dn1 = bf(dqkv @ prm["w_qkv"])
            dxl = bf(dh + S.rmsnorm_input_grad(dn1, v["x"], v["r1"], prm["gamma1"]))
            gr = grads[li]
            gr["w_down"] += dyl.T @ v["s"]
            gr["w_gu"] += dgu.T @ v["n2"]
            gr["gamma2"] += S.rmsnorm_gamma_grad(dn2, v["h"], v["r2"])
            gr["w_o"] += dh.T @ v["a"]
            gr["w_qkv"] += dqkv.T @ v["n1"]
            gr["gamma1"] += S.rmsnorm_gamma_grad(dn1, v["x"], v["r1"])
            dyl = dxl
        dxs.append(dyl)
    return dxs, grads


def replay_errors(c, inp):
    """Relative Frobenius and max-abs errors of the replay against the exact oracle, for every dx
    and every accumulated gradient: {name: (frobenius, max-abs)}."""
    params = synth.params_f64(inp["params"])
    xs = [synth.bf16_to_f64(b) for b in inp["x"]]
    dys = [synth.bf16_to_f64(b) for b in inp["dy"]]
    dx_rep, g_rep = run(c, params, xs, dys)
    orc = S.StageOracle(params, c)
    out = {}
    for i in range(len(xs)):
        orc.forward(i, xs[i])
        out[f"dx{i}"] = errors(dx_rep[i], orc.backward_input(i, dys[i]))
    for i in range(len(xs)):
        orc.backward_weight(i)
    for li in range(len(params)):
        for k, ref in orc.grads[li].items():
            out[f"L{li} d{k}"] = errors(g_rep[li][k], ref)
    return out


if __name__ == "__main__":
    kind = sys.argv[1] if len(sys.argv) > 1 else "causal"
    c = dict(kind="transformer", n_layers=2, hidden=4096, ffn=14336, n_heads=32, n_kv_heads=8, head_dim=128,
             eps=1e-5, attention=kind, seq_len=128 if kind == "causal" else 0)
    inp = synth.stage_inputs("transformer", 2, 4096, 14336, 32, 8, 128, n_mb=2, seed=23, tokens_per_mb=[256, 256])
    for name, (fro, mx) in replay_errors(c, inp).items():
        print(f"{name:16s} frobenius {fro:.3e}  max-abs {mx:.3e}")
