"""Stash-fed parity: every step of every layer of a stage against the float64 oracle, on the
bf16 values the kernels themselves consumed.

A whole-stage comparison against the oracle mixes two things: the error of each kernel, and
the bf16 roundings of every stored activation and gradient, which travel down the layers
(tests/parity.py).  Here the stage runs as usual (F, B, W through the C ABI); after its F and
after its B the test reads the microbatch's activation stash (zb_stage_stash_view), and for
each layer hands the oracle's plain definitions exactly the tensors that layer's kernels read:
its x, rstd, n1, a, h, n2, [g | u] and s from F, its dy, [dg | du], dn2, dh, dqkv and dn1 from B.
Every output a kernel wrote is then compared with the definition at the per-step bar of the
workloads (relative Frobenius <= 5e-3, max-abs <= 2e-2 * max|ref|).  Each such step is one
contraction or elementwise pass with float32 accumulation and one bf16 rounding of its output,
so nothing of the stage's depth enters the bar.  "Zero-Bubble Pipeline Parallelism Guide for
LLMs", section "2. Convergence and Numerical Stability": B and W are the plain backward's
arithmetic, split, so the plain definition is the reference for every step.

The full-size cases (the 8B-shaped and 70B-shaped stages at 4096 tokens) also compare the
stage's dx, every weight gradient and every gamma gradient end to end with the oracle run on
the caller's inputs, at the whole-stage tolerance.
"""
import numpy as np
import pytest
import torch

from backward_split_linear_gb300 import binding as zb
from backward_split_linear_gb300 import synth
from backward_split_linear_gb300.runtime import Stage, bf16_from_bits, f64_from_bf16
from oracle import stage as S
from parity import FRO_TOL, MAX_TOL, errors, stage_fro_tol

pytestmark = pytest.mark.gpu

EPS = 1e-5


@pytest.fixture(autouse=True)
def _status_clean(cuda_device):
    zb.zb_device_status(reset=True)
    yield
    st, code = zb.zb_device_status()
    assert st == 0, f"device status word set: {code}"


class Report:
    """Collects every comparison, fails once at the end with all the misses listed."""

    def __init__(self):
        self.rows, self.misses = [], []

    def check(self, what, got, ref, fro_tol=FRO_TOL, max_tol=MAX_TOL):
        got = np.asarray(got, dtype=np.float64)
        if not np.all(np.isfinite(got)):
            self.misses.append(f"{what}: non-finite values")
            return
        fro, mx = errors(got, ref)
        self.rows.append((what, fro, mx))
        if not (fro <= fro_tol and mx <= max_tol):
            self.misses.append(f"{what}: frobenius {fro:.3e} (tol {fro_tol:.1e}), max {mx:.3e} (tol {max_tol:.1e})")

    def worst(self):
        return max(r[1] for r in self.rows), max(r[2] for r in self.rows)

    def assert_ok(self, title=""):
        assert self.rows, "nothing compared"
        # the worst cases, for the record (shown with pytest -s): per-step comparisons
        # and whole-stage (end-to-end) ones apart, since they answer to different bars
        for kind, rows in (("per step", [r for r in self.rows if not r[0].startswith("end to end")]),
                           ("end to end", [r for r in self.rows if r[0].startswith("end to end")])):
            if rows:
                fro = max(rows, key=lambda r: r[1])
                mx = max(rows, key=lambda r: r[2])
                print(f"\n{title} [{kind}]: {len(rows)} comparisons; worst frobenius {fro[1]:.2e} ({fro[0]}), "
                      f"worst max-abs {mx[2]:.2e} ({mx[0]})")
        assert not self.misses, "\n".join(self.misses)


def fwd_names(shp):
    if shp["kind"] == "mlp":
        return ["x", "rstd2", "n2", "gu", "s"]
    names = ["x", "rstd1", "n1", "a", "h", "rstd2", "n2", "gu", "s"]
    return names + (["qkv"] if shp.get("attention") == "causal" else [])


def bwd_names(shp):
    return ["dy", "gu", "dn2"] + (["dh", "dqkv", "dn1"] if shp["kind"] == "transformer" else [])


def grab(st, mb, n_layers, names):
    """Host copies (exact) of the named stash tensors of every layer of microbatch mb."""
    torch.cuda.synchronize()
    return {(l, n): st.stash(mb, l, n).cpu() for l in range(n_layers) for n in names}


def f64(t):
    return t.double().numpy()


def check_forward(rep, fs, prm, shp, l, y_next, tag):
    """F of layer l: each output from the stashed inputs of its own step."""
    f = lambda n: f64(fs[(l, n)])
    x = f("x")
    if shp["kind"] == "transformer":
        n1, r1 = S.rmsnorm(x, prm["gamma1"], shp["eps"])
        rep.check(f"{tag} L{l} rstd1", f("rstd1")[:, 0], r1)
        rep.check(f"{tag} L{l} n1", f("n1"), n1)
        qkv = f("n1") @ prm["w_qkv"].T
        if shp.get("attention") == "causal":
            rep.check(f"{tag} L{l} qkv", f("qkv"), qkv)
            qkv = f("qkv")
        rep.check(f"{tag} L{l} a", f("a"), S.attention_forward(qkv, shp))
        rep.check(f"{tag} L{l} h", f("h"), x + f("a") @ prm["w_o"].T)
        h = f("h")
    else:
        h = x
    n2, r2 = S.rmsnorm(h, prm["gamma2"], shp["eps"])
    rep.check(f"{tag} L{l} rstd2", f("rstd2")[:, 0], r2)
    rep.check(f"{tag} L{l} n2", f("n2"), n2)
    rep.check(f"{tag} L{l} gu", f("gu"), f("n2") @ prm["w_gu"].T)
    ffn = shp["ffn"]
    gu = f("gu")
    rep.check(f"{tag} L{l} s", f("s"), S.silu(gu[:, :ffn]) * gu[:, ffn:])
    rep.check(f"{tag} L{l} y", y_next, h + f("s") @ prm["w_down"].T)


def check_backward(rep, fs, bs, prm, shp, l, dx_next, tag):
    """B of layer l: each output from the stashed inputs of its own step."""
    f = lambda n: f64(fs[(l, n)])
    b = lambda n: f64(bs[(l, n)])
    ffn = shp["ffn"]
    gu = f("gu")
    dy = b("dy")
    dg, du = S.swiglu_grads(dy @ prm["w_down"], gu[:, :ffn], gu[:, ffn:])
    rep.check(f"{tag} L{l} dgu", b("gu"), np.concatenate([dg, du], axis=1))
    rep.check(f"{tag} L{l} dn2", b("dn2"), b("gu") @ prm["w_gu"])
    h = f("h") if shp["kind"] == "transformer" else f("x")
    dh = dy + S.rmsnorm_input_grad(b("dn2"), h, f("rstd2")[:, 0], prm["gamma2"])
    if shp["kind"] == "mlp":
        rep.check(f"{tag} L{l} dx", dx_next, dh)
        return
    rep.check(f"{tag} L{l} dh", b("dh"), dh)
    da = b("dh") @ prm["w_o"]
    qkv = f("qkv") if shp.get("attention") == "causal" else None
    rep.check(f"{tag} L{l} dqkv", b("dqkv"), S.attention_backward(da, qkv, shp))
    rep.check(f"{tag} L{l} dn1", b("dn1"), b("dqkv") @ prm["w_qkv"])
    dx = b("dh") + S.rmsnorm_input_grad(b("dn1"), f("x"), f("rstd1")[:, 0], prm["gamma1"])
    rep.check(f"{tag} L{l} dx", dx_next, dx)


def add_weight_grads(acc, fs, bs, shp, l):
    """W of layer l from the stashed X and dY pairs: dW += dY^T X, dgamma += sum dn * x r."""
    f = lambda n: f64(fs[(l, n)])
    b = lambda n: f64(bs[(l, n)])
    h = f("h") if shp["kind"] == "transformer" else f("x")
    acc["w_down"] += b("dy").T @ f("s")
    acc["w_gu"] += b("gu").T @ f("n2")
    acc["gamma2"] += S.rmsnorm_gamma_grad(b("dn2"), h, f("rstd2")[:, 0])
    if shp["kind"] == "transformer":
        acc["w_o"] += b("dh").T @ f("a")
        acc["w_qkv"] += b("dqkv").T @ f("n1")
        acc["gamma1"] += S.rmsnorm_gamma_grad(b("dn1"), f("x"), f("rstd1")[:, 0])


def run_stash_fed(c, inp, max_inflight, w_mode="per-microbatch", attention="standin", seq_len=0, end_to_end_tol=None):
    """F of every microbatch, then B of every microbatch, then W (per microbatch, or one flush
    that batches consecutive full slots); the stash is read after each F and each B.  Returns
    the Report and the stage."""
    shp = dict(c, eps=EPS, attention=attention, seq_len=seq_len)
    n_layers, n_mb = c["n_layers"], len(inp["x"])
    max_tokens = max(b.shape[0] for b in inp["x"])
    st = Stage.from_synth(c["kind"], n_layers, c["hidden"], c["ffn"], c["n_heads"], c["n_kv_heads"], c["head_dim"],
                          EPS, max_tokens, max_inflight, inp["params"], attention=attention, seq_len=seq_len)
    xs = [bf16_from_bits(b) for b in inp["x"]]
    dys = [bf16_from_bits(b) for b in inp["dy"]]
    ys = [torch.empty(x.shape[0], c["hidden"], dtype=torch.bfloat16, device="cuda") for x in xs]
    dxs = [torch.empty(x.shape[0], c["hidden"], dtype=torch.bfloat16, device="cuda") for x in xs]
    fstash, bstash = [], []
    for mb in range(n_mb):
        st.forward(mb, xs[mb], ys[mb])
        fstash.append(grab(st, mb, n_layers, fwd_names(shp)))
    for mb in range(n_mb):
        st.backward_input(mb, dys[mb], dxs[mb])
        bstash.append(grab(st, mb, n_layers, bwd_names(shp)))
    if w_mode == "flush":
        st.flush()
    else:
        for mb in range(n_mb):
            st.backward_weight(mb)
    st.sync()
    params = synth.params_f64(inp["params"])
    rep = Report()
    acc = S.zero_grads(params)
    for mb in range(n_mb):
        tag = f"mb{mb}"
        for l in range(n_layers):
            y_next = f64(fstash[mb][(l + 1, "x")]) if l + 1 < n_layers else f64_from_bf16(ys[mb])
            check_forward(rep, fstash[mb], params[l], shp, l, y_next, tag)
            dx_next = f64(bstash[mb][(l - 1, "dy")]) if l > 0 else f64_from_bf16(dxs[mb])
            check_backward(rep, fstash[mb], bstash[mb], params[l], shp, l, dx_next, tag)
            add_weight_grads(acc[l], fstash[mb], bstash[mb], shp, l)
        fstash[mb] = bstash[mb] = None
    for l in range(n_layers):
        for k, ref in acc[l].items():
            rep.check(f"L{l} d{k} ({w_mode} W over {n_mb} microbatches)", st.grads[l][k].cpu().numpy(), ref)
    if end_to_end_tol is not None:
        orc = S.StageOracle(params, shp)
        for mb in range(n_mb):
            orc.forward(mb, synth.bf16_to_f64(inp["x"][mb]))
            rep.check(f"end to end dx mb{mb}", f64_from_bf16(dxs[mb]),
                      orc.backward_input(mb, synth.bf16_to_f64(inp["dy"][mb])), fro_tol=end_to_end_tol)
            orc.backward_weight(mb)
        for l in range(n_layers):
            for k, ref in orc.grads[l].items():
                rep.check(f"end to end L{l} d{k}", st.grads[l][k].cpu().numpy(), ref, fro_tol=end_to_end_tol)
    return rep, st


TINY = dict(kind="mlp", n_layers=2, hidden=256, ffn=1024, n_heads=0, n_kv_heads=0, head_dim=0)
SMALL_TF = dict(kind="transformer", n_layers=2, hidden=256, ffn=512, n_heads=4, n_kv_heads=2, head_dim=64)
LLAMA8B = dict(kind="transformer", n_layers=4, hidden=4096, ffn=14336, n_heads=32, n_kv_heads=8, head_dim=128)
LLAMA70B = dict(kind="transformer", n_layers=2, hidden=8192, ffn=28672, n_heads=64, n_kv_heads=8, head_dim=128)


def test_tiny_config_every_step_flush():
    """The tiny MLP stage (2 layers, 256 / 1024, 128 tokens, m = 4): every step of both layers of all
    four microbatches, W batched by the flush over the four full slots."""
    inp = synth.stage_inputs("mlp", 2, 256, 1024, tokens=128, n_mb=4, seed=0)
    rep, st = run_stash_fed(TINY, inp, 4, w_mode="flush")
    st.close()
    rep.assert_ok("test_tiny_config_every_step_flush")


def test_small_transformer_ragged_every_step():
    """Stand-in transformer layers with ragged microbatches (200, 77, 1 tokens): tails of
    every tile size in T, per-microbatch W."""
    inp = synth.stage_inputs("transformer", 2, 256, 512, 4, 2, 64, n_mb=3, seed=1, tokens_per_mb=[200, 77, 1])
    rep, st = run_stash_fed(SMALL_TF, inp, 3)
    st.close()
    rep.assert_ok("test_small_transformer_ragged_every_step")


def test_causal_8b_widths_every_step():
    """Two 8B-shaped layers (4096 / 14336, 32 / 8 heads) with the causal core, two 512-token
    microbatches in sequences of 256, W in one flush."""
    c = dict(LLAMA8B, n_layers=2)
    inp = synth.stage_inputs("transformer", 2, 4096, 14336, 32, 8, 128, tokens=512, n_mb=2, seed=5)
    rep, st = run_stash_fed(c, inp, 2, w_mode="flush", attention="causal", seq_len=256)
    st.close()
    rep.assert_ok("test_causal_8b_widths_every_step")


def test_llama8b_stage_full_size_every_step_and_end_to_end():
    """At full size: the 8B-shaped 4-layer stage, one 4096-token microbatch.  Every
    step of every layer at the per-step bar (its GEMMs split K in their last wave exactly as in
    the benchmark), then dx, all 16 weight gradients and 8 gamma gradients against the oracle
    run end to end on the caller's inputs, at the 4-layer stage tolerance."""
    inp = synth.stage_inputs("transformer", 4, 4096, 14336, 32, 8, 128, tokens=4096, n_mb=1, seed=0)
    rep, st = run_stash_fed(LLAMA8B, inp, 1, end_to_end_tol=stage_fro_tol(4))
    st.close()
    rep.assert_ok("test_llama8b_stage_full_size_every_step_and_end_to_end")


def test_llama70b_stage_full_size_every_step_and_end_to_end():
    """At full size: the 70B-shaped 2-layer stage (8192 / 28672, 64 / 8 heads), one
    4096-token microbatch, as for the 8B-shaped stage."""
    inp = synth.stage_inputs("transformer", 2, 8192, 28672, 64, 8, 128, tokens=4096, n_mb=1, seed=0)
    rep, st = run_stash_fed(LLAMA70B, inp, 1, end_to_end_tol=stage_fro_tol(2))
    st.close()
    rep.assert_ok("test_llama70b_stage_full_size_every_step_and_end_to_end")
